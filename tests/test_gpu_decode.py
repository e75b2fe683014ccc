"""Sparse MLA decode on the GPU (NVFP4 and FP8 caches) against the float64 oracle.

Decode definition: "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem", section "A kernel that reads four bits directly" (gather the
selected rows, unpack on chip, score / softmax / blend; -1 entries skipped).
Tolerance (bf16 outputs vs float64): max-abs <= 2e-2 max|ref|, relative RMS
<= 5e-3, lse within 1e-3 (1 + |ref|).

The oracle never reads the GPU's pool: it quantizes the same seeded bf16 rows
itself (gpu_helpers.oracle_rows_decode)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMTS = [pytest.param(O.FMT_NVFP4, id="nvfp4"), pytest.param(O.FMT_FP8, id="fp8")]


def quantize_fn(m):
    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)
    return qa


def run_gpu(m, wl, fmt, topk_idx=None, context_lens=None, block_table=None, num_blocks=None):
    dec = m.mla_sparse_decode if fmt == O.FMT_NVFP4 else m.mla_sparse_decode_fp8
    lse = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    out, _ = dec(wl.q_nope, wl.q_rope, wl.pools[fmt], wl.strides[fmt],
                 wl.num_blocks if num_blocks is None else num_blocks,
                 wl.block_table if block_table is None else block_table,
                 wl.context_lens if context_lens is None else context_lens,
                 wl.topk_idx if topk_idx is None else topk_idx, wl.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_request(wl, b, fmt, topk_row=None, ctx=None, bad_blocks=()):
    """Oracle output for request b from the seeded rows of its list entries."""
    idx = (wl.topk_idx[b] if topk_row is None else topk_row).cpu().numpy().astype(np.int64)
    c = int(wl.context_lens[b]) if ctx is None else ctx
    valid = (idx >= 0) & (idx < c)
    if len(bad_blocks):
        valid &= ~np.isin(idx // 64, np.array(list(bad_blocks)))
    pos = torch.from_numpy(np.where(valid, idx, 0)).to(DEV)
    lat, rope = wl.request_rows(b, pos)
    return oracle_rows_decode(u16(wl.q_nope[b]), u16(wl.q_rope[b]), u16(lat), u16(rope), valid, fmt,
                              wl.softmax_scale)


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_config_all_heads(fmt):
    """1 request x 16 heads, 4,096 tokens in 64 shuffled blocks, top-256."""
    m = lib()
    wl = W.tiny_decode(DEV)
    W.fill_pool(wl, fmt, quantize_fn(m))
    out, lse = run_gpu(m, wl, fmt)
    ref, ref_lse = oracle_request(wl, 0, fmt)
    assert_decode_close(out[0], lse[0], ref, ref_lse, "tiny")


def small_workload(batch, heads, topk, ctx_lens, seed, device=DEV):
    def draw(b, c, g):
        n = min(topk, c)
        return W.distinct_uniform(n, 0, c, g, device)
    return W._decode_workload("small", ("small", seed, batch, heads, topk, tuple(ctx_lens)), batch, heads, topk,
                              ctx_lens, device, 0.01, draw)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch,heads,topk,ctx_lens", [
    (3, 32, 300, [5000, 777, 300]),        # ragged stages, second head group
    (2, 16, 2048, [150_000, 2049]),        # full top-k, many splits
    (4, 64, 97, [97, 64, 1, 4096]),        # k not a multiple of 16; ctx < k pads with -1
    (1, 128, 1, [10]),                      # k = 1, eight head groups
    (2, 128, 700, [3000, 650]),             # two 64-head blocks, ragged stages, ctx < k
    (5, 16, 33, [33, 40, 50, 60, 70]),
])
def test_small_shapes(fmt, batch, heads, topk, ctx_lens):
    m = lib()
    wl = small_workload(batch, heads, topk, ctx_lens, seed=batch * 1000 + topk)
    W.fill_pool(wl, fmt, quantize_fn(m))
    out, lse = run_gpu(m, wl, fmt)
    for b in range(batch):
        ref, ref_lse = oracle_request(wl, b, fmt)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("heads", [16, 64])
def test_masked_duplicates_and_bad_blocks(fmt, heads):
    """-1 entries, positions past the context, duplicates, unsorted lists, a
    block id outside the pool and a logical block past the table are all
    handled on the device without faults (64 heads on NVFP4: the
    tensor-memory kernel)."""
    m = lib()
    wl = small_workload(3, heads, 512, [3000, 3000, 700], seed=77)
    W.fill_pool(wl, fmt, quantize_fn(m))
    rng = np.random.default_rng(5)
    idx = wl.topk_idx.cpu().numpy().copy()
    idx[0, ::7] = -1
    idx[0, 1::11] = 2999 + rng.integers(1, 5000, idx[0, 1::11].size)   # past the context
    idx[1] = rng.permutation(idx[1])
    idx[1, :40] = idx[1, 40:80]                                         # duplicates
    idx[2, :] = -1                                                      # nothing valid
    topk = torch.from_numpy(idx).to(DEV)
    bt = wl.block_table.clone()
    bad_logical = 5
    bt[1, bad_logical] = wl.num_blocks + 100                            # block id outside the pool
    out, lse = run_gpu(m, wl, fmt, topk_idx=topk, block_table=bt)
    ref0, l0 = oracle_request(wl, 0, fmt, topk_row=topk[0])
    assert_decode_close(out[0], lse[0], ref0, l0, "masked")
    ref1, l1 = oracle_request(wl, 1, fmt, topk_row=topk[1], bad_blocks=[bad_logical])
    assert_decode_close(out[1], lse[1], ref1, l1, "duplicates + bad block")
    assert not out[2].any() and np.all(np.isneginf(lse[2]))


@pytest.mark.parametrize("fmt", FMTS)
def test_k1_is_the_row_itself(fmt):
    """With one selected row the output is that row's dequantized latent,
    rounded once to bf16 (bit-exact)."""
    m = lib()
    wl = small_workload(2, 16, 1, [500, 64], seed=9)
    W.fill_pool(wl, fmt, quantize_fn(m))
    out, lse = run_gpu(m, wl, fmt)
    for b in range(2):
        t = int(wl.topk_idx[b, 0])
        lat, rope = wl.request_rows(b, torch.tensor([t], device=DEV))
        row = O.quantize_row(u16(lat)[0], u16(rope)[0], fmt)
        c, _ = O.dequant_row(row, fmt)
        want = torch.from_numpy(c).to(torch.bfloat16).float().numpy()
        assert np.array_equal(np.broadcast_to(want, out[b].shape), out[b])


@pytest.mark.parametrize("fmt", FMTS)
def test_tp4_rank_full_size_sampled(fmt):
    """32 requests x 16 heads, 140,000-token contexts, top-2048 (70% prefix +
    30% recent), as timed by bench.py; 4 requests checked against the oracle."""
    m = lib()
    wl = W.tp4_rank_decode(DEV)
    W.fill_pool(wl, fmt, quantize_fn(m))
    out, lse = run_gpu(m, wl, fmt)
    for b in [0, 7, 19, 31]:
        ref, ref_lse = oracle_request(wl, b, fmt)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("fmt", FMTS)
def test_dep_rank_full_size_sampled(fmt):
    """128 requests x 64 heads, contexts 8K-1M (24M tokens in total), top-2048
    uniform; 3 requests checked against the oracle."""
    m = lib()
    wl = W.dep_rank_decode(DEV)
    W.fill_pool(wl, fmt, quantize_fn(m))
    out, lse = run_gpu(m, wl, fmt)
    lens = wl.context_lens.cpu().numpy()
    for b in [int(np.argmax(lens)), int(np.argmin(lens)), 64]:
        ref, ref_lse = oracle_request(wl, b, fmt)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")
    assert np.isfinite(out).all()
    del wl
    torch.cuda.empty_cache()


def test_nvfp4_and_fp8_agree_within_quantization_error():
    """Both paths decode the same bf16 rows; they differ only by the storage
    rounding (a sanity bound, not a parity claim)."""
    m = lib()
    wl = W.tiny_decode(DEV)
    W.fill_pool(wl, O.FMT_NVFP4, quantize_fn(m))
    W.fill_pool(wl, O.FMT_FP8, quantize_fn(m))
    a, _ = run_gpu(m, wl, O.FMT_NVFP4)
    b, _ = run_gpu(m, wl, O.FMT_FP8)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 0 < rel < 0.5


def test_device_fault_word_is_clear():
    m = lib()
    assert m.mla_device_fault(clear=False) == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_block_stride_not_a_whole_number_of_rows(fmt):
    """A pool whose block stride is not a multiple of the row size cannot be
    described to TMA as a tensor of rows; the decode then gathers with
    16-byte cp.async.  Same results against the oracle."""
    m = lib()
    wl = small_workload(3, 32, 700, [5000, 1800, 700], seed=31)
    W.fill_pool(wl, fmt, quantize_fn(m), pad_stride=16)
    assert wl.strides[fmt] % O.row_bytes(fmt) != 0
    out, lse = run_gpu(m, wl, fmt)
    for b in range(wl.batch):
        ref, ref_lse = oracle_request(wl, b, fmt)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")
