"""Several query tokens per request (speculative drafts) on the GPU against
the oracle.

"Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section
"A kernel that reads four bits directly": the native kernel decodes 15 query
tokens per launch.  Each token has its own top-k list; the q_len tokens of a
request are its last q_len positions, so token i sees t < ctx - (q_len-1-i).
Tolerance as for the single-token decode (gpu_helpers)."""
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


def host_pool(wl, fmt):
    """The oracle's own pool: the workload's seeded bf16 rows quantized on the host."""
    rb = O.row_bytes(fmt)
    stride = 64 * rb
    pool = np.zeros(wl.num_blocks * stride, dtype=np.uint8)
    bt = wl.block_table.cpu().numpy()
    for b in range(wl.batch):
        lat, rope = wl.request_rows(b)
        c = lat.shape[0]
        slots = bt[b, np.arange(c) // 64].astype(np.int64) * 64 + np.arange(c) % 64
        O.kv_quantize_append(u16(lat), u16(rope), slots, pool, wl.num_blocks, 64, stride, fmt)
    return pool, stride


def small_draft_workload(batch, heads, topk, ctx_lens, q_len, seed):
    def draw(b, c, g):
        return W.distinct_uniform(min(topk, c), 0, c, g, DEV)
    wl = W._decode_workload("drafts", ("drafts", seed, batch, heads, topk, tuple(ctx_lens)), batch, heads, topk,
                            ctx_lens, DEV, 0.01, draw)
    dq = W.draft_queries(wl, q_len=q_len, keep=0.8, recent=64)
    # every token's list also names the last q_len positions: the causal
    # bound must mask the ones past the token
    idx = dq.topk_idx.clone()
    for b, c in enumerate(ctx_lens):
        tail = torch.arange(max(0, c - q_len), c, device=DEV, dtype=torch.int32)
        idx[b, :, :tail.numel()] = tail
    dq.topk_idx = idx.contiguous()
    return wl, dq


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch,heads,topk,ctx_lens,q_len", [
    (3, 16, 300, [5000, 777, 300], 4),
    (2, 32, 2048, [9000, 2050], 3),
    (2, 16, 64, [3, 1], 4),          # context shorter than q_len: early tokens see nothing
    (1, 64, 97, [4096], 15),
    (2, 64, 2048, [9000, 2050], 3),  # 64-head blocks on NVFP4: tensor-memory kernel, split lists
])
def test_drafts_against_oracle(fmt, batch, heads, topk, ctx_lens, q_len):
    m = lib()
    wl, dq = small_draft_workload(batch, heads, topk, ctx_lens, q_len, seed=topk + q_len)
    W.fill_pool(wl, fmt, quantize_fn(m))
    lse = torch.empty((batch, q_len, heads), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode_mtp(dq.q_nope, dq.q_rope, wl.pools[fmt], wl.strides[fmt], wl.num_blocks,
                                     wl.block_table, wl.context_lens, dq.topk_idx, wl.softmax_scale, fmt=fmt, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    pool, stride = host_pool(wl, fmt)
    ref, ref_lse = O.sparse_decode_mtp(u16(dq.q_nope), u16(dq.q_rope), pool, stride, wl.block_table.cpu().numpy(),
                                       wl.context_lens.cpu().numpy(), dq.topk_idx.cpu().numpy(), 64,
                                       wl.softmax_scale, fmt, threads=O.host_threads())
    for b in range(batch):
        for i in range(q_len):
            assert_decode_close(out[b, i], lse[b, i], ref[b, i], ref_lse[b, i], f"request {b} token {i}")


def test_single_token_equals_plain_decode():
    """q_len = 1 is the plain decode, bit for bit."""
    m = lib()
    wl, dq = small_draft_workload(3, 32, 500, [6000, 900, 4000], 1, seed=11)
    W.fill_pool(wl, O.FMT_NVFP4, quantize_fn(m))
    a, _ = m.mla_sparse_decode_mtp(dq.q_nope, dq.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                   wl.context_lens, dq.topk_idx, wl.softmax_scale)
    b, _ = m.mla_sparse_decode(dq.q_nope[:, 0].contiguous(), dq.q_rope[:, 0].contiguous(), wl.pools[0],
                               wl.strides[0], wl.num_blocks, wl.block_table, wl.context_lens,
                               dq.topk_idx[:, 0].contiguous(), wl.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


@pytest.mark.parametrize("q_len,tokens", [(4, [0, 1, 2, 3]), (15, [0, 7, 14])])
def test_tp4_rank_drafts_full_size_sampled(q_len, tokens):
    """32 requests x q_len tokens x 16 heads, 140,000-token contexts,
    per-token top-2048 lists overlapping 90% (as bench.py times, at 4 tokens
    and at the pages' 15 per launch); 2 requests x a few tokens checked
    against the oracle on the rows each token selects."""
    m = lib()
    wl = W.tp4_rank_decode(DEV)
    dq = W.draft_queries(wl, q_len=q_len)
    W.fill_pool(wl, O.FMT_NVFP4, quantize_fn(m))
    lse = torch.empty((32, q_len, 16), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode_mtp(dq.q_nope, dq.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks,
                                     wl.block_table, wl.context_lens, dq.topk_idx, wl.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    for b in [5, 30]:
        c = int(wl.context_lens[b])
        for i in tokens:
            idx = dq.topk_idx[b, i].cpu().numpy().astype(np.int64)
            valid = (idx >= 0) & (idx < c - (q_len - 1 - i))
            lat, rope = wl.request_rows(b, torch.from_numpy(np.where(valid, idx, 0)).to(DEV))
            ref, ref_lse = oracle_rows_decode(u16(dq.q_nope[b, i]), u16(dq.q_rope[b, i]), u16(lat), u16(rope), valid,
                                              O.FMT_NVFP4, wl.softmax_scale)
            assert_decode_close(out[b, i], lse[b, i], ref, ref_lse, f"request {b} token {i}")
