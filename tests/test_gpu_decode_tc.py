"""Sparse decode with 64-head blocks of NVFP4 rows -- the tensor-memory
(tcgen05) kernel -- against the float64 oracle, on the paths that kernel
adds: the lazy maximum raised in later stages (O rescaled in tensor memory),
a first stage with nothing selected, lists split over several CTAs and
merged by the second kernel, several 64-head blocks per request, and the
same head count on a pool TMA cannot describe (served by the 16-head
kernel).

Decode definition: "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem", section "A kernel that reads four bits directly".  Tolerances are
those of the other decode tests (gpu_helpers.assert_decode_close)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMT = O.FMT_NVFP4


def quantize_fn(m):
    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)
    return qa


def workload(batch, heads, topk, ctx_lens, seed):
    def draw(b, c, g):
        return W.distinct_uniform(min(topk, c), 0, c, g, DEV)
    return W._decode_workload("tc", ("tc", seed, batch, heads, topk, tuple(ctx_lens)), batch, heads, topk, ctx_lens,
                              DEV, 0.01, draw)


def decode(m, wl, topk_idx=None):
    lse = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[FMT], wl.strides[FMT], wl.num_blocks,
                                 wl.block_table, wl.context_lens, wl.topk_idx if topk_idx is None else topk_idx,
                                 wl.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def check(wl, out, lse, b, idx_row=None):
    idx = (wl.topk_idx[b] if idx_row is None else idx_row).cpu().numpy().astype(np.int64)
    c = int(wl.context_lens[b])
    valid = (idx >= 0) & (idx < c)
    lat, rope = wl.request_rows(b, torch.from_numpy(np.where(valid, idx, 0)).to(DEV))
    ref, ref_lse = oracle_rows_decode(u16(wl.q_nope[b]), u16(wl.q_rope[b]), u16(lat), u16(rope), valid, FMT,
                                      wl.softmax_scale)
    assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")


def test_maximum_raised_in_later_stages():
    """The list is ordered by ascending score and the query scaled by 4, so
    every head's running maximum is raised by more than 2^8 in several later
    stages: O is rescaled in tensor memory between P.V steps."""
    m = lib()
    wl = workload(1, 64, 1024, [8192], seed=3)
    wl.q_nope = (wl.q_nope.float() * 4).to(torch.bfloat16)
    wl.q_rope = (wl.q_rope.float() * 4).to(torch.bfloat16)
    W.fill_pool(wl, FMT, quantize_fn(m))
    idx = wl.topk_idx[0]
    lat, rope = wl.request_rows(0, idx.to(torch.int64))
    s = (wl.q_nope[0].float() @ lat.float().T + wl.q_rope[0].float() @ rope.float().T)  # [heads, entries]
    order = torch.argsort(s.mean(0))
    idx_sorted = idx[order].contiguous()
    z2 = (s[:, order] * wl.softmax_scale / math.log(2)).cpu().numpy()
    # the input does what the test is for: each head's scores span > 3 raises
    assert (z2.max(1) - z2.min(1)).min() > 24
    out, lse = decode(m, wl, topk_idx=idx_sorted[None])
    check(wl, out, lse, 0, idx_row=idx_sorted)


def test_first_stage_selects_nothing():
    """The first 200 list entries are -1: the first 128-row stage has no
    valid row, so every maximum is still -inf when the first rows arrive."""
    m = lib()
    wl = workload(2, 64, 600, [5000, 3000], seed=5)
    W.fill_pool(wl, FMT, quantize_fn(m))
    idx = wl.topk_idx.clone()
    idx[:, :200] = -1
    out, lse = decode(m, wl, topk_idx=idx)
    for b in range(2):
        check(wl, out, lse, b, idx_row=idx[b])


@pytest.mark.parametrize("batch,heads,topk,ctx", [
    (1, 64, 2048, 100_000),   # one 64-head block: the list split 16 ways
    (1, 128, 1500, 20_000),   # two blocks, ragged last stage
    (3, 64, 333, 4_000),      # k not a multiple of 128
])
def test_split_lists_merged(batch, heads, topk, ctx):
    """Few requests leave SMs idle, so each list is split over several CTAs
    (partials merged by the second kernel)."""
    m = lib()
    wl = workload(batch, heads, topk, [ctx] * batch, seed=topk)
    W.fill_pool(wl, FMT, quantize_fn(m))
    out, lse = decode(m, wl)
    for b in range(batch):
        check(wl, out, lse, b)


def test_64_heads_on_a_pool_tma_cannot_describe():
    """A block stride that is not a whole number of rows: 64 heads are served
    by the 16-head kernel's cp.async path; same results."""
    m = lib()
    wl = workload(2, 64, 500, [3000, 1200], seed=8)
    W.fill_pool(wl, FMT, quantize_fn(m), pad_stride=16)
    assert wl.strides[FMT] % O.row_bytes(FMT) != 0
    out, lse = decode(m, wl)
    for b in range(2):
        check(wl, out, lse, b)


def test_repeatable():
    """Two launches on the same inputs give bit-identical outputs (the MMA
    accumulation order is fixed)."""
    m = lib()
    wl = workload(4, 64, 900, [7000, 5000, 3000, 900], seed=11)
    W.fill_pool(wl, FMT, quantize_fn(m))
    a, la = decode(m, wl)
    b, lb = decode(m, wl)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
