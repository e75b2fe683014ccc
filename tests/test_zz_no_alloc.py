"""mla_sparse_decode_noalloc: the decode for callers that cannot allocate
device memory (a serving process with a fixed device-memory budget, or a C host
without a device allocator).  Its split-K scratch lives in a fixed array inside
the library; this checks, through the C ABI, that two calls in a row agree with
mla_sparse_decode (which takes caller workspace) within the decode tolerance.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import assert_decode_close, lib

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def build_case(m, maker):
    wl = maker()

    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)

    W.fill_pool(wl, 0, qa)
    return wl


def run_both(m, wl):
    lse_ref = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    ref, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                 wl.context_lens, wl.topk_idx, wl.softmax_scale, lse=lse_ref)
    lse = torch.empty_like(lse_ref)
    out = torch.empty_like(ref)
    L = m.load()
    st = L.mla_sparse_decode_noalloc(
        C.c_void_p(wl.q_nope.data_ptr()), C.c_void_p(wl.q_rope.data_ptr()), C.c_void_p(wl.pools[0].data_ptr()),
        wl.strides[0], wl.num_blocks, C.c_void_p(wl.block_table.data_ptr()), wl.block_table.shape[1],
        C.c_void_p(wl.context_lens.data_ptr()), C.c_void_p(wl.topk_idx.data_ptr()), wl.batch, wl.heads, 64,
        wl.topk, wl.softmax_scale, C.c_void_p(out.data_ptr()), C.c_void_p(lse.data_ptr()),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, m.mla_status_string(st)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy(), lse.cpu().numpy()), (ref.float().cpu().numpy(), lse_ref.cpu().numpy())


def test_no_alloc_decode_matches_workspace_decode_twice():
    m = lib()
    assert m.mla_sparse_decode_workspace_size(32, 16, 2048) <= 16 << 20
    # 8 splits (merged inside a thread-block cluster), 32 and 64 splits
    # (merged by a second kernel), and 64 heads (the tensor-memory kernel,
    # its split lists merged by the second kernel)
    cases = [
        build_case(m, lambda: W.tiny_decode(DEV, seed=3)),
        build_case(m, lambda: W.tp4_rank_decode(DEV, seed=5, batch=8, ctx=20_000)),
        build_case(m, lambda: W.tp4_rank_decode(DEV, seed=6, batch=2, ctx=9_000)),
        build_case(m, lambda: W.tp4_rank_decode(DEV, seed=7, batch=2, ctx=9_000, heads=64)),
    ]
    for wl in cases:  # calls in a row, different shapes sharing the scratch
        assert m.mla_sparse_decode_workspace_size(wl.batch, wl.heads, wl.topk) > 0  # the scratch is used
        (out, lse), (ref, ref_lse) = run_both(m, wl)
        for b in range(wl.batch):
            assert_decode_close(out[b], lse[b], ref[b].astype(np.float64), ref_lse[b].astype(np.float64),
                                f"request {b}")
