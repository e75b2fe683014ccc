"""mla_sparse_decode_noalloc: the decode for callers that cannot allocate
device memory (a serving process with a fixed device-memory budget, or a C host
without a device allocator).  Its split-K scratch lives in a fixed array inside
the library; this checks, through the C ABI, that two calls in a row give the
same bytes as mla_sparse_decode (which takes caller workspace): both run the
same kernels on the same inputs, so anything but bit-identical output would
mean stale or shared scratch leaking into a result.

Collected last on purpose (file name), so a stop-at-first-failure run has
already run every other test."""
import ctypes as C

import pytest
import torch

import workloads as W
from gpu_helpers import lib

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def build_case(m, maker):
    wl = maker()

    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)

    W.fill_pool(wl, 0, qa)
    return wl


def noalloc_call(m, wl, out, lse):
    L = m.load()
    return L.mla_sparse_decode_noalloc(
        C.c_void_p(wl.q_nope.data_ptr()), C.c_void_p(wl.q_rope.data_ptr()), C.c_void_p(wl.pools[0].data_ptr()),
        wl.strides[0], wl.num_blocks, C.c_void_p(wl.block_table.data_ptr()), wl.block_table.shape[1],
        C.c_void_p(wl.context_lens.data_ptr()), C.c_void_p(wl.topk_idx.data_ptr()), wl.batch, wl.heads, 64,
        wl.topk, wl.softmax_scale, C.c_void_p(out.data_ptr()), C.c_void_p(lse.data_ptr()),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))


def run_both(m, wl):
    lse_ref = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    ref, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                 wl.context_lens, wl.topk_idx, wl.softmax_scale, lse=lse_ref)
    outs = []
    for _ in range(2):  # two calls in a row on the same inputs, sharing the scratch
        lse = torch.full_like(lse_ref, float("nan"))
        out = torch.full_like(ref, 0x7FFF)
        st = noalloc_call(m, wl, out, lse)
        assert st == 0, m.mla_status_string(st)
        torch.cuda.synchronize()
        outs.append((out.cpu(), lse.cpu()))
    return outs, (ref.cpu(), lse_ref.cpu())


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
    for wl in cases:  # different shapes in a row, all sharing the one scratch array
        assert m.mla_sparse_decode_workspace_size(wl.batch, wl.heads, wl.topk) > 0  # the scratch is used
        outs, (ref, ref_lse) = run_both(m, wl)
        for out, lse in outs:
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_no_alloc_decode_refuses_too_much_scratch_and_launches_nothing():
    """A shape whose split-K scratch exceeds the fixed array is refused with
    MLA_ERR_WORKSPACE_TOO_SMALL, and the output buffers are left as they were."""
    m = lib()
    wl = build_case(m, lambda: W.tp4_rank_decode(DEV, seed=8, batch=2, ctx=9_000))
    big_batch = 512
    assert m.mla_sparse_decode_workspace_size(big_batch, wl.heads, wl.topk) > 16 << 20
    out = torch.full((big_batch, wl.heads, 512), 0x1234, dtype=torch.int16, device=DEV)
    lse = torch.full((big_batch, wl.heads), 7.0, dtype=torch.float32, device=DEV)
    L = m.load()
    st = L.mla_sparse_decode_noalloc(
        C.c_void_p(wl.q_nope.data_ptr()), C.c_void_p(wl.q_rope.data_ptr()), C.c_void_p(wl.pools[0].data_ptr()),
        wl.strides[0], wl.num_blocks, C.c_void_p(wl.block_table.data_ptr()), wl.block_table.shape[1],
        C.c_void_p(wl.context_lens.data_ptr()), C.c_void_p(wl.topk_idx.data_ptr()), big_batch, wl.heads, 64,
        wl.topk, wl.softmax_scale, C.c_void_p(out.data_ptr()), C.c_void_p(lse.data_ptr()),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 3, m.mla_status_string(st)
    torch.cuda.synchronize()
    assert bool((out == 0x1234).all()) and bool((lse == 7.0).all())
