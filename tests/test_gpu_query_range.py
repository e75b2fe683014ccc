"""The absorbed query over the whole bf16 range, against the float64 oracle.

The pages compute with FP16 operands and FP32 accumulation ("Prime Inference:
serving GLM-5.3 to agents is a KV-cache problem", section "A kernel that reads
four bits directly"), but the query arrives as bf16, whose exponent range is
far wider than FP16's (largest finite 65504, smallest normal 2^-14).  The
kernels scale each head's query by a power of two that brings its largest
magnitude to [2^14, 2^15) and fold the inverse into that head's softmax
scale, which leaves the scores exactly as they were.

Each case multiplies q by a factor f and the softmax scale by 1/f: the scores,
and so the outputs, are those of the unscaled problem, but the query itself
lies far outside FP16's range (f = 2^20, 2^120) or deep below its normal range
(f = 2^-24, 2^-120), or is not a power of two (1e3, 1e-5: the bf16 rounding
of q*f is what the oracle sees).  A mixed case gives neighbouring heads of one
CTA factors 2^40 apart.  Tolerance as for every decode test (gpu_helpers)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMTS = [pytest.param(O.FMT_NVFP4, id="nvfp4"), pytest.param(O.FMT_FP8, id="fp8")]
FACTORS = [pytest.param(2.0 ** 20, id="2^20"), pytest.param(2.0 ** -24, id="2^-24"),
           pytest.param(1e3, id="1e3"), pytest.param(1e-5, id="1e-5"),
           pytest.param(2.0 ** 120, id="2^120"), pytest.param(2.0 ** -120, id="2^-120"),
           pytest.param(None, id="mixed")]


def quantize_fn(m):
    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)
    return qa


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("heads", [16, 64])
@pytest.mark.parametrize("factor", FACTORS)
def test_query_far_outside_fp16_range(fmt, heads, factor):
    m = lib()
    batch, topk, ctx_lens = 2, 512, [3000, 1500]

    def draw(b, c, g):
        return W.distinct_uniform(min(topk, c), 0, c, g, DEV)

    wl = W._decode_workload("qrange", ("qrange", heads), batch, heads, topk, ctx_lens, DEV, 0.01, draw)
    if factor is None:
        # heads alternate between 2^20 and 2^-20 (scale 2^-20): the first kind
        # scores as unscaled, the second has near-zero scores (uniform weights)
        f = torch.where(torch.arange(heads, device=DEV) % 2 == 0, 2.0 ** 20, 2.0 ** -20)[None, :, None]
        scale = wl.softmax_scale * 2.0 ** -20
    else:
        f = factor
        scale = wl.softmax_scale / factor
    wl.q_nope = (wl.q_nope.double() * f).to(torch.bfloat16).contiguous()
    wl.q_rope = (wl.q_rope.double() * f).to(torch.bfloat16).contiguous()
    assert torch.isfinite(wl.q_nope.float()).all() and torch.isfinite(wl.q_rope.float()).all()
    W.fill_pool(wl, fmt, quantize_fn(m))
    dec = m.mla_sparse_decode if fmt == O.FMT_NVFP4 else m.mla_sparse_decode_fp8
    lse = torch.empty((batch, heads), dtype=torch.float32, device=DEV)
    out, _ = dec(wl.q_nope, wl.q_rope, wl.pools[fmt], wl.strides[fmt], wl.num_blocks, wl.block_table,
                 wl.context_lens, wl.topk_idx, scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(batch):
        idx = wl.topk_idx[b].cpu().numpy().astype(np.int64)
        valid = (idx >= 0) & (idx < ctx_lens[b])
        lat, rope = wl.request_rows(b, torch.from_numpy(np.where(valid, idx, 0)).to(DEV))
        ref, ref_lse = oracle_rows_decode(u16(wl.q_nope[b]), u16(wl.q_rope[b]), u16(lat), u16(rope), valid, fmt,
                                          scale)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"request {b}")
