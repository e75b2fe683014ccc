"""Helpers shared by the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

import oracle as O

# Decode tolerance for bf16 outputs against the float64 oracle (workload
# acceptance bar): max-abs <= 2e-2 * max|ref|, relative RMS <= 5e-3; the
# natural-log LSE within 1e-3 * (1 + |ref|).
MAXABS_REL = 2e-2
RMS_REL = 5e-3
LSE_REL = 1e-3


def lib():
    from sparse_mla_decode_kv_gb300 import build
    build.build()
    import sparse_mla_decode_kv_gb300 as m
    m.load()
    return m


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 (or 16-bit) tensor -> numpy uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_rows_decode(q_nope_b, q_rope_b, lat_rows, rope_rows, valid, fmt, scale):
    """Float64 decode of one request whose selected rows are given directly.

    The oracle quantizes the bf16 rows itself into a compact pool (token j of
    the list at logical position j), so nothing from the CUDA path enters it.
    `valid` (bool per list entry) marks entries that are not masked."""
    k = lat_rows.shape[0]
    rb = O.row_bytes(fmt)
    nblk = max(1, (k + 63) // 64)
    stride = 64 * rb
    pool = np.zeros(nblk * stride, dtype=np.uint8)
    O.kv_quantize_append(lat_rows, rope_rows, np.arange(k, dtype=np.int64), pool, nblk, 64, stride, fmt)
    idx = np.where(valid, np.arange(k), -1).astype(np.int32)[None]
    bt = np.arange(nblk, dtype=np.int32)[None]
    out, lse = O.sparse_decode(q_nope_b[None], q_rope_b[None], pool, stride, bt, np.array([k], np.int32), idx, 64,
                               scale, fmt)
    return out[0], lse[0]


def assert_decode_close(out_gpu: np.ndarray, lse_gpu, out_ref: np.ndarray, lse_ref, what=""):
    out_gpu = out_gpu.astype(np.float64)
    scale = np.abs(out_ref).max()
    err = np.abs(out_gpu - out_ref)
    if scale == 0:
        assert err.max() == 0, f"{what}: expected zeros"
    else:
        assert err.max() <= MAXABS_REL * scale, f"{what}: max-abs {err.max():.3e} > {MAXABS_REL} * {scale:.3e}"
        rms = np.sqrt((err ** 2).mean()) / np.sqrt((out_ref ** 2).mean())
        assert rms <= RMS_REL, f"{what}: relative RMS {rms:.3e} > {RMS_REL}"
    if lse_gpu is not None:
        lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
        inf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), inf_ref), f"{what}: -inf pattern of lse differs"
        d = np.abs(lse_gpu[~inf_ref] - lse_ref[~inf_ref])
        assert np.all(d <= LSE_REL * (1 + np.abs(lse_ref[~inf_ref]))), f"{what}: lse off by {d.max():.3e}"
