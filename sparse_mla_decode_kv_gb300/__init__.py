"""Python binding of libmla_nvfp4.so (sparse MLA decode over an NVFP4 paged KV cache).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions carry the C names from ``include/mla_nvfp4.h`` and take
torch tensors (device memory) plus an optional stream; they raise
``MlaError`` on any non-OK status.  There is no fallback: if the library is
not built, loading fails with an explicit error.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import torch

__all__ = [
    "MlaError", "MLA_KV_NVFP4", "MLA_KV_FP8", "library_path", "load",
    "mla_kv_row_bytes", "mla_status_string", "mla_last_cuda_error", "mla_device_fault",
    "mla_kv_quantize_append", "mla_sparse_decode_workspace_size", "mla_sparse_decode_plan",
    "mla_sparse_decode_plan_fmt", "mla_sparse_decode",
    "mla_sparse_decode_fp8", "mla_sparse_decode_noalloc", "mla_topk_workspace_size", "mla_topk",
    "mla_indexer_topk_workspace_size", "mla_indexer_topk", "mla_index_key_quantize_append",
    "mla_staged_pool_bytes", "mla_stage_rows_fp8", "mla_sparse_decode_staged_workspace_size",
    "mla_sparse_decode_staged", "mla_sparse_decode_mtp_workspace_size", "mla_sparse_decode_mtp",
]

MLA_KV_NVFP4 = 0
MLA_KV_FP8 = 1
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmla_nvfp4.so"
_lib = None

_STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_WORKSPACE_TOO_SMALL",
           4: "MLA_ERR_CUDA"}

# Every symbol include/mla_nvfp4.h declares, with (restype, argtypes).
_P, _I32, _I64, _SZ, _F32 = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float
SIGNATURES = {
    "mla_kv_row_bytes": (_SZ, [_I32]),
    "mla_status_string": (C.c_char_p, [_I32]),
    "mla_last_cuda_error": (_I32, [_P]),
    "mla_device_fault": (_I32, [_P, _I32, _P]),
    "mla_kv_quantize_append": (_I32, [_P, _P, _P, _I64, _P, _I64, _I32, _I64, _I32, _P]),
    "mla_sparse_decode_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "mla_sparse_decode_plan": (_I32, [_I32, _I32, _I32, _P, _P, _P]),
    "mla_sparse_decode_plan_fmt": (_I32, [_I32, _I32, _I32, _I32, _I64, _I64, _P, _P, _P, _P]),
    "mla_sparse_decode": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _F32, _P, _P,
                                 _P, _SZ, _P]),
    "mla_sparse_decode_fp8": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _F32, _P,
                                     _P, _P, _SZ, _P]),
    "mla_sparse_decode_noalloc": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _F32, _P,
                                         _P, _P]),
    "mla_topk_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "mla_topk": (_I32, [_P, _I64, _P, _I32, _I32, _I32, _P, _P, _SZ, _P]),
    "mla_indexer_topk_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "mla_indexer_topk": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _I32, _P,
                                _SZ, _P]),
    "mla_index_key_quantize_append": (_I32, [_P, _P, _I64, _P, _I64, _I32, _I64, _P]),
    "mla_sparse_decode_mtp_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "mla_sparse_decode_mtp": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _F32,
                                     _I32, _P, _P, _P, _SZ, _P]),
    "mla_staged_pool_bytes": (_SZ, [_I32, _I32]),
    "mla_stage_rows_fp8": (_I32, [_P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "mla_sparse_decode_staged_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "mla_sparse_decode_staged": (_I32, [_P, _P, _P, _I64, _I64, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _F32, _P,
                                        _P, _P, _SZ, _P]),
}


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = _STATUS.get(status, str(status))
        if status == 4:
            err = C.c_int(0)
            load().mla_last_cuda_error(C.byref(err))
            detail += f" (cudaError {err.value})"
        super().__init__(f"{fn} failed: {detail}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load():
    """Load libmla_nvfp4.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
                               " (or sparse_mla_decode_kv_gb300/build.py); there is no CPU fallback")
        lib = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MlaError(fn, status)


def _contig(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _bits(t: torch.Tensor, name: str) -> torch.Tensor:
    """bf16 tensors are passed as their 16-bit patterns."""
    if t.dtype == torch.bfloat16:
        return _contig(t, torch.bfloat16, name)
    return _contig(t, torch.int16, name) if t.dtype == torch.int16 else _contig(t, torch.uint16, name)


# --------------------------------------------------------------------- misc
def mla_kv_row_bytes(fmt: int) -> int:
    return int(load().mla_kv_row_bytes(fmt))


def mla_status_string(status: int) -> str:
    return load().mla_status_string(status).decode()


def mla_last_cuda_error() -> int:
    err = C.c_int(0)
    load().mla_last_cuda_error(C.byref(err))
    return err.value


def mla_device_fault(clear: bool = False, stream=None) -> int:
    word = C.c_uint(0)
    _check("mla_device_fault", load().mla_device_fault(C.byref(word), int(clear), _stream(stream)))
    return word.value


# --------------------------------------------------------------------- quantize-on-write
def mla_kv_quantize_append(latent: torch.Tensor, rope: torch.Tensor, slot_mapping: torch.Tensor,
                           kv_pool: torch.Tensor, num_blocks: int, block_size: int, kv_block_stride: int,
                           fmt: int = MLA_KV_NVFP4, stream=None) -> None:
    latent = _bits(latent, "latent")
    rope = _bits(rope, "rope")
    slot_mapping = _contig(slot_mapping, torch.int64, "slot_mapping")
    n = slot_mapping.numel()
    if latent.numel() != n * 512 or rope.numel() != n * 64:
        raise ValueError("latent must be [n,512] and rope [n,64] for n = len(slot_mapping)")
    if num_blocks > 0 and kv_pool.numel() * kv_pool.element_size() < (num_blocks - 1) * kv_block_stride + \
            block_size * (352 if fmt == MLA_KV_NVFP4 else 576):
        raise ValueError("kv_pool does not reach the last row of block num_blocks - 1")
    _check("mla_kv_quantize_append",
           load().mla_kv_quantize_append(_ptr(latent), _ptr(rope), _ptr(slot_mapping), n, _ptr(kv_pool),
                                         num_blocks, block_size, kv_block_stride, fmt, _stream(stream)))


def mla_index_key_quantize_append(keys: torch.Tensor, slot_mapping: torch.Tensor, idx_key_pool: torch.Tensor,
                                  num_blocks: int, block_size: int, idx_block_stride: int, stream=None) -> None:
    """Indexer keys bf16 [n, 128] -> 128 e4m3 codes + a float scale per token, by slot."""
    keys = _bits(keys, "keys")
    slot_mapping = _contig(slot_mapping, torch.int64, "slot_mapping")
    n = slot_mapping.numel()
    if keys.numel() != n * 128:
        raise ValueError("keys must be [n,128] for n = len(slot_mapping)")
    if num_blocks > 0 and idx_key_pool.numel() * idx_key_pool.element_size() < (num_blocks - 1) * idx_block_stride + \
            block_size * 132:
        raise ValueError("idx_key_pool does not reach the last scale of block num_blocks - 1")
    _check("mla_index_key_quantize_append",
           load().mla_index_key_quantize_append(_ptr(keys), _ptr(slot_mapping), n, _ptr(idx_key_pool), num_blocks,
                                                block_size, idx_block_stride, _stream(stream)))


# --------------------------------------------------------------------- sparse decode
def mla_sparse_decode_workspace_size(batch: int, num_heads: int, topk: int) -> int:
    return int(load().mla_sparse_decode_workspace_size(batch, num_heads, topk))


def mla_sparse_decode_plan(batch: int, num_heads: int, topk: int) -> dict:
    """{"splits", "rows_per_split", "kernels"} of one decode call on the current device."""
    sp, rows, kern = C.c_int(0), C.c_int(0), C.c_int(0)
    _check("mla_sparse_decode_plan",
           load().mla_sparse_decode_plan(batch, num_heads, topk, C.byref(sp), C.byref(rows), C.byref(kern)))
    return {"splits": sp.value, "rows_per_split": rows.value, "kernels": kern.value}


def mla_sparse_decode_plan_fmt(fmt: int, batch: int, num_heads: int, topk: int, kv_block_stride: int,
                               num_blocks: int) -> dict:
    """The division a decode with this cache format and pool geometry uses,
    including whether it runs the tensor-memory kernel."""
    sp, rows, kern, tm = C.c_int(), C.c_int(), C.c_int(), C.c_int()
    _check("mla_sparse_decode_plan_fmt",
           load().mla_sparse_decode_plan_fmt(fmt, batch, num_heads, topk, kv_block_stride, num_blocks, C.byref(sp),
                                             C.byref(rows), C.byref(kern), C.byref(tm)))
    return {"splits": sp.value, "rows_per_split": rows.value, "kernels": kern.value,
            "tensor_memory": bool(tm.value)}

def _decode(cname: str, q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx,
            softmax_scale, block_size=64, out=None, lse=None, workspace=None, stream=None,
            ws_size=mla_sparse_decode_workspace_size):
    q_nope = _bits(q_nope, "q_nope")
    q_rope = _bits(q_rope, "q_rope")
    block_table = _contig(block_table, torch.int32, "block_table")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    topk_idx = _contig(topk_idx, torch.int32, "topk_idx")
    batch, heads = q_nope.shape[0], q_nope.shape[1]
    topk = topk_idx.shape[1]
    if out is None:
        out = torch.empty((batch, heads, 512), dtype=torch.bfloat16, device=q_nope.device)
    need = ws_size(batch, heads, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = getattr(load(), cname)
    _check(cname, fn(_ptr(q_nope), _ptr(q_rope), _ptr(kv_pool), kv_block_stride, num_blocks, _ptr(block_table),
                     block_table.shape[1], _ptr(context_lens), _ptr(topk_idx), batch, heads, block_size, topk,
                     float(softmax_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse


def mla_sparse_decode(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx,
                      softmax_scale, block_size=64, out=None, lse=None, workspace=None, stream=None):
    """NVFP4 cache.  Returns (out bf16 [B,H,512], lse or None)."""
    return _decode("mla_sparse_decode", q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                   context_lens, topk_idx, softmax_scale, block_size, out, lse, workspace, stream)


def mla_sparse_decode_fp8(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx,
                          softmax_scale, block_size=64, out=None, lse=None, workspace=None, stream=None):
    """FP8 (576-byte) cache.  Returns (out bf16 [B,H,512], lse or None)."""
    return _decode("mla_sparse_decode_fp8", q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                   context_lens, topk_idx, softmax_scale, block_size, out, lse, workspace, stream)


def mla_sparse_decode_staged_workspace_size(batch: int, num_heads: int, topk: int) -> int:
    return int(load().mla_sparse_decode_staged_workspace_size(batch, num_heads, topk))


def mla_sparse_decode_staged(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens,
                             topk_idx, softmax_scale, block_size=64, out=None, lse=None, workspace=None, stream=None):
    """Staged path over the NVFP4 cache (gather to an FP8 copy, then the FP8
    decode).  Returns (out bf16 [B,H,512], lse or None)."""
    return _decode("mla_sparse_decode_staged", q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                   context_lens, topk_idx, softmax_scale, block_size, out, lse, workspace, stream,
                   ws_size=mla_sparse_decode_staged_workspace_size)


def mla_sparse_decode_mtp_workspace_size(batch: int, q_len: int, num_heads: int, topk: int) -> int:
    return int(load().mla_sparse_decode_mtp_workspace_size(batch, q_len, num_heads, topk))


def mla_sparse_decode_mtp(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx,
                          softmax_scale, fmt=MLA_KV_NVFP4, block_size=64, out=None, lse=None, workspace=None,
                          stream=None):
    """Several query tokens per request: q_nope [B,Q,H,512], q_rope [B,Q,H,64],
    topk_idx int32 [B,Q,k].  Returns (out bf16 [B,Q,H,512], lse or None)."""
    q_nope = _bits(q_nope, "q_nope")
    q_rope = _bits(q_rope, "q_rope")
    block_table = _contig(block_table, torch.int32, "block_table")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    topk_idx = _contig(topk_idx, torch.int32, "topk_idx")
    batch, q_len, heads = q_nope.shape[0], q_nope.shape[1], q_nope.shape[2]
    topk = topk_idx.shape[2]
    if out is None:
        out = torch.empty((batch, q_len, heads, 512), dtype=torch.bfloat16, device=q_nope.device)
    need = mla_sparse_decode_mtp_workspace_size(batch, q_len, heads, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("mla_sparse_decode_mtp",
           load().mla_sparse_decode_mtp(_ptr(q_nope), _ptr(q_rope), _ptr(kv_pool), kv_block_stride, num_blocks,
                                        _ptr(block_table), block_table.shape[1], _ptr(context_lens), _ptr(topk_idx),
                                        batch, q_len, heads, block_size, topk, float(softmax_scale), fmt, _ptr(out),
                                        _ptr(lse), _ptr(workspace), ws_bytes, _stream(stream)))
    return out, lse


def mla_staged_pool_bytes(batch: int, topk: int) -> int:
    return int(load().mla_staged_pool_bytes(batch, topk))


def mla_stage_rows_fp8(kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx, block_size=64,
                       staged_pool=None, staged_topk=None, stream=None):
    """Gather step of the staged path.  Returns (staged_pool uint8, staged_topk int32 [B, topk])."""
    block_table = _contig(block_table, torch.int32, "block_table")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    topk_idx = _contig(topk_idx, torch.int32, "topk_idx")
    batch, topk = topk_idx.shape
    dev = topk_idx.device
    if staged_pool is None:
        staged_pool = torch.empty(mla_staged_pool_bytes(batch, topk), dtype=torch.uint8, device=dev)
    if staged_pool.numel() * staged_pool.element_size() < mla_staged_pool_bytes(batch, topk):
        raise ValueError("staged_pool is smaller than mla_staged_pool_bytes(batch, topk)")
    if staged_topk is None:
        staged_topk = torch.empty((batch, topk), dtype=torch.int32, device=dev)
    _check("mla_stage_rows_fp8",
           load().mla_stage_rows_fp8(_ptr(kv_pool), kv_block_stride, num_blocks, _ptr(block_table),
                                     block_table.shape[1], _ptr(context_lens), _ptr(topk_idx), batch, block_size,
                                     topk, _ptr(staged_pool), _ptr(staged_topk), _stream(stream)))
    return staged_pool, staged_topk


def mla_sparse_decode_noalloc(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, context_lens,
                              topk_idx, softmax_scale, block_size=64, out=None, lse=None, stream=None):
    """NVFP4 decode whose split-K scratch is the library's own fixed device
    array (for callers that cannot allocate); same results as
    mla_sparse_decode.  Returns (out bf16 [B,H,512], lse or None)."""
    q_nope = _bits(q_nope, "q_nope")
    q_rope = _bits(q_rope, "q_rope")
    block_table = _contig(block_table, torch.int32, "block_table")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    topk_idx = _contig(topk_idx, torch.int32, "topk_idx")
    batch, heads = q_nope.shape[0], q_nope.shape[1]
    if out is None:
        out = torch.empty((batch, heads, 512), dtype=torch.bfloat16, device=q_nope.device)
    _check("mla_sparse_decode_noalloc",
           load().mla_sparse_decode_noalloc(_ptr(q_nope), _ptr(q_rope), _ptr(kv_pool), kv_block_stride, num_blocks,
                                            _ptr(block_table), block_table.shape[1], _ptr(context_lens),
                                            _ptr(topk_idx), batch, heads, block_size, topk_idx.shape[1],
                                            float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


# --------------------------------------------------------------------- top-k and indexer
def mla_topk_workspace_size(batch: int, max_context_len: int, topk: int) -> int:
    return int(load().mla_topk_workspace_size(batch, max_context_len, topk))


def mla_topk(scores: torch.Tensor, context_lens: torch.Tensor, topk: int, out=None, workspace=None, stream=None):
    """scores float32 [B, max_context_len] -> int32 [B, topk] (ascending, -1 padded)."""
    scores = _contig(scores, torch.float32, "scores")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    batch, max_ctx = scores.shape
    if out is None:
        out = torch.empty((batch, topk), dtype=torch.int32, device=scores.device)
    need = mla_topk_workspace_size(batch, max_ctx, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=scores.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check("mla_topk", load().mla_topk(_ptr(scores), max_ctx, _ptr(context_lens), batch, topk, max_ctx, _ptr(out),
                                       _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def mla_indexer_topk_workspace_size(batch: int, max_context_len: int, topk: int) -> int:
    return int(load().mla_indexer_topk_workspace_size(batch, max_context_len, topk))


def mla_indexer_topk(q_idx, head_w, idx_key_pool, idx_block_stride, num_blocks, block_table, context_lens, topk,
                     max_context_len, block_size=64, topk_out=None, scores_out=None, workspace=None, stream=None):
    """Indexer scores + exact top-k.  Returns (topk_out int32 [B,topk], scores_out or None)."""
    q_idx = _bits(q_idx, "q_idx")
    head_w = _contig(head_w, torch.float32, "head_w")
    block_table = _contig(block_table, torch.int32, "block_table")
    context_lens = _contig(context_lens, torch.int32, "context_lens")
    batch, nh = q_idx.shape[0], q_idx.shape[1]
    if topk_out is None:
        topk_out = torch.empty((batch, topk), dtype=torch.int32, device=q_idx.device)
    need = mla_indexer_topk_workspace_size(batch, max_context_len, topk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_idx.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check("mla_indexer_topk",
           load().mla_indexer_topk(_ptr(q_idx), _ptr(head_w), _ptr(idx_key_pool), idx_block_stride, num_blocks,
                                   _ptr(block_table), block_table.shape[1], _ptr(context_lens), batch, nh, block_size,
                                   topk, _ptr(topk_out), _ptr(scores_out), max_context_len, _ptr(workspace),
                                   ws_bytes, _stream(stream)))
    return topk_out, scores_out
