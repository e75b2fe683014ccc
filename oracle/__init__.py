"""Float64 CPU oracle for sparse MLA decode over an NVFP4 / FP8 paged latent cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never imports, links or calls it, and it shares no
code with the CUDA library: the arithmetic lives in ``mla_oracle.c`` (plain C,
float64, written from the definitions) and this module only marshals numpy
arrays into it through ctypes.

Parity status per function (pins live in ``tests/test_oracle_*.py``):

* e4m3 / e2m1 encode and decode, row quantize / dequantize -- pinned (OCP
  tables, brute-force nearest-even search, hand-worked vectors).
* sparse decode -- pinned (k = 1, identical rows, q = 0, permutation, all
  masked, brute-force un-absorbed dense MLA on tiny inputs).
* indexer score -- pinned (one-hot head weights against an independent
  numpy recomputation from the OCP decode table, relu / sign cases).
* top-k -- pinned (numpy lexsort brute force, all-equal scores, ctx < k).
* several query tokens per request -- pinned (one token equals the single-
  token decode; the last token sees the whole context; causal masking
  against a brute-force softmax over the explicitly visible positions).
* staged FP8 copy of an NVFP4 row -- pinned (nearest-e4m3 brute force over
  the independently decoded values, exactly representable rows, saturation).
* indexer-key quantize -- pinned (nearest-e4m3 brute force on the float
  quotient, power-of-two scaling invariance, amax code, zero key).

Sources: "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem"
(sections "Four bits per latent value" and "A kernel that reads four bits
directly"); "GLM-5.3 PCP/DCP long-context on H200" (sections 1 and 3).
"""
from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .build import build_oracle

FMT_NVFP4 = 0
FMT_FP8 = 1
LATENT = 512
ROPE = 64
IDX_DIM = 128

_lib = None


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = build_oracle()
        L = C.CDLL(path)
        P = C.c_void_p
        i32, i64, f64 = C.c_int, C.c_int64, C.c_double
        L.oracle_bf16_to_double.restype = f64
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_e4m3_to_double.restype = f64
        L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
        L.oracle_e2m1_to_double.restype = f64
        L.oracle_e2m1_to_double.argtypes = [C.c_uint8]
        L.oracle_e4m3_from_double.restype = C.c_uint8
        L.oracle_e4m3_from_double.argtypes = [f64]
        L.oracle_e2m1_from_double.restype = C.c_uint8
        L.oracle_e2m1_from_double.argtypes = [f64]
        L.oracle_e4m3_from_double_array.restype = None
        L.oracle_e4m3_from_double_array.argtypes = [P, i64, P]
        L.oracle_e2m1_from_double_array.restype = None
        L.oracle_e2m1_from_double_array.argtypes = [P, i64, P]
        L.oracle_row_bytes.restype = C.c_size_t
        L.oracle_row_bytes.argtypes = [i32]
        L.oracle_quantize_row_nvfp4.restype = None
        L.oracle_quantize_row_nvfp4.argtypes = [P, P, P]
        L.oracle_quantize_row_fp8.restype = None
        L.oracle_quantize_row_fp8.argtypes = [P, P, P]
        L.oracle_dequant_row.restype = None
        L.oracle_dequant_row.argtypes = [P, i32, P, P]
        L.oracle_kv_quantize_append.restype = i64
        L.oracle_kv_quantize_append.argtypes = [P, P, P, i64, P, i64, i32, i64, i32]
        L.oracle_sparse_decode_request.restype = None
        L.oracle_sparse_decode_request.argtypes = [P, P, P, i64, P, i32, P, i32, i32, i32, f64, i32, P, P]
        L.oracle_indexer_scores_request.restype = None
        L.oracle_indexer_scores_request.argtypes = [P, P, i32, P, i64, P, i32, i32, P]
        L.oracle_topk_request.restype = None
        L.oracle_topk_request.argtypes = [P, i32, i32, P]
        L.oracle_topk_request_f32.restype = None
        L.oracle_topk_request_f32.argtypes = [P, i32, i32, P]
        L.oracle_sparse_decode_mtp.restype = None
        L.oracle_sparse_decode_mtp.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, f64, i32, P, P]
        L.oracle_stage_row_fp8.restype = None
        L.oracle_stage_row_fp8.argtypes = [P, P]
        L.oracle_stage_rows_fp8.restype = None
        L.oracle_stage_rows_fp8.argtypes = [P, i64, i64, P, i32, P, P, i32, i32, i32, P, P]
        L.oracle_quantize_index_key.restype = None
        L.oracle_quantize_index_key.argtypes = [P, P, P]
        L.oracle_index_key_quantize_append.restype = i64
        L.oracle_index_key_quantize_append.argtypes = [P, P, i64, P, i64, i32, i64]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def row_bytes(fmt: int) -> int:
    return int(lib().oracle_row_bytes(fmt))


# ---------------------------------------------------------------- scalars
def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code))


def e2m1_decode(code: int) -> float:
    return lib().oracle_e2m1_to_double(int(code))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_from_double(float(x)))


def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_from_double(float(v)))


def e4m3_encode_array(x) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().oracle_e4m3_from_double_array(_ptr(a), a.size, _ptr(out))
    return out


def e2m1_encode_array(v) -> np.ndarray:
    a = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint8)
    lib().oracle_e2m1_from_double_array(_ptr(a), a.size, _ptr(out))
    return out


# ---------------------------------------------------------------- rows
def quantize_row(latent_bf16: np.ndarray, rope_bf16: np.ndarray, fmt: int) -> np.ndarray:
    lat = np.ascontiguousarray(latent_bf16, dtype=np.uint16).reshape(LATENT)
    rp = np.ascontiguousarray(rope_bf16, dtype=np.uint16).reshape(ROPE)
    out = np.zeros(row_bytes(fmt), dtype=np.uint8)
    fn = lib().oracle_quantize_row_nvfp4 if fmt == FMT_NVFP4 else lib().oracle_quantize_row_fp8
    fn(_ptr(lat), _ptr(rp), _ptr(out))
    return out


def dequant_row(row: np.ndarray, fmt: int):
    r = np.ascontiguousarray(row, dtype=np.uint8).reshape(row_bytes(fmt))
    c = np.zeros(LATENT, dtype=np.float64)
    rp = np.zeros(ROPE, dtype=np.float64)
    lib().oracle_dequant_row(_ptr(r), fmt, _ptr(c), _ptr(rp))
    return c, rp


def kv_quantize_append(latent, rope, slot_mapping, kv_pool: np.ndarray, num_blocks: int,
                       block_size: int, kv_block_stride: int, fmt: int) -> int:
    """Quantize-on-write into ``kv_pool`` (uint8, flat or shaped), in place.

    Tokens whose slot is negative or past the pool are skipped; returns how
    many were skipped."""
    lat = np.ascontiguousarray(latent, dtype=np.uint16)
    rp = np.ascontiguousarray(rope, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    n = sm.shape[0]
    assert lat.size == n * LATENT and rp.size == n * ROPE
    assert kv_pool.dtype == np.uint8 and kv_pool.flags["C_CONTIGUOUS"]
    assert num_blocks == 0 or kv_pool.size >= (num_blocks - 1) * kv_block_stride + block_size * row_bytes(fmt)
    return int(lib().oracle_kv_quantize_append(_ptr(lat), _ptr(rp), _ptr(sm), n, _ptr(kv_pool), num_blocks,
                                               block_size, kv_block_stride, fmt))


# ---------------------------------------------------------------- staged path
def stage_row_fp8(row: np.ndarray) -> np.ndarray:
    """One stored NVFP4 row -> the staged path's 576-byte FP8 row."""
    r = np.ascontiguousarray(row, dtype=np.uint8).reshape(row_bytes(FMT_NVFP4))
    out = np.zeros(row_bytes(FMT_FP8), dtype=np.uint8)
    lib().oracle_stage_row_fp8(_ptr(r), _ptr(out))
    return out


def stage_rows_fp8(kv_pool, kv_block_stride, num_blocks, block_table, context_lens, topk_idx, block_size,
                   staged_pool: np.ndarray) -> np.ndarray:
    """Staged gather of a batch into ``staged_pool`` (uint8, in place; rows of
    masked entries are left untouched).  Returns staged_topk int32 [B, k]:
    j for a valid entry j, -1 for a masked one."""
    pool = np.ascontiguousarray(kv_pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    tk = np.ascontiguousarray(topk_idx, dtype=np.int32)
    B, k = tk.shape
    nblk = (k + block_size - 1) // block_size
    assert staged_pool.dtype == np.uint8 and staged_pool.flags["C_CONTIGUOUS"]
    assert staged_pool.size >= B * nblk * block_size * row_bytes(FMT_FP8)
    out = np.empty((B, k), dtype=np.int32)
    lib().oracle_stage_rows_fp8(_ptr(pool), int(kv_block_stride), int(num_blocks), _ptr(bt), bt.shape[1], _ptr(cl),
                                _ptr(tk), B, block_size, k, _ptr(staged_pool), _ptr(out))
    return out


# ---------------------------------------------------------------- indexer keys
def quantize_index_key(key_bf16) -> tuple:
    """128 bf16 key values -> (128 e4m3 codes uint8, float32 scale)."""
    k = np.ascontiguousarray(key_bf16, dtype=np.uint16).reshape(IDX_DIM)
    codes = np.zeros(IDX_DIM, dtype=np.uint8)
    sc = np.zeros(1, dtype=np.float32)
    lib().oracle_quantize_index_key(_ptr(k), _ptr(codes), _ptr(sc))
    return codes, sc[0]


def index_key_quantize_append(keys, slot_mapping, key_pool: np.ndarray, num_blocks: int, block_size: int,
                              key_block_stride: int) -> int:
    """Indexer-key quantize-on-write into ``key_pool`` (uint8, in place);
    returns the number of skipped tokens."""
    k = np.ascontiguousarray(keys, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    n = sm.shape[0]
    assert k.size == n * IDX_DIM
    assert key_pool.dtype == np.uint8 and key_pool.flags["C_CONTIGUOUS"]
    assert num_blocks == 0 or key_pool.size >= (num_blocks - 1) * key_block_stride + block_size * (IDX_DIM + 4)
    return int(lib().oracle_index_key_quantize_append(_ptr(k), _ptr(sm), n, _ptr(key_pool), num_blocks,
                                                      block_size, key_block_stride))


# ---------------------------------------------------------------- decode
def sparse_decode(q_nope, q_rope, kv_pool, kv_block_stride, block_table, context_lens, topk_idx,
                  block_size: int, softmax_scale: float, fmt: int, requests=None, threads: int = 1):
    """Float64 absorbed-form sparse MLA decode.

    q_nope uint16 [B,H,512], q_rope uint16 [B,H,64], block_table int32
    [B,max_blocks], context_lens int32 [B], topk_idx int32 [B,k].
    Returns (out float64 [R,H,512], lse float64 [R,H]) for the R requests in
    ``requests`` (default: all), computed on ``threads`` host threads.
    """
    qn = np.ascontiguousarray(q_nope, dtype=np.uint16)
    qr = np.ascontiguousarray(q_rope, dtype=np.uint16)
    pool = np.ascontiguousarray(kv_pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    tk = np.ascontiguousarray(topk_idx, dtype=np.int32)
    B, H = qn.shape[0], qn.shape[1]
    k = tk.shape[1]
    reqs = list(range(B)) if requests is None else list(requests)
    out = np.zeros((len(reqs), H, LATENT), dtype=np.float64)
    lse = np.zeros((len(reqs), H), dtype=np.float64)
    L = lib()

    def one(i):
        b = reqs[i]
        o = out[i]
        l = lse[i]
        L.oracle_sparse_decode_request(_ptr(qn[b]), _ptr(qr[b]), _ptr(pool), int(kv_block_stride),
                                       _ptr(bt[b]), int(cl[b]), _ptr(tk[b]), k, H, block_size,
                                       float(softmax_scale), fmt, o.ctypes.data_as(C.c_void_p),
                                       l.ctypes.data_as(C.c_void_p))

    _run(one, len(reqs), threads)
    return out, lse


def sparse_decode_mtp(q_nope, q_rope, kv_pool, kv_block_stride, block_table, context_lens, topk_idx,
                      block_size: int, softmax_scale: float, fmt: int, requests=None, threads: int = 1):
    """Float64 decode of Q query tokens per request, each with its own top-k
    list; token i of request b sees positions < context_lens[b] - (Q-1-i).

    q_nope uint16 [B,Q,H,512], q_rope [B,Q,H,64], topk_idx int32 [B,Q,k].
    Returns (out [R,Q,H,512], lse [R,Q,H]) for the R requests in ``requests``."""
    qn = np.ascontiguousarray(q_nope, dtype=np.uint16)
    qr = np.ascontiguousarray(q_rope, dtype=np.uint16)
    pool = np.ascontiguousarray(kv_pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    tk = np.ascontiguousarray(topk_idx, dtype=np.int32)
    B, Q, H = qn.shape[0], qn.shape[1], qn.shape[2]
    k = tk.shape[2]
    reqs = list(range(B)) if requests is None else list(requests)
    out = np.zeros((len(reqs), Q, H, LATENT), dtype=np.float64)
    lse = np.zeros((len(reqs), Q, H), dtype=np.float64)
    L = lib()

    def one(j):
        b = reqs[j]
        L.oracle_sparse_decode_mtp(_ptr(qn[b]), _ptr(qr[b]), _ptr(pool), int(kv_block_stride), _ptr(bt[b]),
                                   bt.shape[1], _ptr(cl[b:b + 1]), _ptr(tk[b]), 1, Q, H, block_size, k,
                                   float(softmax_scale), fmt, out[j].ctypes.data_as(C.c_void_p),
                                   lse[j].ctypes.data_as(C.c_void_p))

    _run(one, len(reqs), threads)
    return out, lse


# ---------------------------------------------------------------- indexer / top-k
def indexer_scores(q_idx, head_w, idx_key_pool, idx_block_stride, block_table, context_lens,
                   block_size: int, requests=None, threads: int = 1):
    """Float64 indexer scores; returns a list of float64 [ctx_b] arrays."""
    q = np.ascontiguousarray(q_idx, dtype=np.uint16)
    w = np.ascontiguousarray(head_w, dtype=np.float32)
    pool = np.ascontiguousarray(idx_key_pool, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, nh = q.shape[0], q.shape[1]
    reqs = list(range(B)) if requests is None else list(requests)
    res = [np.zeros(int(cl[b]), dtype=np.float64) for b in reqs]
    L = lib()

    def one(i):
        b = reqs[i]
        L.oracle_indexer_scores_request(_ptr(q[b]), _ptr(w[b]), nh, _ptr(pool), int(idx_block_stride),
                                        _ptr(bt[b]), int(cl[b]), block_size, _ptr(res[i]))

    _run(one, len(reqs), threads)
    return res


def topk(scores: np.ndarray, k: int) -> np.ndarray:
    """Exact top-k of one request's scores: ascending indices, -1 padded.

    float64 scores use the double comparison; float32 scores (e.g. a GPU's own
    fp32 scores) are widened exactly, so the float order decides."""
    out = np.empty(k, dtype=np.int32)
    if scores.dtype == np.float32:
        s = np.ascontiguousarray(scores)
        lib().oracle_topk_request_f32(_ptr(s), int(s.shape[0]), int(k), _ptr(out))
    else:
        s = np.ascontiguousarray(scores, dtype=np.float64)
        lib().oracle_topk_request(_ptr(s), int(s.shape[0]), int(k), _ptr(out))
    return out


def _run(fn, n, threads):
    if threads <= 1 or n <= 1:
        for i in range(n):
            fn(i)
        return
    # ctypes releases the GIL around foreign calls, so threads run in parallel.
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fn, range(n)))


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
