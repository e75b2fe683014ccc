"""Indexer score and exact top-k on the GPU against the oracle.

Sources: "GLM-5.3 PCP/DCP long-context on H200", section 1 (the indexer
rates all preceding tokens; attention reads the best 2,048) and section 3 (a
key is 128 e4m3 bytes and a float scale); "Prime Inference:
serving GLM-5.3 to agents is a KV-cache problem", section "Decode: TP4"
(index_topk 2048).

Contract (the score is float32 on the GPU, float64 in the oracle):
  * top-k selection is exact: on synthetic float32 scores fed to both sides
    (mla_topk), the index sets are identical, ties going to the lower index;
  * scores are within 1e-5 (1 + |ref|) of the oracle;
  * the chained top-k equals the exact top-k of the GPU's own scores (checked
    with numpy, not the oracle), and differs from the oracle's top-k only by
    swaps whose two float64 scores lie within that band of the k-th score."""
import zlib

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
SCORE_TOL = 1e-5


def gpu_topk(m, scores: np.ndarray, lens, k):
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).to(DEV)
    cl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = m.mla_topk(s, cl, k)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def lexsort_topk(scores: np.ndarray, k: int) -> np.ndarray:
    s = scores.astype(np.float64) + 0.0  # -0.0 -> +0.0
    order = np.lexsort((np.arange(s.size), -s))
    sel = np.sort(order[:min(k, s.size)])
    out = np.full(k, -1, np.int32)
    out[:sel.size] = sel
    return out


@pytest.mark.parametrize("case", ["normal", "ties", "all_equal", "signed_zero", "negative", "tiny_ctx",
                                  "ctx_eq_k", "ctx_k_plus_1", "empty", "huge_range"])
def test_topk_exact_on_synthetic_scores(case):
    m = lib()
    rng = np.random.default_rng(zlib.crc32(case.encode()))
    B, L, k = 6, 20_000, 2048
    lens = [L, L - 3, 12_345, 4096, 2049, 2048]
    s = rng.standard_normal((B, L)).astype(np.float32) * 30 + 70
    if case == "ties":
        s = rng.integers(0, 40, (B, L)).astype(np.float32) * 0.25
    elif case == "all_equal":
        s[:] = 1.5
    elif case == "signed_zero":
        s = np.where(rng.random((B, L)) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        s[:, ::97] = 1.0
    elif case == "negative":
        s = -np.abs(s)
    elif case == "tiny_ctx":
        lens = [1, 0, 5, 2047, 100, 3]
    elif case == "ctx_eq_k":
        lens = [k] * B
    elif case == "ctx_k_plus_1":
        lens = [k + 1] * B
    elif case == "empty":
        lens = [0] * B
    elif case == "huge_range":
        s = (rng.standard_normal((B, L)) * np.exp(rng.uniform(-80, 80, (B, L)))).astype(np.float32)
    got = gpu_topk(m, s, lens, k)
    for b in range(B):
        ref = O.topk(s[b, :lens[b]], k)
        assert np.array_equal(got[b], ref), f"request {b}"


def oracle_scores(wl, requests, threads):
    return O.indexer_scores(u16(wl.q_idx), wl.head_w.cpu().numpy(), wl.key_pool.cpu().numpy(), wl.key_stride,
                            wl.block_table.cpu().numpy(), wl.context_lens.cpu().numpy(), 64, requests=requests,
                            threads=threads)


def run_indexer(m, wl, max_ctx):
    scores = torch.full((wl.q_idx.shape[0], max_ctx), float("nan"), dtype=torch.float32, device=DEV)
    topk, _ = m.mla_indexer_topk(wl.q_idx, wl.head_w, wl.key_pool, wl.key_stride, wl.num_blocks, wl.block_table,
                                 wl.context_lens, wl.topk, max_ctx, scores_out=scores)
    torch.cuda.synchronize()
    return topk.cpu().numpy(), scores.cpu().numpy()


def check_request(got_idx, got_scores, ref_scores, k):
    n = ref_scores.size
    gs = got_scores[:n].astype(np.float64)
    assert np.all(np.abs(gs - ref_scores) <= SCORE_TOL * (1 + np.abs(ref_scores))), "score accuracy"
    # selection exactness on the GPU's own scores (numpy, not the oracle)
    assert np.array_equal(got_idx, lexsort_topk(got_scores[:n], k)), "top-k of the GPU's scores"
    # against the float64 top-k: only near-tie swaps at the boundary are allowed
    ref_idx = O.topk(ref_scores, k)
    a, b = set(got_idx[got_idx >= 0].tolist()), set(ref_idx[ref_idx >= 0].tolist())
    if a == b:
        return 0
    kth = np.sort(ref_scores)[::-1][min(k, n) - 1]
    band = SCORE_TOL * (1 + abs(kth)) * 2
    for t in a ^ b:
        assert abs(ref_scores[t] - kth) <= band, f"swap of token {t} outside the tie band"
    return len(a ^ b) // 2


@pytest.mark.parametrize("nh,lens", [(32, [3000, 130, 64, 1]), (8, [5000, 4999]), (16, [2048, 2500]),
                                     (64, [1000, 777])])
def test_indexer_small(nh, lens):
    m = lib()
    wl = W.indexer_keys(DEV, seed=nh, batch=len(lens), n_heads=nh, topk=512, ctx_lens=lens)
    max_ctx = max(lens) + 7
    idx, sc = run_indexer(m, wl, max_ctx)
    ref = oracle_scores(wl, None, 1)
    for b in range(len(lens)):
        check_request(idx[b], sc[b], ref[b], wl.topk)
        assert np.all(np.isnan(sc[b, lens[b]:])), "entries past the context are left untouched"


def test_indexer_bad_block_is_minus_inf():
    m = lib()
    wl = W.indexer_keys(DEV, seed=3, batch=2, n_heads=32, topk=64, ctx_lens=[640, 640])
    bt = wl.block_table.clone()
    bt[0, 2] = wl.num_blocks + 5
    bt[1, 9] = -3
    wl.block_table = bt
    idx, sc = run_indexer(m, wl, 640)
    assert np.all(np.isneginf(sc[0, 128:192])) and np.all(np.isneginf(sc[1, 576:640]))
    assert np.all(np.isfinite(sc[0, :128])) and not np.isin(np.arange(128, 192), idx[0]).any()


def test_chained_indexer_topk_decode_full_size():
    """64 requests x 140,000 tokens: indexer + top-2048 on all requests vs the
    oracle, then the NVFP4 decode of 4 requests on the selected rows."""
    m = lib()
    wl = W.indexer_keys(DEV, seed=0, batch=64, ctx=140_000, n_heads=32, topk=2048)
    idx, sc = run_indexer(m, wl, 140_000)
    ref = oracle_scores(wl, None, O.host_threads())
    swaps = sum(check_request(idx[b], sc[b], ref[b], 2048) for b in range(64))
    print(f"near-tie swaps against the float64 top-k over 64 requests: {swaps}")
    # decode on the selected rows (16 MLA heads per request)
    dec = W._decode_workload("chained", ("chained", 0), 64, 16, 2048, [140_000] * 64, DEV, 0.0,
                             lambda b, c, g: torch.from_numpy(idx[b][idx[b] >= 0].astype(np.int64)).to(DEV))

    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)

    W.fill_pool(dec, O.FMT_NVFP4, qa)
    lse = torch.empty((64, 16), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode(dec.q_nope, dec.q_rope, dec.pools[0], dec.strides[0], dec.num_blocks,
                                 dec.block_table, dec.context_lens, dec.topk_idx, dec.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    # the oracle decodes the rows the GPU selected (whatever near-tie swaps
    # the top-k made), so every sampled request is checked
    for b in [0, 21, 42, 63]:
        got = idx[b][idx[b] >= 0].astype(np.int64)
        sel = torch.from_numpy(got).to(DEV)
        lat, rope = dec.request_rows(b, sel)
        valid = np.ones(got.size, bool)
        r, rl = oracle_rows_decode(u16(dec.q_nope[b]), u16(dec.q_rope[b]), u16(lat), u16(rope), valid, 0,
                                   dec.softmax_scale)
        assert_decode_close(out[b], lse[b], r, rl, f"request {b}")


def test_indexer_key_stride_not_a_multiple_of_128():
    """Key blocks 16 bytes apart from the packed layout cannot be TMA tiles;
    the indexer then loads keys directly.  Same contract as the tiled path."""
    m = lib()
    wl = W.indexer_keys(DEV, seed=5, batch=3, n_heads=32, topk=256, ctx_lens=[4000, 1000, 300])
    pad = wl.key_stride + 16
    pool = torch.zeros(wl.num_blocks * pad, dtype=torch.uint8, device=DEV)
    pool.view(wl.num_blocks, pad)[:, :wl.key_stride] = wl.key_pool.view(wl.num_blocks, wl.key_stride)
    ref = oracle_scores(wl, None, 1)
    wl.key_pool, wl.key_stride = pool, pad
    idx, sc = run_indexer(m, wl, 4000)
    for b in range(3):
        check_request(idx[b], sc[b], ref[b], wl.topk)


@pytest.mark.parametrize("nh", [32, 64])
def test_indexer_query_far_below_its_maximum(nh):
    """The tensor-core indexer represents each head's query as two e4m3 parts
    after scaling its largest magnitude into [128, 256): every element is
    exact to within 2^-10 of the scaled unit, i.e. max|q_h| / 128 * 2^-10
    before scaling.  A query with one large element per head and every other
    element 10^-6 .. 10^-2 of it puts most elements in that subnormal range;
    relu is 1-Lipschitz, so every score is within
    sum_h w_h * s_t * sum_d |k_t,d| * max|q_h| / 128 * 2^-10 of the float64
    score, plus the float32 tolerance.  The top-k is exact on the GPU's own
    scores."""
    m = lib()
    lens = [3000, 1000]
    wl = W.indexer_keys(DEV, seed=11 + nh, batch=2, n_heads=nh, topk=256, ctx_lens=lens)
    rng = np.random.default_rng(nh)
    q = rng.standard_normal((2, nh, 128)) * 10.0 ** rng.uniform(-6, -2, (2, nh, 128))
    q[:, :, 0] = rng.choice([-1.0, 1.0], (2, nh)) * 10.0 ** rng.uniform(0, 2, (2, nh))
    wl.q_idx = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16).to(DEV).contiguous()
    idx, sc = run_indexer(m, wl, max(lens))
    ref = oracle_scores(wl, None, 1)
    qb = wl.q_idx.float().cpu().numpy().astype(np.float64)
    w = wl.head_w.cpu().numpy().astype(np.float64)
    err_q = np.abs(qb).max(axis=2) / 128.0 * 2.0 ** -10  # [B, H]: largest representation error
    pool = wl.key_pool.view(-1, wl.key_stride)
    bt = wl.block_table.cpu().numpy()
    for b, c in enumerate(lens):
        nblk = (c + 63) // 64
        blocks = pool[torch.from_numpy(bt[b, :nblk].astype(np.int64)).to(DEV)]
        codes = blocks[:, :64 * 128].contiguous().view(torch.float8_e4m3fn).float().view(nblk * 64, 128)
        scale = blocks[:, 64 * 128:64 * 132].contiguous().view(torch.float32).reshape(nblk * 64)
        kabs = (codes.abs().sum(dim=1) * scale).cpu().numpy().astype(np.float64)[:c]  # sum_d |k_t,d| s_t
        bound = kabs * float(np.dot(w[b], err_q[b])) + 1e-5 * (1 + np.abs(ref[b][:c]))
        diff = np.abs(sc[b, :c].astype(np.float64) - ref[b][:c])
        assert np.all(diff <= bound), f"request {b}: worst excess {np.max(diff - bound):.3e}"
        assert np.array_equal(idx[b], lexsort_topk(sc[b, :c], wl.topk)), "top-k of the GPU's scores"


@pytest.mark.parametrize("padded", [False, True], ids=["tma", "padded"])
@pytest.mark.parametrize("nh", [8, 16, 32, 64])
@pytest.mark.parametrize("factor", [2.0 ** 20, 2.0 ** -24], ids=["2^20", "2^-24"])
def test_indexer_query_outside_fp16_range(nh, factor, padded):
    """q times f with the head weights divided by f gives the same scores
    (relu is positively homogeneous), but puts the query beyond FP16's
    largest value (2^20) or below its normal range (2^-24).  Every score
    kernel -- tensor-memory (32, 64 heads), pipelined (8, 16) and the one for
    key strides TMA cannot tile (padded) -- scales each head by a power of two
    and must still match the float64 oracle within the score tolerance."""
    m = lib()
    lens = [2500, 700]
    wl = W.indexer_keys(DEV, seed=23 + nh, batch=2, n_heads=nh, topk=256, ctx_lens=lens)
    wl.q_idx = (wl.q_idx.double() * factor).to(torch.bfloat16).contiguous()
    wl.head_w = (wl.head_w.double() / factor).float().contiguous()
    if padded:
        pad = wl.key_stride + 16
        pool = torch.zeros(wl.num_blocks * pad, dtype=torch.uint8, device=DEV)
        pool.view(wl.num_blocks, pad)[:, :wl.key_stride] = wl.key_pool.view(wl.num_blocks, wl.key_stride)
        ref = oracle_scores(wl, None, 1)
        wl.key_pool, wl.key_stride = pool, pad
    else:
        ref = oracle_scores(wl, None, 1)
    idx, sc = run_indexer(m, wl, max(lens))
    for b, c in enumerate(lens):
        diff = np.abs(sc[b, :c].astype(np.float64) - ref[b][:c])
        assert np.all(diff <= SCORE_TOL * (1 + np.abs(ref[b][:c]))), f"request {b}: max diff {diff.max():.3e}"
        assert np.array_equal(idx[b], lexsort_topk(sc[b, :c], wl.topk)), "top-k of the GPU's scores"
