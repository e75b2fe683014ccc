"""Pins for the oracle's absorbed-form sparse MLA decode (CPU only).

The decode the oracle computes is the one described in "Prime Inference:
serving GLM-5.3 to agents is a KV-cache problem", section "A kernel that
reads four bits directly" (gather the selected rows, unpack, score, softmax,
blend) with the latent as the value vector ("Prefill topology": all heads
up-project from the same 512-value latent; "GLM-5.3 PCP/DCP long-context on
H200", section 6: sparse_mla_force_mqa keeps every KV row serving all heads).

Pins: closed forms (k = 1, identical rows, q = 0, duplicates), invariances
(permuted top-k list, permuted physical blocks, masked entries), and a
brute-force un-absorbed dense MLA on tiny inputs that reproduces the
absorption identity (q W_UK) . c = q . (W_UK c).  Rows are decoded in the
tests with torch's float8_e4m3fn and the OCP E2M1 value set, not with the
oracle's own decoder.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
BS = 64


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def decode_row_indep(row: np.ndarray, fmt: int):
    """Independent decoder of one stored row -> (c[512], r[64])."""
    if fmt == O.FMT_NVFP4:
        codes = np.empty(512, dtype=np.uint8)
        codes[0::2] = row[:256] & 0xF
        codes[1::2] = row[:256] >> 4
        scales = np.repeat(e4m3_values(row[256:288]), 16)
        return E2M1[codes] * scales, e4m3_values(row[288:352])
    return e4m3_values(row[:512]), e4m3_values(row[512:576])


def bf16(x) -> np.ndarray:
    """float -> bf16 bits by truncation (inputs are arbitrary test data)."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


class Cache:
    """A tiny paged cache built with the oracle's quantizer."""

    def __init__(self, ctx, fmt, seed=0, nblocks_extra=3, rows=None):
        rng = np.random.default_rng(seed)
        self.fmt = fmt
        self.rb = O.row_bytes(fmt)
        self.stride = BS * self.rb + 32
        nblk = (ctx + BS - 1) // BS
        self.num_blocks = nblk + nblocks_extra
        perm = rng.permutation(self.num_blocks)[:nblk].astype(np.int32)
        self.block_table = perm[None, :]
        if rows is None:
            lat = bf16(rng.standard_normal((ctx, 512)))
            rope = bf16(rng.standard_normal((ctx, 64)))
        else:
            lat, rope = rows
        self.pool = np.zeros(self.num_blocks * self.stride, dtype=np.uint8)
        slots = np.array([perm[t // BS] * BS + t % BS for t in range(ctx)], dtype=np.int64)
        O.kv_quantize_append(lat, rope, slots, self.pool, self.num_blocks, BS, self.stride, fmt)
        self.ctx = ctx

    def row(self, t):
        off = int(self.block_table[0, t // BS]) * self.stride + (t % BS) * self.rb
        return self.pool[off:off + self.rb]

    def decode(self, qn, qr, idx, scale, ctx=None):
        idx = np.asarray(idx, dtype=np.int32)[None, :]
        cl = np.array([self.ctx if ctx is None else ctx], dtype=np.int32)
        out, lse = O.sparse_decode(qn[None], qr[None], self.pool, self.stride, self.block_table, cl, idx,
                                   BS, scale, self.fmt)
        return out[0], lse[0]


@pytest.fixture(params=[O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def fmt(request):
    return request.param


def rand_q(H, seed=1):
    rng = np.random.default_rng(seed)
    return bf16(rng.standard_normal((H, 512))), bf16(rng.standard_normal((H, 64)))


def test_k1_returns_the_row_and_its_score(fmt):
    cache = Cache(200, fmt)
    qn, qr = rand_q(4)
    scale = 1 / math.sqrt(192)
    for t in [0, 63, 64, 199]:
        out, lse = cache.decode(qn, qr, [t], scale)
        c, r = decode_row_indep(cache.row(t), fmt)
        for h in range(4):
            assert np.array_equal(out[h], c)
            z = scale * (O.bf16_to_f64(qn[h]) @ c + O.bf16_to_f64(qr[h]) @ r)
            assert lse[h] == pytest.approx(z, rel=1e-12, abs=1e-12)


def test_identical_rows_give_that_row(fmt):
    rng = np.random.default_rng(5)
    one_lat = bf16(rng.standard_normal(512))
    one_rope = bf16(rng.standard_normal(64))
    ctx = 90
    cache = Cache(ctx, fmt, rows=(np.tile(one_lat, (ctx, 1)), np.tile(one_rope, (ctx, 1))))
    qn, qr = rand_q(3)
    idx = np.arange(0, ctx, 3)
    out, lse = cache.decode(qn, qr, idx, 0.1)
    c, r = decode_row_indep(cache.row(0), fmt)
    assert np.allclose(out, c[None, :], rtol=1e-13, atol=1e-13)
    z = 0.1 * (O.bf16_to_f64(qn) @ c + O.bf16_to_f64(qr) @ r)
    assert np.allclose(lse, z + math.log(len(idx)), rtol=1e-12)


def test_zero_query_gives_the_mean_row(fmt):
    cache = Cache(150, fmt, seed=2)
    qn = np.zeros((2, 512), np.uint16)
    qr = np.zeros((2, 64), np.uint16)
    idx = [3, 77, 140, 10, 64]
    out, lse = cache.decode(qn, qr, idx, 1.0)
    rows = np.stack([decode_row_indep(cache.row(t), fmt)[0] for t in idx])
    assert np.allclose(out, rows.mean(axis=0)[None, :], rtol=1e-13, atol=1e-13)
    assert np.allclose(lse, math.log(len(idx)), rtol=1e-13)


def test_duplicate_index_counts_twice(fmt):
    cache = Cache(80, fmt, seed=4)
    qn, qr = rand_q(2, seed=9)
    out1, lse1 = cache.decode(qn, qr, [17], 0.05)
    out2, lse2 = cache.decode(qn, qr, [17, 17], 0.05)
    assert np.array_equal(out1, out2)
    assert np.allclose(lse2, lse1 + math.log(2), rtol=1e-13)


def test_permuted_topk_list_and_masked_entries(fmt):
    cache = Cache(300, fmt, seed=6)
    qn, qr = rand_q(4, seed=3)
    rng = np.random.default_rng(8)
    idx = rng.choice(300, 40, replace=False)
    out, lse = cache.decode(qn, qr, idx, 0.07)
    out_p, lse_p = cache.decode(qn, qr, rng.permutation(idx), 0.07)
    assert np.allclose(out, out_p, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, lse_p, rtol=1e-13)
    # -1 entries and entries at or past the context length are masked away
    noisy = np.concatenate([idx, [-1, -1, 300, 301, -5]])
    out_m, lse_m = cache.decode(qn, qr, rng.permutation(noisy), 0.07)
    assert np.allclose(out, out_m, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, lse_m, rtol=1e-13)
    # a shorter context masks the tail of the list
    short = idx[idx < 120]
    out_s, lse_s = cache.decode(qn, qr, short, 0.07)
    out_c, lse_c = cache.decode(qn, qr, idx, 0.07, ctx=120)
    assert np.allclose(out_s, out_c, rtol=1e-12, atol=1e-14)
    assert np.allclose(lse_s, lse_c, rtol=1e-13)


def test_all_masked_gives_zeros_and_minus_inf(fmt):
    cache = Cache(64, fmt)
    qn, qr = rand_q(2)
    out, lse = cache.decode(qn, qr, [-1, -1, -1, 64, 1000], 0.1)
    assert not out.any()
    assert np.all(np.isneginf(lse))


def test_physical_block_placement_does_not_matter(fmt):
    rng = np.random.default_rng(11)
    ctx = 200
    rows = (bf16(rng.standard_normal((ctx, 512))), bf16(rng.standard_normal((ctx, 64))))
    a = Cache(ctx, fmt, seed=1, rows=rows)
    b = Cache(ctx, fmt, seed=2, rows=rows)
    assert not np.array_equal(a.block_table, b.block_table)
    qn, qr = rand_q(4, seed=12)
    idx = rng.choice(ctx, 50, replace=False)
    oa, la = a.decode(qn, qr, idx, 0.08)
    ob, lb = b.decode(qn, qr, idx, 0.08)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("ctx,H", [(37, 2), (64, 4), (100, 3)])
def test_full_context_equals_brute_force_dense_mla(fmt, ctx, H):
    """top-k = the whole context reproduces un-absorbed dense MLA.

    Per head h: key_t = [W_UK[h] c_t ; r_t], query = [q_n[h] ; q_r[h]],
    value_t = W_UV[h] c_t.  The absorbed query W_UK[h]^T q_n[h] is made of
    small integers so that it is exact in bf16."""
    rng = np.random.default_rng(ctx * 10 + H)
    cache = Cache(ctx, fmt, seed=ctx)
    dn, dv = 128, 128
    w_uk = rng.integers(-1, 2, size=(H, dn, 512)).astype(np.float64)
    w_uv = rng.standard_normal((H, dv, 512))
    q_raw = rng.integers(-2, 3, size=(H, dn)).astype(np.float64)
    q_abs = np.einsum("hd,hdc->hc", q_raw, w_uk)  # integers, |.| <= 256
    assert np.abs(q_abs).max() <= 256
    qn = bf16(q_abs)
    assert np.array_equal(O.bf16_to_f64(qn), q_abs)
    qr = bf16(rng.standard_normal((H, 64)))
    scale = 1.0 / (64 * math.sqrt(192))
    out, lse = cache.decode(qn, qr, np.arange(ctx), scale)

    rows = [decode_row_indep(cache.row(t), fmt) for t in range(ctx)]
    C = np.stack([r[0] for r in rows])  # [ctx, 512]
    R = np.stack([r[1] for r in rows])  # [ctx, 64]
    qrf = O.bf16_to_f64(qr)
    for h in range(H):
        keys = np.concatenate([C @ w_uk[h].T, R], axis=1)  # [ctx, 192]
        query = np.concatenate([q_raw[h], qrf[h]])
        s = scale * keys @ query
        m = s.max()
        p = np.exp(s - m)
        lse_ref = m + math.log(p.sum())
        p /= p.sum()
        vals = C @ w_uv[h].T  # [ctx, 128]
        o_dense = p @ vals
        assert lse[h] == pytest.approx(lse_ref, rel=1e-12, abs=1e-12)
        assert np.allclose(w_uv[h] @ out[h], o_dense, rtol=1e-10, atol=1e-10)
        assert abs(p.sum() - 1.0) < 1e-12


def test_softmax_scale_and_query_scaling_agree(fmt):
    cache = Cache(128, fmt, seed=13)
    rng = np.random.default_rng(14)
    qn_f = np.round(rng.standard_normal((2, 512)) * 4) / 4
    qr_f = np.round(rng.standard_normal((2, 64)) * 4) / 4
    idx = rng.choice(128, 30, replace=False)
    o1, l1 = cache.decode(bf16(qn_f), bf16(qr_f), idx, 0.02)
    o2, l2 = cache.decode(bf16(2 * qn_f), bf16(2 * qr_f), idx, 0.01)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l1, l2, rtol=1e-12)


def test_block_major_pool_slices_match_packed_pools(fmt):
    """Block-major pool ("Prime Inference", section "Moving the cache: 32K
    copies for one request", KV layout figure): layer l's rows live at
    l * 64 * row_bytes inside each block, block stride layers * 64 *
    row_bytes.  Appending into one layer's slice leaves the others untouched,
    and decoding a slice equals decoding a packed single-layer pool."""
    rng = np.random.default_rng(21)
    layers, ctx, nb = 3, 150, 4
    rb = O.row_bytes(fmt)
    sl = BS * rb
    stride = layers * sl
    bt = rng.permutation(nb)[:3].astype(np.int32)[None, :]
    slots = np.array([bt[0, t // BS] * BS + t % BS for t in range(ctx)], dtype=np.int64)
    pool = np.full(nb * stride, 0xEE, dtype=np.uint8)
    qn, qr = rand_q(4, seed=22)
    idx = rng.choice(ctx, 40, replace=False).astype(np.int32)[None, :]
    cl = np.array([ctx], dtype=np.int32)
    for layer in range(layers):
        lat = bf16(rng.standard_normal((ctx, 512)))
        rope = bf16(rng.standard_normal((ctx, 64)))
        view = pool[layer * sl:]
        O.kv_quantize_append(lat, rope, slots, view, nb, BS, stride, fmt)
        blocks = pool.reshape(nb, layers, sl)
        assert np.all(blocks[:, layer + 1:] == 0xEE), "later layers untouched"
        packed = np.full(nb * sl, 0xEE, dtype=np.uint8)
        O.kv_quantize_append(lat, rope, slots, packed, nb, BS, sl, fmt)
        assert np.array_equal(blocks[:, layer].reshape(-1), packed)
        a = O.sparse_decode(qn[None], qr[None], view, stride, bt, cl, idx, BS, 0.05, fmt)
        b = O.sparse_decode(qn[None], qr[None], packed, sl, bt, cl, idx, BS, 0.05, fmt)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_draft_tokens_single_token_and_causal_bounds(fmt):
    """Q query tokens per request, each with its own list (R-causal: token i
    sees positions < ctx - (Q - 1 - i)).  Q = 1 is the single-token decode;
    the last token sees the whole context; the first token with the same
    list equals the single-token decode at ctx - (Q - 1)."""
    cache = Cache(260, fmt, seed=31)
    rng = np.random.default_rng(32)
    Q, H, k = 3, 4, 50
    qn = np.stack([rand_q(H, seed=40 + i)[0] for i in range(Q)])
    qr = np.stack([rand_q(H, seed=40 + i)[1] for i in range(Q)])
    lst = np.concatenate([rng.choice(255, k - 5, replace=False), [255, 256, 257, 258, 259]]).astype(np.int32)
    tk = np.tile(lst, (Q, 1))[None]
    cl = np.array([cache.ctx], dtype=np.int32)
    out, lse = O.sparse_decode_mtp(qn[None], qr[None], cache.pool, cache.stride, cache.block_table, cl, tk, BS,
                                   0.06, fmt)
    for i in range(Q):
        o1, l1 = cache.decode(qn[i], qr[i], lst, 0.06, ctx=cache.ctx - (Q - 1 - i))
        assert np.array_equal(out[0, i], o1) and np.array_equal(lse[0, i], l1)
    one, one_lse = O.sparse_decode_mtp(qn[None, :1], qr[None, :1], cache.pool, cache.stride, cache.block_table, cl,
                                       tk[:, :1], BS, 0.06, fmt)
    o1, l1 = cache.decode(qn[0], qr[0], lst, 0.06)
    assert np.array_equal(one[0, 0], o1) and np.array_equal(one_lse[0, 0], l1)


def test_draft_tokens_brute_force_softmax(fmt):
    """Brute force: per token, an explicit softmax over the visible entries of
    its own list, rows decoded with the OCP tables (not the oracle)."""
    cache = Cache(130, fmt, seed=33)
    rng = np.random.default_rng(34)
    Q, H, k = 4, 2, 20
    qn = np.stack([rand_q(H, seed=50 + i)[0] for i in range(Q)])
    qr = np.stack([rand_q(H, seed=50 + i)[1] for i in range(Q)])
    tk = np.stack([np.concatenate([rng.choice(126, k - 4, replace=False), [126, 127, 128, 129]])
                   for _ in range(Q)]).astype(np.int32)
    tk[1, 0] = -1
    out, lse = O.sparse_decode_mtp(qn[None], qr[None], cache.pool, cache.stride, cache.block_table,
                                   np.array([130], np.int32), tk[None], BS, 0.08, fmt)
    for i in range(Q):
        vis = [t for t in tk[i] if 0 <= t < 130 - (Q - 1 - i)]
        assert len(vis) == k - (Q - 1 - i) - (1 if i == 1 else 0)
        rows = [decode_row_indep(cache.row(t), fmt) for t in vis]
        C_ = np.stack([r[0] for r in rows])
        R_ = np.stack([r[1] for r in rows])
        for h in range(H):
            z = 0.08 * (C_ @ O.bf16_to_f64(qn[i, h]) + R_ @ O.bf16_to_f64(qr[i, h]))
            p = np.exp(z - z.max())
            assert lse[0, i, h] == pytest.approx(z.max() + math.log(p.sum()), rel=1e-12, abs=1e-12)
            assert np.allclose(out[0, i, h], (p / p.sum()) @ C_, rtol=1e-11, atol=1e-12)
