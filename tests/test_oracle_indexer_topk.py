"""Pins for the oracle's indexer score and exact top-k (CPU only).

Source: "GLM-5.3 PCP/DCP long-context on H200", section 1 (the indexer rates
all preceding tokens and attention reads only the 2,048 best) and section 3
(an indexer key is 128 e4m3 bytes and a float scale); "Prime
Inference: serving GLM-5.3 to agents is a KV-cache problem", section "Decode:
TP4, and the copies it keeps" (index_topk 2048).  The score formula
sum_h w_h * relu(s_t * (q_h . k_t)) is the workload definition this library
implements (the pages do not print it).

Pins: special cases that reduce to a library matrix product (one head, unit
weight, positive inputs), relu / sign cases, linearity in the head weights,
block-table indirection, and numpy lexsort brute force for the selection.
"""
import numpy as np
import pytest
import torch

import oracle as O

BS = 64
D = 128


def bf16(x) -> np.ndarray:
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def f8(x) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def f8val(codes) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


class KeyCache:
    """Indexer key pool: per block, bs x 128 e4m3 bytes then bs float32 scales."""

    def __init__(self, keys_codes, scales, seed=0, extra=2):
        ctx = keys_codes.shape[0]
        rng = np.random.default_rng(seed)
        nblk = (ctx + BS - 1) // BS
        self.num_blocks = nblk + extra
        self.stride = BS * (D + 4) + 16 * 3  # padded, still a multiple of 16
        perm = rng.permutation(self.num_blocks)[:nblk].astype(np.int32)
        self.block_table = perm[None, :]
        self.pool = np.zeros(self.num_blocks * self.stride, dtype=np.uint8)
        for t in range(ctx):
            base = int(perm[t // BS]) * self.stride
            self.pool[base + (t % BS) * D: base + (t % BS + 1) * D] = keys_codes[t]
            s = np.array([scales[t]], dtype=np.float32).view(np.uint8)
            self.pool[base + BS * D + (t % BS) * 4: base + BS * D + (t % BS) * 4 + 4] = s
        self.ctx = ctx

    def scores(self, q_bits, w):
        q = q_bits[None]
        w = np.asarray(w, dtype=np.float32)[None]
        return O.indexer_scores(q, w, self.pool, self.stride, self.block_table,
                                np.array([self.ctx], np.int32), BS)[0]


def test_one_head_unit_weight_is_a_matrix_vector_product():
    rng = np.random.default_rng(0)
    ctx = 150
    k = np.abs(rng.standard_normal((ctx, D)))
    codes = f8(k)
    s = rng.uniform(0.5, 2.0, ctx).astype(np.float32)
    q = bf16(np.abs(rng.standard_normal(D)))
    cache = KeyCache(codes, s)
    got = cache.scores(q[None, :], [1.0])
    ref = s.astype(np.float64) * (f8val(codes) @ O.bf16_to_f64(q))  # numpy matmul
    assert np.allclose(got, ref, rtol=1e-13)


def test_relu_drops_negative_head_contributions():
    rng = np.random.default_rng(1)
    ctx = 70
    codes = f8(rng.standard_normal((ctx, D)))
    s = np.ones(ctx, np.float32)
    q = bf16(rng.standard_normal(D))
    cache = KeyCache(codes, s)
    pos = cache.scores(q[None, :], [1.0])
    neg = cache.scores(bf16(-O.bf16_to_f64(q))[None, :], [1.0])
    dots = f8val(codes) @ O.bf16_to_f64(q)
    assert np.array_equal(pos == 0, dots <= 0)
    assert np.array_equal(neg == 0, dots >= 0)
    assert np.allclose(pos - neg, dots, rtol=1e-12, atol=1e-12)  # relu(x) - relu(-x) = x
    assert np.all(pos >= 0) and np.all(neg >= 0)


def test_linear_in_head_weights_and_scale_multiplies():
    rng = np.random.default_rng(2)
    ctx, nh = 130, 8
    codes = f8(rng.standard_normal((ctx, D)))
    s = rng.uniform(0.1, 3, ctx).astype(np.float32)
    q = bf16(rng.standard_normal((nh, D)))
    cache = KeyCache(codes, s)
    w1 = rng.uniform(0, 1, nh).astype(np.float32)
    w2 = rng.uniform(0, 1, nh).astype(np.float32)
    total = cache.scores(q, w1 + w2)
    per = cache.scores(q, w1) + cache.scores(q, w2)
    assert np.allclose(total, per, rtol=1e-6)  # w1 + w2 is rounded to float32
    # each head alone equals w_h * relu(s_t * dot)
    dots = f8val(codes) @ O.bf16_to_f64(q).T  # [ctx, nh]
    for h in range(nh):
        onehot = np.zeros(nh, np.float32)
        onehot[h] = 1.0
        one = cache.scores(q, onehot)
        assert np.allclose(one, np.maximum(0, s.astype(np.float64) * dots[:, h]), rtol=1e-13)


def test_block_placement_does_not_change_scores():
    rng = np.random.default_rng(3)
    ctx = 200
    codes = f8(rng.standard_normal((ctx, D)))
    s = rng.uniform(0.1, 3, ctx).astype(np.float32)
    q = bf16(rng.standard_normal((4, D)))
    w = rng.uniform(0, 1, 4)
    a = KeyCache(codes, s, seed=1).scores(q, w)
    b = KeyCache(codes, s, seed=5).scores(q, w)
    assert np.array_equal(a, b)


def brute_topk(scores: np.ndarray, k: int) -> np.ndarray:
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores.astype(np.float64)))  # score desc, index asc
    sel = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:sel.size] = sel
    return out


@pytest.mark.parametrize("n,k,levels", [(1000, 64, 5), (5000, 2048, 50), (300, 2048, 3), (4096, 1, 1000),
                                        (2049, 2048, 2), (140, 100, 0)])
def test_topk_matches_lexsort_brute_force(n, k, levels):
    rng = np.random.default_rng(n + k)
    if levels:
        sc = rng.integers(0, levels, n).astype(np.float64) * 0.5 - 3.0  # many exact ties
    else:
        sc = rng.standard_normal(n)
    assert np.array_equal(O.topk(sc, k), brute_topk(sc, k))
    f = sc.astype(np.float32)
    assert np.array_equal(O.topk(f, k), brute_topk(f, k))


def test_topk_special_cases():
    # all equal -> the first k indices
    assert np.array_equal(O.topk(np.zeros(5000), 2048), np.arange(2048))
    # context shorter than k -> 0..ctx-1 then -1
    out = O.topk(np.random.default_rng(0).standard_normal(37), 2048)
    assert np.array_equal(out[:37], np.arange(37)) and np.all(out[37:] == -1)
    # empty context -> all -1
    assert np.all(O.topk(np.zeros(0), 16) == -1)
    # -0.0 ties with +0.0 and loses to the lower index
    sc = np.array([1.0, -0.0, 0.0, -0.0, 0.0, -1.0], dtype=np.float32)
    assert np.array_equal(O.topk(sc, 3), [0, 1, 2])
    assert np.array_equal(O.topk(sc[::-1].copy(), 3), [1, 2, 5])
    # output is ascending even when the winners are not in score order
    sc = np.array([0.1, 5.0, 0.2, 4.0, 3.0])
    assert np.array_equal(O.topk(sc, 3), [1, 3, 4])
