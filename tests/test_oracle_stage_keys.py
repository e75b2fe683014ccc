"""Pins for the oracle's staged FP8 copy and indexer-key quantizer (CPU only).

Staged path: "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem", section "A kernel that reads four bits directly", figure "staged vs
native decode" (a gather kernel reads the 352-byte NVFP4 rows and writes a
576-byte FP8 copy that an FP8 attention kernel then reads).  Indexer keys:
"GLM-5.3 PCP/DCP long-context on H200", section 3 (a key is 128 e4m3 bytes
and a float scale).

Every check compares the oracle with something other than its own
arithmetic: the OCP tables through torch's float8_e4m3fn decoder, a
brute-force nearest-even search over all e4m3 values, rows whose values are
exactly representable, and power-of-two scaling invariance."""
import numpy as np
import pytest
import torch

import oracle as O

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def torch_e4m3(codes) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


GRID = torch_e4m3(np.arange(0x7F))  # codes 0x00..0x7E, ascending magnitudes


def brute_e4m3(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 by exhaustive search (ties to the even code), satfinite,
    sign bit from the input."""
    mag = np.minimum(np.abs(x), 1024.0)
    d = np.abs(mag[:, None] - GRID[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.argmax(cand, axis=1)
    two = cand.sum(axis=1) == 2
    idx[two] = np.where(idx[two] % 2 == 0, idx[two], idx[two] + 1)
    return idx.astype(np.uint8) | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)


def decode_nvfp4(row: np.ndarray):
    codes = np.empty(512, dtype=np.uint8)
    codes[0::2] = row[:256] & 0xF
    codes[1::2] = row[:256] >> 4
    return E2M1[codes] * np.repeat(torch_e4m3(row[256:288]), 16)


def random_rows(n, seed):
    """Arbitrary NVFP4 rows: random codes, random finite scales (including
    0x00, subnormals and 448), random finite rope bytes."""
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, 256, (n, 352), dtype=np.uint8)
    for part in (slice(256, 288), slice(288, 352)):
        v = rows[:, part]
        v[(v & 0x7F) == 0x7F] &= 0xFE  # no NaN codes
    rows[0, 256:288] = 0x7E  # 448: products up to 2,688 saturate
    rows[1, 256:288] = np.arange(32, dtype=np.uint8)  # zero and subnormal scales
    return rows


# ------------------------------------------------------------------ staged FP8 copy
def test_stage_row_is_the_nearest_e4m3_of_each_value():
    for i, row in enumerate(random_rows(64, seed=1)):
        got = O.stage_row_fp8(row)
        vals = decode_nvfp4(row)
        assert np.array_equal(got[:512], brute_e4m3(vals)), f"row {i}"
        assert np.array_equal(got[512:], row[288:352]), "rope bytes are copied"


def test_stage_row_is_exact_when_values_are_representable():
    """With scales that are powers of two in [2^-6, 2^6], every e2m1 x S is an
    e4m3 value, so the FP8 copy decodes to exactly the NVFP4 values."""
    rng = np.random.default_rng(2)
    row = rng.integers(0, 256, 352, dtype=np.uint8)
    exps = rng.integers(-6, 7, 32)
    row[256:288] = ((exps + 7) << 3).astype(np.uint8)  # e4m3 1.0 * 2^e
    row[288:352] = rng.integers(0, 0x7F, 64, dtype=np.uint8)
    got = O.stage_row_fp8(row)
    assert np.array_equal(torch_e4m3(got[:512]), decode_nvfp4(row))


def test_stage_row_saturates_and_keeps_signed_zero():
    row = np.zeros(352, dtype=np.uint8)
    row[256:288] = 0x7E            # S = 448
    # elements 2i (low nibble) and 2i+1 (high nibble) of bytes 0..3
    row[:4] = [0x77, 0xFF, 0x08, 0x80]
    got = O.stage_row_fp8(row)
    assert got[0] == 0x7E and got[1] == 0x7E          # 6 * 448 = 2,688 saturates to 448
    assert got[2] == 0xFE and got[3] == 0xFE          # -2,688 saturates to -448
    assert got[4] == 0x80 and got[5] == 0x00          # code 0x8 is -0, code 0x0 is +0
    assert got[6] == 0x00 and got[7] == 0x80


def test_stage_rows_layout_and_masking():
    rng = np.random.default_rng(3)
    bs, rb = 64, 352
    nb = 12
    pool = rng.integers(0, 0x7F, nb * bs * rb, dtype=np.uint8)
    B, k = 3, 70
    bt = np.stack([rng.permutation(nb)[:5] for _ in range(B)]).astype(np.int32)
    bt[1, 2] = nb + 4  # block id outside the pool
    ctx = np.array([300, 320, 10], dtype=np.int32)
    tk = rng.integers(-1, 330, (B, k)).astype(np.int32)
    nblk = (k + bs - 1) // bs
    staged = np.full(B * nblk * bs * 576, 0xAB, dtype=np.uint8)
    st = O.stage_rows_fp8(pool, bs * rb, nb, bt, ctx, tk, bs, staged)
    staged = staged.reshape(B, nblk * bs, 576)
    for b in range(B):
        for j in range(k):
            t = int(tk[b, j])
            ok = 0 <= t < ctx[b] and t // bs < bt.shape[1] and 0 <= bt[b, t // bs] < nb
            assert st[b, j] == (j if ok else -1)
            if ok:
                off = int(bt[b, t // bs]) * bs * rb + (t % bs) * rb
                assert np.array_equal(staged[b, j], O.stage_row_fp8(pool[off:off + rb]))
            else:
                assert np.all(staged[b, j] == 0xAB), "masked entries write no row"
        assert np.all(staged[b, k:] == 0xAB)


# ------------------------------------------------------------------ indexer keys
def bf16_random(shape, seed, spread=8.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(shape) * np.exp(rng.uniform(-spread, spread, shape[:-1] + (1,)))).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def test_index_key_codes_are_the_nearest_e4m3_of_the_float_quotient():
    keys = bf16_random((200, 128), seed=4)
    for n in range(keys.shape[0]):
        codes, s = O.quantize_index_key(keys[n])
        x = bits_to_f32(keys[n])
        amax = np.float32(np.abs(x).max())
        assert s == amax / np.float32(448.0)
        q = (x / np.float32(s)).astype(np.float32)  # single-precision quotient
        assert np.array_equal(codes, brute_e4m3(q.astype(np.float64))), f"key {n}"


def test_index_key_amax_maps_to_448_and_dequant_is_close():
    keys = bf16_random((50, 128), seed=5)
    for n in range(keys.shape[0]):
        codes, s = O.quantize_index_key(keys[n])
        x = bits_to_f32(keys[n]).astype(np.float64)
        assert (codes & 0x7F).max() == 0x7E
        back = torch_e4m3(codes) * float(s)
        # relative step of e4m3 normals is 2^-3; subnormals are 2^-9 * s apart
        assert np.all(np.abs(back - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * float(s)) * (1 + 1e-6))


def test_index_key_power_of_two_scaling_invariance():
    keys = bf16_random((30, 128), seed=6, spread=2.0)
    for n in range(keys.shape[0]):
        c0, s0 = O.quantize_index_key(keys[n])
        scaled = (bits_to_f32(keys[n]) * np.float32(2.0 ** 5)).view(np.uint32) >> 16
        c1, s1 = O.quantize_index_key(scaled.astype(np.uint16))
        assert np.array_equal(c0, c1) and s1 == s0 * np.float32(32.0)


def test_index_key_zero_key():
    codes, s = O.quantize_index_key(np.zeros(128, dtype=np.uint16))
    assert s == 0.0 and not codes.any()
    neg0 = np.full(128, 0x8000, dtype=np.uint16)  # all -0.0
    codes, s = O.quantize_index_key(neg0)
    assert s == 0.0 and not codes.any()


def test_index_key_append_places_codes_and_scales_by_slot():
    rng = np.random.default_rng(7)
    bs, nb = 64, 5
    stride = bs * 132 + 16
    pool = np.full(nb * stride, 0xCD, dtype=np.uint8)
    keys = bf16_random((40, 128), seed=8)
    slots = rng.permutation(nb * bs)[:40].astype(np.int64)
    slots[3] = -1
    slots[7] = nb * bs + 3
    skipped = O.index_key_quantize_append(keys, slots, pool, nb, bs, stride)
    assert skipped == 2
    touched = np.zeros(pool.size, bool)
    for n, slot in enumerate(slots):
        if slot < 0 or slot >= nb * bs:
            continue
        blk, o = divmod(int(slot), bs)
        codes, s = O.quantize_index_key(keys[n])
        base = blk * stride
        assert np.array_equal(pool[base + o * 128: base + o * 128 + 128], codes)
        assert pool[base + bs * 128 + 4 * o: base + bs * 128 + 4 * o + 4].view(np.float32)[0] == s
        touched[base + o * 128: base + o * 128 + 128] = True
        touched[base + bs * 128 + 4 * o: base + bs * 128 + 4 * o + 4] = True
    assert np.all(pool[~touched] == 0xCD)
