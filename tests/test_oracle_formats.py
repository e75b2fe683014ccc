"""Pins for the oracle's number formats and row layout (CPU only).

Each check compares the oracle with something other than itself: the OCP
specification's printed points, a library decoder (torch float8_e4m3fn), a
brute-force nearest-even search (a different algorithm from the oracle's
arithmetic rounding), hand-worked vectors under tests/golden/, and the byte
counts printed on "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem" (section "Four bits per latent value", row table).
"""
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_SET = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX FP4 E2M1 magnitudes


def bf16_bits(values) -> np.ndarray:
    """float values that are exact in bf16 -> their bf16 bit patterns."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


# ------------------------------------------------------------------ decode tables
def test_e2m1_decode_is_the_ocp_value_set():
    got = [O.e2m1_decode(c) for c in range(16)]
    assert got[:8] == E2M1_SET
    neg = got[8:]
    assert [-x for x in E2M1_SET] == neg
    assert np.signbit(neg[0])  # code 0x8 decodes to -0.0


def test_e4m3_decode_matches_torch_float8_e4m3fn_on_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([O.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_spot_values_from_the_spec():
    assert O.e4m3_decode(0x38) == 1.0
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x2A) == 0.3125


def test_e4m3_golden_points():
    for line in open(os.path.join(GOLDEN, "e4m3_points.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        v, code = line.split()
        assert O.e4m3_encode(float(v)) == int(code, 16), line


# ------------------------------------------------------------------ brute-force encoders
def _nearest_even(mag: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value; on an exact tie the even index.

    ``grid`` is sorted ascending and its index is the code (so 'even index'
    is 'even mantissa LSB').  Values past the end pick the last entry, which
    is satfinite."""
    d = np.abs(mag[:, None] - grid[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.argmax(cand, axis=1)
    two = cand.sum(axis=1) == 2
    lo = idx[two]
    idx[two] = np.where(lo % 2 == 0, lo, lo + 1)
    return idx


def brute_e4m3(x: np.ndarray) -> np.ndarray:
    grid = np.array([O.e4m3_decode(c) for c in range(0x7F)])  # 0x00..0x7E, ascending
    # satfinite: magnitudes past 448 clamp to 448 (clamping first also keeps
    # the distances representable for huge inputs)
    code = _nearest_even(np.minimum(np.abs(x), 1024.0), grid).astype(np.uint8)
    return code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)


def brute_e2m1(v: np.ndarray) -> np.ndarray:
    code = _nearest_even(np.minimum(np.abs(v), 16.0), np.array(E2M1_SET)).astype(np.uint8)
    return code | np.where(np.signbit(v), 0x8, 0).astype(np.uint8)


def all_finite_bf16() -> np.ndarray:
    x = O.bf16_to_f64(np.arange(65536, dtype=np.uint16))
    return x[np.isfinite(x)]


def test_e4m3_encoder_equals_brute_force_on_every_bf16():
    x = all_finite_bf16()
    got = O.e4m3_encode_array(x)
    for part in np.array_split(np.arange(x.size), 8):
        assert np.array_equal(got[part], brute_e4m3(x[part]))


def test_e4m3_encoder_equals_torch_in_range():
    x = all_finite_bf16()
    x = x[np.abs(x) < 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode_array(x)
    # torch keeps the sign of values that round to zero too
    assert np.array_equal(got, ref)


def test_e2m1_encoder_equals_brute_force_on_a_dense_sweep():
    v = np.concatenate([np.linspace(-8, 8, 200001), np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, -0.0])])
    assert np.array_equal(O.e2m1_encode_array(v), brute_e2m1(v))


def test_e2m1_ties_go_to_even_codes():
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, code in ties.items():
        assert O.e2m1_encode(v) == code
        assert O.e2m1_encode(-v) == code | 0x8
    assert O.e2m1_encode(6.0) == 7 and O.e2m1_encode(100.0) == 7 and O.e2m1_encode(-1e9) == 0xF


# ------------------------------------------------------------------ fp32 == fp64 for the quantizer
def test_scale_division_fp32_and_fp64_give_the_same_e4m3_code():
    """S = e4m3(amax / 6): an IEEE float32 division and a float64 one round to
    the same code for every non-negative bf16 amax (exhaustive)."""
    amax = all_finite_bf16()
    amax = np.unique(np.abs(amax))
    q64 = amax / 6.0
    q32 = (amax.astype(np.float32) / np.float32(6.0)).astype(np.float64)
    assert np.array_equal(brute_e4m3(q64), brute_e4m3(q32))


def test_code_division_fp32_and_fp64_give_the_same_e2m1_code():
    """code = e2m1(x / S): float32 and float64 division agree for every bf16 x
    and every positive finite e4m3 scale S (exhaustive: 65,024 x 126)."""
    x = all_finite_bf16()
    scales = np.array([O.e4m3_decode(c) for c in range(1, 0x7F)])
    for s in scales:
        v64 = x / s
        with np.errstate(over="ignore"):  # float32 overflow -> inf, which saturates like the double
            v32 = (x.astype(np.float32) / np.float32(s)).astype(np.float64)
        a = O.e2m1_encode_array(v64)
        b = O.e2m1_encode_array(v32)
        assert np.array_equal(a, b), s


def test_dequant_products_are_exact_in_fp16_and_bf16():
    """Every e2m1 value times every finite e4m3 scale is exactly representable
    in float16 and in bfloat16 (so on-chip dequantization is exact)."""
    vals = np.array([O.e2m1_decode(c) for c in range(16)])
    sc = np.array([O.e4m3_decode(c) for c in range(256)])
    sc = sc[np.isfinite(sc)]
    prod = (vals[:, None] * sc[None, :]).ravel()
    assert np.array_equal(prod.astype(np.float16).astype(np.float64), prod)
    b = torch.from_numpy(prod).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(b, prod)


# ------------------------------------------------------------------ row layout
def _parse_vectors():
    recs, cur = [], {}
    for line in open(os.path.join(GOLDEN, "nvfp4_group_vectors.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        cur[key.strip()] = val.strip()
        if key.strip() == "dequant":
            recs.append(cur)
            cur = {}
    return recs


@pytest.mark.parametrize("group", [0, 13, 31])
def test_hand_worked_nvfp4_groups(group):
    recs = _parse_vectors()
    assert len(recs) == 5
    for rec in recs:
        vals = [float(t) for t in rec["input"].split()]
        latent = np.zeros(512, dtype=np.uint16)
        latent[16 * group:16 * group + 16] = bf16_bits(vals)
        rope = np.zeros(64, dtype=np.uint16)
        row = O.quantize_row(latent, rope, O.FMT_NVFP4)
        assert row.size == 352
        want_bytes = np.array([int(t, 16) for t in rec["bytes"].split()], dtype=np.uint8)
        assert np.array_equal(row[8 * group:8 * group + 8], want_bytes), rec["name"]
        assert row[256 + group] == int(rec["scale"], 16), rec["name"]
        others = np.ones(352, dtype=bool)
        others[8 * group:8 * group + 8] = False
        others[256 + group] = False
        assert not row[others].any(), "bytes outside the group must stay zero"
        codes = [int(t, 16) for t in rec["codes"].split()]
        nib = [(row[8 * group + i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
        assert nib == codes, rec["name"]
        c, r = O.dequant_row(row, O.FMT_NVFP4)
        want = np.array([float(t) for t in rec["dequant"].split()])
        assert np.array_equal(c[16 * group:16 * group + 16], want), rec["name"]
        assert np.array_equal(np.signbit(c[16 * group:16 * group + 16]), np.signbit(want)), rec["name"]


def test_row_sizes_match_the_pages_table():
    # NVFP4: 512 x 4 bit + 512 / 16 scales x 1 B + 64 x 1 B = 256 + 32 + 64 = 352
    assert O.row_bytes(O.FMT_NVFP4) == 512 * 4 // 8 + 512 // 16 + 64 == 352
    # FP8: 512 x 1 B + 64 x 1 B = 576, no per-row scale
    assert O.row_bytes(O.FMT_FP8) == 512 + 64 == 576
    # "56.25% of FP8" is the latent alone: (256 + 32) / 512
    assert (256 + 32) / 512 == 0.5625


def test_rope_and_fp8_positions():
    rng = np.random.default_rng(1)
    lat = bf16_bits(np.round(rng.standard_normal(512) * 8) / 8)
    rope = bf16_bits(np.round(rng.standard_normal(64) * 8) / 8)
    r4 = O.quantize_row(lat, rope, O.FMT_NVFP4)
    r8 = O.quantize_row(lat, rope, O.FMT_FP8)
    rope_f = O.bf16_to_f64(rope)
    lat_f = O.bf16_to_f64(lat)
    assert np.array_equal(r4[288:352], brute_e4m3(rope_f))
    assert np.array_equal(r8[512:576], brute_e4m3(rope_f))
    assert np.array_equal(r8[:512], brute_e4m3(lat_f))


def test_random_rows_dequant_to_the_nearest_grid_point():
    """Property: each dequantized latent value is S_g times the nearest-even
    e2m1 point of x / S_g, with S_g the nearest-even e4m3 of amax_g / 6."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        x = rng.standard_normal(512) * np.exp(rng.uniform(np.log(0.1), np.log(10)))
        x[rng.random(512) < 0.01] *= 20
        if trial == 3:
            x[32:48] = 0.0
        lat = (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
        xf = O.bf16_to_f64(lat)
        row = O.quantize_row(lat, np.zeros(64, np.uint16), O.FMT_NVFP4)
        c, _ = O.dequant_row(row, O.FMT_NVFP4)
        for g in range(32):
            xs = xf[16 * g:16 * g + 16]
            s_code = int(brute_e4m3(np.array([np.abs(xs).max() / 6.0]))[0])
            assert row[256 + g] == s_code
            s = O.e4m3_decode(s_code)
            if s_code == 0:
                assert not c[16 * g:16 * g + 16].any()
                continue
            codes = brute_e2m1(xs / s)
            want = np.array([O.e2m1_decode(k) for k in codes]) * s
            assert np.array_equal(c[16 * g:16 * g + 16], want)


def test_quantize_append_places_rows_by_slot_and_skips_negative_slots():
    rng = np.random.default_rng(3)
    n, bs, nb = 10, 64, 4
    stride = bs * 352 + 64  # padded block stride
    lat = (rng.standard_normal((n, 512)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rope = (rng.standard_normal((n, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    slots = np.array([0, 63, 64, 200, -1, 255, 130, -7, 5, 128], dtype=np.int64)
    pool = np.full(nb * stride, 0xCD, dtype=np.uint8)
    assert O.kv_quantize_append(lat, rope, slots, pool, nb, bs, stride, O.FMT_NVFP4) == 2
    touched = np.zeros(pool.size, dtype=bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        off = (s // bs) * stride + (s % bs) * 352
        assert np.array_equal(pool[off:off + 352], O.quantize_row(lat[i], rope[i], O.FMT_NVFP4))
        touched[off:off + 352] = True
    assert np.all(pool[~touched] == 0xCD)
    before = pool.copy()
    assert O.kv_quantize_append(lat[:2], rope[:2], np.array([nb * bs, -3], np.int64), pool, nb, bs, stride,
                                O.FMT_NVFP4) == 2
    assert np.array_equal(pool, before)  # slots past the pool are skipped, nothing is written
