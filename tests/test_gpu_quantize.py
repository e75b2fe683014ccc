"""Quantize-on-write on the GPU is byte-exact against the oracle.

Row format: "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem", section "Four bits per latent value" (576 -> 352 bytes: e2m1
latent with one e4m3 scale per 16 values, e4m3 rope; FP8 row 576 bytes)."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import lib, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def gpu_append(m, lat, rope, slots, num_blocks, fmt, stride=None, fill=0):
    rb = O.row_bytes(fmt)
    stride = stride or 64 * rb
    pool = torch.full((num_blocks * stride,), fill, dtype=torch.uint8, device=DEV)
    m.mla_kv_quantize_append(lat, rope, slots, pool, num_blocks, 64, stride, fmt)
    torch.cuda.synchronize()
    return pool.cpu().numpy(), stride


def oracle_pool(lat, rope, slots, num_blocks, fmt, stride, fill=0):
    pool = np.full(num_blocks * stride, fill, dtype=np.uint8)
    O.kv_quantize_append(u16(lat), u16(rope), slots.cpu().numpy(), pool, num_blocks, 64, stride, fmt)
    return pool


def rows_from_bits(bits: np.ndarray, width: int) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16).reshape(-1, width).copy()).view(
        torch.bfloat16).to(DEV)


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def test_every_bf16_value_in_every_position(fmt):
    """All 65,536 bf16 patterns except NaN/Inf as latent values, in groups
    whose maxima sweep the scale range, and as rope values."""
    m = lib()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(bits)
    bits = bits[np.isfinite(vals)]
    rng = np.random.default_rng(0)
    # latent: shuffle so each 16-group mixes magnitudes (and so many scales occur)
    lat_bits = rng.permutation(bits)
    n_rows = -(-lat_bits.size // 512)
    lat_bits = np.concatenate([lat_bits, np.zeros(n_rows * 512 - lat_bits.size, np.uint16)])
    # plus rows whose groups are sorted by magnitude: groups of similar values
    order = np.argsort(np.abs(O.bf16_to_f64(bits)), kind="stable")
    sorted_bits = bits[order]
    sorted_bits = np.concatenate([sorted_bits, np.zeros(n_rows * 512 - sorted_bits.size, np.uint16)])
    lat = np.concatenate([lat_bits, sorted_bits]).reshape(-1, 512)
    n = lat.shape[0]
    rope_bits = np.concatenate([bits, np.zeros(n * 64 - bits.size, np.uint16)]) if bits.size <= n * 64 else None
    if rope_bits is None:
        reps = -(-bits.size // 64)
        lat = np.concatenate([lat, np.zeros((reps - n, 512), np.uint16)])
        n = reps
        rope_bits = np.concatenate([bits, np.zeros(n * 64 - bits.size, np.uint16)])
    rope = rope_bits.reshape(n, 64)
    slots = torch.arange(n, dtype=torch.int64, device=DEV)
    nb = -(-n // 64)
    lt, rt = rows_from_bits(lat.ravel(), 512), rows_from_bits(rope.ravel(), 64)
    got, stride = gpu_append(m, lt, rt, slots, nb, fmt)
    want = oracle_pool(lt, rt, slots, nb, fmt, stride)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def test_golden_groups_on_gpu(fmt):
    """The hand-worked NVFP4 groups of tests/golden/ reproduce on the GPU."""
    from test_oracle_formats import _parse_vectors, bf16_bits
    m = lib()
    recs = _parse_vectors()
    lat = np.zeros((len(recs), 512), np.uint16)
    for i, rec in enumerate(recs):
        lat[i, 16 * (5 + i):16 * (6 + i)] = bf16_bits([float(t) for t in rec["input"].split()])
    rope = np.zeros((len(recs), 64), np.uint16)
    lt, rt = rows_from_bits(lat.ravel(), 512), rows_from_bits(rope.ravel(), 64)
    slots = torch.arange(len(recs), dtype=torch.int64, device=DEV)
    got, stride = gpu_append(m, lt, rt, slots, 1, fmt)
    rb = O.row_bytes(fmt)
    for i, rec in enumerate(recs):
        row = got[i * rb:(i + 1) * rb]
        if fmt == O.FMT_NVFP4:
            g = 5 + i
            assert np.array_equal(row[8 * g:8 * g + 8], [int(t, 16) for t in rec["bytes"].split()]), rec["name"]
            assert row[256 + g] == int(rec["scale"], 16), rec["name"]
        else:
            assert np.array_equal(row, O.quantize_row(lat[i], rope[i], fmt))


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def test_slot_mapping_skips_and_padded_stride(fmt):
    m = lib()
    rng = np.random.default_rng(1)
    n, nb = 300, 7
    lat = W.bf16_normal((n, 512), torch.Generator(device=DEV).manual_seed(3), DEV)
    rope = W.bf16_normal((n, 64), torch.Generator(device=DEV).manual_seed(4), DEV)
    slots_np = rng.permutation(nb * 64)[:n].astype(np.int64)
    slots_np[::17] = -1            # skipped
    slots_np[5] = nb * 64 + 3      # past the pool: skipped
    slots_np[9] = -(1 << 40)
    slots = torch.from_numpy(slots_np).to(DEV)
    stride = 64 * O.row_bytes(fmt) + 48
    got, _ = gpu_append(m, lat, rope, slots, nb, fmt, stride=stride, fill=0xA5)
    want = oracle_pool(lat, rope, slots, nb, fmt, stride, fill=0xA5)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def test_append_turn_full_size(fmt):
    """64 sessions x 6,000 new tokens (384,000 rows) written through scattered
    block tables: every written row matches the oracle byte for byte, and
    sampled untouched rows stay zero."""
    m = lib()
    wl = W.append_turn(DEV)
    rb = O.row_bytes(fmt)
    stride = 64 * rb
    pool = torch.zeros(wl.num_blocks * stride, dtype=torch.uint8, device=DEV)
    m.mla_kv_quantize_append(wl.latent, wl.rope, wl.slot_mapping, pool, wl.num_blocks, 64, stride, fmt)
    torch.cuda.synchronize()
    slots = wl.slot_mapping
    offs = (slots // 64) * stride + (slots % 64) * rb
    gather = offs[:, None] + torch.arange(rb, device=DEV)[None, :]
    got_rows = pool[gather.view(-1)].view(-1, rb).cpu().numpy()
    lat, rope = u16(wl.latent), u16(wl.rope)
    n = lat.shape[0]
    want_pool = np.zeros(n * rb, dtype=np.uint8)
    O.kv_quantize_append(lat, rope, np.arange(n, dtype=np.int64), want_pool, -(-n // 64), 64, 64 * rb, fmt)
    assert np.array_equal(got_rows, want_pool.reshape(n, rb))
    # untouched rows (prefix positions) are still zero
    untouched = (wl.block_table[:, :100].to(torch.int64) * stride).view(-1)[:500]
    probe = pool[(untouched[:, None] + torch.arange(rb, device=DEV)[None, :]).view(-1)]
    assert int(probe.count_nonzero()) == 0


def test_nvfp4_every_value_under_every_scale():
    """Exhaustive over the code decision x / S: for every positive finite e4m3
    scale S, groups whose maximum is exactly 6 S (so the group's scale is S)
    carry every finite bf16 value x with |x| <= 6 S, both signs."""
    m = lib()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(bits)
    fin = np.isfinite(vals)
    bits, vals = bits[fin], vals[fin]
    groups = []
    for sc in range(1, 0x7F):
        S = O.e4m3_decode(sc)
        amax = 6.0 * S
        amax_bits = (np.array([amax], np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert O.bf16_to_f64(amax_bits)[0] == amax
        xs = bits[np.abs(vals) <= amax]
        pad = (-xs.size) % 15
        xs = np.concatenate([xs, np.zeros(pad, np.uint16)]).reshape(-1, 15)
        groups.append(np.concatenate([np.repeat(amax_bits[None, :], xs.shape[0], 0), xs], axis=1))
    g = np.concatenate(groups)                       # [G, 16]
    pad = (-g.shape[0]) % 32
    g = np.concatenate([g, np.zeros((pad, 16), np.uint16)])
    lat_np = g.reshape(-1, 512)
    n = lat_np.shape[0]
    rope_np = np.zeros((n, 64), np.uint16)
    lat = rows_from_bits(lat_np, 512)
    rope = rows_from_bits(rope_np, 64)
    nb = -(-n // 64)
    slots = torch.arange(n, dtype=torch.int64, device=DEV)
    got, stride = gpu_append(m, lat, rope, slots, nb, O.FMT_NVFP4)
    want = oracle_pool(lat, rope, slots, nb, O.FMT_NVFP4, stride)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ (rows {np.unique(bad // 352)[:5]})"
