"""Indexer-key quantize-on-write and the staged NVFP4 -> FP8 path on the GPU
against the oracle.

Keys: "GLM-5.3 PCP/DCP long-context on H200", section 3 (a key is 128 e4m3
bytes and a float scale) -- byte-exact.  Staged path: "Prime Inference:
serving GLM-5.3 to agents is a KV-cache problem", section "A kernel that
reads four bits directly", figure "staged vs native decode" -- the staged
rows and list are byte-exact; the staged decode is held to the decode
tolerance against the oracle's FP8 decode of the oracle's staged rows.

Inputs of every byte-exact check are host-generated (seeded numpy) and given
to both sides; nothing the GPU computes enters the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from gpu_helpers import assert_decode_close, lib, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BS = 64


def bf16_keys(n, seed, spread=10.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 128)) * np.exp(rng.uniform(-spread, spread, (n, 1)))).astype(np.float32)
    keys = (x.view(np.uint32) >> 16).astype(np.uint16)
    special = [np.zeros(128, np.uint16),                              # zero key
               np.full(128, 0x8000, np.uint16),                       # all -0.0
               rng.integers(0, 0x0080, 128).astype(np.uint16),        # bf16 subnormals
               np.full(128, 0x3F80, np.uint16)]                       # all equal (1.0)
    for i, v in enumerate(special[:n]):
        keys[i] = v
    return keys


@pytest.mark.parametrize("n,nb,pad", [(1, 1, 0), (5, 2, 16), (3000, 60, 0), (20_000, 400, 32), (300_000, 5000, 0)])
def test_index_key_append_bit_exact(n, nb, pad):
    m = lib()
    rng = np.random.default_rng(n)
    keys = bf16_keys(n, seed=n)
    stride = BS * 132 + pad
    slots = rng.permutation(nb * BS)[:n].astype(np.int64)
    slots[1::17] = -1
    if n > 4:
        slots[4] = nb * BS + 5  # past the pool: skipped
    ref = np.full(nb * stride, 0xCD, dtype=np.uint8)
    O.index_key_quantize_append(keys, slots, ref, nb, BS, stride)
    pool = torch.full((nb * stride,), 0xCD, dtype=torch.uint8, device=DEV)
    m.mla_index_key_quantize_append(torch.from_numpy(keys.view(np.int16)).to(DEV), torch.from_numpy(slots).to(DEV),
                                    pool, nb, BS, stride)
    torch.cuda.synchronize()
    got = pool.cpu().numpy()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


def random_nvfp4_pool(nb, seed, stride):
    """Arbitrary 352-byte rows (random codes, finite scales including zero,
    subnormal and 448, finite rope) -- the staged copy must handle any row."""
    rng = np.random.default_rng(seed)
    pool = rng.integers(0, 256, nb * stride, dtype=np.uint8)
    rows = pool.reshape(nb, stride)[:, :BS * 352].reshape(nb * BS, 352)
    for part in (slice(256, 288), slice(288, 352)):
        v = rows[:, part]
        v[(v & 0x7F) == 0x7F] &= 0xFE
    rows[::7, 256:288] = 0x7E
    pool.reshape(nb, stride)[:, :BS * 352] = rows.reshape(nb, BS * 352)
    return pool


@pytest.mark.parametrize("B,k,ctx", [(1, 1, [10]), (3, 70, [300, 320, 10]), (4, 2048, [150_000, 2048, 64, 5000])])
def test_stage_rows_bit_exact(B, k, ctx):
    m = lib()
    rng = np.random.default_rng(B * 100 + k)
    max_blocks = max((c + BS - 1) // BS for c in ctx) + 1
    nb = sum((c + BS - 1) // BS for c in ctx) + 3
    stride = BS * 352 + 16
    pool = random_nvfp4_pool(nb, seed=k, stride=stride)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    perm = rng.permutation(nb)
    o = 0
    for b, c in enumerate(ctx):
        n = (c + BS - 1) // BS
        bt[b, :n] = perm[o:o + n]
        o += n
    if B > 1:
        bt[1, 0] = nb + 9                      # block id outside the pool
    tk = np.stack([rng.integers(-1, c + 40, k) for c in ctx]).astype(np.int32)
    tk[0, :: 5] = -1
    cl = np.array(ctx, dtype=np.int32)
    nblk = (k + BS - 1) // BS
    ref = np.full(B * nblk * BS * 576, 0xAB, dtype=np.uint8)
    ref_tk = O.stage_rows_fp8(pool, stride, nb, bt, cl, tk, BS, ref)
    d = lambda a: torch.from_numpy(a).to(DEV)
    staged = torch.full((m.mla_staged_pool_bytes(B, k),), 0xAB, dtype=torch.uint8, device=DEV)
    got_pool, got_tk = m.mla_stage_rows_fp8(d(pool), stride, nb, d(bt), d(cl), d(tk), staged_pool=staged)
    torch.cuda.synchronize()
    assert np.array_equal(got_tk.cpu().numpy(), ref_tk)
    got = got_pool.cpu().numpy()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


def oracle_staged_decode(qn, qr, pool, stride, nb, bt, cl, tk, scale):
    """Oracle staged path: stage the NVFP4 rows, then the FP8 decode of the copy."""
    B, k = tk.shape
    nblk = (k + BS - 1) // BS
    staged = np.zeros(B * nblk * BS * 576, dtype=np.uint8)
    st = O.stage_rows_fp8(pool, stride, nb, bt, cl, tk, BS, staged)
    sbt = np.arange(B * nblk, dtype=np.int32).reshape(B, nblk)
    scl = np.full(B, nblk * BS, dtype=np.int32)
    return O.sparse_decode(qn, qr, staged, BS * 576, sbt, scl, st, BS, scale, O.FMT_FP8)


@pytest.mark.parametrize("B,H,k,ctx", [(2, 16, 300, [5000, 777]), (3, 32, 2048, [9000, 2049, 2500]),
                                       (1, 64, 97, [97])])
def test_staged_decode_against_oracle(B, H, k, ctx):
    """NVFP4 pool from the oracle's quantizer on seeded bf16 rows; the GPU runs
    the staged decode, the oracle stages and decodes the same pool."""
    m = lib()
    rng = np.random.default_rng(B * 7 + H + k)
    max_blocks = max((c + BS - 1) // BS for c in ctx)
    nb = sum((c + BS - 1) // BS for c in ctx) + 2
    stride = BS * 352
    bt = np.zeros((B, max_blocks), dtype=np.int32)
    perm = rng.permutation(nb)
    pool = np.zeros(nb * stride, dtype=np.uint8)
    o = 0
    for b, c in enumerate(ctx):
        n = (c + BS - 1) // BS
        bt[b, :n] = perm[o:o + n]
        o += n
        lat = (rng.standard_normal((c, 512)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        rope = (rng.standard_normal((c, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        slots = (bt[b, np.arange(c) // BS].astype(np.int64) * BS + np.arange(c) % BS)
        O.kv_quantize_append(lat, rope, slots, pool, nb, BS, stride, O.FMT_NVFP4)
    tk = np.full((B, k), -1, dtype=np.int32)
    for b, c in enumerate(ctx):
        sel = np.sort(rng.choice(c, min(k, c), replace=False))
        tk[b, :sel.size] = sel
    tk[0, 3] = -1
    qn = (rng.standard_normal((B, H, 512)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qr = (rng.standard_normal((B, H, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    cl = np.array(ctx, dtype=np.int32)
    scale = 1 / np.sqrt(192.0)
    ref, ref_lse = oracle_staged_decode(qn, qr, pool, stride, nb, bt, cl, tk, scale)

    d = lambda a: torch.from_numpy(a).to(DEV)
    q_n = d(qn.view(np.int16)).view(torch.bfloat16)
    q_r = d(qr.view(np.int16)).view(torch.bfloat16)
    lse = torch.empty((B, H), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode_staged(q_n, q_r, d(pool), stride, nb, d(bt), d(cl), d(tk), scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        assert_decode_close(out[b], lse[b], ref[b], ref_lse[b], f"staged request {b}")
    # the native decode reads the same pool; the two differ by the e4m3
    # rounding of the staged copy only
    nat, _ = m.mla_sparse_decode(q_n, q_r, d(pool), stride, nb, d(bt), d(cl), d(tk), scale)
    torch.cuda.synchronize()
    nat = nat.float().cpu().numpy()
    rel = np.linalg.norm(nat - out) / np.linalg.norm(nat)
    assert 0 < rel < 0.1


def test_staged_decode_tp4_full_size_sampled():
    """The TP4 rank as bench.py times it (32 requests x 16 heads, 140,000-token
    contexts, top-2048) through the staged path; 3 requests against the
    oracle's staged copies of the same seeded rows."""
    import workloads as W
    m = lib()
    wl = W.tp4_rank_decode(DEV)
    W.fill_pool(wl, O.FMT_NVFP4, lambda lat, rope, slots, pool, nb, stride, fmt:
                m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt))
    lse = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode_staged(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks,
                                        wl.block_table, wl.context_lens, wl.topk_idx, wl.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    k = wl.topk
    for b in [0, 13, 31]:
        lat, rope = wl.request_rows(b, wl.topk_idx[b])
        lat, rope = u16(lat), u16(rope)
        staged = np.zeros((k + 63) // 64 * 64 * 576, dtype=np.uint8).reshape(-1, 576)
        for j in range(k):
            staged[j] = O.stage_row_fp8(O.quantize_row(lat[j], rope[j], O.FMT_NVFP4))
        nblk = (k + 63) // 64
        ref, ref_lse = O.sparse_decode(u16(wl.q_nope[b:b + 1]), u16(wl.q_rope[b:b + 1]), staged.reshape(-1), 64 * 576,
                                       np.arange(nblk, dtype=np.int32)[None], np.array([nblk * 64], np.int32),
                                       np.arange(k, dtype=np.int32)[None], 64, wl.softmax_scale, O.FMT_FP8)
        assert_decode_close(out[b], lse[b], ref[0], ref_lse[0], f"staged request {b}")
