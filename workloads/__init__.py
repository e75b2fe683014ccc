"""Seeded synthetic workloads shaped like the pages' decode traffic.

This module only draws random numbers and lays out tables (block tables, slot
mappings, top-k lists).  It holds none of the method's arithmetic: no
quantization, no scoring, no attention.  Both the CUDA path's tests/bench and
the oracle consume what it returns.

Shapes follow "Prime Inference: serving GLM-5.3 to agents is a KV-cache
problem" (section "The workload": each agent turn appends roughly 6,000 new tokens
after a roughly 140,000-token prefix; section "Decode: TP4": 64 heads split four ways -> 16 per rank,
top-k 2,048) and "GLM-5.3 PCP/DCP long-context on H200" (1M-token contexts,
all 64 heads per DP rank, indexer keys of 128 e4m3 bytes and a float scale).  The
AgentX traces the pages benchmark on are not available; these seeded draws
stand in for them.

Every tensor is drawn from a torch.Generator seeded by ``sub_seed(config,
name, index)``, so any request's rows can be regenerated on their own.
"""
from __future__ import annotations

import hashlib
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

BLOCK = 64
LATENT = 512
ROPE = 64
IDX_DIM = 128
NVFP4_ROW = 352
FP8_ROW = 576
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)  # 128 nope + 64 rope query dims


def sub_seed(*parts) -> int:
    h = hashlib.sha256(repr(parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def generator(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(*parts))
    return g


def bf16_normal(shape, gen: torch.Generator, device, outlier_frac: float = 0.0, outlier_scale: float = 20.0,
                row_scale: Optional[torch.Tensor] = None) -> torch.Tensor:
    """N(0,1) values as bf16; a fraction scaled up as outliers; optional per-row scale."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_frac > 0:
        m = torch.rand(shape, generator=gen, device=device) < outlier_frac
        x = torch.where(m, x * outlier_scale, x)
    if row_scale is not None:
        x = x * row_scale.reshape(-1, *([1] * (len(shape) - 1)))
    return x.to(torch.bfloat16)


def scattered_block_tables(n_req: int, blocks_per_req: List[int], gen: torch.Generator, device,
                           extra_blocks: int = 0):
    """Blocks of all requests scattered over one shared pool.

    Returns (block_table int32 [n_req, max_blocks] padded with -1, num_blocks)."""
    total = sum(blocks_per_req) + extra_blocks
    perm = torch.randperm(total, generator=gen, device=device).to(torch.int32)
    mx = max(blocks_per_req) if blocks_per_req else 1
    bt = torch.full((n_req, mx), -1, dtype=torch.int32, device=device)
    off = 0
    for r, nb in enumerate(blocks_per_req):
        bt[r, :nb] = perm[off:off + nb]
        off += nb
    return bt, total


def slots_for_positions(block_table_row: torch.Tensor, positions: torch.Tensor) -> torch.Tensor:
    """Slot index (block * 64 + offset) of logical positions through one request's table."""
    pos = positions.to(torch.int64)
    return block_table_row.to(torch.int64)[pos // BLOCK] * BLOCK + pos % BLOCK


def distinct_uniform(n: int, lo: int, hi: int, gen: torch.Generator, device) -> torch.Tensor:
    """n distinct integers drawn uniformly from [lo, hi)."""
    span = hi - lo
    if n >= span:
        return torch.arange(lo, hi, device=device, dtype=torch.int64)
    if span <= 4 * n or span <= 1 << 22:
        return torch.randperm(span, generator=gen, device=device)[:n] + lo
    out = torch.empty(0, dtype=torch.int64, device=device)
    while out.numel() < n:  # rejection of duplicates on a large range
        draw = torch.randint(lo, hi, (2 * n,), generator=gen, device=device)
        out = torch.unique(torch.cat([out, draw]))
    return out[torch.randperm(out.numel(), generator=gen, device=device)[:n]]


@dataclass
class DecodeWorkload:
    """One decode layer: queries, paged cache geometry, top-k lists."""
    name: str
    batch: int
    heads: int
    topk: int
    q_nope: torch.Tensor                 # bf16 [B,H,512]
    q_rope: torch.Tensor                 # bf16 [B,H,64]
    block_table: torch.Tensor            # int32 [B, max_blocks]
    num_blocks: int
    context_lens: torch.Tensor           # int32 [B]
    topk_idx: torch.Tensor               # int32 [B, k]
    softmax_scale: float = SOFTMAX_SCALE
    seed_parts: tuple = ()
    outlier_frac: float = 0.0
    pools: Dict[int, torch.Tensor] = field(default_factory=dict)  # fmt -> uint8 pool
    strides: Dict[int, int] = field(default_factory=dict)

    def request_rows(self, b: int, positions: Optional[torch.Tensor] = None):
        """Regenerate request b's bf16 latent/rope rows (all positions, or a subset)."""
        ctx = int(self.context_lens[b])
        gen = generator(self.q_nope.device, *self.seed_parts, "rows", b)
        lat = bf16_normal((ctx, LATENT), gen, self.q_nope.device, self.outlier_frac)
        rope = bf16_normal((ctx, ROPE), gen, self.q_nope.device, self.outlier_frac)
        if positions is not None:
            p = positions.to(torch.int64).to(lat.device)
            return lat[p], rope[p]
        return lat, rope


def _decode_workload(name, seed_parts, batch, heads, topk, ctx_lens: List[int], device, outlier_frac, topk_draw):
    gq = generator(device, *seed_parts, "q")
    q_nope = bf16_normal((batch, heads, LATENT), gq, device)
    q_rope = bf16_normal((batch, heads, ROPE), gq, device)
    gb = generator(device, *seed_parts, "block_table")
    bt, nb = scattered_block_tables(batch, [(c + BLOCK - 1) // BLOCK for c in ctx_lens], gb, device)
    idx = torch.full((batch, topk), -1, dtype=torch.int32, device=device)
    for b in range(batch):
        sel = topk_draw(b, ctx_lens[b], generator(device, *seed_parts, "topk", b))
        sel = torch.sort(sel.to(torch.int64)).values.to(torch.int32)
        idx[b, :sel.numel()] = sel
    cl = torch.tensor(ctx_lens, dtype=torch.int32, device=device)
    return DecodeWorkload(name, batch, heads, topk, q_nope, q_rope, bt, nb, cl, idx, seed_parts=seed_parts,
                          outlier_frac=outlier_frac)


def tiny_decode(device, seed: int = 0) -> DecodeWorkload:
    """1 request x 16 heads, 4,096 cached tokens (64 shuffled blocks), 256
    distinct random top-k indices, scale 1/sqrt(192)."""
    return _decode_workload("tiny: 1 request x 16 heads, 4,096 tokens, top-256", ("tiny", seed), 1, 16, 256, [4096],
                            device, 0.0,
                            lambda b, ctx, g: distinct_uniform(256, 0, ctx, g, device))


def tp4_rank_decode(device, seed: int = 0, batch: int = 32, ctx: int = 140_000, heads: int = 16,
                    topk: int = 2048, recent: int = 6000) -> DecodeWorkload:
    """A TP4 decode rank: 32 requests x 16 heads, 140,000-token contexts,
    top-2048 = 70% uniform over the prefix + 30% from the last 6,000 tokens
    (1,434 + 614), 1% of cache values x20 outliers."""
    n_recent = round(0.3 * topk)
    n_old = topk - n_recent

    def draw(b, c, g):
        old = distinct_uniform(n_old, 0, c - recent, g, device)
        new = distinct_uniform(n_recent, c - recent, c, g, device)
        return torch.cat([old, new])

    return _decode_workload(f"TP4 rank: {batch} requests x {heads} heads, {ctx:,}-token contexts, top-{topk}",
                            ("tp4", seed, batch, ctx, heads, topk), batch, heads, topk, [ctx] * batch, device, 0.01,
                            draw)


@dataclass
class DraftQueries:
    """q_len query tokens per request of a decode workload: queries and one
    top-k list per token."""
    q_len: int
    q_nope: torch.Tensor     # bf16 [B,Q,H,512]
    q_rope: torch.Tensor     # bf16 [B,Q,H,64]
    topk_idx: torch.Tensor   # int32 [B,Q,k]


def draft_queries(wl: DecodeWorkload, q_len: int = 4, keep: float = 0.9, recent: int = 6000,
                  seed: int = 0) -> DraftQueries:
    """Speculative draft tokens for the requests of `wl` (its context lengths
    count the q_len new tokens).  Token i's list keeps a random `keep`
    fraction of the request's list in `wl` and fills the rest with distinct
    positions from the last `recent` tokens (lists of neighbouring tokens
    overlap, as an indexer's would); ascending."""
    dev = wl.q_nope.device
    B, H, k = wl.batch, wl.heads, wl.topk
    gq = generator(dev, *wl.seed_parts, "draft", seed, "q")
    qn = bf16_normal((B, q_len, H, LATENT), gq, dev)
    qr = bf16_normal((B, q_len, H, ROPE), gq, dev)
    idx = torch.full((B, q_len, k), -1, dtype=torch.int32, device=dev)
    for b in range(B):
        base = wl.topk_idx[b]
        base = base[base >= 0].to(torch.int64)
        n = base.numel()
        c = int(wl.context_lens[b])
        for i in range(q_len):
            g = generator(dev, *wl.seed_parts, "draft", seed, "topk", b, i)
            n_keep = int(round(keep * n))
            kept = base[torch.randperm(n, generator=g, device=dev)[:n_keep]]
            lo = max(0, c - recent)
            cand = distinct_uniform(min(c - lo, 3 * (n - n_keep) + 64), lo, c, g, dev).to(torch.int64)
            cand = cand[~torch.isin(cand, kept)][:n - n_keep]
            sel = torch.sort(torch.cat([kept, cand])).values.to(torch.int32)
            idx[b, i, :sel.numel()] = sel
    return DraftQueries(q_len, qn, qr, idx)


def dep_rank_context_lens(seed: int = 0, batch: int = 128, lo: int = 8192, hi: int = 1 << 20,
                          cap: int = 24_000_000) -> List[int]:
    """Context lengths log-uniform in [lo, hi]; if they sum past `cap` they are
    scaled down by cap / sum (floored, at least lo)."""
    g = torch.Generator()
    g.manual_seed(sub_seed("dep", seed, "ctx"))
    u = torch.rand(batch, generator=g, dtype=torch.float64)
    ctx = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
    total = float(ctx.sum())
    if total > cap:
        ctx = torch.clamp(torch.floor(ctx * (cap / total)), min=lo)
    return [int(x) for x in ctx]


def dep_rank_decode(device, seed: int = 0, batch: int = 128, heads: int = 64, topk: int = 2048,
                    cap: int = 24_000_000) -> DecodeWorkload:
    """All heads per rank (DEP-style): 128 requests x 64 heads, contexts
    log-uniform in [8,192, 1,048,576] capped at `cap` tokens in total (24M),
    top-2048 uniform without replacement over each context."""
    ctx = dep_rank_context_lens(seed, batch, cap=cap)
    seed_parts = ("dep", seed, batch, heads, topk) if cap == 24_000_000 else ("dep", seed, batch, heads, topk, cap)
    return _decode_workload(f"DEP rank: {batch} requests x {heads} heads, contexts 8K-1M (sum {sum(ctx):,}), top-{topk}",
                            seed_parts, batch, heads, topk, ctx, device, 0.0,
                            lambda b, c, g: distinct_uniform(min(topk, c), 0, c, g, device))


def fill_pool(wl: DecodeWorkload, fmt: int, quantize_append, pad_stride: int = 0, requests=None) -> torch.Tensor:
    """Allocate a pool for `fmt` and write every request's rows through
    `quantize_append(latent, rope, slot_mapping, pool, num_blocks, stride, fmt)`."""
    rb = NVFP4_ROW if fmt == 0 else FP8_ROW
    stride = BLOCK * rb + pad_stride
    pool = torch.zeros(wl.num_blocks * stride, dtype=torch.uint8, device=wl.q_nope.device)
    for b in (range(wl.batch) if requests is None else requests):
        lat, rope = wl.request_rows(b)
        ctx = int(wl.context_lens[b])
        slots = slots_for_positions(wl.block_table[b], torch.arange(ctx, device=lat.device))
        quantize_append(lat, rope, slots, pool, wl.num_blocks, stride, fmt)
    wl.pools[fmt] = pool
    wl.strides[fmt] = stride
    return pool


@dataclass
class AppendWorkload:
    """Quantize-on-write of one turn: `sessions` x `new_tokens` rows."""
    name: str
    latent: torch.Tensor         # bf16 [N,512]
    rope: torch.Tensor           # bf16 [N,64]
    slot_mapping: torch.Tensor   # int64 [N]
    num_blocks: int
    block_table: torch.Tensor


def append_turn(device, seed: int = 0, sessions: int = 64, prefix: int = 140_000, new_tokens: int = 6000,
                zero_group_frac: float = 0.001) -> AppendWorkload:
    """64 sessions each appending a 6,000-token turn at positions
    140,000..145,999 through its own scattered block table; rows ~N(0,1) times
    a per-row scale log-uniform in [0.1, 10]; 0.1% of 16-value latent groups
    set to exact zero."""
    n = sessions * new_tokens
    g = generator(device, "append", seed, "rows")
    u = torch.rand(n, generator=g, device=device)
    row_scale = torch.exp(math.log(0.1) + u * (math.log(10.0) - math.log(0.1)))
    lat = bf16_normal((n, LATENT), g, device, row_scale=row_scale)
    rope = bf16_normal((n, ROPE), g, device, row_scale=row_scale)
    zero = torch.rand((n, LATENT // 16), generator=g, device=device) < zero_group_frac
    lat = lat.view(n, LATENT // 16, 16).masked_fill(zero[..., None], 0).view(n, LATENT)
    total = prefix + new_tokens
    gb = generator(device, "append", seed, "block_table")
    bt, nb = scattered_block_tables(sessions, [(total + BLOCK - 1) // BLOCK] * sessions, gb, device)
    pos = torch.arange(prefix, total, device=device)
    slots = torch.cat([slots_for_positions(bt[s], pos) for s in range(sessions)])
    return AppendWorkload(f"append: {sessions} sessions x {new_tokens:,} new tokens after a {prefix:,}-token prefix",
                          lat, rope, slots, nb, bt)


@dataclass
class IndexerWorkload:
    """Indexer keys + queries for B requests (and the MLA decode that follows)."""
    name: str
    q_idx: torch.Tensor          # bf16 [B, n_heads, 128]
    head_w: torch.Tensor         # float32 [B, n_heads]
    key_pool: torch.Tensor       # uint8, per block: 64 x 128 e4m3 then 64 float32 scales
    key_stride: int
    block_table: torch.Tensor    # int32 [B, max_blocks]
    num_blocks: int
    context_lens: torch.Tensor   # int32 [B]
    topk: int


def indexer_keys(device, seed: int = 0, batch: int = 64, ctx: int = 140_000, n_heads: int = 32, topk: int = 2048,
                 ctx_lens: Optional[List[int]] = None) -> IndexerWorkload:
    """Keys k~N(0,1) [ctx,128] per token, scale s_t = max|k|/448, stored as
    e4m3(k / s_t) (torch's float8_e4m3fn conversion) plus s_t; query 32 x 128
    ~N(0,1) bf16; head weights ~U(0,1)."""
    lens = ctx_lens if ctx_lens is not None else [ctx] * batch
    gq = generator(device, "indexer", seed, "q")
    q = bf16_normal((batch, n_heads, IDX_DIM), gq, device)
    w = torch.rand((batch, n_heads), generator=gq, device=device, dtype=torch.float32)
    gb = generator(device, "indexer", seed, "block_table")
    bt, nb = scattered_block_tables(batch, [(c + BLOCK - 1) // BLOCK for c in lens], gb, device)
    stride = BLOCK * (IDX_DIM + 4)
    pool = torch.zeros(nb * stride, dtype=torch.uint8, device=device)
    blocks = pool.view(nb, stride)
    for b, c in enumerate(lens):
        gk = generator(device, "indexer", seed, "keys", b)
        nblk = (c + BLOCK - 1) // BLOCK
        k = torch.randn((nblk * BLOCK, IDX_DIM), generator=gk, device=device, dtype=torch.float32)
        s = k.abs().amax(dim=1) / 448.0
        codes = (k / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
        phys = bt[b, :nblk].to(torch.int64)
        blocks[phys, :BLOCK * IDX_DIM] = codes.view(nblk, BLOCK * IDX_DIM)
        blocks[phys, BLOCK * IDX_DIM:] = s.to(torch.float32).view(torch.uint8).view(nblk, BLOCK * 4)
    return IndexerWorkload(f"indexer: {batch} requests x {n_heads} index heads, {max(lens):,}-token contexts, "
                           f"top-{topk}", q, w, pool, stride, bt, nb, torch.tensor(lens, dtype=torch.int32,
                                                                                   device=device), topk)
