"""Benchmark: sparse-MLA decode rows/s per layer, HBM GB/s and % of roofline (NVFP4 vs FP8).

Workload (one GPU): a TP4 decode rank -- 32 requests x 16 heads, each with a
140,000-token paged cache (block 64, blocks scattered over one pool), top-2048
per request (70% uniform over the prefix + 30% from the last 6,000 tokens),
seeded synthetic data shaped like the pages' agent traffic ("Prime
Inference: serving GLM-5.3 to agents is a KV-cache problem", sections "The
workload" and "Decode: TP4").

A step is one decode token through L layers: for each of L distinct layer
caches (own pool, own top-k lists, own queries) one NVFP4 sparse decode.  The
L layers are captured in one CUDA graph; their caches together are far larger
than L2, so every layer reads its rows from HBM.  The FP8 (576-byte row)
decode of the same rows is timed the same way and reported beside it; the
quantize-on-write (64 sessions x 6,000 rows) and indexer + top-k (64 x 140,000
tokens) steps of the path are timed on their own workloads in the same run.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs its own replica of the workload (requests are
independent: weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode rows/s per layer, HBM GB/s and % of roofline (NVFP4 vs FP8)"
UNIT = "rows/s"
ROW_NVFP4, ROW_FP8 = 352, 576
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--layers", type=int, default=0, help="distinct layer caches (0: enough to defeat L2)")
    p.add_argument("--no-extras", action="store_true", help="skip the append / indexer sub-measurements")
    p.add_argument("--ctx", type=int, default=140_000,
                   help="context length per request (smaller values only shrink the pools, for profiling)")
    p.add_argument("--append-sessions", type=int, default=64, help="sessions in the quantize-on-write sub-benchmark")
    p.add_argument("--indexer-batch", type=int, default=64, help="requests in the indexer + top-k sub-benchmark")
    p.add_argument("--only-extras", action="store_true", help="time only the sub-benchmarks (profiling)")
    p.add_argument("--draft-tokens", type=str, default="4,15",
                   help="query tokens per request in the draft-token timings (comma-separated; the pages' "
                        "native kernel decodes 15 per launch)")
    p.add_argument("--no-chain", action="store_true", help="skip the chained indexer + top-k + decode timing")
    p.add_argument("--no-dep", action="store_true", help="skip the 128 x 64-head (DEP rank) decode timing")
    p.add_argument("--dep-tokens", type=int, default=24_000_000,
                   help="cached tokens of the DEP rank in total (a smaller pool, same 128 x 2,048 selected rows)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# DRAM traffic of one NVFP4 decode launch of the TP4-rank workload
# (dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture of one
# launch over 65,536 selected rows, `ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum --clock-control none -k regex:sparse_decode_kernel
# -s 1 -c 1` on `bench.py --ctx 16384 --layers 2 --no-extras`), and a digest
# of the kernel source it was taken on: once the source differs, the figure
# no longer describes the kernel and is reported as null.


def e2e_chunks(n_layers):
    """Layers per copy chunk of the end-to-end pass: small chunks at both ends
    (the first chunk's inputs and the last chunk's outputs are the copies no
    decode hides), chunks of at most six layers in between; 1, 2, 4, 6, 6, 3, 1
    for 23 layers."""
    head, tail, rest = [], [], n_layers
    for s in (1, 2, 4):
        if rest > s + 4:
            head.append(s)
            rest -= s
    for s in (1, 3):
        if rest > s + 4:
            tail.insert(0, s)
            rest -= s
    n_mid = max(1, -(-rest // 6)) if rest > 0 else 0
    mid = [rest // n_mid + (1 if i < rest % n_mid else 0) for i in range(n_mid)]
    return head + mid + tail
DECODE_NVFP4_TRAFFIC = {"bytes": 29_498_112 + 2_304, "source_digest": "0fad475c4951d847"}
KERNEL_SOURCES = ("sparse_mla_decode_kv_gb300/csrc/sparse_decode.cu", "sparse_mla_decode_kv_gb300/csrc/mla_device.cuh")


def kernel_source_digest():
    """sha256 over the decode kernel's sources with comments and blank lines
    removed (a comment edit does not change the kernel)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        for line in open(os.path.join(ROOT, rel)):
            code = re.sub(r"//.*$", "", line).strip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def decode_traffic():
    t = DECODE_NVFP4_TRAFFIC
    return t["bytes"] if kernel_source_digest() == t["source_digest"] else None


GB300_L2_BYTES = 132 * 2 ** 20  # used only when no GPU is visible (reference arm on a host without one)


def step_config(ctx, layers, l2_bytes, world):
    """The `config` of the JSON line, shared by both arms so that the driver
    compares like with like."""
    layer_bytes = decode_bytes(32, 16, 2048, ROW_NVFP4)
    return {"workload": f"TP4 rank decode: 32 requests x 16 heads, {ctx:,}-token contexts, top-2048 "
                        "(70% prefix + 30% last 6,000), NVFP4 352-byte rows, block 64",
            "layers_per_step": layers, "block_table": "one per request, shared by the layers",
            "l2": f"inputs larger than L2: {layers} distinct layer caches, "
                  f"{layers * layer_bytes / 1e6:.0f} MB read per step vs {l2_bytes / 1e6:.0f} MB L2",
            "global_batch": 32 * world, "seq_len": ctx, "parallelism": f"replicas x{world}"}


def layers_per_step(requested, l2_bytes):
    return requested or max(8, math.ceil(4 * l2_bytes / decode_bytes(32, 16, 2048, ROW_NVFP4)))


def decode_bytes(batch, heads, topk, row_bytes):
    """Algorithmic bytes of one decode layer: every selected row plus its int32
    index, and per (request, head) the bf16 query (576 values), bf16 output
    (512 values) and float lse."""
    return batch * topk * (row_bytes + 4) + batch * heads * (576 * 2 + 512 * 2 + 4)


def decode_flops(batch, heads, topk):
    """2 * (576 + 512) FLOP per head per selected row (QK over 576, PV over 512)."""
    return batch * heads * topk * 2 * (576 + 512)


def max_over_ranks(x, dist=None, device=None):
    """The slowest rank's value of a per-rank time (a no-op on one rank).
    Every rank gets the maximum back."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def whole_job_rate(units_per_rank, world, seconds):
    """Units processed by all ranks (each runs its own replica) per second of
    the slowest rank's time."""
    return units_per_rank * world / seconds


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed
    region runs: NVML through ctypes every ~1 ms (read-only queries), or
    nvidia-smi every 200 ms if NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str, smi_index: int = 0):
        self.pci = pci_bus_id
        self.smi_index = smi_index
        self.samples = []  # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _nvml(self):
        import ctypes as C
        lib = C.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = C.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(self.pci.encode(), C.byref(h)) != 0:
            raise OSError("no NVML handle for " + self.pci)
        mx = C.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, C.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        clk, rs = C.c_uint(0), C.c_ulonglong(0)

        def loop():
            while not self._stop.is_set():
                if lib.nvmlDeviceGetClockInfo(h, 1, C.byref(clk)) == 0 and get_reasons(h, C.byref(rs)) == 0:
                    self.samples.append((float(clk.value), int(rs.value)))
                time.sleep(0.001)
        return loop

    def __enter__(self):
        try:
            loop = self._nvml()
            self.source = "nvml"
            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
        except Exception:
            self.source = "nvidia-smi"
            fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                      "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                      "clocks_event_reasons.sw_power_cap")
            try:
                self._proc = subprocess.Popen(["nvidia-smi", "-i", str(self.smi_index), f"--query-gpu={fields}",
                                               "--format=csv,noheader,nounits", "-lms", "200"],
                                              stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self._thread = threading.Thread(target=self._read_smi, daemon=True)
                self._thread.start()
            except FileNotFoundError:
                self._proc = None
        return self

    def _read_smi(self):
        bits = [0x8, 0x40, 0x20, 0x4]
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                sm, self.max_mhz = float(parts[0]), float(parts[1])
            except (ValueError, IndexError):
                continue
            mask = sum(b for b, v in zip(bits, parts[2:6]) if v.lower() == "active")
            self.samples.append((sm, mask))

    def __exit__(self, *a):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self):
        sm = [s for s, _ in self.samples]
        mask = 0
        for _, r in self.samples:
            mask |= r
        reasons = sorted(n for b, n in self.REASONS.items() if mask & b)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(sm), "source": self.source}


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args, rank, world):
    import numpy as np
    import oracle as O
    if rank != 0:
        return
    batch, heads, topk, ctx = 32, 16, 2048, args.ctx
    l2 = GB300_L2_BYTES
    try:
        import torch
        if torch.cuda.is_available():
            l2 = torch.cuda.get_device_properties(0).L2_cache_size
    except Exception:
        pass
    rng = np.random.default_rng(0)
    threads = O.host_threads()
    # Bounded sample per step: 8 requests' decodes of one layer (float64), rows
    # drawn and quantized by the oracle itself.
    n_req = 8
    qn = (rng.standard_normal((n_req, heads, 512)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qr = (rng.standard_normal((n_req, heads, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    lat = (rng.standard_normal((n_req * topk, 512)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rope = (rng.standard_normal((n_req * topk, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    nblk = n_req * topk // 64
    pool = np.zeros(nblk * 64 * ROW_NVFP4, np.uint8)
    O.kv_quantize_append(lat, rope, np.arange(n_req * topk, dtype=np.int64), pool, nblk, 64, 64 * ROW_NVFP4, 0)
    bt = np.arange(nblk, dtype=np.int32).reshape(n_req, topk // 64)
    bt_full = np.full((n_req, (ctx + 63) // 64), 0, np.int32)
    bt_full[:, :topk // 64] = bt
    idx = np.tile(np.arange(topk, dtype=np.int32), (n_req, 1))
    cl = np.full(n_req, ctx, np.int32)

    def step():
        O.sparse_decode(qn, qr, pool, 64 * ROW_NVFP4, bt_full, cl, idx, 64, 1 / math.sqrt(192), 0, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = n_req * topk / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": step_config(args.ctx, layers_per_step(args.layers, l2), l2, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{n_req} of 32 requests of one layer per step ({n_req} x {topk} rows), "
                                       f"float64, {threads} host threads"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch

    import sparse_mla_decode_kv_gb300 as m
    import workloads as W
    from sparse_mla_decode_kv_gb300 import build as libbuild

    libbuild.build()
    m.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    hbm, tf_burst, tf_sust, peak_kind = peaks()
    if args.only_extras:
        stream = torch.cuda.Stream(device=dev)
        print(json.dumps(sub_measurements(m, W, dev, stream, args, hbm)), flush=True)
        return
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    B, H, K = 32, 16, 2048
    layer_bytes4 = decode_bytes(B, H, K, ROW_NVFP4)
    layer_bytes8 = decode_bytes(B, H, K, ROW_FP8)
    L = layers_per_step(args.layers, l2)

    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)

    layers = []
    for li in range(L):
        wl = W.tp4_rank_decode(dev, seed=1000 * rank + li, ctx=args.ctx)
        if layers:
            # a paged cache keeps one block table per request for every layer
            # (each layer has its own pool, addressed by the same block ids)
            wl.block_table, wl.num_blocks = layers[0].block_table, layers[0].num_blocks
        W.fill_pool(wl, 0, qa)
        W.fill_pool(wl, 1, qa)
        wl.out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
        wl.lse = torch.empty((B, H), dtype=torch.float32, device=dev)
        layers.append(wl)
    ws_bytes = m.mla_sparse_decode_workspace_size(B, H, K)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    # The staged path: every layer gets its own FP8 copy (576-byte rows, with
    # the identity block table and list the copy kernel writes beside it), and
    # a step first stages all L layers, then runs the L FP8 decodes on the
    # copies.  The L copies together are far larger than L2, so the copy is
    # written to and read back from HBM, as on the pages.
    nblk_st = (K + 63) // 64
    st_pool_bytes = m.mla_staged_pool_bytes(B, K)
    staged = [{"pool": torch.empty(st_pool_bytes, dtype=torch.uint8, device=dev),
               "list": torch.empty((B, K), dtype=torch.int32, device=dev)} for _ in range(L)]
    st_table = torch.arange(B * nblk_st, dtype=torch.int32, device=dev).view(B, nblk_st)
    st_ctx = torch.full((B,), nblk_st * 64, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)

    def decode_all(fmt):
        # fmt 0: native NVFP4, 1: FP8 cache
        fn = {0: m.mla_sparse_decode, 1: m.mla_sparse_decode_fp8}[fmt]
        for wl in layers:
            fn(wl.q_nope, wl.q_rope, wl.pools[fmt], wl.strides[fmt], wl.num_blocks, wl.block_table,
               wl.context_lens, wl.topk_idx, wl.softmax_scale, out=wl.out, lse=wl.lse, workspace=workspace,
               stream=stream)

    def staged_all():
        # staged NVFP4: gather every layer's selected rows into its FP8 copy, then decode the copies
        for wl, st in zip(layers, staged):
            m.mla_stage_rows_fp8(wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table, wl.context_lens,
                                 wl.topk_idx, staged_pool=st["pool"], staged_topk=st["list"], stream=stream)
        for wl, st in zip(layers, staged):
            m.mla_sparse_decode_fp8(wl.q_nope, wl.q_rope, st["pool"], 64 * ROW_FP8, B * nblk_st, st_table, st_ctx,
                                    st["list"], wl.softmax_scale, out=wl.out, lse=wl.lse, workspace=workspace,
                                    stream=stream)

    # Draft tokens: Q query tokens per request, each with its own top-k list
    # (90% shared with its neighbours), over the same layer caches; one
    # timing per Q (4, and the pages' 15 per launch).
    draft_qs = [int(x) for x in args.draft_tokens.split(",") if x.strip()]
    draft_sets = {}
    for Q in draft_qs:
        draft_sets[Q] = {
            "drafts": [W.draft_queries(wl, q_len=Q) for wl in layers],
            "ws": torch.empty(max(m.mla_sparse_decode_mtp_workspace_size(B, Q, H, K), 256), dtype=torch.uint8,
                              device=dev),
            "out": torch.empty((B, Q, H, 512), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((B, Q, H), dtype=torch.float32, device=dev)}

    def drafts_all(Q):
        d = draft_sets[Q]
        for wl, dq in zip(layers, d["drafts"]):
            m.mla_sparse_decode_mtp(dq.q_nope, dq.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                    wl.context_lens, dq.topk_idx, wl.softmax_scale, out=d["out"], lse=d["lse"],
                                    workspace=d["ws"], stream=stream)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()  # warm the launch path outside capture
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        return g

    graphs = {0: capture(lambda: decode_all(0)), 1: capture(lambda: decode_all(1)), 2: capture(staged_all)}
    for Q in draft_qs:
        graphs[("mtp", Q)] = capture(lambda Q=Q: drafts_all(Q))
    torch.cuda.synchronize()

    def timed(g, steps, warmup):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
        stream.synchronize()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / steps, pg, dev)

    props = torch.cuda.get_device_properties(dev)
    pci = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
    with ClockSampler(pci, local) as clocks:
        ms4 = timed(graphs[0], args.steps, args.warmup)
        ms8 = timed(graphs[1], args.steps, args.warmup)
        ms_st = timed(graphs[2], args.steps, args.warmup)
        ms_mtp = {Q: timed(graphs[("mtp", Q)], args.steps, args.warmup) for Q in draft_qs}
    clk = clocks.summary()
    plan = m.mla_sparse_decode_plan(B, H, K)
    launches_per_step = L * plan["kernels"]

    per_layer4 = ms4 / L * 1e-3
    per_layer8 = ms8 / L * 1e-3
    per_layer_st = ms_st / L * 1e-3

    def draft_entry(Q):
        per_layer = ms_mtp[Q] / L * 1e-3
        dq0 = draft_sets[Q]["drafts"][0]
        # rows a layer must read at least once: distinct valid entries over a request's Q lists (layer 0)
        distinct = sum(int(torch.unique(dq0.topk_idx[b][dq0.topk_idx[b] >= 0]).numel()) for b in range(B))
        return {"q_len": Q, "value": whole_job_rate(B * Q * K, world, per_layer), "unit": UNIT,
                "per_layer_us": per_layer * 1e6, "vs_single_token": per_layer / per_layer4,
                "distinct_rows_per_layer": distinct,
                "hbm_gbs_distinct_rows": (distinct * (ROW_NVFP4 + 4) + B * Q * H * 2180) / per_layer / 1e9,
                "note": f"{Q} query tokens per request, each with its own top-2048 list (90% shared), one "
                        "launch per layer"}
    rows = B * K
    value = whole_job_rate(rows, world, per_layer4)
    ach4 = layer_bytes4 / per_layer4 / 1e9
    ach8 = layer_bytes8 / per_layer8 / 1e9
    fl = decode_flops(B, H, K)
    roof_t4 = max(layer_bytes4 / (hbm * 1e9), fl / (tf_burst * 1e12))
    roof_t8 = max(layer_bytes8 / (hbm * 1e9), fl / (tf_burst * 1e12))

    # ---- end to end through the C ABI with host buffers (pinned): per step,
    # every layer's packed inputs (q_nope, q_rope, top-k list, context
    # lengths) are copied H2D, the L decodes run on views of that device
    # buffer, and every layer's packed outputs (out, lse) are copied D2H; the
    # copies go in a few large chunks on a second stream, overlapping the
    # decodes, all captured in one CUDA graph.  (Copying per layer cost ~14 us
    # of copy-engine time per layer, more than the decode.)
    names = ("q_nope", "q_rope", "topk_idx", "context_lens")

    def layout(tensors):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    in_offs, in_bytes = layout([getattr(layers[0], k) for k in names])
    out_like = [layers[0].out, layers[0].lse]
    out_offs, out_bytes = layout(out_like)
    host_in = torch.empty(L * in_bytes, dtype=torch.uint8).pin_memory()
    for li, wl in enumerate(layers):
        for k, o in zip(names, in_offs):
            t = getattr(wl, k).contiguous().cpu()
            n = t.numel() * t.element_size()
            host_in[li * in_bytes + o:li * in_bytes + o + n].copy_(t.view(-1).view(torch.uint8))

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    d_in_buf = torch.empty(L * in_bytes, dtype=torch.uint8, device=dev)
    d_out_buf = torch.empty(L * out_bytes, dtype=torch.uint8, device=dev)
    h_out_buf = torch.empty(L * out_bytes, dtype=torch.uint8).pin_memory()
    d_in = [{k: view(d_in_buf, li * in_bytes + o, getattr(layers[0], k)) for k, o in zip(names, in_offs)}
            for li in range(L)]
    d_out = [[view(d_out_buf, li * out_bytes + o, t) for o, t in zip(out_offs, out_like)] for li in range(L)]
    h2d = in_bytes * L
    d2h = out_bytes * L

    # The step's layers in chunks (e2e_chunks): a second stream copies the
    # inputs of the chunks ahead and the outputs of the chunks done while a
    # chunk decodes.
    bounds, lo = [], 0
    for n in e2e_chunks(L):
        bounds.append((lo, lo + n))
        lo += n
    copy_stream = torch.cuda.Stream(device=dev)

    def e2e_step():
        copy_stream.wait_stream(stream)
        h2d_done = []
        with torch.cuda.stream(copy_stream):
            for lo, hi in bounds:
                d_in_buf[lo * in_bytes:hi * in_bytes].copy_(host_in[lo * in_bytes:hi * in_bytes], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                h2d_done.append(ev)
        dec_done = []
        for (lo, hi), ev in zip(bounds, h2d_done):
            stream.wait_event(ev)
            for li in range(lo, hi):
                wl, x = layers[li], d_in[li]
                m.mla_sparse_decode(x["q_nope"], x["q_rope"], wl.pools[0], wl.strides[0], wl.num_blocks,
                                    wl.block_table, x["context_lens"], x["topk_idx"], wl.softmax_scale,
                                    out=d_out[li][0], lse=d_out[li][1], workspace=workspace, stream=stream)
            ev2 = torch.cuda.Event()
            ev2.record(stream)
            dec_done.append(ev2)
        with torch.cuda.stream(copy_stream):
            for (lo, hi), ev2 in zip(bounds, dec_done):
                copy_stream.wait_event(ev2)
                h_out_buf[lo * out_bytes:hi * out_bytes].copy_(d_out_buf[lo * out_bytes:hi * out_bytes],
                                                               non_blocking=True)
        stream.wait_stream(copy_stream)

    g_e2e = capture(e2e_step)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_e2e.replay()
        stream.synchronize()
        if pg:
            pg.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g_e2e.replay()
        e1.record(stream)
    e1.synchronize()
    # the end-to-end path computes exactly what a device-resident call computes
    wl = layers[-1]
    ref, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                 wl.context_lens, wl.topk_idx, wl.softmax_scale, workspace=workspace, stream=stream)
    stream.synchronize()
    ref = ref.cpu()
    if not torch.equal(view(h_out_buf, (L - 1) * out_bytes + out_offs[0], ref), ref):
        raise RuntimeError("end-to-end decode output differs from the device-resident call")
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, pg, dev)
    e2e_value = whole_job_rate(rows * L, world, ms_e2e * 1e-3)

    extras = {}
    if not args.no_extras:
        del graphs
        extras = sub_measurements(m, W, dev, stream, args, hbm)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms4, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": step_config(args.ctx, L, l2, world),
        "per_layer_us": per_layer4 * 1e6,
        "hbm_gbs": ach4,
        "roofline": {"bound": "hbm" if layer_bytes4 / hbm / 1e9 >= fl / tf_burst / 1e12 else "tensor",
                     "achieved": ach4, "peak": hbm, "unit": "GB/s", "frac": ach4 / hbm, "traffic": decode_traffic(),
                     "kernel": ("sparse_decode_kernel<NVFP4>, splits merged inside their cluster (one launch per layer)"
                                if plan["kernels"] == 1 else
                                "sparse_decode_kernel<NVFP4> + splitk_merge_kernel (one decode layer)"),
                     "plan": plan,
                     "algorithmic_bytes_per_launch": layer_bytes4, "peak_source": peak_kind,
                     "roofline_us": roof_t4 * 1e6, "frac_of_roofline_time": roof_t4 / per_layer4,
                     "vs_nominal_8tbs": ach4 / 8000.0},
        "fp8": {"value": whole_job_rate(rows, world, per_layer8), "unit": UNIT, "per_layer_us": per_layer8 * 1e6,
                "hbm_gbs": ach8, "frac": ach8 / hbm, "roofline_us": roof_t8 * 1e6,
                "bytes_per_row": ROW_FP8 + 4},
        "staged": {"value": whole_job_rate(rows, world, per_layer_st), "unit": UNIT,
                   "per_layer_us": per_layer_st * 1e6, "vs_native": per_layer_st / per_layer4,
                   "vs_fp8": per_layer_st / per_layer8,
                   "algorithmic_bytes_per_row": ROW_NVFP4 + 4 + 2 * (ROW_FP8 + 4),
                   "note": f"a step gathers every layer's selected rows into its own 576-byte FP8 copy "
                           f"({L} copies of {st_pool_bytes / 1e6:.1f} MB, far beyond L2), then runs the {L} FP8 "
                           "decodes on the copies"},
        "drafts": [draft_entry(Q) for Q in draft_qs],
        "nvfp4_bytes_per_row": ROW_NVFP4 + 4,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    line.update(extras)
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(m, W, dev)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def sub_measurements(m, W, dev, stream, args, hbm):
    """Quantize-on-write and indexer + top-k, each timed with CUDA events."""
    import torch
    out = {}
    wl = W.append_turn(dev, sessions=args.append_sessions)
    n = wl.slot_mapping.numel()
    res = {}
    for fmt, rb in ((0, ROW_NVFP4), (1, ROW_FP8)):
        stride = 64 * rb
        pool = torch.zeros(wl.num_blocks * stride, dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                m.mla_kv_quantize_append(wl.latent, wl.rope, wl.slot_mapping, pool, wl.num_blocks, 64, stride, fmt,
                                         stream=stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                m.mla_kv_quantize_append(wl.latent, wl.rope, wl.slot_mapping, pool, wl.num_blocks, 64, stride, fmt,
                                         stream=stream)
            e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1) / args.steps * 1e-3
        bytes_ = n * (512 * 2 + 64 * 2 + 8 + rb)
        res["nvfp4" if fmt == 0 else "fp8"] = {"rows_per_s": n / t, "us": t * 1e6, "hbm_gbs": bytes_ / t / 1e9,
                                               "frac": bytes_ / t / 1e9 / hbm}
        del pool
    out["append"] = {"workload": wl.name, **res}
    # indexer-key quantize-on-write of the same new tokens (the keys are
    # seeded bf16 values, here the first 128 latent values of each token)
    keys = wl.latent[:, :128].contiguous()
    kstride = 64 * 132
    kpool = torch.zeros(wl.num_blocks * kstride, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            m.mla_index_key_quantize_append(keys, wl.slot_mapping, kpool, wl.num_blocks, 64, kstride, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            m.mla_index_key_quantize_append(keys, wl.slot_mapping, kpool, wl.num_blocks, 64, kstride, stream=stream)
        e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / args.steps * 1e-3
    kbytes = n * (128 * 2 + 8 + 132)
    out["index_key_append"] = {"workload": f"{n:,} new tokens' indexer keys (128 bf16 -> 128 e4m3 + float scale)",
                               "rows_per_s": n / t, "us": t * 1e6, "hbm_gbs": kbytes / t / 1e9,
                               "frac": kbytes / t / 1e9 / hbm}
    del kpool, keys
    del wl
    torch.cuda.empty_cache()

    nb = args.indexer_batch
    iw = W.indexer_keys(dev, seed=0, batch=nb, ctx=140_000, n_heads=32, topk=2048)
    max_ctx = 140_000
    ws = torch.empty(m.mla_indexer_topk_workspace_size(nb, max_ctx, 2048), dtype=torch.uint8, device=dev)
    tk = torch.empty((nb, 2048), dtype=torch.int32, device=dev)

    def run():
        m.mla_indexer_topk(iw.q_idx, iw.head_w, iw.key_pool, iw.key_stride, iw.num_blocks, iw.block_table,
                           iw.context_lens, 2048, max_ctx, topk_out=tk, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            run()
        e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / args.steps * 1e-3
    tokens = nb * 140_000
    key_bytes = tokens * 132
    out["indexer_topk"] = {"workload": iw.name, "us": t * 1e6, "tokens_per_s": tokens / t,
                           "key_hbm_gbs": key_bytes / t / 1e9, "frac": key_bytes / t / 1e9 / hbm}
    if not args.no_chain:
        out["chain"] = chain_measurement(m, W, dev, stream, args, hbm, iw, ws, tk)
    del iw, ws
    torch.cuda.empty_cache()
    if not args.no_dep:
        out["dep_rank"] = dep_measurement(m, W, dev, stream, args, hbm)
    return out


def chain_measurement(m, W, dev, stream, args, hbm, iw, ws, tk):
    """The whole path of one decode step and layer: the indexer scores every
    cached token of the 64 requests (140,000 each), keeps the exact top-2048,
    and the NVFP4 sparse decode of 16 MLA heads reads those rows -- the two
    calls captured in one CUDA graph and timed together."""
    import torch
    _, tf_burst, _, _ = peaks()
    nb = iw.q_idx.shape[0]
    kv = W.tp4_rank_decode(dev, seed=77, batch=nb, ctx=140_000)

    def qa(lat, rope, slots, pool, n_blocks, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, n_blocks, 64, stride, fmt)

    W.fill_pool(kv, 0, qa)
    H, K = kv.heads, 2048
    dws = torch.empty(max(m.mla_sparse_decode_workspace_size(nb, H, K), 256), dtype=torch.uint8, device=dev)
    out_t = torch.empty((nb, H, 512), dtype=torch.bfloat16, device=dev)
    lse_t = torch.empty((nb, H), dtype=torch.float32, device=dev)
    max_ctx = 140_000

    def chain():
        m.mla_indexer_topk(iw.q_idx, iw.head_w, iw.key_pool, iw.key_stride, iw.num_blocks, iw.block_table,
                           iw.context_lens, K, max_ctx, topk_out=tk, workspace=ws, stream=stream)
        m.mla_sparse_decode(kv.q_nope, kv.q_rope, kv.pools[0], kv.strides[0], kv.num_blocks, kv.block_table,
                            kv.context_lens, tk, kv.softmax_scale, out=out_t, lse=lse_t, workspace=dws, stream=stream)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        chain()
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            chain()
        for _ in range(args.warmup):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    t = e0.elapsed_time(e1) / args.steps * 1e-3
    tokens = nb * max_ctx
    idx_bytes = tokens * 132 + nb * 32 * (128 * 2 + 4) + nb * K * 4
    dec_bytes = decode_bytes(nb, H, K, ROW_NVFP4)
    flops = tokens * 32 * 128 * 2 + decode_flops(nb, H, K)
    roof = max((idx_bytes + dec_bytes) / (hbm * 1e9), flops / (tf_burst * 1e12))
    res = {"workload": f"{nb} requests x {max_ctx:,} tokens: indexer (32 heads x 128, e4m3 keys) + exact "
                       f"top-{K} + NVFP4 sparse decode of {H} heads on the selected rows, one CUDA graph",
           "us": t * 1e6, "algorithmic_bytes": idx_bytes + dec_bytes, "hbm_gbs": (idx_bytes + dec_bytes) / t / 1e9,
           "roofline_us": roof * 1e6, "frac_of_roofline_time": roof / t,
           "note": "the float32 score row of every request (35.8 MB in all) is scratch between the indexer and the "
                   "top-k and is not counted"}
    del kv, dws
    torch.cuda.empty_cache()
    return res


def dep_measurement(m, W, dev, stream, args, hbm):
    """All heads on one rank: 128 requests x 64 heads, contexts 8K-1M (24M
    cached tokens), top-2048, NVFP4.  Each launch is timed alone with CUDA
    events after an L2 flush (the selected rows of one layer fit in L2)."""
    import torch
    _, tf_burst, _, _ = peaks()
    wl = W.dep_rank_decode(dev, cap=args.dep_tokens)

    def qa(lat, rope, slots, pool, nb, stride, fmt):
        m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt)

    W.fill_pool(wl, 0, qa)
    B, H, K = wl.batch, wl.heads, wl.topk
    ws = torch.empty(max(m.mla_sparse_decode_workspace_size(B, H, K), 256), dtype=torch.uint8, device=dev)
    out_t = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def run():
        m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                            wl.context_lens, wl.topk_idx, wl.softmax_scale, out=out_t, workspace=ws, stream=stream)

    total_ms = 0.0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run()
        steps = max(3, args.steps // 4)
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            e1.synchronize()
            total_ms += e0.elapsed_time(e1)
    t = total_ms / steps * 1e-3
    rows = int((wl.topk_idx >= 0).sum())
    bytes_ = rows * (ROW_NVFP4 + 4) + B * H * (576 * 2 + 512 * 2 + 4)
    flops = decode_flops(B, H, K)
    roof = max(bytes_ / (hbm * 1e9), flops / (tf_burst * 1e12))
    plan = m.mla_sparse_decode_plan_fmt(0, B, H, K, wl.strides[0], wl.num_blocks)
    kernel = ("sparse_decode_tc_kernel (tcgen05.mma, accumulators in tensor memory)" if plan["tensor_memory"]
              else "sparse_decode_kernel<NVFP4> (mma.sync)")
    res = {"workload": wl.name, "kernel": kernel, "plan": plan, "us": t * 1e6, "rows_per_s": rows / t,
           "hbm_gbs": bytes_ / t / 1e9,
           "tflops": flops / t / 1e12, "tensor_frac_of_bf16_peak": flops / t / 1e12 / tf_burst,
           "roofline_us": roof * 1e6, "frac_of_roofline_time": roof / t}
    del wl, flush, ws
    torch.cuda.empty_cache()
    return res


def cpu_baseline(m, W, dev):
    """The float64 oracle on a bounded sample of the same workload (one layer's
    32 requests), timed on all host cores and single-threaded."""
    import numpy as np
    import torch
    import oracle as O

    def u16(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    wl = W.tp4_rank_decode(dev, seed=0)
    reqs = list(range(wl.batch))
    threads = O.host_threads()
    pools, qn, qr = [], u16(wl.q_nope[reqs]), u16(wl.q_rope[reqs])
    K = wl.topk
    nblk = K // 64
    pool = np.zeros(len(reqs) * nblk * 64 * ROW_NVFP4, np.uint8)
    for i, b in enumerate(reqs):
        lat, rope = wl.request_rows(b, wl.topk_idx[b])
        O.kv_quantize_append(u16(lat), u16(rope), np.arange(i * K, (i + 1) * K, dtype=np.int64), pool,
                             len(reqs) * nblk, 64, 64 * ROW_NVFP4, 0)
    bt = np.arange(len(reqs) * nblk, dtype=np.int32).reshape(len(reqs), nblk)
    idx = np.tile(np.arange(K, dtype=np.int32), (len(reqs), 1))
    cl = np.full(len(reqs), K, np.int32)
    # Median of 3 timed runs, on all host cores (one layer: 32 requests) and
    # single-threaded (8 of the 32 requests, to stay bounded).
    def median_rate(n_req, n_threads):
        times = []
        for _ in range(3):
            t0 = time.perf_counter()
            O.sparse_decode(qn[:n_req], qr[:n_req], pool, 64 * ROW_NVFP4, bt[:n_req], cl[:n_req], idx[:n_req], 64,
                            wl.softmax_scale, 0, threads=n_threads)
            times.append(time.perf_counter() - t0)
        return n_req * K / statistics.median(times), statistics.median(times)

    all_rate, all_t = median_rate(len(reqs), threads)
    one_rate, one_t = median_rate(8, 1)
    return {"value": all_rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"one layer ({len(reqs)} requests x {K} rows of 352 B), float64, median of 3 runs "
                      f"({all_t:.3f} s each) on {threads} threads",
            "single_thread": {"value": one_rate, "unit": UNIT, "cores": 1,
                              "sample": f"8 requests x {K} rows, float64, median of 3 runs ({one_t:.3f} s each)"}}


if __name__ == "__main__":
    main()
