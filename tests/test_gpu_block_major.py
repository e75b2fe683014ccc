"""Block-major pool: every layer's slice of a block stored together.

"Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section
"Moving the cache: 32K copies for one request" and its KV layout figure: in
the block-major (BLHNC) layout one block's data for all layers is
contiguous, so a block is one transfer region.  Here the
pool is [num_blocks][layers][64 rows][row bytes]: layer l's view starts at
l * 64 * row bytes and its block stride is layers * 64 * row bytes.

Checks: quantize-on-write into one layer's slice leaves the other layers'
bytes untouched; the decode of each layer from the block-major pool equals,
bit for bit, the decode of the same rows from a packed single-layer pool;
and one layer is checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LAYERS = 3


def layer_workloads():
    def draw(b, c, g):
        return W.distinct_uniform(min(400, c), 0, c, g, DEV)
    # same geometry (block tables, lists) for every layer; different rows and queries
    wls = [W._decode_workload("block-major", ("bm", l), 3, 32, 400, [3000, 900, 5000], DEV, 0.01, draw)
           for l in range(LAYERS)]
    for wl in wls[1:]:
        wl.block_table, wl.num_blocks, wl.topk_idx = wls[0].block_table, wls[0].num_blocks, wls[0].topk_idx
    return wls


@pytest.mark.parametrize("fmt", [O.FMT_NVFP4, O.FMT_FP8], ids=["nvfp4", "fp8"])
def test_block_major_pool(fmt):
    m = lib()
    rb = O.row_bytes(fmt)
    slice_bytes = 64 * rb
    stride = LAYERS * slice_bytes
    wls = layer_workloads()
    nb = wls[0].num_blocks
    pool = torch.full((nb * stride,), 0xEE, dtype=torch.uint8, device=DEV)

    def append_into(layer):
        view = pool[layer * slice_bytes:]

        def qa(lat, rope, slots, _pool, num_blocks, _stride, f):
            m.mla_kv_quantize_append(lat, rope, slots, view, num_blocks, 64, stride, f)
        wl = wls[layer]
        for b in range(wl.batch):
            lat, rope = wl.request_rows(b)
            slots = W.slots_for_positions(wl.block_table[b], torch.arange(lat.shape[0], device=DEV))
            qa(lat, rope, slots, None, nb, stride, fmt)

    # writing layer 1 only leaves layers 0 and 2 untouched
    append_into(1)
    torch.cuda.synchronize()
    blocks = pool.view(nb, LAYERS, slice_bytes)
    assert bool((blocks[:, 0] == 0xEE).all()) and bool((blocks[:, 2] == 0xEE).all())
    append_into(0)
    append_into(2)

    dec = m.mla_sparse_decode if fmt == O.FMT_NVFP4 else m.mla_sparse_decode_fp8
    for layer, wl in enumerate(wls):
        view = pool[layer * slice_bytes:]
        out_bm, _ = dec(wl.q_nope, wl.q_rope, view, stride, nb, wl.block_table, wl.context_lens, wl.topk_idx,
                        wl.softmax_scale)
        packed = torch.full((nb * slice_bytes,), 0xEE, dtype=torch.uint8, device=DEV)
        for b in range(wl.batch):
            lat, rope = wl.request_rows(b)
            slots = W.slots_for_positions(wl.block_table[b], torch.arange(lat.shape[0], device=DEV))
            m.mla_kv_quantize_append(lat, rope, slots, packed, nb, 64, slice_bytes, fmt)
        out_pk, _ = dec(wl.q_nope, wl.q_rope, packed, slice_bytes, nb, wl.block_table, wl.context_lens,
                        wl.topk_idx, wl.softmax_scale)
        torch.cuda.synchronize()
        assert torch.equal(out_bm, out_pk), f"layer {layer}: block-major and packed pools decode differently"
        # the packed pool's bytes equal this layer's slice of every block
        assert torch.equal(packed.view(nb, slice_bytes), pool.view(nb, LAYERS, slice_bytes)[:, layer])

    # one layer against the oracle
    wl = wls[2]
    lse = torch.empty((wl.batch, wl.heads), dtype=torch.float32, device=DEV)
    out, _ = dec(wl.q_nope, wl.q_rope, pool[2 * slice_bytes:], stride, nb, wl.block_table, wl.context_lens,
                 wl.topk_idx, wl.softmax_scale, lse=lse)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(wl.batch):
        idx = wl.topk_idx[b].cpu().numpy().astype(np.int64)
        valid = (idx >= 0) & (idx < int(wl.context_lens[b]))
        lat, rope = wl.request_rows(b, torch.from_numpy(np.where(valid, idx, 0)).to(DEV))
        ref, ref_lse = oracle_rows_decode(u16(wl.q_nope[b]), u16(wl.q_rope[b]), u16(lat), u16(rope), valid, fmt,
                                          wl.softmax_scale)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"block-major layer 2 request {b}")
