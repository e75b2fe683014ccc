"""Split merge inside the decode launch, for every cluster size.

"Prime Inference: serving GLM-5.3 to agents is a KV-cache problem", section
"A kernel that reads four bits directly": the CTAs that share a request's
list merge their partial outputs in-cluster.  Here the splits of one
(request, head group) form a thread-block cluster when there are 2 to 8 of
them and merge after a cluster barrier; more splits go through a second
kernel.  For each split count 2..8 the batch is chosen (through the plan
query, on this device) so that the decode plans exactly that many splits,
and sampled requests are checked against the oracle at the decode tolerance.
The decode is also deterministic: two calls give the same bits."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import assert_decode_close, lib, oracle_rows_decode, u16

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
HEADS, TOPK, CTX = 16, 2048, 2560


def batch_for_splits(m, splits):
    for batch in range(1, 600):
        if m.mla_sparse_decode_plan(batch, HEADS, TOPK)["splits"] == splits:
            return batch
    return None


def workload(batch, seed):
    def draw(b, c, g):
        return W.distinct_uniform(TOPK, 0, c, g, DEV)
    return W._decode_workload("cluster sizes", ("cluster", seed, batch), batch, HEADS, TOPK, [CTX] * batch, DEV,
                              0.01, draw)


@pytest.mark.parametrize("splits", [2, 3, 4, 5, 6, 7, 8])
def test_every_cluster_size_against_oracle(splits):
    m = lib()
    batch = batch_for_splits(m, splits)
    if batch is None:
        pytest.skip(f"no batch of {HEADS}-head requests plans {splits} splits on this device")
    plan = m.mla_sparse_decode_plan(batch, HEADS, TOPK)
    assert plan["kernels"] == 1  # merged inside the decode launch
    wl = workload(batch, seed=splits)
    W.fill_pool(wl, O.FMT_NVFP4, lambda lat, rope, slots, pool, nb, stride, fmt:
                m.mla_kv_quantize_append(lat, rope, slots, pool, nb, 64, stride, fmt))
    lse = torch.empty((batch, HEADS), dtype=torch.float32, device=DEV)
    out, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks, wl.block_table,
                                 wl.context_lens, wl.topk_idx, wl.softmax_scale, lse=lse)
    again, _ = m.mla_sparse_decode(wl.q_nope, wl.q_rope, wl.pools[0], wl.strides[0], wl.num_blocks,
                                   wl.block_table, wl.context_lens, wl.topk_idx, wl.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, again), "two calls on the same inputs differ"
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    for b in sorted({0, batch // 2, batch - 1}):
        idx = wl.topk_idx[b]
        lat, rope = wl.request_rows(b, idx)
        ref, ref_lse = oracle_rows_decode(u16(wl.q_nope[b]), u16(wl.q_rope[b]), u16(lat), u16(rope),
                                          np.ones(TOPK, dtype=bool), O.FMT_NVFP4, wl.softmax_scale)
        assert_decode_close(out[b], lse[b], ref, ref_lse, f"{splits} splits, request {b}")
