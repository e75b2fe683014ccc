// Staged path: the selected NVFP4 rows re-stored as 576-byte FP8 rows, for
// the FP8 decode to read (an ablation of the native kernel).
//
// "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem",
// section "A kernel that reads four bits directly", figure "staged vs native
// decode": the first version gathered the rows the indexer selected, wrote
// an FP8 copy of each to GPU memory and ran the existing FP8 attention kernel
// on it; per selected row that moves 352 + 576 + 576 bytes through HBM
// instead of 352.  Each latent value e2m1 x S is re-encoded as e4m3
// (nearest-even, satfinite, sign kept); the rope bytes are copied.
//
// Layout of the staged copy: request b's entry j lands in row
// (b * nblk * 64 + j) of a 576-byte paged pool with nblk = ceil(topk / 64)
// blocks per request, so block table [b, i] = b * nblk + i and context
// length nblk * 64 make it an ordinary FP8 pool; the staged list holds j for
// a valid entry and -1 for a masked one (masked entries write no row).
//
// One warp per 4 list entries: lanes 0-3 resolve the four rows (index, then
// block table), then every lane converts its 16-value group of each row
// (8 code bytes + 1 scale byte in, 16 bytes out) and lanes 0-3 copy the
// rope.  All loads of the four rows are issued before any conversion.
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kRowsPerWarp = 4;

struct StageArgs {
  const uint8_t* pool;
  int64_t block_stride;
  int64_t num_blocks;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  uint8_t* staged;
  int32_t* staged_topk;
  int32_t* staged_bt;   // optional: identity block table [batch, nblk]
  int32_t* staged_ctx;  // optional: [batch] = nblk * 64
  int64_t entries;      // batch * topk
  int max_blocks;
  int topk;
  int nblk;
  int batch;
};

__global__ void __launch_bounds__(kWarps * 32) stage_rows_fp8_kernel(const StageArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (a.staged_bt != nullptr)
    for (int64_t i = gtid; i < static_cast<int64_t>(a.batch) * a.nblk; i += nthreads)
      a.staged_bt[i] = static_cast<int32_t>(i);
  if (a.staged_ctx != nullptr)
    for (int64_t i = gtid; i < a.batch; i += nthreads) a.staged_ctx[i] = a.nblk * kBlock;

  const int64_t warp_global = gtid >> 5;
  const int64_t warp_stride = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t e0 = warp_global * kRowsPerWarp; e0 < a.entries; e0 += warp_stride * kRowsPerWarp) {
    // ---- resolve four entries (lanes 0..3)
    int64_t off = -1;
    int64_t dst_row = 0;
    if (lane < kRowsPerWarp && e0 + lane < a.entries) {
      const int64_t e = e0 + lane;
      const int b = static_cast<int>(e / a.topk);
      const int j = static_cast<int>(e - static_cast<int64_t>(b) * a.topk);
      const int t = __ldg(a.topk_idx + e);
      bool ok = t >= 0 && t < __ldg(a.ctx_lens + b) && t / kBlock < a.max_blocks;
      const int64_t blk = ok ? __ldg(a.block_table + static_cast<int64_t>(b) * a.max_blocks + t / kBlock) : -1;
      ok = ok && blk >= 0 && blk < a.num_blocks;
      a.staged_topk[e] = ok ? j : -1;
      off = ok ? blk * a.block_stride + static_cast<int64_t>(t % kBlock) * kRowNvfp4 : -1;
      dst_row = static_cast<int64_t>(b) * a.nblk * kBlock + j;
    }
    int64_t offs[kRowsPerWarp], dsts[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      offs[r] = __shfl_sync(0xFFFFFFFFu, off, r);
      dsts[r] = __shfl_sync(0xFFFFFFFFu, dst_row, r);
    }
    // ---- loads of all four rows first
    uint2 codes[kRowsPerWarp];
    uint32_t scale[kRowsPerWarp];
    uint4 rope[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      codes[r] = make_uint2(0, 0);
      scale[r] = 0;
      rope[r] = make_uint4(0, 0, 0, 0);
      if (offs[r] >= 0) {
        const uint8_t* row = a.pool + offs[r];
        codes[r] = __ldg(reinterpret_cast<const uint2*>(row) + lane);
        scale[r] = __ldg(row + kScaleOff + lane);
        if (lane < 4) rope[r] = __ldg(reinterpret_cast<const uint4*>(row + kRopeOffNvfp4) + lane);
      }
    }
    // ---- convert and store
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (offs[r] < 0) continue;
      const uint32_t s2 = e4m3x2_to_f16x2(scale[r] | (scale[r] << 8));  // {S, S}
      const uint32_t cw[2] = {codes[r].x, codes[r].y};
      uint32_t outw[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          // bytes 2q, 2q+1 of word h -> values 4(2h+q) .. 4(2h+q)+3
          const uint32_t v01 = hmul2(e2m1x2_to_f16x2((cw[h] >> (16 * q)) & 0xFFu), s2);  // exact in f16
          const uint32_t v23 = hmul2(e2m1x2_to_f16x2((cw[h] >> (16 * q + 8)) & 0xFFu), s2);
          const float f0 = __half2float(__ushort_as_half(static_cast<unsigned short>(v01 & 0xFFFFu)));
          const float f1 = __half2float(__ushort_as_half(static_cast<unsigned short>(v01 >> 16)));
          const float f2 = __half2float(__ushort_as_half(static_cast<unsigned short>(v23 & 0xFFFFu)));
          const float f3 = __half2float(__ushort_as_half(static_cast<unsigned short>(v23 >> 16)));
          outw[2 * h + q] = f32x2_to_e4m3x2(f1, f0) | (f32x2_to_e4m3x2(f3, f2) << 16);
        }
      }
      uint8_t* dst = a.staged + dsts[r] * kRowFp8;
      *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
      if (lane < 4) *reinterpret_cast<uint4*>(dst + kRopeOffFp8 + 16 * lane) = rope[r];
    }
  }
}

}  // namespace

cudaError_t launch_stage_rows_fp8(const void* pool, int64_t block_stride, int64_t num_blocks,
                                  const int32_t* block_table, int max_blocks_per_req, const int32_t* context_lens,
                                  const int32_t* topk_idx, int batch, int topk, void* staged, int32_t* staged_topk,
                                  int32_t* staged_bt, int32_t* staged_ctx, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  StageArgs a;
  a.pool = static_cast<const uint8_t*>(pool);
  a.block_stride = block_stride;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.ctx_lens = context_lens;
  a.topk_idx = topk_idx;
  a.staged = static_cast<uint8_t*>(staged);
  a.staged_topk = staged_topk;
  a.staged_bt = staged_bt;
  a.staged_ctx = staged_ctx;
  a.entries = static_cast<int64_t>(batch) * topk;
  a.max_blocks = max_blocks_per_req;
  a.topk = topk;
  a.nblk = (topk + kBlock - 1) / kBlock;
  a.batch = batch;
  const int64_t per_block = static_cast<int64_t>(kWarps) * kRowsPerWarp;
  const int64_t want = (a.entries + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;  // grid-stride beyond 8 blocks per SM
  const int grid = static_cast<int>(want < cap ? want : cap);
  stage_rows_fp8_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
