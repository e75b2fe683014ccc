// Indexer score and exact top-k selection.
//
// "GLM-5.3 PCP/DCP long-context on H200", section 1: the indexer rates all
// preceding tokens and attention reads only the 2,048 best; section 3: an
// indexer key is 128 e4m3 bytes and a float scale.  The score
// is sum_h w_h * relu(s_t * (q_h . k_t)).
//
// indexer_scores_kernel: one CTA = 4 warps over 512 tokens of one request.
// Each warp takes 16-token m-tiles; the keys are loaded straight from the
// paged pool (8 bytes per lane per 32-dim chunk, prefetched one m-tile
// ahead), converted e4m3x2 -> f16x2 into mma.sync A fragments and multiplied
// by the n_heads query rows held as B fragments; the epilogue applies the
// per-token scale, relu and head weights and reduces over heads with two
// shuffles.  HBM-bound at 132 bytes per token.
//
// Top-k in two kernels.  Scores map to order-preserving 32-bit keys (with
// -0.0 folded into +0.0).  topk_collect_kernel: 8 CTAs per request each draw
// the same strided sample of 2,048 keys of the whole row, take from it a
// threshold expected to keep ~2.5 k elements (two radix passes over the
// sample), and collect the elements of their eighth of the row at or above
// it into global lists in index order.  topk_kernel: one 1,024-thread CTA
// per request concatenates the 8 lists in order; three histogram passes over
// 11 + 11 + 10 key bits find the k-th largest key T among the candidates and
// how many ties at T are taken, and an ordered compaction writes every index
// with key > T and the lowest-index ties in ascending order.  If the
// threshold kept too few or too many elements, the same selection runs over
// the whole row instead.
#include <cuda_fp16.h>

#include <algorithm>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kIdxWarps = 4;
constexpr int kIdxTokensPerCta = 512;
constexpr int kIdxBlockBytesKeys = kBlock * kIdxDim;  // 8,192 key bytes, then 64 float scales

__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t two) {
  return f32x2_to_f16x2_sat(bf16_bits_to_f32(two & 0xFFFFu), bf16_bits_to_f32(two >> 16));
}

struct IdxArgs {
  const uint16_t* q;
  const float* w;
  const uint8_t* pool;
  int64_t block_stride;
  int64_t num_blocks;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  float* scores;
  int64_t scores_stride;
  int max_blocks;
  int n_heads;
  int max_ctx;
  int batch;
};

// Row address of token t's key (nullptr when masked) and its scale.
__device__ __forceinline__ const uint8_t* key_row(const IdxArgs& a, const int32_t* bt_row, int t, int ctx,
                                                  float* scale) {
  if (t >= ctx) return nullptr;
  const int lb = t / kBlock;
  if (lb >= a.max_blocks) return nullptr;
  const int pb = __ldg(bt_row + lb);
  if (pb < 0 || pb >= a.num_blocks) return nullptr;
  const uint8_t* blk = a.pool + static_cast<int64_t>(pb) * a.block_stride;
  *scale = __ldg(reinterpret_cast<const float*>(blk + kIdxBlockBytesKeys) + (t % kBlock));
  return blk + (t % kBlock) * kIdxDim;
}

template <int NT>  // n-tiles of 8 heads
__global__ void __launch_bounds__(kIdxWarps * 32, 3) indexer_scores_kernel(const IdxArgs a) {
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
  const int t_begin = blockIdx.x * kIdxTokensPerCta;
  if (t_begin >= ctx) return;
  const int32_t* bt_row = a.block_table + static_cast<int64_t>(b) * a.max_blocks;

  // Query B fragments (K = 128 dims permuted like the keys, N = 8*NT heads) and head weights.
  uint32_t bq[8][NT][2];
  float wh[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int h = 8 * n + g;
    const uint16_t* qh = a.q + (static_cast<int64_t>(b) * a.n_heads + h) * kIdxDim;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + 32 * q + 8 * c));
      bq[2 * q][n][0] = bf16pair_to_f16x2(v.x);
      bq[2 * q][n][1] = bf16pair_to_f16x2(v.y);
      bq[2 * q + 1][n][0] = bf16pair_to_f16x2(v.z);
      bq[2 * q + 1][n][1] = bf16pair_to_f16x2(v.w);
    }
    const float* wb = a.w + static_cast<int64_t>(b) * a.n_heads;
    wh[n][0] = __ldg(wb + 8 * n + 2 * c);
    wh[n][1] = __ldg(wb + 8 * n + 2 * c + 1);
  }

  float* out_row = a.scores + static_cast<int64_t>(b) * a.scores_stride;
  const int n_mt = kIdxTokensPerCta / 16;
  // Software pipeline: the keys and scales of the warp's next m-tile are
  // loaded while the current one is multiplied.
  auto load_tile = [&](int mt, uint2 (&v0)[4], uint2 (&v1)[4], float& s0, float& s1, bool& ok0, bool& ok1) {
    const int t0 = t_begin + 16 * mt + g;
    const uint8_t* k0 = key_row(a, bt_row, t0, ctx, &s0);
    const uint8_t* k1 = key_row(a, bt_row, t0 + 8, ctx, &s1);
    ok0 = k0 != nullptr;
    ok1 = k1 != nullptr;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v0[q] = k0 ? __ldg(reinterpret_cast<const uint2*>(k0 + 32 * q + 8 * c)) : make_uint2(0, 0);
      v1[q] = k1 ? __ldg(reinterpret_cast<const uint2*>(k1 + 32 * q + 8 * c)) : make_uint2(0, 0);
    }
  };
  uint2 v0[4], v1[4];
  float s0 = 0.f, s1 = 0.f;
  bool ok0 = false, ok1 = false;
  int mt = warp;
  if (t_begin + 16 * mt < ctx) load_tile(mt, v0, v1, s0, s1, ok0, ok1);
  for (; mt < n_mt && t_begin + 16 * mt < ctx; mt += kIdxWarps) {
    const int t0 = t_begin + 16 * mt + g;
    const int t1 = t0 + 8;
    const int nmt = mt + kIdxWarps;
    uint2 n0[4], n1[4];
    float ns0 = 0.f, ns1 = 0.f;
    bool nok0 = false, nok1 = false;
    if (nmt < n_mt && t_begin + 16 * nmt < ctx) load_tile(nmt, n0, n1, ns0, ns1, nok0, nok1);
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x0[2], x1[2], y0[2], y1[2];
      e4m3x4_to_f16x2x2(v0[q].x, x0);
      e4m3x4_to_f16x2x2(v1[q].x, x1);
      e4m3x4_to_f16x2x2(v0[q].y, y0);
      e4m3x4_to_f16x2x2(v1[q].y, y1);
      uint32_t A0[4] = {x0[0], x1[0], x0[1], x1[1]};
      uint32_t A1[4] = {y0[0], y1[0], y0[1], y1[1]};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma_f16(acc[n], A0, bq[2 * q][n][0], bq[2 * q][n][1]);
        mma_f16(acc[n], A1, bq[2 * q + 1][n][0], bq[2 * q + 1][n][1]);
      }
    }
    // sum_h w_h * relu(s_t * dot): this lane holds heads 8n + 2c + {0,1}.
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      p0 += wh[n][0] * fmaxf(s0 * acc[n][0], 0.f) + wh[n][1] * fmaxf(s0 * acc[n][1], 0.f);
      p1 += wh[n][0] * fmaxf(s1 * acc[n][2], 0.f) + wh[n][1] * fmaxf(s1 * acc[n][3], 0.f);
    }
    p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 1);
    p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 2);
    p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 1);
    p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 2);
    if (c == 0) {
      if (t0 < ctx) out_row[t0] = ok0 ? p0 : -INFINITY;
      if (t1 < ctx) out_row[t1] = ok1 ? p1 : -INFINITY;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v0[q] = n0[q];
      v1[q] = n1[q];
    }
    s0 = ns0;
    s1 = ns1;
    ok0 = nok0;
    ok1 = nok1;
  }
}

// TMA variant (the pool's block stride is a multiple of 128 bytes, so the key
// pool is a 2-D tensor of 128-byte rows): the CTA's 8 key blocks (64 tokens
// x 128 bytes each) land in shared memory as 8 tiles with the 128-byte
// swizzle, their scales as 8 bulk copies of 256 bytes, all issued at entry
// (66 KB in flight per CTA); each block has its own mbarrier so the warps
// start on block 0 while the rest arrive.  The swizzle puts the 16-byte
// chunk j of tile row r at chunk j ^ (r & 7), so the 8 rows a fragment load
// touches hit 8 different bank groups.
constexpr int kIdxBlocksPerCta = kIdxTokensPerCta / kBlock;  // 8

struct alignas(1024) IdxSmem {
  uint8_t keys[kIdxBlocksPerCta][kBlock][kIdxDim];  // 8 KB per block, 1024-byte aligned (swizzle atom)
  float scales[kIdxBlocksPerCta][kBlock];
  uint64_t bar[kIdxBlocksPerCta];
  int32_t pblk[kIdxBlocksPerCta];  // physical block, -1 if invalid or past the context
};

template <int NT>  // n-tiles of 8 heads
__global__ void __launch_bounds__(kIdxWarps * 32, 3)
    indexer_scores_tma_kernel(const IdxArgs a, const __grid_constant__ CUtensorMap tmap, unsigned int* fault_word) {
  extern __shared__ uint8_t idx_smem_raw[];
  // The swizzled tiles need a 1024-byte aligned base.
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>(idx_smem_raw + ((1024u - (smem_u32(idx_smem_raw) & 1023u)) & 1023u));
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
  const int t_begin = blockIdx.x * kIdxTokensPerCta;
  if (t_begin >= ctx) return;
  const int32_t* bt_row = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
  const int lb0 = t_begin / kBlock;

  if (threadIdx.x < kIdxBlocksPerCta) {
    const int lb = lb0 + threadIdx.x;
    int pb = -1;
    if (lb * kBlock < ctx && lb < a.max_blocks) {
      pb = __ldg(bt_row + lb);
      if (pb < 0 || pb >= a.num_blocks) pb = -1;
    }
    sm.pblk[threadIdx.x] = pb;
    mbar_init(&sm.bar[threadIdx.x], 1);
  }
  fence_mbar_init();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int64_t rows_per_block = a.block_stride / kIdxDim;
#pragma unroll 1
    for (int i = 0; i < kIdxBlocksPerCta; ++i) {
      const int pb = sm.pblk[i];
      if (pb < 0) continue;
      mbar_expect_tx(&sm.bar[i], kIdxBlockBytesKeys + kBlock * 4);
      tma_load_2d(sm.keys[i][0], &tmap, 0, static_cast<int>(pb * rows_per_block), &sm.bar[i]);
      bulk_load(sm.scales[i], a.pool + static_cast<int64_t>(pb) * a.block_stride + kIdxBlockBytesKeys, kBlock * 4,
                &sm.bar[i]);
    }
  }

  // Query B fragments (K = 128 dims permuted like the keys, N = 8*NT heads) and head weights.
  uint32_t bq[8][NT][2];
  float wh[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int h = 8 * n + g;
    const uint16_t* qh = a.q + (static_cast<int64_t>(b) * a.n_heads + h) * kIdxDim;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + 32 * q + 8 * c));
      bq[2 * q][n][0] = bf16pair_to_f16x2(v.x);
      bq[2 * q][n][1] = bf16pair_to_f16x2(v.y);
      bq[2 * q + 1][n][0] = bf16pair_to_f16x2(v.z);
      bq[2 * q + 1][n][1] = bf16pair_to_f16x2(v.w);
    }
    const float* wb = a.w + static_cast<int64_t>(b) * a.n_heads;
    wh[n][0] = __ldg(wb + 8 * n + 2 * c);
    wh[n][1] = __ldg(wb + 8 * n + 2 * c + 1);
  }

  float* out_row = a.scores + static_cast<int64_t>(b) * a.scores_stride;
  constexpr int kTiles = kIdxTokensPerCta / 16;
  for (int mt = warp; mt < kTiles && t_begin + 16 * mt < ctx; mt += kIdxWarps) {
    const int blk = mt / (kBlock / 16);
    const int r0 = (mt % (kBlock / 16)) * 16 + g;  // tile rows r0 and r0 + 8; (r & 7) == g for both
    const int t0 = t_begin + 16 * mt + g;
    const int t1 = t0 + 8;
    if (sm.pblk[blk] < 0) {  // block id outside the pool: the block's tokens score -inf
      if (c == 0) {
        if (t0 < ctx) out_row[t0] = -INFINITY;
        if (t1 < ctx) out_row[t1] = -INFINITY;
      }
      continue;
    }
    if (!mbar_wait_bounded(&sm.bar[blk], 0u, fault_word, kFaultIndexerWait)) continue;
    const uint8_t* row0 = sm.keys[blk][r0];
    const uint8_t* row1 = sm.keys[blk][r0 + 8];
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int off = (((2 * q + (c >> 1)) ^ g) << 4) + 8 * (c & 1);
      const uint2 v0 = *reinterpret_cast<const uint2*>(row0 + off);
      const uint2 v1 = *reinterpret_cast<const uint2*>(row1 + off);
      uint32_t x0[2], x1[2], y0[2], y1[2];
      e4m3x4_to_f16x2x2(v0.x, x0);
      e4m3x4_to_f16x2x2(v1.x, x1);
      e4m3x4_to_f16x2x2(v0.y, y0);
      e4m3x4_to_f16x2x2(v1.y, y1);
      uint32_t A0[4] = {x0[0], x1[0], x0[1], x1[1]};
      uint32_t A1[4] = {y0[0], y1[0], y0[1], y1[1]};
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        mma_f16(acc[n], A0, bq[2 * q][n][0], bq[2 * q][n][1]);
        mma_f16(acc[n], A1, bq[2 * q + 1][n][0], bq[2 * q + 1][n][1]);
      }
    }
    const float s0 = sm.scales[blk][r0];
    const float s1 = sm.scales[blk][r0 + 8];
    // sum_h w_h * relu(s_t * dot): this lane holds heads 8n + 2c + {0,1}.
    float p0 = 0.f, p1 = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      p0 += wh[n][0] * fmaxf(s0 * acc[n][0], 0.f) + wh[n][1] * fmaxf(s0 * acc[n][1], 0.f);
      p1 += wh[n][0] * fmaxf(s1 * acc[n][2], 0.f) + wh[n][1] * fmaxf(s1 * acc[n][3], 0.f);
    }
    p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 1);
    p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 2);
    p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 1);
    p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 2);
    if (c == 0) {
      if (t0 < ctx) out_row[t0] = p0;
      if (t1 < ctx) out_row[t1] = p1;
    }
  }
}

// Pipelined variant (TMA, up to 32 index heads): a persistent grid of two
// CTAs per SM, each walking a contiguous range of 256-token chunks (request
// major, so the query changes rarely).  A producer warp resolves each
// chunk's four block ids (eight chunks per batch of lookups, one lane per
// block) and loads its keys (64 x 128-byte TMA tiles, 128-byte swizzle) and
// scales (256-byte bulk copies) into a three-slot ring, up to three chunks
// ahead; four compute warps take row group w of every block, two 16-token
// tiles at a time so that eight accumulator chains are in flight, and hand
// the slot back.  Compared with one CTA per 512 tokens, no chunk waits for
// its own block-table lookups and copies: they were issued while the
// previous chunks were multiplied.
constexpr int kPipeChunk = 256;                  // tokens per chunk
constexpr int kPipeBlocks = kPipeChunk / kBlock;  // 4 key blocks
constexpr int kPipeSlots = 3;
constexpr int kPipeComputeWarps = 4;
constexpr int kPipeThreads = (kPipeComputeWarps + 1) * 32;
constexpr uint32_t kPipeBlockBytes = kIdxBlockBytesKeys + kBlock * 4;  // 8,448 bytes per block

struct alignas(1024) IdxPipeSmem {
  uint8_t keys[kPipeSlots][kPipeBlocks][kBlock][kIdxDim];  // 8 KB per block (1024-byte aligned)
  float scales[kPipeSlots][kPipeBlocks][kBlock];
  int32_t pblk[kPipeSlots][kPipeBlocks];  // physical block; -1: outside the pool (-inf); -2: past the context
  uint64_t full[kPipeSlots];
  uint64_t empty[kPipeSlots];
  int abort_flag;
};

template <int NT>  // n-tiles of 8 heads
__global__ void __launch_bounds__(kPipeThreads, 2)
    indexer_scores_pipe_kernel(const IdxArgs a, const __grid_constant__ CUtensorMap tmap, unsigned int* fault_word) {
  extern __shared__ uint8_t idx_smem_raw[];
  IdxPipeSmem& sm =
      *reinterpret_cast<IdxPipeSmem*>(idx_smem_raw + ((1024u - (smem_u32(idx_smem_raw) & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunk = (a.max_ctx + kPipeChunk - 1) / kPipeChunk;
  const int64_t n_items = static_cast<int64_t>(a.batch) * n_chunk;
  const int64_t per = (n_items + gridDim.x - 1) / gridDim.x;
  const int64_t it_begin = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t it_end = min(n_items, it_begin + per);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPipeSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kPipeComputeWarps);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kPipeComputeWarps) {
    // ------------------------------------------------------------ producer
    const int64_t rows_per_block = a.block_stride / kIdxDim;
    int s = 0;
    bool stop = false;
    for (int64_t base = it_begin; base < it_end && !stop; base += 8) {
      // lane l: block l % 4 of item base + l / 4
      const int64_t item = base + lane / 4;
      int pb = -2;
      bool live = false;
      if (item < it_end) {
        const int b = static_cast<int>(item / n_chunk);
        const int chunk = static_cast<int>(item - static_cast<int64_t>(b) * n_chunk);
        const int ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
        live = chunk * kPipeChunk < ctx;
        const int lb = chunk * kPipeBlocks + (lane & 3);
        if (lb * kBlock < ctx) {
          pb = -1;
          if (lb < a.max_blocks) {
            const int p = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_blocks + lb);
            if (p >= 0 && p < a.num_blocks) pb = p;
          }
        }
      }
      const uint32_t live_mask = __ballot_sync(0xFFFFFFFFu, live);
      const uint32_t valid_mask = __ballot_sync(0xFFFFFFFFu, pb >= 0);
      for (int k = 0; k < 8; ++k) {
        if (!((live_mask >> (4 * k)) & 1u)) continue;  // empty item (past the context): nothing to load
        const int slot = s % kPipeSlots;
        bool ok = true;
        if (lane == 0 && s >= kPipeSlots)
          ok = mbar_wait_or_abort(&sm.empty[slot], static_cast<uint32_t>(s / kPipeSlots - 1) & 1u, &sm.abort_flag,
                                  fault_word, kFaultIndexerWait);
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
          if (lane == 0) sm.abort_flag = 1;
          stop = true;
          break;
        }
        const bool mine = (lane >> 2) == k;
        if (mine) sm.pblk[slot][lane & 3] = pb;
        __syncwarp();
        if (lane == 0)
          mbar_expect_tx(&sm.full[slot], __popc((valid_mask >> (4 * k)) & 0xFu) * kPipeBlockBytes);
        __syncwarp();
        if (mine && pb >= 0) {
          tma_load_2d(sm.keys[slot][lane & 3][0], &tmap, 0, static_cast<int>(pb * rows_per_block), &sm.full[slot]);
          bulk_load(sm.scales[slot][lane & 3], a.pool + static_cast<int64_t>(pb) * a.block_stride + kIdxBlockBytesKeys,
                    kBlock * 4, &sm.full[slot]);
        }
        ++s;
      }
    }
    // no copy may be in flight when the CTA exits
    if (lane == 0)
      for (int j = max(0, s - kPipeSlots); j < s; ++j)
        mbar_wait_bounded(&sm.full[j % kPipeSlots], static_cast<uint32_t>(j / kPipeSlots) & 1u, fault_word,
                          kFaultIndexerWait);
    return;
  }

  // ------------------------------------------------------------ compute warps
  const int g = lane >> 2, c = lane & 3;
  uint32_t bq[8][NT][2];
  float wh[NT][2];
  int cur_b = -1, ctx = 0;
  int s = 0;
  for (int64_t item = it_begin; item < it_end; ++item) {
    const int b = static_cast<int>(item / n_chunk);
    const int chunk = static_cast<int>(item - static_cast<int64_t>(b) * n_chunk);
    if (b != cur_b) {
      // the request's query (B fragments, K permuted like the keys) and head weights
      cur_b = b;
      ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const uint16_t* qh = a.q + (static_cast<int64_t>(b) * a.n_heads + 8 * n + g) * kIdxDim;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + 32 * q + 8 * c));
          bq[2 * q][n][0] = bf16pair_to_f16x2(v.x);
          bq[2 * q][n][1] = bf16pair_to_f16x2(v.y);
          bq[2 * q + 1][n][0] = bf16pair_to_f16x2(v.z);
          bq[2 * q + 1][n][1] = bf16pair_to_f16x2(v.w);
        }
        const float* wb = a.w + static_cast<int64_t>(b) * a.n_heads;
        wh[n][0] = __ldg(wb + 8 * n + 2 * c);
        wh[n][1] = __ldg(wb + 8 * n + 2 * c + 1);
      }
    }
    if (chunk * kPipeChunk >= ctx) continue;
    const int slot = s % kPipeSlots;
    const bool ok = mbar_wait_or_abort(&sm.full[slot], static_cast<uint32_t>(s / kPipeSlots) & 1u, &sm.abort_flag,
                                       fault_word, kFaultIndexerWait);
    if (!__all_sync(0xFFFFFFFFu, ok)) {
      if (lane == 0) sm.abort_flag = 1;
      break;
    }
    float* out_row = a.scores + static_cast<int64_t>(b) * a.scores_stride;
    const int t_base = chunk * kPipeChunk;
#pragma unroll 1
    for (int p = 0; p < 2; ++p) {
      // tiles (row group `warp` of blocks 2p and 2p + 1)
      const int blk0 = 2 * p, blk1 = 2 * p + 1;
      const int r0 = 16 * warp + g;  // tile rows r0 and r0 + 8; (r & 7) == g
      const int pb0 = sm.pblk[slot][blk0], pb1 = sm.pblk[slot][blk1];
      float acc0[NT][4], acc1[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc0[n][e] = acc1[n][e] = 0.f;
      const uint8_t* k00 = sm.keys[slot][blk0][r0];
      const uint8_t* k01 = sm.keys[slot][blk0][r0 + 8];
      const uint8_t* k10 = sm.keys[slot][blk1][r0];
      const uint8_t* k11 = sm.keys[slot][blk1][r0 + 8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int off = (((2 * q + (c >> 1)) ^ g) << 4) + 8 * (c & 1);
        const uint2 u00 = *reinterpret_cast<const uint2*>(k00 + off);
        const uint2 u01 = *reinterpret_cast<const uint2*>(k01 + off);
        const uint2 u10 = *reinterpret_cast<const uint2*>(k10 + off);
        const uint2 u11 = *reinterpret_cast<const uint2*>(k11 + off);
        uint32_t x00[2], x01[2], y00[2], y01[2], x10[2], x11[2], y10[2], y11[2];
        e4m3x4_to_f16x2x2(u00.x, x00);
        e4m3x4_to_f16x2x2(u01.x, x01);
        e4m3x4_to_f16x2x2(u00.y, y00);
        e4m3x4_to_f16x2x2(u01.y, y01);
        e4m3x4_to_f16x2x2(u10.x, x10);
        e4m3x4_to_f16x2x2(u11.x, x11);
        e4m3x4_to_f16x2x2(u10.y, y10);
        e4m3x4_to_f16x2x2(u11.y, y11);
        const uint32_t A00[4] = {x00[0], x01[0], x00[1], x01[1]};
        const uint32_t A01[4] = {y00[0], y01[0], y00[1], y01[1]};
        const uint32_t A10[4] = {x10[0], x11[0], x10[1], x11[1]};
        const uint32_t A11[4] = {y10[0], y11[0], y10[1], y11[1]};
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_f16(acc0[n], A00, bq[2 * q][n][0], bq[2 * q][n][1]);
          mma_f16(acc1[n], A10, bq[2 * q][n][0], bq[2 * q][n][1]);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          mma_f16(acc0[n], A01, bq[2 * q + 1][n][0], bq[2 * q + 1][n][1]);
          mma_f16(acc1[n], A11, bq[2 * q + 1][n][0], bq[2 * q + 1][n][1]);
        }
      }
      // sum_h w_h * relu(s_t * dot): this lane holds heads 8n + 2c + {0,1}
#pragma unroll
      for (int tt = 0; tt < 2; ++tt) {
        const int blk = tt ? blk1 : blk0;
        const int pbk = tt ? pb1 : pb0;
        const float(&acc)[NT][4] = tt ? acc1 : acc0;
        const float s0 = sm.scales[slot][blk][r0];
        const float s1 = sm.scales[slot][blk][r0 + 8];
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          p0 += wh[n][0] * fmaxf(s0 * acc[n][0], 0.f) + wh[n][1] * fmaxf(s0 * acc[n][1], 0.f);
          p1 += wh[n][0] * fmaxf(s1 * acc[n][2], 0.f) + wh[n][1] * fmaxf(s1 * acc[n][3], 0.f);
        }
        p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 1);
        p0 += __shfl_xor_sync(0xFFFFFFFFu, p0, 2);
        p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 1);
        p1 += __shfl_xor_sync(0xFFFFFFFFu, p1, 2);
        const int t0 = t_base + blk * kBlock + r0;
        if (c == 0 && pbk != -2) {  // -2: the whole block lies past the context
          if (t0 < ctx) out_row[t0] = pbk >= 0 ? p0 : -INFINITY;
          if (t0 + 8 < ctx) out_row[t0 + 8] = pbk >= 0 ? p1 : -INFINITY;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
    ++s;
  }
}

// ----------------------------------------------------------------- top-k
constexpr int kTopkThreads = 1024;
constexpr int kHistBins = 2048;

__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);  // -0.0 + 0.0 = +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Adds 1 to hist[bin] with one shared atomic per distinct bin in the warp.
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
  const uint32_t mask = __ballot_sync(0xFFFFFFFFu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(mask, bin);
  if ((__ffs(peers) - 1) == static_cast<int>(threadIdx.x & 31)) atomicAdd(hist + bin, __popc(peers));
}

// Block-wide exclusive prefix sum of one value per thread; also returns the total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, s, off);
      if (lane >= off) s += y;
    }
    warp_sums[lane] = s;  // inclusive
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

// Given hist[2048] (count per bin) and `need` (>= 1) elements still to pick
// among them, find the bin holding the need-th largest element.  Returns the
// bin; *need_in_bin = how many of that bin's elements are taken.
__device__ __forceinline__ uint32_t select_bin(const uint32_t* hist, uint32_t need, uint32_t* warp_sums,
                                               uint32_t* sel_bin, uint32_t* sel_need) {
  // Thread i owns bins in descending order: 2047 - 2i and 2046 - 2i.
  const int i = threadIdx.x;
  const uint32_t hA = hist[kHistBins - 1 - 2 * i], hB = hist[kHistBins - 2 - 2 * i];
  uint32_t total;
  const uint32_t above = block_exclusive_scan(hA + hB, warp_sums, &total);  // elements in higher bins
  if (above < need && above + hA >= need) {
    *sel_bin = kHistBins - 1 - 2 * i;
    *sel_need = need - above;
  } else if (above + hA < need && above + hA + hB >= need) {
    *sel_bin = kHistBins - 2 - 2 * i;
    *sel_need = need - above - hA;
  }
  __syncthreads();
  return *sel_bin;
}

// Sample-select parameters: a strided sample of kSample keys fixes a
// threshold T0 expected to keep ~2.5 k elements; one order-preserving pass
// collects every element >= T0 into per-warp lists (warp w scans a contiguous
// chunk, so concatenating the lists keeps index order); the exact selection
// then runs on the candidates in shared memory.  If a list overflows or fewer
// than k elements reach T0, the kernel falls back to radix passes over the
// whole row.
constexpr int kSample = 2048;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kWarpCap = 512;
constexpr int kCandCap = kWarpCap * kTopkWarps;  // 16,384 candidates

struct TopkSmem {
  uint32_t cand_key[kCandCap];
  int32_t cand_idx[kCandCap];
  uint32_t sample[kSample];
  uint32_t hist[kHistBins];
  uint32_t warp_sums[32];
  uint32_t warp_cnt[32];
  uint32_t warp_off[32];
  uint32_t sel_bin, sel_need, run_gt, run_eq;
};

// Exact selection over `count` elements given in ascending index order by
// `src(j) -> (order key, index)`: three radix passes find the k-th largest key
// T and how many ties at T are taken, then an ordered compaction writes every
// element with key > T and the lowest-index ties, ascending, to orow[0..k).
template <class Src>
__device__ void select_and_compact(const Src& src, int count, int topk, int32_t* orow, TopkSmem& sm) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, need = topk;
  const int shifts[3] = {21, 10, 0};
  const uint32_t widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    for (int j = tid; j < kHistBins; j += kTopkThreads) sm.hist[j] = 0;
    __syncthreads();
    const int sh = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int hi_shift = sh + static_cast<int>(widths[pass]);
    for (int base = 0; base < count; base += 4 * kTopkThreads) {
      uint32_t key[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = base + u * kTopkThreads + tid;
        key[u] = j < count ? src.key(j) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = base + u * kTopkThreads + tid;
        const bool match = j < count && (pass == 0 || (key[u] >> hi_shift) == prefix);
        hist_add(sm.hist, (key[u] >> sh) & bmask, match);
      }
    }
    __syncthreads();
    if (tid == 0) sm.sel_bin = sm.sel_need = 0;
    __syncthreads();
    const uint32_t bin = select_bin(sm.hist, need, sm.warp_sums, &sm.sel_bin, &sm.sel_need);
    need = sm.sel_need;
    prefix = (pass == 0) ? bin : ((prefix << widths[pass]) | bin);
    __syncthreads();
  }
  const uint32_t T = prefix;
  // element j goes to position G(j) + min(E(j), need), G / E counting keys > T / == T before j
  if (tid == 0) sm.run_gt = sm.run_eq = 0;
  __syncthreads();
  constexpr int kPer = 4;
  for (int base = 0; base < count; base += kTopkThreads * kPer) {
    uint32_t keys[kPer];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = base + tid * kPer + i;
      keys[i] = j < count ? src.key(j) : 0u;
      ngt += (j < count && keys[i] > T);
      neq += (j < count && keys[i] == T);
    }
    uint32_t tot;
    const uint32_t packed = block_exclusive_scan((ngt << 16) | neq, sm.warp_sums, &tot);
    uint32_t G = sm.run_gt + (packed >> 16), E = sm.run_eq + (packed & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = base + tid * kPer + i;
      if (j >= count) break;
      if (keys[i] > T) {
        orow[G + min(E, need)] = src.idx(j);
        ++G;
      } else if (keys[i] == T) {
        if (E < need) orow[G + E] = src.idx(j);
        ++E;
      }
    }
    __syncthreads();
    if (tid == 0) {
      sm.run_gt += tot >> 16;
      sm.run_eq += tot & 0xFFFFu;
    }
    __syncthreads();
  }
}

struct RowSrc {
  const float* row;
  __device__ uint32_t key(int j) const { return order_key(__ldg(row + j)); }
  __device__ int32_t idx(int j) const { return j; }
};
struct CandSrc {
  const TopkSmem* sm;
  __device__ uint32_t key(int j) const { return sm->cand_key[j]; }
  __device__ int32_t idx(int j) const { return sm->cand_idx[j]; }
};

// ---- parallel candidate collection: kParts CTAs per request ---------------
// Every part CTA draws the same strided sample of the whole row and takes
// the same threshold T0 from it (two radix passes over the sample give the
// lower bound of the 22-bit key bin holding the sample's r0-th largest key);
// it then collects its part's elements with key >= T0, in index order, into
// global memory.  The selection kernel concatenates the parts in order.
constexpr int kParts = 8;
constexpr int kPartThreads = 256;
constexpr int kPartWarps = kPartThreads / 32;
constexpr int kPartCap = kCandCap / kParts;          // 2,048 candidates per part
constexpr int kPartWarpCap = kPartCap / kPartWarps;  // 256 per warp

struct CollectSmem {
  uint32_t hist[kHistBins];
  uint32_t cand_key[kPartCap];
  int32_t cand_idx[kPartCap];
  uint32_t scan[kPartWarps];
  uint32_t warp_cnt[kPartWarps];
  uint32_t sel_bin, sel_need;
};

// The bin holding the need-th largest element of hist[] (descending), with
// 256 threads owning 8 bins each; *need_in_bin as in select_bin.
__device__ __forceinline__ uint32_t select_bin_256(const uint32_t* hist, uint32_t need, CollectSmem& sm) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t h[8], sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    h[k] = hist[kHistBins - 1 - 8 * t - k];
    sum += h[k];
  }
  uint32_t x = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sm.scan[warp] = x;
  __syncthreads();
  uint32_t acc = x - sum;
  for (int w = 0; w < warp; ++w) acc += sm.scan[w];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (acc < need && acc + h[k] >= need) {
      sm.sel_bin = kHistBins - 1 - 8 * t - k;
      sm.sel_need = need - acc;
    }
    acc += h[k];
  }
  __syncthreads();
  return sm.sel_bin;
}

__global__ void __launch_bounds__(kPartThreads)
    topk_collect_kernel(const float* __restrict__ scores, int64_t row_stride, const int32_t* __restrict__ ctx_lens,
                        int topk, int max_ctx, uint32_t* __restrict__ cand_key, int32_t* __restrict__ cand_idx,
                        int32_t* __restrict__ cand_cnt) {
  __shared__ CollectSmem sm;
  const int part = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = max(0, min(__ldg(ctx_lens + b), max_ctx));
  if (n <= topk) return;  // the selection kernel takes everything
  const float* row = scores + static_cast<int64_t>(b) * row_stride;

  // 1. Threshold from the strided sample of the whole row.
  uint32_t key[kSample / kPartThreads];
#pragma unroll
  for (int u = 0; u < kSample / kPartThreads; ++u) {
    const int i = tid + u * kPartThreads;
    key[u] = order_key(__ldg(row + static_cast<int>((static_cast<int64_t>(i) * n) / kSample)));
  }
  const int r0 = min(kSample - 1, static_cast<int>((2.5 * topk * kSample) / n) + 8);
  uint32_t need = r0 + 1, prefix = 0;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    for (int j = tid; j < kHistBins; j += kPartThreads) sm.hist[j] = 0;
    if (tid == 0) sm.sel_bin = sm.sel_need = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kSample / kPartThreads; ++u) {
      if (pass == 0) hist_add(sm.hist, key[u] >> 21, true);
      else hist_add(sm.hist, (key[u] >> 10) & 0x7FFu, (key[u] >> 21) == prefix);
    }
    __syncthreads();
    const uint32_t bin = select_bin_256(sm.hist, need, sm);
    need = sm.sel_need;
    prefix = pass == 0 ? bin : ((prefix << 11) | bin);
    __syncthreads();
  }
  const uint32_t T0 = prefix << 10;  // lower bound of the selected 22-bit bin

  // 2. Collect this part's elements >= T0, order-preserving per warp chunk.
  const int chunk = (n + kParts - 1) / kParts;
  const int lo = part * chunk, hi = min(n, lo + chunk);
  const int wchunk = (max(0, hi - lo) + kPartWarps - 1) / kPartWarps;
  const int wlo = lo + warp * wchunk, whi = min(hi, wlo + wchunk);
  uint32_t cnt = 0;
  constexpr int kBatch = 8;  // independent loads in flight per lane
  for (int base = wlo; base < whi; base += 32 * kBatch) {
    uint32_t k[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = base + 32 * u + lane;
      k[u] = j < whi ? order_key(__ldg(row + j)) : 0u;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = base + 32 * u + lane;
      const bool take = j < whi && k[u] >= T0;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, take);
      const uint32_t pos = cnt + __popc(m & ((1u << lane) - 1u));
      if (take && pos < kPartWarpCap) {
        sm.cand_key[warp * kPartWarpCap + pos] = k[u];
        sm.cand_idx[warp * kPartWarpCap + pos] = j;
      }
      cnt += __popc(m);
    }
  }
  if (lane == 0) sm.warp_cnt[warp] = cnt;
  __syncthreads();
  uint32_t off = 0, total = 0;
  bool overflow = false;
  for (int w = 0; w < kPartWarps; ++w) {
    if (w == warp) off = total;
    total += sm.warp_cnt[w];
    overflow |= sm.warp_cnt[w] > static_cast<uint32_t>(kPartWarpCap);
  }
  const int64_t slot = static_cast<int64_t>(b) * kParts + part;
  if (overflow) {
    if (tid == 0) cand_cnt[slot] = -1;  // the selection kernel falls back to the whole row
    return;
  }
  for (uint32_t e = lane; e < cnt; e += 32) {
    cand_key[slot * kPartCap + off + e] = sm.cand_key[warp * kPartWarpCap + e];
    cand_idx[slot * kPartCap + off + e] = sm.cand_idx[warp * kPartWarpCap + e];
  }
  if (tid == 0) cand_cnt[slot] = static_cast<int32_t>(total);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t row_stride,
                                                            const int32_t* __restrict__ ctx_lens, int topk,
                                                            int max_ctx, const uint32_t* __restrict__ cand_key,
                                                            const int32_t* __restrict__ cand_idx,
                                                            const int32_t* __restrict__ cand_cnt,
                                                            int32_t* __restrict__ out) {
  extern __shared__ __align__(16) uint8_t topk_smem_raw[];
  TopkSmem& sm = *reinterpret_cast<TopkSmem*>(topk_smem_raw);
  const int b = blockIdx.x;
  const int n = max(0, min(__ldg(ctx_lens + b), max_ctx));
  const float* row = scores + static_cast<int64_t>(b) * row_stride;
  int32_t* orow = out + static_cast<int64_t>(b) * topk;
  const int tid = threadIdx.x;

  if (n <= topk) {  // everything is selected
    for (int j = tid; j < topk; j += kTopkThreads) orow[j] = j < n ? j : -1;
    return;
  }
  // The parts' candidate lists, concatenated in part order (index order kept).
  const int64_t slot0 = static_cast<int64_t>(b) * kParts;
  int cnt[kParts];
  int total = 0;
  bool overflow = false;
#pragma unroll
  for (int p = 0; p < kParts; ++p) {
    cnt[p] = __ldg(cand_cnt + slot0 + p);
    overflow |= cnt[p] < 0;
    total += max(cnt[p], 0);
  }
  if (overflow || total < topk) {
    // Rare: the sample threshold kept too many or too few: exact selection
    // over the whole row.
    select_and_compact(RowSrc{row}, n, topk, orow, sm);
    return;
  }
  int off = 0;
#pragma unroll
  for (int p = 0; p < kParts; ++p) {
    for (int e = tid; e < cnt[p]; e += kTopkThreads) {
      sm.cand_key[off + e] = __ldg(cand_key + (slot0 + p) * kPartCap + e);
      sm.cand_idx[off + e] = __ldg(cand_idx + (slot0 + p) * kPartCap + e);
    }
    off += cnt[p];
  }
  __syncthreads();
  select_and_compact(CandSrc{&sm}, total, topk, orow, sm);
}

}  // namespace

size_t topk_workspace_bytes(int batch, int, int) {
  if (batch <= 0) return 0;
  const size_t lists = static_cast<size_t>(batch) * kParts * kPartCap * sizeof(uint32_t);
  return 2 * ((lists + 255) / 256 * 256) + (static_cast<size_t>(batch) * kParts * sizeof(int32_t) + 255) / 256 * 256;
}

cudaError_t launch_topk(const float* scores, int64_t row_stride, const int32_t* context_lens, int batch, int topk,
                        int max_context_len, int32_t* out, void* workspace, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  if (workspace == nullptr) return cudaErrorInvalidValue;
  const size_t lists = (static_cast<size_t>(batch) * kParts * kPartCap * sizeof(uint32_t) + 255) / 256 * 256;
  uint32_t* cand_key = static_cast<uint32_t*>(workspace);
  int32_t* cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + lists);
  int32_t* cand_cnt = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + 2 * lists);
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(topk_kernel),
                                      static_cast<int>(sizeof(TopkSmem)), &configured);
  if (e != cudaSuccess) return e;
  topk_collect_kernel<<<dim3(kParts, batch), kPartThreads, 0, stream>>>(scores, row_stride, context_lens, topk,
                                                                       max_context_len, cand_key, cand_idx, cand_cnt);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_kernel<<<batch, kTopkThreads, sizeof(TopkSmem), stream>>>(scores, row_stride, context_lens, topk,
                                                                  max_context_len, cand_key, cand_idx, cand_cnt, out);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_idx_pipe(const IdxArgs& a, const CUtensorMap& map, unsigned int* fw, cudaStream_t stream) {
  const size_t smem = sizeof(IdxPipeSmem) + 1024;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(indexer_scores_pipe_kernel<NT>),
                                      static_cast<int>(smem), &configured);
  if (e != cudaSuccess) return e;
  const int64_t n_items = static_cast<int64_t>(a.batch) * ((a.max_ctx + kPipeChunk - 1) / kPipeChunk);
  const int64_t grid = std::min<int64_t>(n_items, 2 * static_cast<int64_t>(device_sm_count()));
  indexer_scores_pipe_kernel<NT><<<static_cast<unsigned>(grid), kPipeThreads, smem, stream>>>(a, map, fw);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_idx_tma(const IdxArgs& a, const CUtensorMap& map, unsigned int* fw, dim3 grid, size_t smem,
                           cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(indexer_scores_tma_kernel<NT>),
                                      static_cast<int>(smem), &configured);
  if (e != cudaSuccess) return e;
  indexer_scores_tma_kernel<NT><<<grid, kIdxWarps * 32, smem, stream>>>(a, map, fw);
  return cudaGetLastError();
}

cudaError_t launch_indexer_scores(const uint16_t* q_idx, const float* head_w, const void* key_pool,
                                  int64_t block_stride, int64_t num_blocks, const int32_t* block_table,
                                  int max_blocks_per_req, const int32_t* context_lens, int batch, int n_heads,
                                  int max_context_len, float* scores, int64_t scores_stride, cudaStream_t stream) {
  if (batch <= 0 || max_context_len <= 0) return cudaSuccess;
  IdxArgs a;
  a.q = q_idx;
  a.w = head_w;
  a.pool = static_cast<const uint8_t*>(key_pool);
  a.block_stride = block_stride;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.ctx_lens = context_lens;
  a.scores = scores;
  a.scores_stride = scores_stride;
  a.max_blocks = max_blocks_per_req;
  a.n_heads = n_heads;
  a.max_ctx = max_context_len;
  a.batch = batch;
  dim3 grid((max_context_len + kIdxTokensPerCta - 1) / kIdxTokensPerCta, batch);
  CUtensorMap map;
  const int64_t rows = num_blocks * (block_stride / kIdxDim);
  unsigned int* fw = fault_word_ptr();
  if (fw != nullptr && num_blocks > 0 && block_stride % kIdxDim == 0 && rows <= 0x7FFFFFFF &&
      encode_tensor_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, key_pool, kIdxDim, rows, kIdxDim, kIdxDim, kBlock,
                           CU_TENSOR_MAP_SWIZZLE_128B)) {
    const size_t smem = sizeof(IdxSmem) + 1024;
    switch (n_heads / 8) {
      case 1: return launch_idx_pipe<1>(a, map, fw, stream);
      case 2: return launch_idx_pipe<2>(a, map, fw, stream);
      case 4: return launch_idx_pipe<4>(a, map, fw, stream);
      case 8: return launch_idx_tma<8>(a, map, fw, grid, smem, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (n_heads / 8) {
    case 1: indexer_scores_kernel<1><<<grid, kIdxWarps * 32, 0, stream>>>(a); break;
    case 2: indexer_scores_kernel<2><<<grid, kIdxWarps * 32, 0, stream>>>(a); break;
    case 4: indexer_scores_kernel<4><<<grid, kIdxWarps * 32, 0, stream>>>(a); break;
    case 8: indexer_scores_kernel<8><<<grid, kIdxWarps * 32, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mla
