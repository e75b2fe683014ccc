// Indexer score and exact top-k selection.
//
// "GLM-5.3 PCP/DCP long-context on H200", section 1: the indexer rates all
// preceding tokens and attention reads only the 2,048 best; section 3: an
// indexer key is 128 e4m3 bytes and a float scale.  The score
// is sum_h w_h * relu(s_t * (q_h . k_t)).
//
// Three score kernels, by the key pool's stride and the number of heads:
//  * indexer_scores_tc_kernel (key blocks TMA can tile, 32 or 64 heads): a
//    persistent grid; a producer warp loads 128-token chunks of key tiles
//    into a ring, the products run on the tcgen05 tensor cores with e4m3
//    operands (keys as stored, the query split into two e4m3 parts) and
//    accumulators in tensor memory, and four warps apply relu, the token
//    scale and the head weights, one token per thread.
//  * indexer_scores_pipe_kernel (TMA-tileable pools, 8 or 16 heads): the
//    same persistent ring, products on mma.sync with the query in registers.
//  * indexer_scores_kernel (other strides): one CTA = 4 warps over 512 tokens
//    of one request, keys loaded straight from the paged pool one m-tile
//    ahead, mma.sync.
// The two mma.sync kernels take the query as FP16 after scaling each head by
// a power of two 2^k (its largest magnitude into [2^14, 2^15)) and its weight
// by 2^-k, which leaves every score unchanged (relu is positively
// homogeneous) and keeps the whole bf16 range.
// All are HBM-bound at 132 bytes per token.
//
// Top-k in two kernels.  Scores map to order-preserving 32-bit keys (with
// -0.0 folded into +0.0).  topk_collect_kernel: 8 CTAs per request each draw
// the same sample of 2,048 keys of the whole row (256 runs of 8), take from it a
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

__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t two, float mul) {
  return f32x2_to_f16x2_sat(bf16_bits_to_f32(two & 0xFFFFu) * mul, bf16_bits_to_f32(two >> 16) * mul);
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

// The query of request b as mma.sync B fragments (K = 128 dims permuted like
// the keys, N = 8 NT heads) in FP16, and the head weights of this lane's
// epilogue heads (8n + 2c, 8n + 2c + 1).  The bf16 query does not fit FP16's
// exponent range in general, so each head is scaled by a power of two 2^k
// that brings its largest magnitude into [2^14, 2^15) and its weight by 2^-k:
// w relu(s 2^k dot) 2^-k = w relu(s dot), exactly.  Lane (g, c) holds dims
// 32q + 8c .. + 8 of head 8n + g; the four lanes of a head reduce its maximum.
template <int NT>
__device__ __forceinline__ void load_query_fragments(const IdxArgs& a, int b, int g, int c,
                                                     uint32_t (&bq)[8][NT][2], float (&wh)[NT][2]) {
  const float* wb = a.w + static_cast<int64_t>(b) * a.n_heads;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const uint16_t* qh = a.q + (static_cast<int64_t>(b) * a.n_heads + 8 * n + g) * kIdxDim;
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldg(reinterpret_cast<const uint4*>(qh + 32 * q + 8 * c));
    uint32_t m = max(max(bf16x8_absmax_bits(v[0]), bf16x8_absmax_bits(v[1])),
                     max(bf16x8_absmax_bits(v[2]), bf16x8_absmax_bits(v[3])));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    const int k = query_shift(m);
    const float mul = pow2f(k);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      bq[2 * q][n][0] = bf16pair_to_f16x2(v[q].x, mul);
      bq[2 * q][n][1] = bf16pair_to_f16x2(v[q].y, mul);
      bq[2 * q + 1][n][0] = bf16pair_to_f16x2(v[q].z, mul);
      bq[2 * q + 1][n][1] = bf16pair_to_f16x2(v[q].w, mul);
    }
    // the shifts of heads 8n + 2c and 8n + 2c + 1 (held by lanes 4 (2c) and 4 (2c + 1))
    const int k0 = __shfl_sync(0xFFFFFFFFu, k, 8 * c);
    const int k1 = __shfl_sync(0xFFFFFFFFu, k, 8 * c + 4);
    wh[n][0] = __ldg(wb + 8 * n + 2 * c) * pow2f(-k0);
    wh[n][1] = __ldg(wb + 8 * n + 2 * c + 1) * pow2f(-k1);
  }
}

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

template <int NT>  // n-tiles of 8 heads (64 heads: two CTAs per SM, their query fragments take 128 registers)
__global__ void __launch_bounds__(kIdxWarps * 32, NT == 8 ? 2 : 3) indexer_scores_kernel(const IdxArgs a) {
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
  load_query_fragments<NT>(a, b, g, c, bq, wh);

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
      load_query_fragments<NT>(a, b, g, c, bq, wh);
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

// Tensor-memory variant (TMA key tiles, 32 or 64 index heads): the products
// run on the fifth-generation tensor cores with 8-bit operands, the keys
// straight from the TMA tiles.  The bf16 query of head h is scaled by a
// power of two 2^k_h that brings its largest magnitude into [128, 256) and
// split into two e4m3 parts, hi = e4m3(q 2^k_h) and lo = e4m3(q 2^k_h - hi):
// a bf16 value has 8 significant bits and each part 4, so hi + lo is exact
// for every element of at least 2^-2 (after scaling), and within 2^-10 (the
// e4m3 subnormal step) for the smaller ones.  B = [hi rows; lo rows], N = 2
// x heads, so one MMA chain gives both partial dot products of every head:
// D[t, h] + D[t, H + h] = 2^k_h (q_h . k_t) for the 128 tokens t of a chunk
// (M = 128, four K = 32 steps over the 128 dims).  Roles: warp 4 loads key
// tiles and scales into a three-slot ring (as the pipelined kernel); warp 5
// owns the tensor memory (two accumulators of N columns) and one of its
// lanes issues the MMAs; warps 0-3 -- tensor-memory lanes 0-127, one token
// each -- read the accumulator, apply relu, the token scale and the head
// weights (times 2^-k_h), store the score, and write the split query when
// the request changes.
constexpr int kTcIdxChunk = 128;                    // tokens per chunk = MMA M
constexpr int kTcIdxBlocks = kTcIdxChunk / kBlock;  // 2 key blocks
constexpr int kTcIdxSlots = 3;
// CTAs per SM: three for 32 heads (60 KB of shared memory and 128
// tensor-memory columns each); two for 64 heads, whose 256 columns per CTA
// would not fit three times in an SM's 512.
__host__ __device__ constexpr int tc_idx_ctas_per_sm(int heads) { return heads <= 32 ? 3 : 2; }
constexpr int kTcIdxEpiWarps = 4;
constexpr int kTcIdxThreads = (kTcIdxEpiWarps + 2) * 32;
constexpr int kTcIdxItemsPerLookup = 32 / kTcIdxBlocks;

template <int H>
struct alignas(1024) TcIdxSmem {
  uint8_t keys[kTcIdxSlots][kTcIdxBlocks][kBlock][kIdxDim];  // 16 KB per slot, 128-byte swizzle (TMA)
  uint8_t qop[2 * H][kIdxDim];  // B operand: rows 0..H-1 hi parts, H..2H-1 lo parts, 128-byte swizzle
  float scales[kTcIdxSlots][kTcIdxBlocks][kBlock];
  float wq[H];  // w_h * 2^-k_h
  int32_t pblk[kTcIdxSlots][kTcIdxBlocks];  // physical block; -1: outside the pool (-inf); -2: past the context
  uint64_t raw_full[kTcIdxSlots], raw_empty[kTcIdxSlots], acc_full[2], acc_empty[2], b_ready;
  uint32_t tmem_base;
  int abort_flag;
};

template <int H>
__global__ void __launch_bounds__(kTcIdxThreads, tc_idx_ctas_per_sm(H))
    indexer_scores_tc_kernel(const IdxArgs a, const __grid_constant__ CUtensorMap tmap, unsigned int* fault_word) {
  constexpr int N = 2 * H;                                  // accumulator columns per chunk
  constexpr uint32_t kCols = 2 * N;                         // two accumulators
  constexpr uint32_t kIdesc = umma_idesc_f32acc(kTcIdxChunk, N, 0, 0);  // e4m3 x e4m3 -> f32
  static_assert(N % 16 == 0 && N <= 256 && (kCols & (kCols - 1)) == 0, "tensor-memory shape");
  extern __shared__ uint8_t idx_smem_raw[];
  TcIdxSmem<H>& sm =
      *reinterpret_cast<TcIdxSmem<H>*>(idx_smem_raw + ((1024u - (smem_u32(idx_smem_raw) & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_chunk = (a.max_ctx + kTcIdxChunk - 1) / kTcIdxChunk;
  const int64_t n_items = static_cast<int64_t>(a.batch) * n_chunk;
  const int64_t per = (n_items + gridDim.x - 1) / gridDim.x;
  const int64_t it_begin = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t it_end = min(n_items, it_begin + per);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcIdxSlots; ++i) {
      mbar_init(&sm.raw_full[i], 1);
      mbar_init(&sm.raw_empty[i], kTcIdxEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], kTcIdxEpiWarps);
    }
    mbar_init(&sm.b_ready, kTcIdxEpiWarps);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kTcIdxEpiWarps + 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  const uint32_t tbase = sm.tmem_base;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait_or_abort(bar, parity, &sm.abort_flag, fault_word, kFaultIndexerWait);
    if (!ok) *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
    return ok;
  };

  if (warp == kTcIdxEpiWarps) {
    // ------------------------------------------------------------ producer
    const int64_t rows_per_block = a.block_stride / kIdxDim;
    int s = 0;
    bool stop = false;
    for (int64_t base = it_begin; base < it_end && !stop; base += kTcIdxItemsPerLookup) {
      const int64_t item = base + lane / kTcIdxBlocks;  // lane l: block l % 2 of item base + l / 2
      int pb = -2;
      bool live = false;
      if (item < it_end) {
        const int b = static_cast<int>(item / n_chunk);
        const int chunk = static_cast<int>(item - static_cast<int64_t>(b) * n_chunk);
        const int ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
        live = chunk * kTcIdxChunk < ctx;
        const int lb = chunk * kTcIdxBlocks + lane % kTcIdxBlocks;
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
      for (int k = 0; k < kTcIdxItemsPerLookup; ++k) {
        if (!((live_mask >> (kTcIdxBlocks * k)) & 1u)) continue;  // empty item (past the context)
        const int slot = s % kTcIdxSlots;
        bool ok = true;
        if (lane == 0 && s >= kTcIdxSlots) ok = wait(&sm.raw_empty[slot], static_cast<uint32_t>(s / kTcIdxSlots - 1) & 1u);
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) {
          stop = true;
          break;
        }
        const bool mine = lane / kTcIdxBlocks == k;
        const int j = lane % kTcIdxBlocks;
        if (mine) sm.pblk[slot][j] = pb;
        __syncwarp();
        if (lane == 0)
          mbar_expect_tx(&sm.raw_full[slot], __popc((valid_mask >> (kTcIdxBlocks * k)) & 3u) * (kIdxBlockBytesKeys + kBlock * 4));
        __syncwarp();
        if (mine && pb >= 0) {
          tma_load_2d(sm.keys[slot][j][0], &tmap, 0, static_cast<int>(pb * rows_per_block), &sm.raw_full[slot]);
          bulk_load(sm.scales[slot][j], a.pool + static_cast<int64_t>(pb) * a.block_stride + kIdxBlockBytesKeys,
                    kBlock * 4, &sm.raw_full[slot]);
        }
        ++s;
      }
    }
    // no copy may be in flight when the CTA leaves
    if (lane == 0)
      for (int j = max(0, s - kTcIdxSlots); j < s; ++j)
        mbar_wait_bounded(&sm.raw_full[j % kTcIdxSlots], static_cast<uint32_t>(j / kTcIdxSlots) & 1u, fault_word,
                          kFaultIndexerWait);
  } else if (warp == kTcIdxEpiWarps + 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint64_t b_desc = umma_desc_sw128(smem_u32(sm.qop));
      int s = 0, cur_b = -1, cur_ctx_b = -1, ctx = 0, changes = 0;
      for (int64_t item = it_begin; item < it_end; ++item) {
        const int b = static_cast<int>(item / n_chunk);
        const int chunk = static_cast<int>(item - static_cast<int64_t>(b) * n_chunk);
        if (b != cur_ctx_b) {
          cur_ctx_b = b;
          ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
        }
        if (chunk * kTcIdxChunk >= ctx) continue;
        if (b != cur_b) {  // the epilogue warps have written this request's split query
          if (!wait(&sm.b_ready, static_cast<uint32_t>(changes) & 1u)) break;
          ++changes;
          cur_b = b;
        }
        const int slot = s % kTcIdxSlots, acc = s & 1;
        if (!wait(&sm.raw_full[slot], static_cast<uint32_t>(s / kTcIdxSlots) & 1u)) break;
        if (s >= 2 && !wait(&sm.acc_empty[acc], static_cast<uint32_t>(s / 2 - 1) & 1u)) break;
        tcgen05_fence_after();
        const uint64_t a_desc = umma_desc_sw128(smem_u32(sm.keys[slot][0][0]));
#pragma unroll
        for (int kk = 0; kk < kIdxDim / 32; ++kk)  // K = 32 e4m3 values = 32 bytes per step: +2 in the address field
          umma_f8(tbase + static_cast<uint32_t>(acc * N), a_desc + 2 * kk, b_desc + 2 * kk, kIdesc, kk > 0);
        umma_commit(&sm.acc_full[acc]);
        ++s;
      }
      // every MMA issued above has completed once the last commit has arrived
      if (s > 0)
        mbar_wait_bounded(&sm.acc_full[(s - 1) & 1], static_cast<uint32_t>((s - 1) / 2) & 1u, fault_word,
                          kFaultIndexerWait);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- epilogue (warps 0-3)
    const int t = threadIdx.x;  // token row of the chunk = tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    int s = 0, cur_b = -1, cur_ctx_b = -1, ctx = 0;
    // After a timed-out wait the warp keeps walking its items without waiting
    // or computing, so that every epilogue warp still meets the barriers of
    // the query rewrites.
    bool aborted = false;
    for (int64_t item = it_begin; item < it_end; ++item) {
      const int b = static_cast<int>(item / n_chunk);
      const int chunk = static_cast<int>(item - static_cast<int64_t>(b) * n_chunk);
      if (b != cur_ctx_b) {
        cur_ctx_b = b;
        ctx = min(__ldg(a.ctx_lens + b), a.max_ctx);
      }
      if (chunk * kTcIdxChunk >= ctx) continue;
      if (b != cur_b) {
        // The split query of request b.  Every MMA of earlier requests has
        // completed (this warp waited for all their accumulators) and the MMA
        // lane waits for b_ready before the next one, so B can be rewritten.
        cur_b = b;
        for (int u = t; u < H * 4; u += kTcIdxEpiWarps * 32) {
          const int h = u >> 2, qd = u & 3;  // head h, dims 32 qd .. 32 qd + 31 (lanes 4g .. 4g+3 share h)
          const uint4* qh = reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.n_heads + h) * kIdxDim +
                                                           32 * qd);
          uint4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = __ldg(qh + i);
          uint32_t m = max(max(bf16x8_absmax_bits(v[0]), bf16x8_absmax_bits(v[1])),
                           max(bf16x8_absmax_bits(v[2]), bf16x8_absmax_bits(v[3])));
          m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
          m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
          // largest |q| into [128, 256): k = 7 - exponent (a subnormal maximum counts as -127)
          const int k = m == 0 ? 0 : min(126, max(-120, 7 - (static_cast<int>(m >> 7) - 127)));
          const float mul = pow2f(k);
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int p = 0; p < 2; ++p) {  // four values -> one word of hi and one of lo
              const float f0 = bf16_bits_to_f32(w4[2 * p] & 0xFFFFu) * mul;
              const float f1 = bf16_bits_to_f32(w4[2 * p] >> 16) * mul;
              const float f2 = bf16_bits_to_f32(w4[2 * p + 1] & 0xFFFFu) * mul;
              const float f3 = bf16_bits_to_f32(w4[2 * p + 1] >> 16) * mul;
              const uint32_t hw = f32x2_to_e4m3x2(f1, f0) | (f32x2_to_e4m3x2(f3, f2) << 16);
              uint32_t back[2];
              e4m3x4_to_f16x2x2(hw, back);
              const float2 b01 = __half22float2(*reinterpret_cast<const __half2*>(&back[0]));
              const float2 b23 = __half22float2(*reinterpret_cast<const __half2*>(&back[1]));
              hi[2 * i + p] = hw;
              lo[2 * i + p] = f32x2_to_e4m3x2(f1 - b01.y, f0 - b01.x) | (f32x2_to_e4m3x2(f3 - b23.y, f2 - b23.x) << 16);
            }
          }
          // bytes 32 qd .. 32 qd + 31 of rows h (hi) and H + h (lo): 16-byte
          // chunks 2 qd and 2 qd + 1, at chunk ^ (row % 8) (128-byte swizzle)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int ch = 2 * qd + c;
            *reinterpret_cast<uint4*>(&sm.qop[h][(ch ^ (h & 7)) * 16]) =
                make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
            *reinterpret_cast<uint4*>(&sm.qop[H + h][(ch ^ ((H + h) & 7)) * 16]) =
                make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
          }
          if (qd == 0) sm.wq[h] = __ldg(a.w + static_cast<int64_t>(b) * a.n_heads + h) * pow2f(-k);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.b_ready);
        named_bar_sync(1, kTcIdxEpiWarps * 32);  // every head weight written before any epilogue reads it
      }
      if (aborted) continue;
      const int slot = s % kTcIdxSlots, acc = s & 1;
      bool ok = wait(&sm.acc_full[acc], static_cast<uint32_t>(s / 2) & 1u);
      // the producer's block ids and scales of this slot (already complete)
      ok = ok && wait(&sm.raw_full[slot], static_cast<uint32_t>(s / kTcIdxSlots) & 1u);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        aborted = true;
        continue;
      }
      tcgen05_fence_after();
      const int blk = t / kBlock, r = t % kBlock;
      const float st = sm.scales[slot][blk][r];
      float score = 0.f;
#pragma unroll
      for (int hg = 0; hg < H; hg += 32) {
        uint32_t hv[32], lv[32];
        tmem_load_32cols(tbase + lane_base + static_cast<uint32_t>(acc * N + hg), hv);
        tmem_load_32cols(tbase + lane_base + static_cast<uint32_t>(acc * N + H + hg), lv);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          score += sm.wq[hg + j] * fmaxf(st * (__uint_as_float(hv[j]) + __uint_as_float(lv[j])), 0.f);
      }
      tcgen05_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[acc]);
      const int pb = sm.pblk[slot][blk];
      const int tok = chunk * kTcIdxChunk + t;
      if (pb != -2 && tok < ctx)
        a.scores[static_cast<int64_t>(b) * a.scores_stride + tok] = pb >= 0 ? score : -INFINITY;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.raw_empty[slot]);
      ++s;
    }
  }

  // ---- teardown: every copy and MMA has completed (the producer and the MMA
  // lane waited for them); free the tensor memory
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  if (warp == kTcIdxEpiWarps + 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kCols) : "memory");
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

// Selection kernel: the candidates every collection CTA kept (keys >= the
// sample threshold T0, in index order) are concatenated in shared memory and
// the exact selection runs on them.  If a list overflowed or fewer than k
// elements reached T0, it falls back to radix passes over the whole row.
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kWarpCap = 512;
constexpr int kCandCap = kWarpCap * kTopkWarps;  // 16,384 candidates

struct TopkSmem {
  uint32_t cand_key[kCandCap];
  int32_t cand_idx[kCandCap];
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
  // The passes resolve the k-th largest key 11, 11 and 10 bits at a time.
  // Once the bin holding it contains exactly the `need` elements still to
  // take, every element of the bin is taken and its lower bits do not
  // matter: the selection stops there (prefix compared at `t_shift`).
  int t_shift = 0;
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
    const bool whole_bin = sm.hist[bin] == need;
    t_shift = sh;
    __syncthreads();
    if (whole_bin) break;
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
      keys[i] = j < count ? (src.key(j) >> t_shift) : 0u;
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
// Every part CTA draws the same sample of the whole row and takes
// the same threshold T0 from it (two radix passes over the sample give the
// lower bound of the 22-bit key bin holding the sample's r0-th largest key);
// it then collects its part's elements with key >= T0, in index order, into
// global memory.  The selection kernel concatenates the parts in order.
constexpr int kParts = 8;
constexpr int kPartThreads = 256;
constexpr int kPartWarps = kPartThreads / 32;
constexpr int kPartCap = kCandCap / kParts;          // 2,048 candidates per part
constexpr int kPartWarpCap = kPartCap / kPartWarps;  // 256 per warp
constexpr int kCollectSample = 2048;  // sample of the row that sets the threshold (256 runs of 8)

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
  // The selection kernel is launched as a programmatic dependent of this
  // one: it may become resident now and waits for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int part = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = max(0, min(__ldg(ctx_lens + b), max_ctx));
  if (n <= topk) return;  // the selection kernel takes everything
  const float* row = scores + static_cast<int64_t>(b) * row_stride;

  // 1. Threshold from a sample of the whole row: 256 runs of 8 consecutive
  // scores spread evenly over it.  Eight lanes read one run (one 32-byte
  // sector), so the sample costs 256 sector requests per CTA rather than
  // 2,048 scattered ones (all parts of a request draw the same sample).
  uint32_t key[kCollectSample / kPartThreads];
  {
    constexpr int kRuns = kCollectSample / 8;
#pragma unroll
    for (int u = 0; u < kCollectSample / kPartThreads; ++u) {
      const int r = (tid >> 3) + (kPartThreads / 8) * u;
      const int pos = static_cast<int>((static_cast<int64_t>(r) * n) / kRuns) & ~7;
      key[u] = order_key(__ldg(row + min(pos + (tid & 7), n - 1)));
    }
  }
  const int r0 = min(kCollectSample - 1, static_cast<int>((2.5 * topk * kCollectSample) / n) + 8);
  uint32_t need = r0 + 1, prefix = 0;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    for (int j = tid; j < kHistBins; j += kPartThreads) sm.hist[j] = 0;
    if (tid == 0) sm.sel_bin = sm.sel_need = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kCollectSample / kPartThreads; ++u) {
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
  // A programmatic dependent of the collection kernel: nothing is read
  // before that grid has completed and its candidate lists are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  // Candidate j of the concatenation lies in the last part whose start is
  // <= j; each thread issues all its loads before storing any (one L2 round
  // trip for the whole list instead of one per part).
  int start[kParts];
  start[0] = 0;
#pragma unroll
  for (int p = 1; p < kParts; ++p) start[p] = start[p - 1] + cnt[p - 1];
  constexpr int kLoadsPerThread = 4;
  for (int base = 0; base < total; base += kLoadsPerThread * kTopkThreads) {
    uint32_t kv[kLoadsPerThread];
    int32_t iv[kLoadsPerThread];
#pragma unroll
    for (int u = 0; u < kLoadsPerThread; ++u) {
      const int j = base + u * kTopkThreads + tid;
      int p = 0;
#pragma unroll
      for (int q = 1; q < kParts; ++q) p += j >= start[q];
      const int64_t src = (slot0 + p) * kPartCap + (j - start[p]);
      kv[u] = j < total ? __ldg(cand_key + src) : 0u;
      iv[u] = j < total ? __ldg(cand_idx + src) : 0;
    }
#pragma unroll
    for (int u = 0; u < kLoadsPerThread; ++u) {
      const int j = base + u * kTopkThreads + tid;
      if (j < total) {
        sm.cand_key[j] = kv[u];
        sm.cand_idx[j] = iv[u];
      }
    }
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
  // the selection as a programmatic dependent: its launch overlaps the tail
  // of the collection (it waits for the whole grid before reading)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = sizeof(TopkSmem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, topk_kernel, scores, row_stride, context_lens, topk, max_context_len,
                         static_cast<const uint32_t*>(cand_key), static_cast<const int32_t*>(cand_idx),
                         static_cast<const int32_t*>(cand_cnt), out);
  return e != cudaSuccess ? e : cudaGetLastError();
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

template <int H>
cudaError_t launch_idx_tc(const IdxArgs& a, const CUtensorMap& map, unsigned int* fw, cudaStream_t stream) {
  const size_t smem = sizeof(TcIdxSmem<H>) + 1024;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(indexer_scores_tc_kernel<H>),
                                      static_cast<int>(smem), &configured);
  if (e != cudaSuccess) return e;
  const int64_t n_items = static_cast<int64_t>(a.batch) * ((a.max_ctx + kTcIdxChunk - 1) / kTcIdxChunk);
  const int64_t grid =
      std::min<int64_t>(n_items, tc_idx_ctas_per_sm(H) * static_cast<int64_t>(device_sm_count()));
  indexer_scores_tc_kernel<H><<<static_cast<unsigned>(grid), kTcIdxThreads, smem, stream>>>(a, map, fw);
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
    switch (n_heads / 8) {
      case 1: return launch_idx_pipe<1>(a, map, fw, stream);
      case 2: return launch_idx_pipe<2>(a, map, fw, stream);
      case 4: return launch_idx_tc<32>(a, map, fw, stream);
      case 8: return launch_idx_tc<64>(a, map, fw, stream);
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
