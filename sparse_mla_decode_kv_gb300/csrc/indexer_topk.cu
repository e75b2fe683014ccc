// Indexer score and exact top-k selection.
//
// "GLM-5.3 PCP/DCP long-context on H200", section 1: an indexer scores every
// earlier token and sparse MLA attends to the 2,048 it picks; section 3:
// indexer keys are 128 FP8 values plus a 4-byte scale per token.  The score
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
// topk_kernel: one 1,024-thread CTA per request.  Scores map to order-
// preserving 32-bit keys (with -0.0 folded into +0.0); three histogram
// passes over 11 + 11 + 10 key bits find the k-th largest key T and how
// many ties at T are taken; a final pass writes every index with key > T and
// the lowest-index ties, in ascending index order, using block-wide prefix
// counts.  The scores stay L2-resident between passes.
#include <cuda_fp16.h>

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
__global__ void __launch_bounds__(kIdxWarps * 32) indexer_scores_kernel(const IdxArgs a) {
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
  for (int mt = warp; mt < n_mt; mt += kIdxWarps) {
    const int t0 = t_begin + 16 * mt + g;
    const int t1 = t0 + 8;
    if (t_begin + 16 * mt >= ctx) break;
    float s0 = 0.f, s1 = 0.f;
    const uint8_t* k0 = key_row(a, bt_row, t0, ctx, &s0);
    const uint8_t* k1 = key_row(a, bt_row, t1, ctx, &s1);
    uint2 v0[4], v1[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v0[q] = k0 ? __ldg(reinterpret_cast<const uint2*>(k0 + 32 * q + 8 * c)) : make_uint2(0, 0);
      v1[q] = k1 ? __ldg(reinterpret_cast<const uint2*>(k1 + 32 * q + 8 * c)) : make_uint2(0, 0);
    }
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t A0[4] = {e4m3x2_to_f16x2(v0[q].x), e4m3x2_to_f16x2(v1[q].x), e4m3x2_to_f16x2(v0[q].x >> 16),
                        e4m3x2_to_f16x2(v1[q].x >> 16)};
      uint32_t A1[4] = {e4m3x2_to_f16x2(v0[q].y), e4m3x2_to_f16x2(v1[q].y), e4m3x2_to_f16x2(v0[q].y >> 16),
                        e4m3x2_to_f16x2(v1[q].y >> 16)};
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
      if (t0 < ctx) out_row[t0] = k0 ? p0 : -INFINITY;
      if (t1 < ctx) out_row[t1] = k1 ? p1 : -INFINITY;
    }
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

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ scores, int64_t row_stride,
                                                            const int32_t* __restrict__ ctx_lens, int topk,
                                                            int max_ctx, int32_t* __restrict__ out) {
  __shared__ uint32_t hist[kHistBins];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t sel_bin, sel_need;
  __shared__ uint32_t run_gt, run_eq;
  const int b = blockIdx.x;
  const int n = max(0, min(__ldg(ctx_lens + b), max_ctx));
  const float* row = scores + static_cast<int64_t>(b) * row_stride;
  int32_t* orow = out + static_cast<int64_t>(b) * topk;
  const int tid = threadIdx.x;

  if (n <= topk) {  // everything is selected
    for (int j = tid; j < topk; j += kTopkThreads) orow[j] = j < n ? j : -1;
    return;
  }

  // Three radix passes: key bits [31:21], [20:10], [9:0].
  uint32_t prefix = 0, need = topk;
  const int shifts[3] = {21, 10, 0};
  const uint32_t widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    for (int j = tid; j < kHistBins; j += kTopkThreads) hist[j] = 0;
    __syncthreads();
    const int sh = shifts[pass];
    const uint32_t bmask = (1u << widths[pass]) - 1u;
    const int hi_shift = sh + static_cast<int>(widths[pass]);  // bits above this pass must equal `prefix`
    for (int base = 0; base < n; base += kTopkThreads) {
      const int j = base + tid;
      const bool in = j < n;
      const uint32_t key = in ? order_key(__ldg(row + j)) : 0u;
      const bool match = in && (pass == 0 || (key >> hi_shift) == prefix);
      hist_add(hist, (key >> sh) & bmask, match);
    }
    __syncthreads();
    if (tid == 0) sel_bin = sel_need = 0;
    __syncthreads();
    const uint32_t bin = select_bin(hist, need, warp_sums, &sel_bin, &sel_need);
    need = sel_need;
    prefix = (pass == 0) ? bin : ((prefix << widths[pass]) | bin);
    __syncthreads();
  }
  const uint32_t T = prefix;  // the k-th largest key; `need` ties at T are taken

  // Compaction in index order: element j goes to position G(j) + min(E(j), need)
  // where G / E count the keys > T / == T before j.
  if (tid == 0) run_gt = run_eq = 0;
  __syncthreads();
  constexpr int kPer = 4;
  for (int base = 0; base < n; base += kTopkThreads * kPer) {
    uint32_t keys[kPer];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = base + tid * kPer + i;
      keys[i] = j < n ? order_key(__ldg(row + j)) : 0u;
      ngt += (j < n && keys[i] > T);
      neq += (j < n && keys[i] == T);
    }
    uint32_t tot;
    const uint32_t packed = block_exclusive_scan((ngt << 16) | neq, warp_sums, &tot);
    uint32_t G = run_gt + (packed >> 16), E = run_eq + (packed & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = base + tid * kPer + i;
      if (j >= n) break;
      if (keys[i] > T) {
        orow[G + min(E, need)] = j;
        ++G;
      } else if (keys[i] == T) {
        if (E < need) orow[G + E] = j;
        ++E;
      }
    }
    __syncthreads();
    if (tid == 0) {
      run_gt += tot >> 16;
      run_eq += tot & 0xFFFFu;
    }
    __syncthreads();
  }
}

}  // namespace

size_t topk_workspace_bytes(int, int, int) { return 0; }

cudaError_t launch_topk(const float* scores, int64_t row_stride, const int32_t* context_lens, int batch, int topk,
                        int max_context_len, int32_t* out, void*, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  topk_kernel<<<batch, kTopkThreads, 0, stream>>>(scores, row_stride, context_lens, topk, max_context_len, out);
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
  dim3 grid((max_context_len + kIdxTokensPerCta - 1) / kIdxTokensPerCta, batch);
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
