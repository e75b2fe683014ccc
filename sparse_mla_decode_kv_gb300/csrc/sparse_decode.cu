// Absorbed-form sparse MLA decode over the paged NVFP4 (352-byte) or FP8
// (576-byte) latent cache, plus the split-K log-sum-exp merge.
//
// What it computes: "Prime Inference: serving GLM-5.3 to agents is a
// KV-cache problem", section "A kernel that reads four bits directly" -- one
// kernel reads the selected 352-byte rows, unpacks them on chip and scores,
// soft-maxes and blends them with FP16 operands and FP32 accumulation; -1
// entries of the top-k list are skipped rather than read.  The value vector
// is the 512-value latent itself (absorbed form: every row serves all heads,
// "GLM-5.3 PCP/DCP long-context on H200", section 6).
//
// Design on sm_103a (the page's GB200 kernel is prior art, not a blueprint):
//
//  * One CTA = one request x 16 heads x one contiguous slice of its top-k
//    list.  Warp 4 is the producer: each lane resolves one selected row
//    through the block table and issues one cp.async.bulk copy of the whole
//    row (352 or 576 bytes, 16-byte aligned) into a 4-stage shared-memory
//    ring; rows that are masked (-1, past the context, bad block id) are
//    zero-filled instead of read.  Stage completion is an mbarrier with
//    transaction bytes.
//  * Warps 0-3 consume 16-row m-tiles.  Warp w owns latent dims
//    [128w, 128w+128) and rope dims [16w, 16w+16): it unpacks only those
//    bytes, straight into mma.sync A fragments (cvt e2m1x2 / e4m3x2 -> f16x2,
//    times the group's e4m3 scale; the products are exact in FP16), and
//    computes its partial Q.K^T with the 16 heads' absorbed query held in
//    registers as B fragments.  The four partial score tiles are summed
//    through shared memory; warp w then owns the online softmax of heads
//    [4w, 4w+4) and publishes P (f16) and the rescale factors.
//  * P.V reuses the same A fragments: the transpose of each 8x8 tile
//    (movmatrix) is exactly the B fragment of the [tokens x dims] value
//    operand, so every stored value is unpacked once per CTA.  Warp w keeps
//    O[16 heads x its 128 dims] in 64 fp32 registers.
//  * The K dimension inside each 32-dim chunk is permuted so that one
//    4-byte (NVFP4) or 8-byte (FP8) shared load per row feeds two k-steps;
//    the query fragments use the same permutation and the output is written
//    back in natural order.
//  * When a request's list is split over several CTAs, each writes its
//    normalised partial output and base-2 LSE to the workspace and a small
//    merge kernel combines them (the pages merge in-cluster through DSMEM;
//    this build uses a second launch).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageRows = 32;
constexpr int kStages = 4;
constexpr int kHeadsPerCta = 16;
constexpr int kMaxRows = 2048;  // rows of one CTA's slice (top-k <= 2048)
constexpr int kRedPitch = 24;  // floats per token row of the partial-score exchange
constexpr int kPPitch = 24;    // halfs per head row of P (48 bytes: ldmatrix conflict-free)
constexpr float kLn2 = 0.6931471805599453f;

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {
  static constexpr int kRowBytes = kRowNvfp4;
  static constexpr int kPitch = kRowNvfp4 + 16;  // 368: conflict-free fragment loads
  static constexpr int kRopeOff = kRopeOffNvfp4;
};
template <>
struct Fmt<1> {
  static constexpr int kRowBytes = kRowFp8;
  static constexpr int kPitch = kRowFp8 + 16;  // 592
  static constexpr int kRopeOff = kRopeOffFp8;
};

template <int FMT>
struct alignas(128) Smem {
  uint8_t rows[kStages][kStageRows][Fmt<FMT>::kPitch];
  float red[kConsumerWarps][16][kRedPitch];
  __half pbuf[kHeadsPerCta][kPPitch];
  float alpha[kHeadsPerCta];
  float mfin[kHeadsPerCta];
  float lfin[kHeadsPerCta];
  int32_t tok_all[kMaxRows];  // token of each row of the slice, -1 if masked
  int32_t pb_all[kMaxRows];   // its physical block
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort_flag;
};

struct DecodeArgs {
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  const uint8_t* pool;
  int64_t block_stride;
  int64_t num_blocks;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  uint16_t* out;
  float* lse;
  float* part_o;    // [B*H, splits, 512] (splits > 1)
  float* part_lse;  // [B*H, splits], base-2
  int max_blocks;
  int topk;
  int num_heads;
  int splits;
  int rows_per_split;
  float scale_log2;  // softmax_scale * log2(e)
  unsigned int* fault_word;
};

__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t two) {
  return f32x2_to_f16x2_sat(bf16_bits_to_f32(two & 0xFFFFu), bf16_bits_to_f32(two >> 16));
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) sparse_decode_kernel(const DecodeArgs args) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<FMT>& sm = *reinterpret_cast<Smem<FMT>*>(smem_raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x / args.splits;
  const int sp = blockIdx.x % args.splits;
  const int hg = blockIdx.y;
  const int row_begin = sp * args.rows_per_split;
  const int row_end = min(args.topk, row_begin + args.rows_per_split);
  const int n_rows = max(0, row_end - row_begin);
  const int n_stages = (n_rows + kStageRows - 1) / kStageRows;
  const int ctx = __ldg(args.ctx_lens + b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Resolve the rows of the slice: the first kStages stages first (so their
    // copies can start one index + one block-table round trip after launch),
    // then the rest while those copies are in flight.  Loads are batched so
    // that each lane has up to 8 independent requests outstanding.
    const int32_t* topk_row = args.topk_idx + static_cast<int64_t>(b) * args.topk + row_begin;
    const int32_t* bt_row = args.block_table + static_cast<int64_t>(b) * args.max_blocks;
    const int n_slots = n_stages * kStageRows;
    auto resolve = [&](int lo, int hi) {
      for (int base = lo; base < hi; base += 8 * 32) {
        int t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = base + u * 32 + lane;
          t[u] = (j < hi && j < n_rows) ? __ldg(topk_row + j) : -1;
        }
        int pb[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool ok = t[u] >= 0 && t[u] < ctx && t[u] / kBlock < args.max_blocks;
          pb[u] = ok ? __ldg(bt_row + t[u] / kBlock) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = base + u * 32 + lane;
          const bool ok = pb[u] >= 0 && pb[u] < args.num_blocks;
          if (j < hi) {
            sm.tok_all[j] = ok ? t[u] : -1;
            sm.pb_all[j] = ok ? pb[u] : -1;
          }
        }
      }
    };
    const int first = min(n_slots, kStages * kStageRows);
    resolve(0, first);
    __syncwarp();
    int issued = 0;
    for (int it = 0; it < n_stages; ++it) {
      const int slot = it % kStages;
      const uint32_t round = it / kStages;
      const bool ok = mbar_wait_bounded(&sm.empty[slot], (round & 1u) ^ 1u, args.fault_word, kFaultDecodeWait);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;  // warp-uniform decision
      const int j = it * kStageRows + lane;
      const int t = sm.tok_all[j];
      uint8_t* dst = sm.rows[slot][lane];
      if (t < 0) {
#pragma unroll
        for (int i = 0; i < F::kRowBytes / 16; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
      }
      const uint32_t valid = __ballot_sync(0xFFFFFFFFu, t >= 0);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], __popc(valid) * F::kRowBytes);
      __syncwarp();
      if (t >= 0) {
        const uint8_t* src = args.pool + static_cast<int64_t>(sm.pb_all[j]) * args.block_stride +
                             static_cast<int64_t>(t % kBlock) * F::kRowBytes;
        bulk_g2s(dst, src, F::kRowBytes, &sm.full[slot]);
      }
      issued = it + 1;
      if (it == min(n_stages, kStages) - 1 && n_slots > first) {
        resolve(first, n_slots);  // the remaining rows, behind the first copies
        __syncwarp();
      }
    }
    // Never leave with copies in flight: wait for the last stages issued.
    for (int it = max(0, issued - kStages); it < issued; ++it)
      mbar_wait_bounded(&sm.full[it % kStages], (static_cast<uint32_t>(it / kStages)) & 1u, args.fault_word, kFaultDecodeWait);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2;
  const int c = lane & 3;
  const int w = warp;

  // Absorbed query as B fragments (K = this warp's 144 dims, N = 16 heads).
  uint32_t bq[9][2][2];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int h = hg * kHeadsPerCta + 8 * n + g;
    const uint16_t* qn = args.q_nope + (static_cast<int64_t>(b) * args.num_heads + h) * kLatent;
    const uint16_t* qr = args.q_rope + (static_cast<int64_t>(b) * args.num_heads + h) * kRope;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(qn + 128 * w + 32 * q + 8 * c));
      bq[2 * q][n][0] = bf16pair_to_f16x2(v.x);
      bq[2 * q][n][1] = bf16pair_to_f16x2(v.y);
      bq[2 * q + 1][n][0] = bf16pair_to_f16x2(v.z);
      bq[2 * q + 1][n][1] = bf16pair_to_f16x2(v.w);
    }
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(qr + 16 * w + 4 * c));
    bq[8][n][0] = bf16pair_to_f16x2(r.x);
    bq[8][n][1] = bf16pair_to_f16x2(r.y);
  }

  float o[8][2][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[ks][be][e] = 0.f;

  // Online-softmax state of the two heads this lane tracks as head owner.
  const int hown = 4 * w + 2 * (lane & 1);
  const int tloc = lane >> 1;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  bool aborted = false;

  for (int it = 0; it < n_stages && !aborted; ++it) {
    const int slot = it % kStages;
    const uint32_t round = it / kStages;
    const bool ok = mbar_wait_bounded(&sm.full[slot], round & 1u, args.fault_word, kFaultDecodeWait);
    if (!__all_sync(0xFFFFFFFFu, ok) && lane == 0) sm.abort_flag = 1;  // all warps leave after the next barrier
    const uint8_t* base = sm.rows[slot][0];

#pragma unroll 1
    for (int mt = 0; mt < 2; ++mt) {
      const uint8_t* row0 = base + (16 * mt + g) * F::kPitch;
      const uint8_t* row1 = row0 + 8 * F::kPitch;
      uint32_t a[9][4];
      if constexpr (FMT == 0) {
        // Scales of groups 8w + 2q + (c>>1), q = 0..3: one 8-byte load per row,
        // two byte permutes, two conversions, then {S, S} duplicates.
        const uint32_t sel = (c >> 1) ? 0x3131u : 0x2020u;
        const uint2 sw0 = *reinterpret_cast<const uint2*>(row0 + kScaleOff + 8 * w);
        const uint2 sw1 = *reinterpret_cast<const uint2*>(row1 + kScaleOff + 8 * w);
        const uint32_t s0_01 = e4m3x2_to_f16x2(__byte_perm(sw0.x, 0, sel));
        const uint32_t s0_23 = e4m3x2_to_f16x2(__byte_perm(sw0.y, 0, sel));
        const uint32_t s1_01 = e4m3x2_to_f16x2(__byte_perm(sw1.x, 0, sel));
        const uint32_t s1_23 = e4m3x2_to_f16x2(__byte_perm(sw1.y, 0, sel));
        const uint32_t sc0[4] = {__byte_perm(s0_01, 0, 0x1010), __byte_perm(s0_01, 0, 0x3232),
                                 __byte_perm(s0_23, 0, 0x1010), __byte_perm(s0_23, 0, 0x3232)};
        const uint32_t sc1[4] = {__byte_perm(s1_01, 0, 0x1010), __byte_perm(s1_01, 0, 0x3232),
                                 __byte_perm(s1_23, 0, 0x1010), __byte_perm(s1_23, 0, 0x3232)};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = 64 * w + 16 * q + 4 * c;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(row0 + off);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(row1 + off);
          const uint32_t s0 = sc0[q];
          const uint32_t s1 = sc1[q];
          a[2 * q][0] = hmul2(e2m1x2_to_f16x2(w0 & 0xFFu), s0);
          a[2 * q][1] = hmul2(e2m1x2_to_f16x2(w1 & 0xFFu), s1);
          a[2 * q][2] = hmul2(e2m1x2_to_f16x2((w0 >> 8) & 0xFFu), s0);
          a[2 * q][3] = hmul2(e2m1x2_to_f16x2((w1 >> 8) & 0xFFu), s1);
          a[2 * q + 1][0] = hmul2(e2m1x2_to_f16x2((w0 >> 16) & 0xFFu), s0);
          a[2 * q + 1][1] = hmul2(e2m1x2_to_f16x2((w1 >> 16) & 0xFFu), s1);
          a[2 * q + 1][2] = hmul2(e2m1x2_to_f16x2(w0 >> 24), s0);
          a[2 * q + 1][3] = hmul2(e2m1x2_to_f16x2(w1 >> 24), s1);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = 128 * w + 32 * q + 8 * c;
          const uint2 v0 = *reinterpret_cast<const uint2*>(row0 + off);
          const uint2 v1 = *reinterpret_cast<const uint2*>(row1 + off);
          a[2 * q][0] = e4m3x2_to_f16x2(v0.x);
          a[2 * q][1] = e4m3x2_to_f16x2(v1.x);
          a[2 * q][2] = e4m3x2_to_f16x2(v0.x >> 16);
          a[2 * q][3] = e4m3x2_to_f16x2(v1.x >> 16);
          a[2 * q + 1][0] = e4m3x2_to_f16x2(v0.y);
          a[2 * q + 1][1] = e4m3x2_to_f16x2(v1.y);
          a[2 * q + 1][2] = e4m3x2_to_f16x2(v0.y >> 16);
          a[2 * q + 1][3] = e4m3x2_to_f16x2(v1.y >> 16);
        }
      }
      {
        const int off = F::kRopeOff + 16 * w + 4 * c;
        const uint32_t x0 = *reinterpret_cast<const uint32_t*>(row0 + off);
        const uint32_t x1 = *reinterpret_cast<const uint32_t*>(row1 + off);
        a[8][0] = e4m3x2_to_f16x2(x0);
        a[8][1] = e4m3x2_to_f16x2(x1);
        a[8][2] = e4m3x2_to_f16x2(x0 >> 16);
        a[8][3] = e4m3x2_to_f16x2(x1 >> 16);
      }

      // Partial scores over this warp's 144 dims: S^T [16 tokens x 16 heads].
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      float sodd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // second chain: shorter dependency
#pragma unroll
      for (int ks = 0; ks < 9; ks += 2) {
        mma_f16(sacc[0], a[ks], bq[ks][0][0], bq[ks][0][1]);
        mma_f16(sacc[1], a[ks], bq[ks][1][0], bq[ks][1][1]);
        if (ks + 1 < 9) {
          mma_f16(sodd[0], a[ks + 1], bq[ks + 1][0][0], bq[ks + 1][0][1]);
          mma_f16(sodd[1], a[ks + 1], bq[ks + 1][1][0], bq[ks + 1][1][1]);
        }
      }
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[n][e] += sodd[n][e];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        *reinterpret_cast<float2*>(&sm.red[w][g][8 * n + 2 * c]) = make_float2(sacc[n][0], sacc[n][1]);
        *reinterpret_cast<float2*>(&sm.red[w][g + 8][8 * n + 2 * c]) = make_float2(sacc[n][2], sacc[n][3]);
      }
      named_bar_sync(1, kConsumerWarps * 32);
      if (sm.abort_flag) {
        aborted = true;
        break;
      }

      // Head owner: heads hown, hown+1 for token tloc of this m-tile.
      {
        float2 s = *reinterpret_cast<const float2*>(&sm.red[0][tloc][hown]);
#pragma unroll
        for (int ww = 1; ww < kConsumerWarps; ++ww) {
          const float2 v = *reinterpret_cast<const float2*>(&sm.red[ww][tloc][hown]);
          s.x += v.x;
          s.y += v.y;
        }
        const bool valid = sm.tok_all[it * kStageRows + 16 * mt + tloc] >= 0;
        float z[2] = {valid ? s.x * args.scale_log2 : -INFINITY, valid ? s.y * args.scale_log2 : -INFINITY};
        __half ph[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = z[e];
#pragma unroll
          for (int off = 2; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
          const float m_new = fmaxf(m_run[e], mx);
          const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run[e] - m_new);
          const float p = (z[e] == -INFINITY) ? 0.f : ex2(z[e] - m_new);
          ph[e] = __float2half_rn(p);
          l_run[e] = l_run[e] * alpha + __half2float(ph[e]);
          m_run[e] = m_new;
          if (tloc == 0) sm.alpha[hown + e] = alpha;
        }
        sm.pbuf[hown][tloc] = ph[0];
        sm.pbuf[hown + 1][tloc] = ph[1];
      }
      named_bar_sync(1, kConsumerWarps * 32);

      // O[16 heads x 128 dims] += P[16 x 16 tokens] . V[16 tokens x 128 dims].
      uint32_t pa[4];
      ldmatrix_x4(pa, smem_u32(&sm.pbuf[lane & 15][(lane >> 4) * 8]));
      const float al0 = sm.alpha[g];
      const float al1 = sm.alpha[g + 8];
      if (__any_sync(0xFFFFFFFFu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
#pragma unroll
          for (int be = 0; be < 2; ++be) {
            o[ks][be][0] *= al0;
            o[ks][be][1] *= al0;
            o[ks][be][2] *= al1;
            o[ks][be][3] *= al1;
          }
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_f16(o[ks][0], pa, movmatrix_t(a[ks][0]), movmatrix_t(a[ks][1]));
        mma_f16(o[ks][1], pa, movmatrix_t(a[ks][2]), movmatrix_t(a[ks][3]));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);
  }
  if (aborted) return;

  // ---------------------------------------------------------------- finish
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float l = l_run[e];
#pragma unroll
    for (int off = 2; off < 32; off <<= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
    if (tloc == 0) {
      sm.mfin[hown + e] = m_run[e];
      sm.lfin[hown + e] = l;
    }
  }
  named_bar_sync(1, kConsumerWarps * 32);

  const int h0 = hg * kHeadsPerCta + g;  // rows g and g+8 of this thread's O fragments
  const float l0 = sm.lfin[g], l1 = sm.lfin[g + 8];
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float lse2_0 = l0 > 0.f ? sm.mfin[g] + lg2(l0) : -INFINITY;
  const float lse2_1 = l1 > 0.f ? sm.mfin[g + 8] + lg2(l1) : -INFINITY;
  const int64_t bh0 = static_cast<int64_t>(b) * args.num_heads + h0;
  const int64_t bh1 = bh0 + 8;

  if (args.splits == 1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int dim = 128 * w + 32 * q + 8 * c;
      uint32_t r0[4], r1[4];
#pragma unroll
      for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int be = 0; be < 2; ++be) {
          __nv_bfloat162 x0 = __floats2bfloat162_rn(o[2 * q + s][be][0] * inv0, o[2 * q + s][be][1] * inv0);
          __nv_bfloat162 x1 = __floats2bfloat162_rn(o[2 * q + s][be][2] * inv1, o[2 * q + s][be][3] * inv1);
          r0[2 * s + be] = *reinterpret_cast<uint32_t*>(&x0);
          r1[2 * s + be] = *reinterpret_cast<uint32_t*>(&x1);
        }
      *reinterpret_cast<uint4*>(args.out + bh0 * kLatent + dim) = make_uint4(r0[0], r0[1], r0[2], r0[3]);
      *reinterpret_cast<uint4*>(args.out + bh1 * kLatent + dim) = make_uint4(r1[0], r1[1], r1[2], r1[3]);
    }
    if (args.lse != nullptr && w == 0 && c == 0) {
      args.lse[bh0] = lse2_0 * kLn2;
      args.lse[bh1] = lse2_1 * kLn2;
    }
  } else {
    float* p0 = args.part_o + (bh0 * args.splits + sp) * kLatent;
    float* p1 = args.part_o + (bh1 * args.splits + sp) * kLatent;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int dim = 128 * w + 32 * q + 8 * c;
      *reinterpret_cast<float4*>(p0 + dim) = make_float4(o[2 * q][0][0] * inv0, o[2 * q][0][1] * inv0,
                                                        o[2 * q][1][0] * inv0, o[2 * q][1][1] * inv0);
      *reinterpret_cast<float4*>(p0 + dim + 4) = make_float4(o[2 * q + 1][0][0] * inv0, o[2 * q + 1][0][1] * inv0,
                                                            o[2 * q + 1][1][0] * inv0, o[2 * q + 1][1][1] * inv0);
      *reinterpret_cast<float4*>(p1 + dim) = make_float4(o[2 * q][0][2] * inv1, o[2 * q][0][3] * inv1,
                                                        o[2 * q][1][2] * inv1, o[2 * q][1][3] * inv1);
      *reinterpret_cast<float4*>(p1 + dim + 4) = make_float4(o[2 * q + 1][0][2] * inv1, o[2 * q + 1][0][3] * inv1,
                                                            o[2 * q + 1][1][2] * inv1, o[2 * q + 1][1][3] * inv1);
    }
    if (w == 0 && c == 0) {
      args.part_lse[bh0 * args.splits + sp] = lse2_0;
      args.part_lse[bh1 * args.splits + sp] = lse2_1;
    }
  }
}

// Combine `splits` normalised partial outputs with their base-2 LSEs:
// LSE = log2 sum_s 2^lse_s, out = sum_s 2^(lse_s - LSE) * O_s.  One CTA per
// (request, head); thread i handles dims [4i, 4i+4).
__global__ void __launch_bounds__(128) splitk_merge_kernel(const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse, int splits,
                                                           uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int64_t bh = blockIdx.x;
  const int t = threadIdx.x;
  const float* pl = part_lse + bh * splits;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, __ldg(pl + s));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx != -INFINITY) {
    const float4* src = reinterpret_cast<const float4*>(part_o + bh * splits * kLatent) + t;
    for (int s = 0; s < splits; ++s) {
      const float ws = ex2(__ldg(pl + s) - mx);
      const float4 v = __ldg(src + s * (kLatent / 4));
      wsum += ws;
      acc.x += ws * v.x;
      acc.y += ws * v.y;
      acc.z += ws * v.z;
      acc.w += ws * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out + bh * kLatent + 4 * t) =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lse != nullptr && t == 0) lse[bh] = wsum > 0.f ? (mx + lg2(wsum)) * kLn2 : -INFINITY;
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& a, int batch, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<FMT>);
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(sparse_decode_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(batch * a.splits, a.num_heads / kHeadsPerCta);
  sparse_decode_kernel<FMT><<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

DecodePlan plan_sparse_decode(int batch, int num_heads, int topk) {
  DecodePlan p{1, 0, 0};
  const int groups = batch * (num_heads / kHeadsPerCta);
  const int slots = 2 * device_sm_count();  // two CTAs per SM fit (registers, shared memory)
  int splits = groups > 0 ? slots / groups : 1;
  const int max_splits = (topk + kStageRows - 1) / kStageRows;
  splits = splits < 1 ? 1 : (splits > max_splits ? max_splits : splits);
  int rows = (topk + splits - 1) / splits;
  rows = (rows + 15) / 16 * 16;
  splits = (topk + rows - 1) / rows;
  p.splits = splits;
  p.rows_per_split = rows;
  if (splits > 1) {
    const size_t n_bh = static_cast<size_t>(batch) * num_heads;
    size_t o_bytes = n_bh * splits * kLatent * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    p.workspace = o_bytes + ((n_bh * splits * sizeof(float) + 255) / 256 * 256);
  }
  return p;
}

cudaError_t launch_sparse_decode(int fmt, const uint16_t* q_nope, const uint16_t* q_rope, const void* pool,
                                 int64_t block_stride, int64_t num_blocks, const int32_t* block_table,
                                 int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                 int batch, int num_heads, int topk, float softmax_scale, uint16_t* out, float* lse,
                                 void* workspace, const DecodePlan& plan, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  DecodeArgs a;
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.pool = static_cast<const uint8_t*>(pool);
  a.block_stride = block_stride;
  a.num_blocks = num_blocks;
  a.block_table = block_table;
  a.ctx_lens = context_lens;
  a.topk_idx = topk_idx;
  a.out = out;
  a.lse = lse;
  a.max_blocks = max_blocks_per_req;
  a.topk = topk;
  a.num_heads = num_heads;
  a.splits = plan.splits;
  a.rows_per_split = plan.rows_per_split;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.fault_word = fault_word_ptr();
  if (a.fault_word == nullptr) return cudaErrorInvalidDevicePointer;
  if (plan.splits > 1) {
    const size_t n_bh = static_cast<size_t>(batch) * num_heads;
    size_t o_bytes = n_bh * plan.splits * kLatent * sizeof(float);
    o_bytes = (o_bytes + 255) / 256 * 256;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + o_bytes);
  }
  cudaError_t e = fmt == 0 ? launch_fmt<0>(a, batch, stream) : launch_fmt<1>(a, batch, stream);
  if (e != cudaSuccess || plan.splits == 1) return e;
  const int64_t n_bh = static_cast<int64_t>(batch) * num_heads;
  splitk_merge_kernel<<<static_cast<unsigned>(n_bh), 128, 0, stream>>>(a.part_o, a.part_lse, plan.splits, out, lse);
  return cudaGetLastError();
}

}  // namespace mla
