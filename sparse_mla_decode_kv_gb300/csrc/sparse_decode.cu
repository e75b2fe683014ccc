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
//    list; four warps, all of which load, unpack and compute.  At entry the
//    CTA resolves every row of its slice (top-k index, then block table) in
//    batches of independent loads and keeps the row positions in shared
//    memory; rows that are masked (-1, past the context, logical block past
//    the table, block id outside the pool) get -1.
//  * Rows travel in stages of 32 through a ring of shared-memory slots (4
//    for NVFP4, 3 for FP8).  When the pool's block stride is a whole number
//    of rows, the pool is a 2-D tensor of rows to TMA and each warp gathers
//    its 8 rows of a stage with two 4-row tile::gather4 copies (a masked row
//    is coordinate -1 and reads zeros), one stage ahead.  Other pools use
//    16-byte cp.async from every thread, arriving on the slot's mbarrier.
//  * Warp w owns latent dims [128w, 128w+128) and rope dims [16w, 16w+16):
//    it unpacks only those bytes of both 16-row m-tiles, straight into
//    mma.sync A fragments (cvt e2m1x2 / e4m3x2 -> f16x2, times the group's
//    e4m3 scale; the products are exact in FP16), and computes its partial
//    Q.K^T against the 16 heads' absorbed query (B fragments kept in shared
//    memory in fragment order).  The four partial score tiles are summed
//    through shared memory; warp w then owns the online softmax of heads
//    [4w, 4w+4) with lane = token, and publishes P (f16) and the rescale
//    factors.  The running maximum is lazy: it is raised only when a score
//    exceeds it by more than 2^8, so most stages need no rescale.
//  * P.V reuses the same A fragments: the transpose of each 8x8 tile
//    (movmatrix) is exactly the B fragment of the [tokens x dims] value
//    operand, so every stored value is unpacked once per CTA.  Warp w keeps
//    O[16 heads x its 128 dims] in 64 fp32 registers.
//  * The K dimension inside each 32-dim chunk is permuted so that one
//    4-byte (NVFP4) or 8-byte (FP8) shared load per row feeds two k-steps;
//    the query fragments use the same permutation and the output is written
//    back in natural order.
//  * When a request's list is split over several CTAs, each writes its
//    normalised partial output (f16) and base-2 LSE to the workspace.  Up to
//    8 splits form a thread-block cluster and merge inside this kernel after
//    a cluster barrier, as the pages' kernel merges in-cluster; more splits
//    are merged by a small kernel launched as a programmatic dependent.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstring>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = kConsumerWarps * 32;  // all warps consume; warp 0 also refills stages
constexpr int kStageRows = 32;  // one stage = one phase = two 16-row m-tiles
constexpr int kHeadsPerCta = 16;
constexpr int kMaxRows = 1024;  // list entries of one CTA's slice (the plan never exceeds it)
constexpr int kRedPitch = 24;  // floats per token row of the partial-score exchange
constexpr int kPPitch = 40;    // halfs per head row of P (80 bytes: ldmatrix conflict-free)
constexpr int kKSteps = 9;     // k-steps of 16 dims per consumer warp (128 latent + 16 rope)
// Splits of one (request, head group) up to this many form a thread-block
// cluster and merge their partials inside the decode kernel.
constexpr int kMaxClusterSplits = 8;
// Lazy softmax maximum: scores are exponentiated against a reference maximum
// that is raised only when a score exceeds it by more than kLazy (base 2), so
// P stays <= 2^kLazy (fine in f16) and the common path needs no reduction.
constexpr float kLazy = 8.f;
constexpr float kLn2 = 0.6931471805599453f;

template <int FMT>
struct Fmt;
template <>
struct Fmt<0> {
  static constexpr int kRowBytes = kRowNvfp4;
  static constexpr int kPitch = kRowNvfp4 + 16;  // 368: conflict-free fragment loads
  static constexpr int kRopeOff = kRopeOffNvfp4;
  static constexpr int kStages = 4;
};
template <>
struct Fmt<1> {
  static constexpr int kRowBytes = kRowFp8;
  static constexpr int kPitch = kRowFp8 + 16;  // 592
  static constexpr int kRopeOff = kRopeOffFp8;
  static constexpr int kStages = 3;  // two CTAs per SM still fit
};

// Row pitch in the shared-memory ring: the 16-byte pad that makes the
// fragment loads conflict-free is only possible with per-chunk copies; a
// 4-row TMA gather writes its rows back to back.
template <int FMT, bool TMA>
constexpr int row_pitch() { return TMA ? Fmt<FMT>::kRowBytes : Fmt<FMT>::kPitch; }

template <int FMT, bool TMA>
struct alignas(128) Smem {
  uint8_t rows[Fmt<FMT>::kStages][kStageRows][row_pitch<FMT, TMA>()];
  uint4 qfrag[kConsumerWarps][kKSteps][32];  // query B fragments, fragment order
  float red[kConsumerWarps][kStageRows][kRedPitch];
  __half pbuf[kHeadsPerCta][kPPitch];
  float alpha[kHeadsPerCta];
  int rescale[kConsumerWarps];
  float mfin[kHeadsPerCta];
  uint32_t qmax[kConsumerWarps][kHeadsPerCta];  // per warp and head: largest |q| (bf16 magnitude bits)
  float lfin[kHeadsPerCta];
  int64_t row_off[kMaxRows];  // per row of the slice: byte offset in the pool (TMA: row index), -1 if masked
  int32_t tok_all[kMaxRows];  // token of each row of the slice, -1 if masked
  uint64_t full[Fmt<FMT>::kStages];
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
  __half* part_o;   // [B*H, splits, 512] normalised partial O in f16 (splits > 1)
  float* part_lse;  // [B*H, splits], base-2
  int max_blocks;
  int topk;
  int q_len;  // query tokens per request (1 for plain decode)
  int num_heads;
  int splits;
  int rows_per_split;
  int cluster_merge;  // 1: the splits of a (request, head group) are one cluster, merged through DSMEM
  float scale_log2;  // softmax_scale * log2(e)
  unsigned int* fault_word;
};

// Two floats to f16 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 half2_floats(uint32_t bits) {
  return __half22float2(*reinterpret_cast<const __half2*>(&bits));
}

// Two bf16 query values times 2^k (`mul`) to f16x2; exact for every value
// that lands in f16's normal range.
__device__ __forceinline__ uint32_t bf16pair_to_f16x2(uint32_t two, float mul) {
  return f32x2_to_f16x2_sat(bf16_bits_to_f32(two & 0xFFFFu) * mul, bf16_bits_to_f32(two >> 16) * mul);
}

// Cluster merge: the splits of one (request, head group) are the CTAs of a
// cluster.  Each has written its normalised partial O (f16) and base-2 LSE to
// the workspace (through L2: distributed shared memory has a fraction of L2's
// bandwidth per SM); after the cluster barrier (release/acquire at cluster
// scope) CTA r combines the 8-value units r*128 + t + k*S*128 of the 16 x 512
// output tile from every split: LSE = log2 sum_r 2^lse_r and
// out = sum_r 2^(lse_r - max) O_r / sum_r 2^(lse_r - max).
__device__ __forceinline__ void cluster_merge(const DecodeArgs& args, int v, int hg, int sp) {
  cluster_sync_all();
  const int S = args.splits;
  const int64_t bh_base = static_cast<int64_t>(v) * args.num_heads + hg * kHeadsPerCta;
  // unit u = (head u / 64, dims 8 (u % 64) .. + 8) of the 16 x 512 tile; a
  // thread loads the LSEs and partials of two units before using any (one
  // L2 round trip) and forms the split weights itself
  constexpr int kPerHead = kLatent / 8;
  constexpr int kUnits = kHeadsPerCta * kPerHead;
  const uint4* part = reinterpret_cast<const uint4*>(args.part_o);
  for (int u0 = sp * kThreads + static_cast<int>(threadIdx.x); u0 < kUnits; u0 += 2 * S * kThreads) {
    uint4 pv[2][kMaxClusterSplits];
    float ls[2][kMaxClusterSplits];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int u = u0 + i * S * kThreads;
      const int64_t row = (bh_base + u / kPerHead) * S;
#pragma unroll
      for (int r = 0; r < kMaxClusterSplits; ++r) {
        const bool in = u < kUnits && r < S;
        ls[i][r] = in ? __ldcg(args.part_lse + row + r) : -INFINITY;
        pv[i][r] = in ? __ldcg(part + (row + r) * kPerHead + u % kPerHead) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int u = u0 + i * S * kThreads;
      if (u < kUnits) {
        const int h = u / kPerHead;
        float mx = -INFINITY;
#pragma unroll
        for (int r = 0; r < kMaxClusterSplits; ++r) mx = fmaxf(mx, ls[i][r]);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float wsum = 0.f;
#pragma unroll
        for (int r = 0; r < kMaxClusterSplits; ++r) {
          const float ws = mx == -INFINITY ? 0.f : ex2(ls[i][r] - mx);  // 0 for an empty split
          wsum += ws;
          const uint32_t wd[4] = {pv[i][r].x, pv[i][r].y, pv[i][r].z, pv[i][r].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = half2_floats(wd[k]);
            acc[2 * k] += ws * f.x;
            acc[2 * k + 1] += ws * f.y;
          }
        }
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        uint32_t ob[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 x = __floats2bfloat162_rn(acc[2 * k] * inv, acc[2 * k + 1] * inv);
          ob[k] = *reinterpret_cast<const uint32_t*>(&x);
        }
        *reinterpret_cast<uint4*>(args.out + (bh_base + h) * kLatent + 8 * (u % kPerHead)) =
            make_uint4(ob[0], ob[1], ob[2], ob[3]);
        if (args.lse != nullptr && u % kPerHead == 0)
          args.lse[bh_base + h] = wsum > 0.f ? (mx + lg2(wsum)) * kLn2 : -INFINITY;
      }
    }
  }
}

// TMA = true: rows are gathered by TMA, 4 rows per instruction (the pool's
// block stride is a whole number of rows, so the pool is a 2-D tensor of
// rows); false: every thread copies 16-byte chunks with cp.async.
template <int FMT, bool TMA>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_decode_kernel(const DecodeArgs args, const __grid_constant__ CUtensorMap tmap) {
  using F = Fmt<FMT>;
  constexpr int kStages = F::kStages;
  constexpr int kPitchB = row_pitch<FMT, TMA>();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem<FMT, TMA>& sm = *reinterpret_cast<Smem<FMT, TMA>*>(smem_raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // v = (request, query token) pair: queries, list, output and partials are
  // indexed by v; the block table and context length by the request b.
  // The head groups of one slice are adjacent in the grid, so they run
  // together and all but the first read the slice's rows from L2.
  // Cluster merge: the splits of one (request, head group) are adjacent
  // instead, and the split index is the CTA's rank in its cluster.
  const int n_hg = args.num_heads / kHeadsPerCta;
  const int hg = args.cluster_merge ? (blockIdx.x / args.splits) % n_hg : blockIdx.x % n_hg;
  const int v = args.cluster_merge ? blockIdx.x / (args.splits * n_hg) : blockIdx.x / (n_hg * args.splits);
  const int b = v / args.q_len;
  const int sp = args.cluster_merge ? blockIdx.x % args.splits : (blockIdx.x / n_hg) % args.splits;
  const int row_begin = sp * args.rows_per_split;
  const int row_end = min(args.topk, row_begin + args.rows_per_split);
  const int n_rows = max(0, row_end - row_begin);
  const int n_stages = (n_rows + kStageRows - 1) / kStageRows;

  // This grid is launched as a programmatic dependent of whatever precedes it
  // on the stream: its CTAs may be resident early, but nothing is read before
  // the preceding grid has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // query token i of the request's q_len sees t < ctx_b - (q_len - 1 - i)
  const int ctx = __ldg(args.ctx_lens + b) - (args.q_len - 1 - (v - b * args.q_len));
  // The split merge (launched as a programmatic dependent) may start its
  // launch now; it waits for this whole grid before reading any partial.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], TMA ? kConsumerWarps : kThreads);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  const int g = lane >> 2;
  const int c = lane & 3;
  const int w = warp;

  // The absorbed query of this warp's dims, loaded first: it does not depend
  // on the row resolution below, so its latency overlaps it.
  const int h0 = hg * kHeadsPerCta + g;
  const uint16_t* qn0 = args.q_nope + (static_cast<int64_t>(v) * args.num_heads + h0) * kLatent + 128 * w + 8 * c;
  const uint16_t* qr0 = args.q_rope + (static_cast<int64_t>(v) * args.num_heads + h0) * kRope + 16 * w + 4 * c;
  uint4 qv0[4], qv1[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    qv0[q] = __ldg(reinterpret_cast<const uint4*>(qn0 + 32 * q));
    qv1[q] = __ldg(reinterpret_cast<const uint4*>(qn0 + 8 * kLatent + 32 * q));  // head h0 + 8
  }
  const uint2 qr_0 = __ldg(reinterpret_cast<const uint2*>(qr0));
  const uint2 qr_1 = __ldg(reinterpret_cast<const uint2*>(qr0 + 8 * kRope));

  // ---------------------------------------------------------------- rows
  // Resolve every row of the slice (top-k index, then block table) with all
  // threads, in batches of independent loads: two round trips in total.
  const int32_t* topk_row = args.topk_idx + static_cast<int64_t>(v) * args.topk + row_begin;
  const int32_t* bt_row = args.block_table + static_cast<int64_t>(b) * args.max_blocks;
  const int n_slots = n_stages * kStageRows;
  for (int base = 0; base < n_slots; base += 4 * kThreads) {
    int t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * kThreads + threadIdx.x;
      t[u] = (j < n_rows) ? __ldg(topk_row + j) : -1;
    }
    int pb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = t[u] >= 0 && t[u] < ctx && t[u] / kBlock < args.max_blocks;
      pb[u] = ok ? __ldg(bt_row + t[u] / kBlock) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = base + u * kThreads + threadIdx.x;
      const bool ok = pb[u] >= 0 && pb[u] < args.num_blocks;
      if (j < n_slots) {
        sm.tok_all[j] = ok ? t[u] : -1;
        if constexpr (TMA)
          sm.row_off[j] = ok ? static_cast<int64_t>(pb[u]) * (args.block_stride / F::kRowBytes) + t[u] % kBlock : -1;
        else
          sm.row_off[j] = ok ? static_cast<int64_t>(pb[u]) * args.block_stride +
                                   static_cast<int64_t>(t[u] % kBlock) * F::kRowBytes
                             : -1;
      }
    }
  }
  // Largest |q| of heads h0 and h0 + 8 over this warp's dims (the four lanes
  // of a row group hold disjoint dims), for the per-head power-of-two shift.
  {
    uint32_t m0 = max(bf16x2_absmax_bits(qr_0.x), bf16x2_absmax_bits(qr_0.y));
    uint32_t m1 = max(bf16x2_absmax_bits(qr_1.x), bf16x2_absmax_bits(qr_1.y));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      m0 = max(m0, bf16x8_absmax_bits(qv0[q]));
      m1 = max(m1, bf16x8_absmax_bits(qv1[q]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      m0 = max(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, off));
      m1 = max(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, off));
    }
    if (c == 0) {
      sm.qmax[w][g] = m0;
      sm.qmax[w][g + 8] = m1;
    }
  }
  __syncthreads();  // barrier init, the resolved rows and the query maxima are visible

  // Fill stage `it` into its ring slot; masked rows arrive as zeros.
  // TMA: lane 0 of every warp posts its share of the stage's bytes on
  // full[slot] and issues two 4-row gathers (rows 8w .. 8w+7).  cp.async:
  // every thread copies its 16-byte chunks, then arrives on full[slot] when
  // they land.
  constexpr int kChunks = F::kRowBytes / 16;
  auto fill_stage = [&](int it) {
    const int slot = it % kStages;
    if constexpr (TMA) {
      if (lane == 0) {
        constexpr int kWarpRows = kStageRows / kConsumerWarps;  // 8
        mbar_expect_tx(&sm.full[slot], kWarpRows * F::kRowBytes);
        const int64_t* y = sm.row_off + it * kStageRows + kWarpRows * warp;
#pragma unroll
        for (int k = 0; k < kWarpRows / 4; ++k)
          tma_gather4(sm.rows[slot][kWarpRows * warp + 4 * k], &tmap, static_cast<int>(y[4 * k]),
                      static_cast<int>(y[4 * k + 1]), static_cast<int>(y[4 * k + 2]), static_cast<int>(y[4 * k + 3]),
                      &sm.full[slot]);
      }
    } else {
      for (int i = threadIdx.x; i < kStageRows * kChunks; i += kThreads) {
        const int r = i / kChunks, k = i - (i / kChunks) * kChunks;
        const int64_t off = sm.row_off[it * kStageRows + r];
        const uint8_t* src = args.pool + (off >= 0 ? off : 0) + 16 * k;
        cp_async16(sm.rows[slot][r] + 16 * k, src, off >= 0 ? 16u : 0u);
      }
      cp_async_arrive(&sm.full[slot]);
    }
  };
  // One stage up front: the copies of every CTA start together, and any
  // deeper initial burst only delays the first stage behind the others (all
  // of them compete for HBM at once).  The next stages are issued at the
  // following stage boundaries.
  constexpr int kInitialStages = 1;
  int next_fill = 0;
  for (; next_fill < min(n_stages, kInitialStages); ++next_fill) fill_stage(next_fill);

  // Per-head shift k (largest |q| into [2^14, 2^15)): heads h0 and h0 + 8 for
  // the fragments, heads 4w .. 4w + 3 (softmax owner) for the scale 2^-k.
  auto head_shift = [&](int h) {
    return query_shift(max(max(sm.qmax[0][h], sm.qmax[1][h]), max(sm.qmax[2][h], sm.qmax[3][h])));
  };
  const float qmul0 = pow2f(head_shift(g));
  const float qmul1 = pow2f(head_shift(g + 8));
  float scale_h[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) scale_h[e] = args.scale_log2 * pow2f(-head_shift(4 * w + e));

  // Stage the query as B fragments (K = this warp's 144 dims in the permuted
  // order, N = 16 heads) in fragment order: one 16-byte load per k-step.
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    sm.qfrag[w][2 * q][lane] = make_uint4(bf16pair_to_f16x2(qv0[q].x, qmul0), bf16pair_to_f16x2(qv0[q].y, qmul0),
                                          bf16pair_to_f16x2(qv1[q].x, qmul1), bf16pair_to_f16x2(qv1[q].y, qmul1));
    sm.qfrag[w][2 * q + 1][lane] =
        make_uint4(bf16pair_to_f16x2(qv0[q].z, qmul0), bf16pair_to_f16x2(qv0[q].w, qmul0),
                   bf16pair_to_f16x2(qv1[q].z, qmul1), bf16pair_to_f16x2(qv1[q].w, qmul1));
  }
  sm.qfrag[w][8][lane] = make_uint4(bf16pair_to_f16x2(qr_0.x, qmul0), bf16pair_to_f16x2(qr_0.y, qmul0),
                                    bf16pair_to_f16x2(qr_1.x, qmul1), bf16pair_to_f16x2(qr_1.y, qmul1));
  __syncwarp();

  // -------------------------------------------------------------- consumers
  float o[8][2][4];
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
#pragma unroll
    for (int be = 0; be < 2; ++be)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[ks][be][e] = 0.f;

  // Softmax state: as head owner, warp w tracks heads 4w..4w+3 and lane =
  // token of the stage; m_ref is warp-uniform, l_run is this lane's share.
  float m_ref[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float l_run[4] = {0.f, 0.f, 0.f, 0.f};
  bool aborted = false;
  int abort_it = 0;

  for (int it = 0; it < n_stages && !aborted; ++it) {
    const int slot = it % kStages;
    const uint32_t round = it / kStages;
    if constexpr (TMA) {
      // One stage ahead: stage it + 1 is issued as stage it begins (its slot
      // held stage it - 1, which every warp finished reading before that
      // stage's first barrier).  Prefetching deeper measured slower: the
      // extra bytes in flight delay the stage being waited on.
      for (; next_fill < n_stages && next_fill <= min(it + 1, it - 1 + kStages); ++next_fill) fill_stage(next_fill);
    }
    const bool ok = mbar_wait_bounded(&sm.full[slot], round & 1u, args.fault_word, kFaultDecodeWait);
    if (!__all_sync(0xFFFFFFFFu, ok) && lane == 0) sm.abort_flag = 1;  // all warps leave after the next barrier
    const uint8_t* base = sm.rows[slot][0];

    // ---- unpack this warp's dims of both m-tiles straight into A fragments
    uint32_t a[2][kKSteps][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint8_t* row0 = base + (16 * mt + g) * kPitchB;
      const uint8_t* row1 = row0 + 8 * kPitchB;
      if constexpr (FMT == 0) {
        // Scales of groups 8w + 2q + (c>>1), q = 0..3: one 8-byte load per row,
        // a byte permute and a conversion per pair, then {S, S} duplicates.
        const uint32_t sel = (c >> 1) ? 0x3131u : 0x2020u;
        const uint2 sw0 = *reinterpret_cast<const uint2*>(row0 + kScaleOff + 8 * w);
        const uint2 sw1 = *reinterpret_cast<const uint2*>(row1 + kScaleOff + 8 * w);
        const uint32_t s0_01 = e4m3x2_to_f16x2(__byte_perm(sw0.x, 0, sel));
        const uint32_t s0_23 = e4m3x2_to_f16x2(__byte_perm(sw0.y, 0, sel));
        const uint32_t s1_01 = e4m3x2_to_f16x2(__byte_perm(sw1.x, 0, sel));
        const uint32_t s1_23 = e4m3x2_to_f16x2(__byte_perm(sw1.y, 0, sel));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = 64 * w + 16 * q + 4 * c;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(row0 + off);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(row1 + off);
          const uint32_t s0 = __byte_perm(q < 2 ? s0_01 : s0_23, 0, (q & 1) ? 0x3232 : 0x1010);
          const uint32_t s1 = __byte_perm(q < 2 ? s1_01 : s1_23, 0, (q & 1) ? 0x3232 : 0x1010);
          uint32_t d0[4], d1[4];
          e2m1x8_to_f16x2x4(w0, d0);
          e2m1x8_to_f16x2x4(w1, d1);
          a[mt][2 * q][0] = hmul2(d0[0], s0);
          a[mt][2 * q][1] = hmul2(d1[0], s1);
          a[mt][2 * q][2] = hmul2(d0[1], s0);
          a[mt][2 * q][3] = hmul2(d1[1], s1);
          a[mt][2 * q + 1][0] = hmul2(d0[2], s0);
          a[mt][2 * q + 1][1] = hmul2(d1[2], s1);
          a[mt][2 * q + 1][2] = hmul2(d0[3], s0);
          a[mt][2 * q + 1][3] = hmul2(d1[3], s1);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int off = 128 * w + 32 * q + 8 * c;
          const uint2 v0 = *reinterpret_cast<const uint2*>(row0 + off);
          const uint2 v1 = *reinterpret_cast<const uint2*>(row1 + off);
          uint32_t lo0[2], lo1[2], hi0[2], hi1[2];
          e4m3x4_to_f16x2x2(v0.x, lo0);
          e4m3x4_to_f16x2x2(v1.x, lo1);
          e4m3x4_to_f16x2x2(v0.y, hi0);
          e4m3x4_to_f16x2x2(v1.y, hi1);
          a[mt][2 * q][0] = lo0[0];
          a[mt][2 * q][1] = lo1[0];
          a[mt][2 * q][2] = lo0[1];
          a[mt][2 * q][3] = lo1[1];
          a[mt][2 * q + 1][0] = hi0[0];
          a[mt][2 * q + 1][1] = hi1[0];
          a[mt][2 * q + 1][2] = hi0[1];
          a[mt][2 * q + 1][3] = hi1[1];
        }
      }
      const int roff = F::kRopeOff + 16 * w + 4 * c;
      const uint32_t x0 = *reinterpret_cast<const uint32_t*>(row0 + roff);
      const uint32_t x1 = *reinterpret_cast<const uint32_t*>(row1 + roff);
      {
        uint32_t r0[2], r1[2];
        e4m3x4_to_f16x2x2(x0, r0);
        e4m3x4_to_f16x2x2(x1, r1);
        a[mt][8][0] = r0[0];
        a[mt][8][1] = r1[0];
        a[mt][8][2] = r0[1];
        a[mt][8][3] = r1[1];
      }
    }

    // ---- partial scores over this warp's 144 dims: S^T [32 tokens x 16 heads]
    float sacc[2][2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int n = 0; n < 2; ++n) sacc[mt][n][0] = sacc[mt][n][1] = sacc[mt][n][2] = sacc[mt][n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kKSteps; ++ks) {
      const uint4 qb = sm.qfrag[w][ks][lane];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mma_f16(sacc[mt][0], a[mt][ks], qb.x, qb.y);
        mma_f16(sacc[mt][1], a[mt][ks], qb.z, qb.w);
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        *reinterpret_cast<float2*>(&sm.red[w][16 * mt + g][8 * n + 2 * c]) = make_float2(sacc[mt][n][0], sacc[mt][n][1]);
        *reinterpret_cast<float2*>(&sm.red[w][16 * mt + g + 8][8 * n + 2 * c]) =
            make_float2(sacc[mt][n][2], sacc[mt][n][3]);
      }
    named_bar_sync(1, kConsumerWarps * 32);
    if (sm.abort_flag) {
      aborted = true;
      abort_it = it;
      break;
    }
    // Every warp has finished reading the rows of stages <= it, so stages up
    // to it + kStages may be issued; at most two per boundary.
    if constexpr (!TMA)
      for (int k = 0; k < 2 && next_fill < n_stages && next_fill <= it + kStages; ++k) fill_stage(next_fill++);

    // ---- head owner: heads 4w..4w+3 of token `lane`
    {
      float4 s4 = *reinterpret_cast<const float4*>(&sm.red[0][lane][4 * w]);
#pragma unroll
      for (int ww = 1; ww < kConsumerWarps; ++ww) {
        const float4 v = *reinterpret_cast<const float4*>(&sm.red[ww][lane][4 * w]);
        s4.x += v.x;
        s4.y += v.y;
        s4.z += v.z;
        s4.w += v.w;
      }
      const bool valid = sm.tok_all[it * kStageRows + lane] >= 0;
      float z[4] = {s4.x, s4.y, s4.z, s4.w};
      bool need = false;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        z[e] = valid ? z[e] * scale_h[e] : -INFINITY;
        need |= z[e] > m_ref[e] + kLazy;
      }
      float alpha[4] = {1.f, 1.f, 1.f, 1.f};
      if (__any_sync(0xFFFFFFFFu, need)) {  // rare: raise the reference maxima
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float mx = z[e];
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
          if (mx > m_ref[e] + kLazy) {
            alpha[e] = ex2(m_ref[e] - mx);  // 0 when m_ref was -inf (nothing accumulated yet)
            m_ref[e] = mx;
          }
        }
      }
      int any_rescale = 0;
      __half ph[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = (z[e] == -INFINITY) ? 0.f : ex2(z[e] - m_ref[e]);
        ph[e] = __float2half_rn(p);
        l_run[e] = l_run[e] * alpha[e] + __half2float(ph[e]);
        sm.pbuf[4 * w + e][lane] = ph[e];
        any_rescale |= alpha[e] != 1.f;
      }
      if (lane == 0) {
        *reinterpret_cast<float4*>(&sm.alpha[4 * w]) = make_float4(alpha[0], alpha[1], alpha[2], alpha[3]);
        sm.rescale[w] = any_rescale;
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);

    // ---- O[16 heads x 128 dims] += P[16 x 32 tokens] . V[32 tokens x 128 dims]
    const int4 rf = *reinterpret_cast<const int4*>(sm.rescale);
    if (rf.x | rf.y | rf.z | rf.w) {
      const float al0 = sm.alpha[g];
      const float al1 = sm.alpha[g + 8];
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
    for (int mt = 0; mt < 2; ++mt) {
      uint32_t pa[4];
      ldmatrix_x4(pa, smem_u32(&sm.pbuf[lane & 15][16 * mt + (lane >> 4) * 8]));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma_f16(o[ks][0], pa, movmatrix_t(a[mt][ks][0]), movmatrix_t(a[mt][ks][1]));
        mma_f16(o[ks][1], pa, movmatrix_t(a[mt][ks][2]), movmatrix_t(a[mt][ks][3]));
      }
    }
  }
  if (aborted) {
    // Leave no copy in flight: wait (bounded) for the stages issued but not
    // yet consumed (abort_it .. next_fill - 1).
    for (int it2 = abort_it; it2 < next_fill; ++it2)
        mbar_wait_bounded(&sm.full[it2 % kStages], static_cast<uint32_t>(it2 / kStages) & 1u, args.fault_word,
                          kFaultDecodeWait);
    if (!args.cluster_merge) return;
    // Every CTA of a cluster must reach the cluster barrier: this one joins
    // the merge as an empty split.
#pragma unroll
    for (int e = 0; e < 4; ++e) l_run[e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int be = 0; be < 2; ++be)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[ks][be][e] = 0.f;
  }

  // ---------------------------------------------------------------- finish
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float l = l_run[e];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
    if (lane == 0) {
      sm.mfin[4 * w + e] = m_ref[e];
      sm.lfin[4 * w + e] = l;
    }
  }
  named_bar_sync(1, kConsumerWarps * 32);

  // rows g and g+8 of this thread's O fragments are heads h0 and h0 + 8
  const float l0 = sm.lfin[g], l1 = sm.lfin[g + 8];
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const float lse2_0 = l0 > 0.f ? sm.mfin[g] + lg2(l0) : -INFINITY;
  const float lse2_1 = l1 > 0.f ? sm.mfin[g + 8] + lg2(l1) : -INFINITY;
  const int64_t bh0 = static_cast<int64_t>(v) * args.num_heads + h0;
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
    // The normalised partial is a convex combination of dequantised values
    // (|x| <= 6 x 448), so f16 holds it with 11 significant bits.
    __half* p0 = args.part_o + (bh0 * args.splits + sp) * kLatent;
    __half* p1 = args.part_o + (bh1 * args.splits + sp) * kLatent;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int dim = 128 * w + 32 * q + 8 * c;
      *reinterpret_cast<uint4*>(p0 + dim) =
          make_uint4(half2_bits(o[2 * q][0][0] * inv0, o[2 * q][0][1] * inv0),
                     half2_bits(o[2 * q][1][0] * inv0, o[2 * q][1][1] * inv0),
                     half2_bits(o[2 * q + 1][0][0] * inv0, o[2 * q + 1][0][1] * inv0),
                     half2_bits(o[2 * q + 1][1][0] * inv0, o[2 * q + 1][1][1] * inv0));
      *reinterpret_cast<uint4*>(p1 + dim) =
          make_uint4(half2_bits(o[2 * q][0][2] * inv1, o[2 * q][0][3] * inv1),
                     half2_bits(o[2 * q][1][2] * inv1, o[2 * q][1][3] * inv1),
                     half2_bits(o[2 * q + 1][0][2] * inv1, o[2 * q + 1][0][3] * inv1),
                     half2_bits(o[2 * q + 1][1][2] * inv1, o[2 * q + 1][1][3] * inv1));
    }
    if (w == 0 && c == 0) {
      args.part_lse[bh0 * args.splits + sp] = lse2_0;
      args.part_lse[bh1 * args.splits + sp] = lse2_1;
    }
    if (args.cluster_merge) cluster_merge(args, v, hg, sp);
  }
}

// Combine `splits` normalised partial outputs with their base-2 LSEs:
// LSE = log2 sum_s 2^lse_s, out = sum_s 2^(lse_s - LSE) * O_s.  One CTA per
// (request, head); thread i handles dims [4i, 4i+4).  The partials are read
// in chunks of kMergeChunk splits whose loads are all issued before any is
// used (one L2 round trip per chunk, not per split); a running maximum
// rescales the sums between chunks.
constexpr int kMergeChunk = 8;
__global__ void __launch_bounds__(128) splitk_merge_kernel(const __half* __restrict__ part_o,
                                                           const float* __restrict__ part_lse, int splits,
                                                           uint16_t* __restrict__ out, float* __restrict__ lse) {
  // Launched as a programmatic dependent of the decode: wait until that grid
  // has completed and its partials are visible.  What follows on the stream
  // may launch early (it waits for this grid the same way).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t bh = blockIdx.x;
  const int t = threadIdx.x;
  const float* pl = part_lse + bh * splits;
  const uint2* src = reinterpret_cast<const uint2*>(part_o + bh * splits * kLatent) + t;
  float mx = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  for (int s0 = 0; s0 < splits; s0 += kMergeChunk) {
    float ls[kMergeChunk];
    float4 v[kMergeChunk];
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      const bool in = s0 + u < splits;
      ls[u] = in ? __ldg(pl + s0 + u) : -INFINITY;
      const uint2 hv = in ? __ldg(src + (s0 + u) * (kLatent / 4)) : make_uint2(0, 0);
      const float2 a = half2_floats(hv.x), b = half2_floats(hv.y);
      v[u] = make_float4(a.x, a.y, b.x, b.y);
    }
    float cm = mx;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) cm = fmaxf(cm, ls[u]);
    if (cm == -INFINITY) continue;  // nothing selected so far
    const float al = ex2(mx - cm);  // 0 while mx is -inf
    wsum *= al;
    acc.x *= al;
    acc.y *= al;
    acc.z *= al;
    acc.w *= al;
    mx = cm;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      const float ws = ex2(ls[u] - mx);  // 0 for an empty split (lse -inf)
      wsum += ws;
      acc.x += ws * v[u].x;
      acc.y += ws * v[u].y;
      acc.z += ws * v[u].z;
      acc.w += ws * v[u].w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out + bh * kLatent + 4 * t) =
      make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  if (lse != nullptr && t == 0) lse[bh] = wsum > 0.f ? (mx + lg2(wsum)) * kLn2 : -INFINITY;
}

// The pool as a 2-D tensor of rows for the 4-row gather: [rows][row bytes / 8]
// with 8-byte elements, rows row_bytes apart (the block stride is a whole
// number of rows), box one row high.  False if the pool cannot be described.
bool make_row_tensor_map(CUtensorMap* map, const void* pool, int64_t block_stride, int64_t num_blocks, int row_bytes) {
  if (block_stride % row_bytes != 0 || num_blocks <= 0) return false;
  const int64_t rows = num_blocks * (block_stride / row_bytes);
  if (rows > 0x7FFFFFFF) return false;  // row coordinates are 32-bit
  return encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, pool, row_bytes / 8, rows, row_bytes,
                              row_bytes / 8, 1, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <int FMT, bool TMA>
cudaError_t launch_variant(const DecodeArgs& a, const CUtensorMap& map, int pairs, cudaStream_t stream) {
  const size_t smem = sizeof(Smem<FMT, TMA>);
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(sparse_decode_kernel<FMT, TMA>),
                                      static_cast<int>(smem), &configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pairs * a.splits * (a.num_heads / kHeadsPerCta));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.cluster_merge ? static_cast<unsigned>(a.splits) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster_merge ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, sparse_decode_kernel<FMT, TMA>, a, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& a, int pairs, cudaStream_t stream) {
  CUtensorMap map;
  if (make_row_tensor_map(&map, a.pool, a.block_stride, a.num_blocks, Fmt<FMT>::kRowBytes))
    return launch_variant<FMT, true>(a, map, pairs, stream);
  memset(&map, 0, sizeof(map));
  return launch_variant<FMT, false>(a, map, pairs, stream);
}

}  // namespace

DecodePlan plan_sparse_decode(int batch, int num_heads, int topk) {
  DecodePlan p{1, 0, false, 0};
  const int groups = batch * (num_heads / kHeadsPerCta);
  const int slots = 2 * device_sm_count();  // two CTAs per SM fit (registers, shared memory)
  const int max_splits = (topk + kStageRows - 1) / kStageRows;
  const int min_splits = (topk + kMaxRows - 1) / kMaxRows;  // a slice fits the CTA's row tables
  // Modelled time: waves of CTAs x (32-row stages per CTA + ~2 stages of
  // start-up latency per CTA); the fewest splits among the cheapest.
  int splits = min_splits;
  long long best = -1;
  for (int s = min_splits; s <= max_splits && groups > 0; ++s) {
    const long long waves = (static_cast<long long>(groups) * s + slots - 1) / slots;
    const int st = ((topk + s - 1) / s + kStageRows - 1) / kStageRows;
    const long long cost = waves * (st + 2);
    if (best < 0 || cost < best) {
      best = cost;
      splits = s;
    }
  }
  // The critical path is the number of 32-row stages per CTA: keep it, but
  // with as few splits as give it (fewer, fuller CTAs and partials to merge).
  const int stages = ((topk + splits - 1) / splits + kStageRows - 1) / kStageRows;
  splits = (topk + stages * kStageRows - 1) / (stages * kStageRows);
  int rows = (topk + splits - 1) / splits;
  rows = (rows + 15) / 16 * 16;
  splits = (topk + rows - 1) / rows;
  p.splits = splits;
  p.rows_per_split = rows;
  p.cluster = splits > 1 && splits <= kMaxClusterSplits;
  if (splits > 1) {
    const size_t n_bh = static_cast<size_t>(batch) * num_heads;
    size_t o_bytes = n_bh * splits * kLatent * sizeof(__half);
    o_bytes = (o_bytes + 255) / 256 * 256;
    p.workspace = o_bytes + ((n_bh * splits * sizeof(float) + 255) / 256 * 256);
  }
  return p;
}

cudaError_t launch_sparse_decode(int fmt, const uint16_t* q_nope, const uint16_t* q_rope, const void* pool,
                                 int64_t block_stride, int64_t num_blocks, const int32_t* block_table,
                                 int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                 int batch, int q_len, int num_heads, int topk, float softmax_scale, uint16_t* out,
                                 float* lse, void* workspace, const DecodePlan& plan, cudaStream_t stream) {
  const int pairs = batch * q_len;  // (request, query token) pairs
  if (pairs <= 0) return cudaSuccess;
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
  a.q_len = q_len;
  a.num_heads = num_heads;
  a.splits = plan.splits;
  a.rows_per_split = plan.rows_per_split;
  a.cluster_merge = plan.cluster ? 1 : 0;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.part_o = nullptr;
  a.part_lse = nullptr;
  a.fault_word = fault_word_ptr();
  if (a.fault_word == nullptr) return cudaErrorInvalidDevicePointer;
  if (plan.splits > 1) {
    const size_t n_bh = static_cast<size_t>(pairs) * num_heads;
    size_t o_bytes = n_bh * plan.splits * kLatent * sizeof(__half);
    o_bytes = (o_bytes + 255) / 256 * 256;
    a.part_o = static_cast<__half*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + o_bytes);
  }
  // 64-head blocks of NVFP4 rows in a pool TMA can describe go to the
  // tensor-memory kernel; it splits a list at most plan.splits ways, so the
  // workspace sized for this plan holds its partials (same layout), which
  // the merge kernel below combines.
  int merge_splits = plan.cluster ? 1 : plan.splits;
  cudaError_t e = cudaSuccess;
  CUtensorMap tc_map;
  if (sparse_decode_tc_supported(fmt, num_heads) &&
      make_row_tensor_map(&tc_map, pool, block_stride, num_blocks, kRowNvfp4)) {
    TcDecodeParams p;
    p.q_nope = q_nope;
    p.q_rope = q_rope;
    p.block_stride = block_stride;
    p.num_blocks = num_blocks;
    p.block_table = block_table;
    p.max_blocks_per_req = max_blocks_per_req;
    p.context_lens = context_lens;
    p.topk_idx = topk_idx;
    p.pairs = pairs;
    p.q_len = q_len;
    p.num_heads = num_heads;
    p.topk = topk;
    p.splits = plan_sparse_decode_tc(pairs, num_heads, topk, plan.splits);
    p.softmax_scale = softmax_scale;
    p.out = out;
    p.lse = lse;
    p.part_o = a.part_o;
    p.part_lse = a.part_lse;
    p.fault_word = a.fault_word;
    merge_splits = p.splits;
    e = launch_sparse_decode_tc(p, tc_map, stream);
  } else {
    e = fmt == 0 ? launch_fmt<0>(a, pairs, stream) : launch_fmt<1>(a, pairs, stream);
  }
  if (e != cudaSuccess || merge_splits == 1) return e;
  const int64_t n_bh = static_cast<int64_t>(pairs) * num_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_bh));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, splitk_merge_kernel, static_cast<const __half*>(a.part_o),
                         static_cast<const float*>(a.part_lse), merge_splits, out, lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
