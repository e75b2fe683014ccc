// Sparse MLA decode on the fifth-generation tensor cores (tcgen05, tensor
// memory) for head counts that are multiples of 64, NVFP4 rows gathered by
// TMA.  Same result as the 16-head kernel ("Prime Inference: serving GLM-5.3
// to agents is a KV-cache problem", section "A kernel that reads four bits
// directly": the selected rows are unpacked on chip and both products use
// FP16 operands with FP32 accumulation).
//
// One CTA = one (request, query token) x 64 heads x a slice of its top-k
// list, in stages of 128 selected rows.  Ten warps:
//   * warp 8 resolves each stage's rows (top-k index, block table) and
//     gathers them into one of two raw-row slots with 4-row TMA gathers;
//   * warp 9 allocates 512 tensor-memory columns and one lane issues every
//     tcgen05.mma;
//   * warps 0-7 unpack the raw rows into f16 operand chunks in shared
//     memory (16 KB each, three buffers; a chunk is converted in registers
//     before its buffer is waited for), run the online softmax and write
//     the output.
// Per stage:
//   S[128 rows x 64 heads] = K[128 x 576] . Q^T   (M = 128, N = 64, 36 MMAs:
//       nine 64-dim chunks of the rows, K-major; Q K-major, resident)
//   O^T[512 x 64] += V^T[512 x 128] . P^T          (M = 128 dims, N = 64,
//       32 MMAs: 64-row x 128-dim chunks of the same rows, unpacked a second
//       time, read MN-major; P written by the softmax warps, MN-major)
// S lives in tensor-memory columns 0-63 (lane = row), O^T in columns 64-319
// (lane = latent dim within a 128-dim block, column = head).  The softmax
// keeps a lazy per-head maximum (raised only when a score exceeds it by 2^8),
// so O is rescaled in tensor memory only on the rare stages that raise it.
// Every wait is bounded; a timeout sets the library's fault bit and the CTA
// leaves after its copies and MMAs in flight have drained.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kTcHeads = 64;
constexpr int kTcRows = 128;  // selected rows per stage
constexpr int kTcUnpackWarps = 8;
constexpr int kTcUnpackThreads = kTcUnpackWarps * 32;
constexpr int kTcThreads = kTcUnpackThreads + 64;  // + producer warp + MMA warp
constexpr int kTcQkChunks = 9;                     // 8 x 64 latent dims + 64 rope dims
constexpr int kTcPvChunks = 8;                     // 2 row halves x 4 blocks of 128 dims
constexpr int kTcChunkBytes = 16384;
constexpr int kTcChunkBufs = 3;
constexpr int kTcQBytes = kTcHeads * (kLatent + kRope) * 2;  // 73,728
constexpr int kTcQHeadGroupBytes = (kLatent + kRope) / 8 * 128;  // 9,216: 8 heads x 576 dims
constexpr int kTcRawBytes = kTcRows * kRowNvfp4;                // 45,056
constexpr int kTcPBytes = kTcRows * kTcHeads * 2;               // 16,384
constexpr uint32_t kTcCols = 512;                               // tensor-memory columns allocated
constexpr uint32_t kTcOCol = 64;                                // first column of O^T
constexpr float kTcLazy = 8.f;
constexpr float kTcLn2 = 0.6931471805599453f;

struct TcArgs {
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  const int32_t* topk_idx;
  uint16_t* out;
  float* lse;
  __half* part_o;
  float* part_lse;
  int64_t rows_per_block;  // pool rows per block (block stride / row bytes)
  int64_t num_blocks;
  int max_blocks;
  int topk;
  int q_len;
  int num_heads;
  int splits;
  int rows_per_split;
  float scale_log2;
  unsigned int* fault_word;
};

struct alignas(1024) TcSmem {
  uint8_t q_op[kTcQBytes];               // Q, K-major core matrices: (h/8)*9216 + (d/8)*128 + (h%8)*16
  uint8_t raw[2][kTcRawBytes];           // gathered rows, back to back
  uint8_t chunk[kTcChunkBufs][kTcChunkBytes];  // unpacked operand chunks
  uint8_t p_op[kTcPBytes];               // P, MN-major: (h/8)*2048 + (r/8)*128 + (r%8)*16 + (h%8)*2
  int32_t tok[2][kTcRows];               // token of each row of the slot's stage, -1 if masked
  // per-warp, per-head reduction scratch of the softmax; before the first
  // stage, its first 64 words hold each head's largest |q| (bf16 magnitude bits)
  float red[kTcUnpackWarps][32];
  float m_ref[2][32];                    // running (lazy) maximum per head, base 2, per head half
  float alpha[2][32];                    // rescale factor of the last raise, per head half
  float qscale[kTcHeads];                // per head: softmax scale (base 2) x 2^-shift of its query
  uint64_t raw_full[2], raw_free[2], chunk_full[kTcChunkBufs], chunk_free[kTcChunkBufs], s_full, p_full, done;
  uint32_t tmem_base;
  int abort_flag;
};

static_assert(sizeof(TcSmem) <= 227 * 1024, "one CTA per SM must fit");

// ---- tcgen05 wrappers -------------------------------------------------------
// Shared-memory matrix descriptor, no swizzle: start address, leading and
// stride byte offsets (>> 4), descriptor version 1 (bit 46).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, the
// majorness of A and B (0 = K-major, 1 = MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t tc_idesc(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// 32 consecutive columns of this warp's 32 lanes (one 32-bit value each).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// OR of `pred` over the first `threads` threads of the CTA (named barrier 2).
__device__ __forceinline__ bool bar_red_or(bool pred, int threads) {
  uint32_t out;
  asm volatile(
      "{ .reg .pred pi, po; setp.ne.u32 pi, %1, 0; barrier.cta.red.or.pred po, 2, %2, pi; selp.u32 %0, 1, 0, po; }"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(pred)), "r"(threads)
      : "memory");
  return out != 0;
}

// The same, polling without the suspend hint: for the chunk hand-offs, where
// the phase usually completes within a few hundred cycles.
__device__ __forceinline__ bool tc_wait_spin(TcSmem& sm, uint64_t* bar, uint32_t parity, unsigned int* fault_word) {
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
  }
  atomicOr(fault_word, kFaultDecodeWait);
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  return false;
}
// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool tc_wait(TcSmem& sm, uint64_t* bar, uint32_t parity, unsigned int* fault_word) {
  for (uint32_t i = 0; i < kSpinPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
  }
  uint32_t ns = 64;
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
    if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) return false;
  }
  atomicOr(fault_word, kFaultDecodeWait);
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  return false;
}

// Two bf16 query values times 2^k (`mul`) to f16x2.
__device__ __forceinline__ uint32_t tc_bf16pair_to_f16x2(uint32_t two, float mul) {
  return f32x2_to_f16x2_sat(bf16_bits_to_f32(two & 0xFFFFu) * mul, bf16_bits_to_f32(two >> 16) * mul);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    sparse_decode_tc_kernel(const TcArgs args, const __grid_constant__ CUtensorMap tmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  TcSmem& sm = *reinterpret_cast<TcSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_hb = args.num_heads / kTcHeads;
  const int sp = blockIdx.x % args.splits;
  const int hb = (blockIdx.x / args.splits) % n_hb;
  const int v = blockIdx.x / (args.splits * n_hb);
  const int b = v / args.q_len;
  const int row_begin = sp * args.rows_per_split;
  const int row_end = min(args.topk, row_begin + args.rows_per_split);
  const int n_rows = max(0, row_end - row_begin);
  const int n_stages = (n_rows + kTcRows - 1) / kTcRows;
  const int h0 = hb * kTcHeads;
  unsigned int* fw = args.fault_word;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.raw_full[i], 1);
      mbar_init(&sm.raw_free[i], kTcUnpackThreads);
    }
    for (int i = 0; i < kTcChunkBufs; ++i) {
      mbar_init(&sm.chunk_full[i], kTcUnpackThreads);
      mbar_init(&sm.chunk_free[i], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, kTcUnpackThreads);
    mbar_init(&sm.done, 1);
    sm.abort_flag = 0;
    for (int j = 0; j < 64; ++j) sm.m_ref[j >> 5][j & 31] = -INFINITY;
    for (int j = 0; j < kTcHeads; ++j) reinterpret_cast<uint32_t*>(&sm.red[0][0])[j] = 0;
    fence_mbar_init();
  }
  if (warp == kTcUnpackWarps + 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                 "r"(kTcCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  int issued_last[2] = {-1, -1};  // producer: last stage gathered into each slot

  if (warp == kTcUnpackWarps) {
    // ------------------------------------------------------------ producer
    const int ctx = __ldg(args.ctx_lens + b) - (args.q_len - 1 - (v - b * args.q_len));
    const int32_t* topk_row = args.topk_idx + static_cast<int64_t>(v) * args.topk;
    const int32_t* bt_row = args.block_table + static_cast<int64_t>(b) * args.max_blocks;
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s & 1;
      // this lane's rows 4 lane .. 4 lane + 3 of the stage: top-k index,
      // then block table; masked rows get coordinate -1 (reads zeros)
      int t[4], rc[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = row_begin + s * kTcRows + 4 * lane + e;
        t[e] = j < row_end ? __ldg(topk_row + j) : -1;
      }
      int pb[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = t[e] >= 0 && t[e] < ctx && t[e] / kBlock < args.max_blocks;
        pb[e] = ok ? __ldg(bt_row + t[e] / kBlock) : -1;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool ok = pb[e] >= 0 && pb[e] < args.num_blocks;
        rc[e] = ok ? static_cast<int>(static_cast<int64_t>(pb[e]) * args.rows_per_block + t[e] % kBlock) : -1;
        t[e] = ok ? t[e] : -1;
      }
      bool ok = true;
      if (s >= 2) ok = tc_wait(sm, &sm.raw_free[slot], static_cast<uint32_t>((s >> 1) - 1) & 1u, fw);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
#pragma unroll
      for (int e = 0; e < 4; ++e) sm.tok[slot][4 * lane + e] = t[e];
      __syncwarp();
      if (lane == 0) mbar_expect_tx(&sm.raw_full[slot], kTcRawBytes);
      __syncwarp();
      tma_gather4(sm.raw[slot] + 4 * lane * kRowNvfp4, &tmap, rc[0], rc[1], rc[2], rc[3], &sm.raw_full[slot]);
      issued_last[slot] = s;
    }
  } else if (warp == kTcUnpackWarps + 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t kIdescQk = tc_idesc(128, kTcHeads, 0, 0);
      constexpr uint32_t kIdescPv = tc_idesc(128, kTcHeads, 1, 1);
      const uint32_t q_base = smem_u32(sm.q_op);
      const uint32_t p_base = smem_u32(sm.p_op);
      const uint32_t ch_base0 = smem_u32(sm.chunk[0]);
      int q = 0;
      bool ok = true;
      for (int s = 0; s < n_stages && ok; ++s) {
        // S = K . Q^T over nine 64-dim chunks (four K = 16 steps each)
        for (int c = 0; c < kTcQkChunks; ++c, ++q) {
          const int bb = q % kTcChunkBufs;
          ok = tc_wait_spin(sm, &sm.chunk_full[bb], static_cast<uint32_t>(q / kTcChunkBufs) & 1u, fw);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = ch_base0 + bb * kTcChunkBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(tbase, tc_desc(a0 + 256 * j, 128, 1024),
                   tc_desc(q_base + (8 * c + 2 * j) * 128, 128, kTcQHeadGroupBytes), kIdescQk, (c | j) != 0);
          tc_commit(&sm.chunk_free[bb]);
        }
        if (!ok) break;
        tc_commit(&sm.s_full);
        ok = tc_wait(sm, &sm.p_full, static_cast<uint32_t>(s) & 1u, fw);
        if (!ok) break;
        tc_fence_after();
        // O^T += V^T . P^T: row half hf, 128-dim block blk (four K = 16 steps)
        for (int c = 0; c < kTcPvChunks; ++c, ++q) {
          const int hf = c >> 2, blk = c & 3;
          const int bb = q % kTcChunkBufs;
          ok = tc_wait_spin(sm, &sm.chunk_full[bb], static_cast<uint32_t>(q / kTcChunkBufs) & 1u, fw);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a0 = ch_base0 + bb * kTcChunkBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(tbase + kTcOCol + 64 * blk, tc_desc(a0 + 256 * j, 128, 1024),
                   tc_desc(p_base + (8 * hf + 2 * j) * 128, 128, 2048), kIdescPv, (s | hf | j) != 0);
          tc_commit(&sm.chunk_free[bb]);
        }
      }
      tc_commit(&sm.done);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ unpack, softmax, output
    const int w = warp;
    const int quad = w & 3;  // tensor-memory lanes 32 quad .. 32 quad + 31
    const int half = w >> 2;  // heads 32 half .. 32 half + 31
    const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
    const int t_lo = lane & 7;
    const int dg_lo = lane >> 3;
    float l_part[32];  // this row's share of each head's softmax denominator
#pragma unroll
    for (int j = 0; j < 32; ++j) l_part[j] = 0.f;
    const float* m_ref = sm.m_ref[half];
    {
      // The absorbed query of the 64 heads, bf16 -> f16, as K-major core
      // matrices (8 heads x 8 dims per 128 bytes); all loads issued before
      // any is used, while the producer gathers the first stage.  The proxy
      // fence before the first chunk's arrival publishes it to the MMAs.
      const int64_t qrow = static_cast<int64_t>(v) * args.num_heads + h0;
      constexpr int kDimGroups = (kLatent + kRope) / 8;
      constexpr int kQPer = kTcHeads * kDimGroups / kTcUnpackThreads;  // 18
      uint4 xs[kQPer];
#pragma unroll
      for (int i = 0; i < kQPer; ++i) {
        const int u = threadIdx.x + i * kTcUnpackThreads;
        const int h = u / kDimGroups;
        const int dg = u - h * kDimGroups;
        xs[i] = dg < kLatent / 8
                    ? __ldg(reinterpret_cast<const uint4*>(args.q_nope + (qrow + h) * kLatent) + dg)
                    : __ldg(reinterpret_cast<const uint4*>(args.q_rope + (qrow + h) * kRope) + (dg - kLatent / 8));
      }
      // Per-head power-of-two shift bringing the largest |q| into
      // [2^14, 2^15) (FP16 operands), undone in the head's softmax scale.
      uint32_t* qmax = reinterpret_cast<uint32_t*>(&sm.red[0][0]);
#pragma unroll
      for (int i = 0; i < kQPer; ++i) {
        const int u = threadIdx.x + i * kTcUnpackThreads;
        atomicMax(&qmax[u / kDimGroups], bf16x8_absmax_bits(xs[i]));
      }
      named_bar_sync(1, kTcUnpackThreads);
      if (threadIdx.x < kTcHeads)
        sm.qscale[threadIdx.x] = args.scale_log2 * pow2f(-query_shift(qmax[threadIdx.x]));
#pragma unroll
      for (int i = 0; i < kQPer; ++i) {
        const int u = threadIdx.x + i * kTcUnpackThreads;
        const int h = u / kDimGroups;
        const int dg = u - h * kDimGroups;
        const float mul = pow2f(query_shift(qmax[h]));
        *reinterpret_cast<uint4*>(sm.q_op + (h >> 3) * kTcQHeadGroupBytes + dg * 128 + (h & 7) * 16) =
            make_uint4(tc_bf16pair_to_f16x2(xs[i].x, mul), tc_bf16pair_to_f16x2(xs[i].y, mul),
                       tc_bf16pair_to_f16x2(xs[i].z, mul), tc_bf16pair_to_f16x2(xs[i].w, mul));
      }
      fence_async_smem();
    }
    int q = 0;
    bool aborted = false;
    for (int s = 0; s < n_stages; ++s) {
      const int slot = s & 1;
      bool ok = tc_wait(sm, &sm.raw_full[slot], static_cast<uint32_t>(s >> 1) & 1u, fw);
      const uint8_t* raw = sm.raw[slot];
      // ---- K operand chunks: rows 0..127 x dims 64c .. 64c + 63, K-major
      // core matrices (r/8)*1024 + (d/8)*128 + (r%8)*16; lane -> row r with
      // r % 8 = lane % 8 (conflict-free 16-byte stores), 8-dim group lane / 8
      for (int c = 0; c < kTcQkChunks; ++c, ++q) {
        const int bb = q % kTcChunkBufs;
        uint32_t hvs[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 8 * (w + 8 * (i & 1)) + t_lo;
          const int dg = dg_lo + 4 * (i >> 1);
          const uint8_t* row = raw + r * kRowNvfp4;
          uint32_t (&hv)[4] = hvs[i];
          if (c < 8) {
            const uint32_t codes = *reinterpret_cast<const uint32_t*>(row + 32 * c + 4 * dg);
            const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint32_t>(row[kScaleOff + 4 * c + (dg >> 1)]) * 0x0101u);
            e2m1x8_to_f16x2x4(codes, hv);
#pragma unroll
            for (int k = 0; k < 4; ++k) hv[k] = hmul2(hv[k], s2);
          } else {
            const uint2 rb = *reinterpret_cast<const uint2*>(row + kRopeOffNvfp4 + 8 * dg);
            uint32_t lo[2], hi[2];
            e4m3x4_to_f16x2x2(rb.x, lo);
            e4m3x4_to_f16x2x2(rb.y, hi);
            hv[0] = lo[0];
            hv[1] = lo[1];
            hv[2] = hi[0];
            hv[3] = hi[1];
          }
        }
        if (ok && q >= kTcChunkBufs)
          ok = tc_wait_spin(sm, &sm.chunk_free[bb], static_cast<uint32_t>(q / kTcChunkBufs + 1) & 1u, fw);
        if (!ok) continue;
        uint8_t* dst = sm.chunk[bb];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 8 * (w + 8 * (i & 1)) + t_lo;
          const int dg = dg_lo + 4 * (i >> 1);
          *reinterpret_cast<uint4*>(dst + (r >> 3) * 1024 + dg * 128 + (r & 7) * 16) =
              make_uint4(hvs[i][0], hvs[i][1], hvs[i][2], hvs[i][3]);
        }
        fence_async_smem();
        mbar_arrive(&sm.chunk_full[bb]);
      }
      if (ok) ok = tc_wait(sm, &sm.s_full, static_cast<uint32_t>(s) & 1u, fw);
      // every unpack thread takes the same branch at every named barrier
      if (bar_red_or(!ok, kTcUnpackThreads)) {
        aborted = true;
        break;
      }
      tc_fence_after();

      // ---- softmax: this thread owns row r of the stage for 32 heads
      uint32_t sr[32];
      tmem_ld32(tbase + lane_base + 32 * half, sr);
      const int r = 32 * quad + lane;
      const bool valid = sm.tok[slot][r] >= 0;
      float z[32];
      bool need = false;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        z[j] = valid ? __uint_as_float(sr[j]) * sm.qscale[32 * half + j] : -INFINITY;
        need |= z[j] > m_ref[j] + kTcLazy;
      }
      bool rescale = false;
      if (bar_red_or(need, kTcUnpackThreads)) {
        // per-head maximum over the 128 rows: warp butterfly, then lane j of
        // the half's first warp combines the four warps for head j
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float m = z[j];
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
          if (lane == 0) sm.red[w][j] = m;
        }
        named_bar_sync(1, kTcUnpackThreads);
        if (quad == 0) {
          const float m = fmaxf(fmaxf(sm.red[4 * half][lane], sm.red[4 * half + 1][lane]),
                                fmaxf(sm.red[4 * half + 2][lane], sm.red[4 * half + 3][lane]));
          const float old = sm.m_ref[half][lane];
          float al = 1.f;
          if (m > old + kTcLazy) {
            al = ex2(old - m);  // 0 while the maximum is -inf
            sm.m_ref[half][lane] = m;
          }
          sm.alpha[half][lane] = al;
        }
        named_bar_sync(1, kTcUnpackThreads);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float al = sm.alpha[half][j];
          l_part[j] *= al;
          rescale |= al != 1.f;
        }
      }
      // O^T columns of this half x alpha (identical decision in the 4 warps of
      // the half; nothing to scale before the first P.V)
      if (rescale && s > 0) {
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          const uint32_t ta = tbase + lane_base + kTcOCol + 64 * blk + 32 * half;
          uint32_t o[32];
          tmem_ld32(ta, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * sm.alpha[half][j]);
          tmem_st32(ta, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      }
      // P (f16) into the MN-major operand: head group 4 half + g, row r
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float p0 = z[j] == -INFINITY ? 0.f : ex2(z[j] - m_ref[j]);
        const float p1 = z[j + 1] == -INFINITY ? 0.f : ex2(z[j + 1] - m_ref[j + 1]);
        const __half2 ph = __floats2half2_rn(p0, p1);
        l_part[j] += __low2float(ph);
        l_part[j + 1] += __high2float(ph);
        pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&ph);
      }
#pragma unroll
      for (int g = 0; g < 4; ++g)
        *reinterpret_cast<uint4*>(sm.p_op + (4 * half + g) * 2048 + r * 16) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.p_full);

      // ---- V operand chunks: rows 64 hf .. 64 hf + 63 x dims 128 blk ..
      // 128 blk + 127, MN-major core matrices (d/8)*1024 + (r/8)*128 + (r%8)*16
      for (int c = 0; c < kTcPvChunks; ++c, ++q) {
        const int hf = c >> 2, blk = c & 3;
        const int bb = q % kTcChunkBufs;
        const int rr = 8 * w + t_lo;
        const uint8_t* row = raw + (64 * hf + rr) * kRowNvfp4;
        uint32_t hvs[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int dg = dg_lo + 4 * i;
          const uint32_t codes = *reinterpret_cast<const uint32_t*>(row + 64 * blk + 4 * dg);
          const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint32_t>(row[kScaleOff + 8 * blk + (dg >> 1)]) * 0x0101u);
          e2m1x8_to_f16x2x4(codes, hvs[i]);
#pragma unroll
          for (int k = 0; k < 4; ++k) hvs[i][k] = hmul2(hvs[i][k], s2);
        }
        if (ok && q >= kTcChunkBufs)
          ok = tc_wait_spin(sm, &sm.chunk_free[bb], static_cast<uint32_t>(q / kTcChunkBufs + 1) & 1u, fw);
        if (!ok) continue;
        uint8_t* dst = sm.chunk[bb];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint4*>(dst + (dg_lo + 4 * i) * 1024 + rr * 16) =
              make_uint4(hvs[i][0], hvs[i][1], hvs[i][2], hvs[i][3]);
        fence_async_smem();
        mbar_arrive(&sm.chunk_full[bb]);
      }
      if (ok) mbar_arrive(&sm.raw_free[slot]);
      if (bar_red_or(!ok, kTcUnpackThreads)) {
        aborted = true;
        break;
      }
    }
    bool ok = !aborted && tc_wait(sm, &sm.done, 0u, fw);
    if (!bar_red_or(!ok, kTcUnpackThreads)) {
      tc_fence_after();
      // l per head: sum of this half's 128 row partials; lane j of the
      // half's first warp finishes head j (denominator, LSE)
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float l = l_part[j];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, off);
        if (lane == 0) sm.red[w][j] = l;
      }
      named_bar_sync(1, kTcUnpackThreads);
      const int64_t bh0 = static_cast<int64_t>(v) * args.num_heads + h0 + 32 * half;
      if (quad == 0) {
        const float l = (sm.red[4 * half][lane] + sm.red[4 * half + 1][lane]) +
                        (sm.red[4 * half + 2][lane] + sm.red[4 * half + 3][lane]);
        sm.alpha[half][lane] = l > 0.f ? 1.f / l : 0.f;  // reused: 1 / l, 0 when nothing was selected
        const float lse2 = l > 0.f ? sm.m_ref[half][lane] + lg2(l) : -INFINITY;
        if (args.splits == 1) {
          if (args.lse != nullptr) args.lse[bh0 + lane] = lse2 * kTcLn2;
        } else {
          args.part_lse[(bh0 + lane) * args.splits + sp] = lse2;
        }
      }
      named_bar_sync(1, kTcUnpackThreads);
#pragma unroll 1
      for (int blk = 0; blk < 4; ++blk) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_base + kTcOCol + 64 * blk + 32 * half, o);
        const int dim = 128 * blk + 32 * quad + lane;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float inv = sm.alpha[half][j];
          const float x = inv > 0.f ? __uint_as_float(o[j]) * inv : 0.f;
          if (args.splits == 1)
            args.out[(bh0 + j) * kLatent + dim] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
          else
            args.part_o[((bh0 + j) * args.splits + sp) * kLatent + dim] = __float2half_rn(x);
        }
      }
    }
  }

  // ---- teardown: no copy or MMA may still be in flight when the CTA leaves
  // or frees its tensor memory
  if (warp == kTcUnpackWarps && lane == 0) {
    for (int i = 0; i < 2; ++i)
      if (issued_last[i] >= 0)
        mbar_wait_bounded(&sm.raw_full[i], static_cast<uint32_t>(issued_last[i] >> 1) & 1u, fw, kFaultDecodeWait);
  }
  if (warp == kTcUnpackWarps + 1 && lane == 0) mbar_wait_bounded(&sm.done, 0u, fw, kFaultDecodeWait);
  tc_fence_before();
  __syncthreads();
  if (warp == kTcUnpackWarps + 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTcCols) : "memory");
  }
}

}  // namespace

bool sparse_decode_tc_supported(int fmt, int num_heads) {
  return fmt == 0 && num_heads >= kTcHeads && num_heads % kTcHeads == 0;
}

// The same conditions as the dispatch in launch_sparse_decode: the format
// and head count, a pool the row tensor map can describe (a stride of whole
// rows, at least one block, row coordinates within 32 bits) and a driver
// that can encode tensor maps.
bool sparse_decode_uses_tc(int fmt, int num_heads, int64_t block_stride, int64_t num_blocks) {
  if (!sparse_decode_tc_supported(fmt, num_heads) || num_blocks <= 0 || block_stride % kRowNvfp4 != 0) return false;
  return num_blocks * (block_stride / kRowNvfp4) <= 0x7FFFFFFF && tensor_maps_available();
}

int plan_sparse_decode_tc(int pairs, int num_heads, int topk, int max_splits) {
  const int groups = pairs * (num_heads / kTcHeads);
  const int stages = (topk + kTcRows - 1) / kTcRows;
  int splits = groups > 0 ? device_sm_count() / groups : 1;  // one CTA per SM
  splits = max(1, min(splits, min(stages, max_splits)));
  return splits;
}

cudaError_t launch_sparse_decode_tc(const TcDecodeParams& p, const CUtensorMap& map, cudaStream_t stream) {
  const size_t smem = sizeof(TcSmem);
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(sparse_decode_tc_kernel),
                                      static_cast<int>(smem), &configured);
  if (e != cudaSuccess) return e;
  TcArgs a;
  a.q_nope = p.q_nope;
  a.q_rope = p.q_rope;
  a.block_table = p.block_table;
  a.ctx_lens = p.context_lens;
  a.topk_idx = p.topk_idx;
  a.out = p.out;
  a.lse = p.lse;
  a.part_o = static_cast<__half*>(p.part_o);
  a.part_lse = p.part_lse;
  a.rows_per_block = p.block_stride / kRowNvfp4;
  a.num_blocks = p.num_blocks;
  a.max_blocks = p.max_blocks_per_req;
  a.topk = p.topk;
  a.q_len = p.q_len;
  a.num_heads = p.num_heads;
  a.splits = p.splits;
  a.rows_per_split = (p.topk + p.splits - 1) / p.splits;
  a.scale_log2 = p.softmax_scale * 1.4426950408889634f;
  a.fault_word = p.fault_word;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.pairs * (p.num_heads / kTcHeads) * p.splits));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, sparse_decode_tc_kernel, a, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
