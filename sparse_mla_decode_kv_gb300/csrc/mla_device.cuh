// Device-side helpers shared by the library's kernels: row layout constants,
// inline-PTX conversions, warp-level tensor-core MMA, bulk async copies and
// bounded mbarrier waits.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace mla {

// ---- row layout ("Prime Inference", section "Four bits per latent value":
// 512 x 4 bit codes + 32 one-byte scales + 64 one-byte rope = 352 bytes; the
// FP8 row is 512 + 64 bytes).  Offsets inside the row are this library's.
constexpr int kLatent = 512;
constexpr int kRope = 64;
constexpr int kGroup = 16;                 // latent values per e4m3 scale
constexpr int kRowNvfp4 = 352;
constexpr int kRowFp8 = 576;
constexpr int kScaleOff = 256;             // NVFP4: scales after the codes
constexpr int kRopeOffNvfp4 = 288;
constexpr int kRopeOffFp8 = 512;
constexpr int kBlock = 64;                 // tokens per paged block
constexpr int kIdxDim = 128;               // indexer key width (e4m3)

// Bits of the library-wide device fault word (a __device__ variable in
// mla_api.cu whose address kernels receive as an argument).
constexpr unsigned int kFaultDecodeWait = 1u;
constexpr unsigned int kFaultIndexerWait = 2u;
// Poll budget of the back-off phase of a bounded wait (each poll sleeps a
// few microseconds): about a second in total, with the hinted phase before
// it, far beyond any legitimate wait in these kernels (microseconds).  Polls
// do not advance while the context is switched out, so time-slicing with
// other work does not make a wait give up early.
constexpr uint32_t kWaitPolls = 1u << 18;

// ---- conversions -----------------------------------------------------------
// Two e2m1 codes (low nibble -> low half) to two exact f16 values.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  asm("{ .reg .b8 b; cvt.u8.u32 b, %1; cvt.rn.f16x2.e2m1x2 %0, b; }" : "=r"(d) : "r"(byte));
  return d;
}
// Eight e2m1 codes (one 32-bit word, element 2i in the low nibble of byte i)
// to four f16x2 (byte i -> d[i]); the word is split into its bytes by a
// register unpack, not by shifts.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&d)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(w));
}
// Four e4m3 bytes to two f16x2 (low half-word -> d[0]).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t (&d)[2]) {
  asm("{ .reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h1; }"
      : "=r"(d[0]), "=r"(d[1])
      : "r"(w));
}
// Two e4m3 bytes (low byte -> low half) to two exact f16 values.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t d;
  uint16_t h = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(h));
  return d;
}
// Two floats to e4m3, round-to-nearest-even, satfinite.  `hi` lands in the
// high byte, `lo` in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two floats to e2m1, round-to-nearest-even, satfinite.  `hi` lands in the
// high nibble, `lo` in the low nibble; the sign of a value that rounds to
// zero is kept (code 0x8).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float hi, float lo) {
  uint32_t r;
  asm("{ .reg .b8 b; cvt.rn.satfinite.e2m1x2.f32 b, %1, %2; cvt.u32.u8 %0, b; }" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two floats to f16x2 (lo -> low half), round-to-nearest-even, saturating at
// +-65504.
__device__ __forceinline__ uint32_t f32x2_to_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- query range --------------------------------------------------------------
// The absorbed query arrives as bf16 (8 exponent bits) but feeds FP16
// operands (5 exponent bits): a head whose values lie beyond +-65504 would
// saturate and values below 2^-14 would lose bits.  Each head is therefore
// scaled by a power of two 2^k that brings its largest magnitude into
// [2^14, 2^15), and the head's softmax scale is multiplied by 2^-k: the
// scaled scores are exactly the unscaled ones (powers of two are exact).
//
// Largest magnitude of the two bf16 values in `two`, as the 15 bits of the
// magnitude (ordered like the values for every finite input).
__device__ __forceinline__ uint32_t bf16x2_absmax_bits(uint32_t two) {
  return max(two & 0x7FFFu, (two >> 16) & 0x7FFFu);
}
__device__ __forceinline__ uint32_t bf16x8_absmax_bits(uint4 v) {
  return max(max(bf16x2_absmax_bits(v.x), bf16x2_absmax_bits(v.y)),
             max(bf16x2_absmax_bits(v.z), bf16x2_absmax_bits(v.w)));
}
// The shift k for a head whose largest bf16 magnitude has bits `m`: 0 for an
// all-zero head, else 14 - exponent, clamped so that 2^k and 2^-k are normal
// floats (a subnormal maximum counts as exponent -127).
__device__ __forceinline__ int query_shift(uint32_t m) {
  if (m == 0) return 0;
  const int e = static_cast<int>(m >> 7) - 127;
  return min(126, max(-113, 14 - e));
}
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((127 + k) << 23); }

// ---- warp-level tensor core (m16n8k16, f16 x f16 -> f32) -------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Transpose of an 8x8 16-bit tile held in the standard fragment layout
// (lane l holds row l/4, columns 2(l%4) and 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t smem_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr));
}

// ---- shared memory, mbarriers and bulk copies -----------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.release.cta.shared::cta.b64 st, [%0]; }" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: the thread may sleep in hardware (up to
// `hint_ns`) until the phase completes instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  The first kSpinPolls
// tries sleep in hardware between polls (woken when the phase completes);
// after them the loop backs off with nanosleep.  Returns false (after
// setting `fault` in *fault_word) if the phase never completed.
constexpr uint32_t kSpinPolls = 1u << 14;
constexpr uint32_t kSleepHintNs = 20000;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned int* fault_word,
                                                  unsigned int fault) {
  for (uint32_t i = 0; i < kSpinPolls; ++i)
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
  uint32_t ns = 64;
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
    if (mbar_try_wait(bar, parity)) return true;
  }
  atomicOr(fault_word, fault);
  return false;
}
// The same bounded wait, but it also gives up (returning false, without
// setting a fault bit) as soon as another warp of the CTA has set
// *abort_flag -- that warp timed out, and the phase may never complete.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, const int* abort_flag,
                                                   unsigned int* fault_word, unsigned int fault) {
  const volatile int* flag = abort_flag;
  for (uint32_t i = 0; i < kSpinPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*flag) return false;
  }
  uint32_t ns = 64;
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    __nanosleep(ns);
    if (ns < 1024) ns <<= 1;
    if (mbar_try_wait(bar, parity)) return true;
    if (*flag) return false;
  }
  atomicOr(fault_word, fault);
  return false;
}
// 16-byte global -> shared copy (cp.async, L2 only).  With src_bytes == 0
// nothing is read and the 16 destination bytes are zero-filled.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
               "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed;
// the arrival counts toward the barrier's expected count (no increment).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// ---- TMA (bulk tensor copies) -----------------------------------------------
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// 4-row TMA gather: rows y0..y3 of a 2-D tensor (x = 0), one row high per box;
// a negative row index reads zeros.  Completion is signalled on `bar` as
// transaction bytes.
__device__ __forceinline__ void tma_gather4(void* dst, const void* tmap, int y0, int y1, int y2, int y3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(0), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
      : "memory");
}
// One 2-D TMA tile (the tensor map's box) at coordinates (x, y).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Contiguous global -> shared bulk copy (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ---- fifth-generation tensor cores (tcgen05) --------------------------------
// Shared-memory matrix descriptor of a K-major operand stored in 128-byte
// swizzle atoms -- 8 rows of 128 bytes, the 16-byte chunk j of row r at
// chunk j ^ (r % 8), which is what a TMA tile loaded with the 128-byte
// swizzle writes.  Fields: start address >> 4, leading byte offset 16 (not
// used by a swizzled K-major operand whose K step fits one atom), stride
// between 8-row groups 1024 bytes, descriptor version 1, layout type 2
// (128-byte swizzle).  The atom base must be 1024-byte aligned; a K step
// inside the atom advances the start address by its byte offset.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}
// Instruction descriptor, dense MMA with an f32 accumulator, A and B both
// K-major: A / B format codes (kind::f8f6f4: 0 = e4m3), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t umma_idesc_f32acc(int m, int n, int a_fmt, int b_fmt) {
  return (1u << 4) | (static_cast<uint32_t>(a_fmt) << 7) | (static_cast<uint32_t>(b_fmt) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
// D (tensor memory) [+]= A . B^T with 8-bit floating-point operands from
// shared memory, issued by one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tcgen05_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tcgen05_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_load_32cols(uint32_t taddr, uint32_t (&r)[32]) {
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

// ---- thread-block clusters ------------------------------------------------
// Barrier over every thread of every CTA of the cluster; the release/acquire
// pair (cluster scope) makes every write before it, to shared or global
// memory, visible to the cluster's threads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace mla
