// Quantize-on-write of MLA latent rows into the paged cache.
//
// "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem",
// section "Four bits per latent value": the 512-value latent is stored as
// four-bit values with one FP8 scale per 16 values, the 64 rope values stay
// FP8, 576 -> 352 bytes per row.  The FP8 comparison row keeps all 576 values
// as e4m3 with no scale.
//
// One warp per token.  Lane g owns latent group g (16 values, 32 bytes of
// bf16) and rope values 2g, 2g+1, so the warp reads its 1,152 input bytes
// with fully used 16-byte loads and writes the 352 (or 576) output bytes as
// contiguous 8-, 1- and 2-byte lanes.  The kernel is HBM-bound: 1,160 bytes
// in (latent + rope + slot) and 352 out per token.
//
// The indexer's keys have their own quantize-on-write below (128 e4m3 values
// and a float scale per token).
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;

// x / d (d > 0) rounded to nearest-even, i.e. the IEEE float32 quotient,
// from the correctly rounded reciprocal and one FMA correction step
// (Markstein's theorem: with r = RN(1/d) and q0 = RN(x r),
// RN(q0 + RN(x - q0 d) r) = RN(x/d) while quotient and residual stay in the
// normal range).  Tiny quotients (x subnormal) round to 0 in both e2m1 and
// e4m3 whichever way their last bit goes.  The correction turns -0 into +0,
// so the quotient takes x's sign explicitly.
__device__ __forceinline__ float div_rn(float x, float d, float r) {
  const float q0 = __fmul_rn(x, r);
  const float e = __fmaf_rn(-q0, d, x);
  return copysignf(__fmaf_rn(e, r, q0), x);
}

template <int FMT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    quantize_append_kernel(const uint16_t* __restrict__ latent, const uint16_t* __restrict__ rope,
                           const int64_t* __restrict__ slot_mapping, int64_t n_tokens, uint8_t* __restrict__ pool,
                           int64_t num_blocks, int64_t block_stride) {
  constexpr int kUnroll = 2;  // tokens per warp per iteration: all their loads are issued first
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t n0 = warp_global; n0 < n_tokens; n0 += kUnroll * warp_stride) {
    int64_t slot[kUnroll];
    uint4 v0[kUnroll], v1[kUnroll];
    uint32_t rope2[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t n = n0 + u * warp_stride;
      slot[u] = -1;
      if (n < n_tokens) {
        slot[u] = __ldg(slot_mapping + n);
        // 16 latent values of group `lane`, as two 16-byte loads.
        const uint4* src = reinterpret_cast<const uint4*>(latent + n * kLatent + lane * kGroup);
        v0[u] = __ldg(src);
        v1[u] = __ldg(src + 1);
        rope2[u] = __ldg(reinterpret_cast<const uint32_t*>(rope + n * kRope) + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (slot[u] < 0 || slot[u] / kBlock >= num_blocks) continue;  // skipped (warp-uniform)
      uint8_t* row =
          pool + (slot[u] / kBlock) * block_stride + (slot[u] % kBlock) * (FMT == 0 ? kRowNvfp4 : kRowFp8);
      const uint32_t w[8] = {v0[u].x, v0[u].y, v0[u].z, v0[u].w, v1[u].x, v1[u].y, v1[u].z, v1[u].w};
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
        x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
      }
      const uint32_t rope_e4m3x2 =
          f32x2_to_e4m3x2(bf16_bits_to_f32(rope2[u] >> 16), bf16_bits_to_f32(rope2[u] & 0xFFFFu));

      if constexpr (FMT == 0) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
        // S = e4m3(amax / 6): IEEE division, then round-to-nearest-even.
        const uint32_t s_code = f32x2_to_e4m3x2(0.f, __fdiv_rn(amax, 6.0f)) & 0xFFu;
        const uint32_t s_f16 = e4m3x2_to_f16x2(s_code) & 0xFFFFu;
        const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(s_f16)));
        uint32_t lo = 0, hi = 0;  // 16 codes: element 2i in the low nibble of byte i
        if (s_code != 0) {
          const float r = __frcp_rn(s);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo |= f32x2_to_e2m1x2(div_rn(x[2 * i + 1], s, r), div_rn(x[2 * i], s, r)) << (8 * i);
            hi |= f32x2_to_e2m1x2(div_rn(x[8 + 2 * i + 1], s, r), div_rn(x[8 + 2 * i], s, r)) << (8 * i);
          }
        }
        *reinterpret_cast<uint2*>(row + lane * 8) = make_uint2(lo, hi);
        row[kScaleOff + lane] = static_cast<uint8_t>(s_code);
        *reinterpret_cast<uint16_t*>(row + kRopeOffNvfp4 + 2 * lane) = static_cast<uint16_t>(rope_e4m3x2);
      } else {
        uint32_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          b[i] = f32x2_to_e4m3x2(x[4 * i + 1], x[4 * i]) | (f32x2_to_e4m3x2(x[4 * i + 3], x[4 * i + 2]) << 16);
        *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(b[0], b[1], b[2], b[3]);
        *reinterpret_cast<uint16_t*>(row + kRopeOffFp8 + 2 * lane) = static_cast<uint16_t>(rope_e4m3x2);
      }
    }
  }
}

// Indexer keys ("GLM-5.3 PCP/DCP long-context on H200", section 3: a key is
// 128 e4m3 bytes and a float scale): s = amax / 448 and codes
// e4m3(k / s), both divisions IEEE single precision; a zero key stores s = 0
// and zero codes.  Four lanes per token: lane l of the four owns values
// [32l, 32l+32) (four 16-byte loads, two 16-byte stores), so the per-token
// scale and reciprocal are shared by 32 values per lane; the amax is a
// 4-lane shuffle reduction.  Block layout: 64 x 128 code bytes, then 64
// floats.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    index_key_append_kernel(const uint16_t* __restrict__ keys, const int64_t* __restrict__ slot_mapping,
                            int64_t n_tokens, uint8_t* __restrict__ pool, int64_t num_blocks,
                            int64_t block_stride) {
  constexpr int kUnroll = 1;  // groups of 8 tokens per warp per iteration (loads of the group issued first)
  const int lane = threadIdx.x & 31;
  const int tok = lane >> 2;  // token of the group
  const int lt = lane & 3;    // lane within the token
  const int64_t warp_global = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
  for (int64_t quad0 = warp_global; 8 * quad0 < n_tokens; quad0 += kUnroll * warp_stride) {
    int64_t slots[kUnroll];
    uint4 vv[kUnroll][4];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t n = 8 * (quad0 + u * warp_stride) + tok;
      const bool in = n < n_tokens;
      slots[u] = in ? __ldg(slot_mapping + n) : -1;
      const uint4* src = reinterpret_cast<const uint4*>(keys + n * kIdxDim) + 4 * lt;
#pragma unroll
      for (int k = 0; k < 4; ++k) vv[u][k] = in ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (8 * (quad0 + u * warp_stride) >= n_tokens) break;  // warp-uniform
      const int64_t slot = slots[u];
      const bool ok = slot >= 0 && slot / kBlock < num_blocks;
      float x[32];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {vv[u][k].x, vv[u][k].y, vv[u][k].z, vv[u][k].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[8 * k + 2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
          x[8 * k + 2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
      for (int off = 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      if (!ok) continue;
      const float s = amax == 0.f ? 0.f : __fdiv_rn(amax, 448.0f);
      uint32_t q[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // 32 codes, value 4k + j in byte j of q[k]
      if (amax != 0.f && s >= 1.17549435e-38f) {  // normal scale: reciprocal and one correction
        const float r = __frcp_rn(s);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          q[k] = f32x2_to_e4m3x2(div_rn(x[4 * k + 1], s, r), div_rn(x[4 * k], s, r)) |
                 (f32x2_to_e4m3x2(div_rn(x[4 * k + 3], s, r), div_rn(x[4 * k + 2], s, r)) << 16);
      } else if (amax != 0.f) {  // subnormal scale (1/s overflows): plain IEEE division
#pragma unroll
        for (int k = 0; k < 8; ++k)
          q[k] = f32x2_to_e4m3x2(__fdiv_rn(x[4 * k + 1], s), __fdiv_rn(x[4 * k], s)) |
                 (f32x2_to_e4m3x2(__fdiv_rn(x[4 * k + 3], s), __fdiv_rn(x[4 * k + 2], s)) << 16);
      }
      uint8_t* blk = pool + (slot / kBlock) * block_stride;
      const int64_t o = slot % kBlock;
      *reinterpret_cast<uint4*>(blk + o * kIdxDim + 32 * lt) = make_uint4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<uint4*>(blk + o * kIdxDim + 32 * lt + 16) = make_uint4(q[4], q[5], q[6], q[7]);
      if (lt == 0) *reinterpret_cast<float*>(blk + static_cast<int64_t>(kBlock) * kIdxDim + 4 * o) = s;
    }
  }
}

}  // namespace

cudaError_t launch_index_key_append(const uint16_t* keys, const int64_t* slot_mapping, int64_t n_tokens, void* pool,
                                    int64_t num_blocks, int64_t block_stride, cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  const int64_t quads = (n_tokens + 7) / 8;
  int64_t want = (quads + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  index_key_append_kernel<<<grid, kWarpsPerBlock * 32, 0, stream>>>(keys, slot_mapping, n_tokens,
                                                                     static_cast<uint8_t*>(pool), num_blocks,
                                                                     block_stride);
  return cudaGetLastError();
}

cudaError_t launch_quantize_append(const uint16_t* latent, const uint16_t* rope, const int64_t* slot_mapping,
                                   int64_t n_tokens, void* pool, int64_t num_blocks, int64_t block_stride, int fmt,
                                   cudaStream_t stream) {
  if (n_tokens <= 0) return cudaSuccess;
  int sms = device_sm_count();
  int64_t want = (n_tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  int64_t cap = static_cast<int64_t>(sms) * 16;  // grid-stride beyond 16 blocks per SM
  int grid = static_cast<int>(want < cap ? want : cap);
  if (fmt == 0)
    quantize_append_kernel<0><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        latent, rope, slot_mapping, n_tokens, static_cast<uint8_t*>(pool), num_blocks, block_stride);
  else
    quantize_append_kernel<1><<<grid, kWarpsPerBlock * 32, 0, stream>>>(
        latent, rope, slot_mapping, n_tokens, static_cast<uint8_t*>(pool), num_blocks, block_stride);
  return cudaGetLastError();
}

}  // namespace mla
