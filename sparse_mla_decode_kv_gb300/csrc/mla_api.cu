// The C ABI of libmla_nvfp4.so (declared in include/mla_nvfp4.h): host-side
// argument validation, workspace sizing and kernel dispatch.  Nothing here
// allocates device memory; every launch goes to the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mla_nvfp4.h"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace mla {

// Set by bounded device waits that run out (bits in mla_device.cuh); read and
// cleared through mla_device_fault().
__device__ unsigned int g_fault_word = 0;

namespace {

thread_local int t_last_cuda_error = 0;

mla_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  t_last_cuda_error = static_cast<int>(e);
  return MLA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// block_size: 64 is supported; other powers of two are valid but unsupported.
mla_status_t check_block_size(int block_size) {
  if (block_size <= 0 || (block_size & (block_size - 1)) != 0) return MLA_ERR_INVALID_ARG;
  return block_size == kBlock ? MLA_OK : MLA_ERR_UNSUPPORTED;
}

int row_bytes(int fmt) { return fmt == MLA_KV_NVFP4 ? kRowNvfp4 : fmt == MLA_KV_FP8 ? kRowFp8 : 0; }

mla_status_t check_decode_args(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                               int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                               int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                               int batch, int num_heads, int block_size, int topk, float softmax_scale,
                               const uint16_t* out, int fmt) {
  if (batch < 0) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_block_size(block_size);
  if (s != MLA_OK) return s;
  if (num_heads < 16 || num_heads > 128 || num_heads % 16 != 0) return MLA_ERR_INVALID_ARG;
  if (topk < 1 || topk > 2048) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q_nope || !q_rope || !kv_pool || !block_table || !context_lens || !topk_idx || !out)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(q_rope, 8) || !aligned(kv_pool, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(topk_idx, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 0 || max_blocks_per_req < 1) return MLA_ERR_INVALID_ARG;
  if (kv_block_stride % 16 != 0 || kv_block_stride < static_cast<int64_t>(block_size) * row_bytes(fmt))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

constexpr int kMaxQueryTokens = 64;

mla_status_t decode_impl(int fmt, const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                         int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                         int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx, int batch,
                         int q_len, int num_heads, int block_size, int topk, float softmax_scale, uint16_t* out,
                         float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (q_len < 1 || q_len > kMaxQueryTokens) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_decode_args(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                                     max_blocks_per_req, context_lens, topk_idx, batch, num_heads, block_size,
                                     topk, softmax_scale, out, fmt);
  if (s != MLA_OK || batch == 0) return s;
  if (lse && !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
  const DecodePlan plan = plan_sparse_decode(batch * q_len, num_heads, topk);
  if (plan.workspace > 0) {
    if (workspace_bytes < plan.workspace) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  }
  return cuda_status(launch_sparse_decode(fmt, q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                                          max_blocks_per_req, context_lens, topk_idx, batch, q_len, num_heads, topk,
                                          softmax_scale, out, lse, workspace, plan, stream));
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

namespace {
// Per-device caches of the SM count and the fault word's device address.
// Host threads may drive different devices at once: each device has its own
// slot (an atomic, so the fast path takes no lock), filled once under a
// mutex.  A device index past the table is looked up on every call.
constexpr int kMaxCachedDevices = 64;
std::mutex g_cache_mutex;
std::atomic<int> g_sm_count[kMaxCachedDevices];
std::atomic<unsigned int*> g_fault_word_ptr[kMaxCachedDevices];

int query_sm_count(int dev) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  return sms;
}
unsigned int* query_fault_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(p);
}
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev < 0 || dev >= kMaxCachedDevices) return query_sm_count(dev);
  int sms = g_sm_count[dev].load(std::memory_order_acquire);
  if (sms > 0) return sms;
  std::lock_guard<std::mutex> lock(g_cache_mutex);
  sms = g_sm_count[dev].load(std::memory_order_relaxed);
  if (sms <= 0) {
    sms = query_sm_count(dev);
    g_sm_count[dev].store(sms, std::memory_order_release);
  }
  return sms;
}

// The address is cached per device for the life of the process; after a
// cudaDeviceReset the library's device variables may move, so a process that
// resets a device must not call into the library on it again.
unsigned int* fault_word_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxCachedDevices) return query_fault_word();
  unsigned int* p = g_fault_word_ptr[dev].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(g_cache_mutex);
  p = g_fault_word_ptr[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    p = query_fault_word();
    if (p != nullptr) g_fault_word_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); null if unavailable.
EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool tensor_maps_available() { return encode_tiled() != nullptr; }

cudaError_t set_smem_limit_once(const void* kernel, int bytes, std::atomic<uint64_t>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done->load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done->fetch_or(bit, std::memory_order_release);
  return e;
}

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t row_stride, uint32_t box_inner, uint32_t box_rows,
                          CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_kv_row_bytes(mla_kv_format_t fmt) { return static_cast<size_t>(row_bytes(fmt)); }

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
  }
  return "MLA_ERR_UNKNOWN";
}

mla_status_t mla_last_cuda_error(int* cuda_err) {
  if (!cuda_err) return MLA_ERR_INVALID_ARG;
  *cuda_err = t_last_cuda_error;
  return MLA_OK;
}

mla_status_t mla_device_fault(unsigned int* word, int clear, mla_stream_t stream) {
  if (!word) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_fault_word, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_fault_word, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  return cuda_status(e);
}

mla_status_t mla_kv_quantize_append(const uint16_t* latent, const uint16_t* rope, const int64_t* slot_mapping,
                                    int64_t n_tokens, void* kv_pool, int64_t num_blocks, int block_size,
                                    int64_t kv_block_stride, mla_kv_format_t fmt, mla_stream_t stream) {
  if (n_tokens < 0 || num_blocks < 0) return MLA_ERR_INVALID_ARG;
  if (fmt != MLA_KV_NVFP4 && fmt != MLA_KV_FP8) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_block_size(block_size);
  if (s != MLA_OK) return s;
  if (kv_block_stride % 16 != 0 || kv_block_stride < static_cast<int64_t>(block_size) * row_bytes(fmt))
    return MLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return MLA_OK;
  if (!latent || !rope || !slot_mapping || !kv_pool) return MLA_ERR_INVALID_ARG;
  if (!aligned(latent, 16) || !aligned(rope, 4) || !aligned(slot_mapping, 8) || !aligned(kv_pool, 16))
    return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_append(latent, rope, slot_mapping, n_tokens, kv_pool, num_blocks,
                                            kv_block_stride, fmt, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mla_sparse_decode_workspace_size(int batch, int num_heads, int topk) {
  if (batch <= 0 || num_heads < 16 || num_heads % 16 != 0 || topk < 1) return 0;
  return plan_sparse_decode(batch, num_heads, topk).workspace;
}

mla_status_t mla_sparse_decode_plan(int batch, int num_heads, int topk, int* splits, int* rows_per_split,
                                    int* kernels) {
  if (batch <= 0 || num_heads < 16 || num_heads % 16 != 0 || topk < 1) return MLA_ERR_INVALID_ARG;
  const DecodePlan plan = plan_sparse_decode(batch, num_heads, topk);
  if (splits) *splits = plan.splits;
  if (rows_per_split) *rows_per_split = plan.rows_per_split;
  if (kernels) *kernels = (plan.splits > 1 && !plan.cluster) ? 2 : 1;
  return MLA_OK;
}

mla_status_t mla_sparse_decode_plan_fmt(int fmt, int batch, int num_heads, int topk, int64_t kv_block_stride,
                                        int64_t num_blocks, int* splits, int* rows_per_split, int* kernels,
                                        int* tensor_memory) {
  if (fmt != MLA_KV_NVFP4 && fmt != MLA_KV_FP8) return MLA_ERR_INVALID_ARG;
  if (batch <= 0 || num_heads < 16 || num_heads % 16 != 0 || topk < 1) return MLA_ERR_INVALID_ARG;
  const DecodePlan plan = plan_sparse_decode(batch, num_heads, topk);
  const bool tc = sparse_decode_uses_tc(fmt, num_heads, kv_block_stride, num_blocks);
  int s = plan.splits, rows = plan.rows_per_split, k = (plan.splits > 1 && !plan.cluster) ? 2 : 1;
  if (tc) {
    s = plan_sparse_decode_tc(batch, num_heads, topk, plan.splits);
    rows = (topk + s - 1) / s;
    k = s > 1 ? 2 : 1;
  }
  if (splits) *splits = s;
  if (rows_per_split) *rows_per_split = rows;
  if (kernels) *kernels = k;
  if (tensor_memory) *tensor_memory = tc ? 1 : 0;
  return MLA_OK;
}

mla_status_t mla_sparse_decode(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                               int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                               int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                               int batch, int num_heads, int block_size, int topk, float softmax_scale,
                               uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                               mla_stream_t stream) {
  return decode_impl(MLA_KV_NVFP4, q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                     max_blocks_per_req, context_lens, topk_idx, batch, 1, num_heads, block_size, topk,
                     softmax_scale, out, lse, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

mla_status_t mla_sparse_decode_fp8(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                   int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                   int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                   int batch, int num_heads, int block_size, int topk, float softmax_scale,
                                   uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                   mla_stream_t stream) {
  return decode_impl(MLA_KV_FP8, q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                     max_blocks_per_req, context_lens, topk_idx, batch, 1, num_heads, block_size, topk,
                     softmax_scale, out, lse, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

mla_status_t mla_index_key_quantize_append(const uint16_t* keys, const int64_t* slot_mapping, int64_t n_tokens,
                                           void* idx_key_pool, int64_t num_blocks, int block_size,
                                           int64_t idx_block_stride, mla_stream_t stream) {
  if (n_tokens < 0 || num_blocks < 0) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_block_size(block_size);
  if (s != MLA_OK) return s;
  if (idx_block_stride % 16 != 0 || idx_block_stride < static_cast<int64_t>(block_size) * (kIdxDim + 4))
    return MLA_ERR_INVALID_ARG;
  if (n_tokens == 0) return MLA_OK;
  if (!keys || !slot_mapping || !idx_key_pool) return MLA_ERR_INVALID_ARG;
  if (!aligned(keys, 16) || !aligned(slot_mapping, 8) || !aligned(idx_key_pool, 16)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_index_key_append(keys, slot_mapping, n_tokens, idx_key_pool, num_blocks,
                                             idx_block_stride, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mla_staged_pool_bytes(int batch, int topk) {
  if (batch <= 0 || topk < 1) return 0;
  const int64_t nblk = (topk + kBlock - 1) / kBlock;
  return static_cast<size_t>(batch) * nblk * kBlock * kRowFp8;
}

mla_status_t mla_stage_rows_fp8(const void* kv_pool, int64_t kv_block_stride, int64_t num_blocks,
                                const int32_t* block_table, int max_blocks_per_req, const int32_t* context_lens,
                                const int32_t* topk_idx, int batch, int block_size, int topk, void* staged_pool,
                                int32_t* staged_topk, mla_stream_t stream) {
  if (batch < 0 || topk < 1 || topk > 2048) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_block_size(block_size);
  if (s != MLA_OK) return s;
  if (batch == 0) return MLA_OK;
  if (!kv_pool || !block_table || !context_lens || !topk_idx || !staged_pool || !staged_topk)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(kv_pool, 16) || !aligned(staged_pool, 16) || !aligned(block_table, 4) ||
      !aligned(context_lens, 4) || !aligned(topk_idx, 4) || !aligned(staged_topk, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 0 || max_blocks_per_req < 1) return MLA_ERR_INVALID_ARG;
  if (kv_block_stride % 16 != 0 || kv_block_stride < static_cast<int64_t>(block_size) * kRowNvfp4)
    return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_stage_rows_fp8(kv_pool, kv_block_stride, num_blocks, block_table, max_blocks_per_req,
                                           context_lens, topk_idx, batch, topk, staged_pool, staged_topk, nullptr,
                                           nullptr, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// Workspace of the staged decode: staged rows | staged list | identity block
// table | context lengths | the FP8 decode's own split-K workspace.
struct StagedLayout {
  size_t rows, list, table, ctx, decode, total;
};
StagedLayout staged_layout(int batch, int num_heads, int topk) {
  StagedLayout l{};
  const int64_t nblk = (topk + kBlock - 1) / kBlock;
  l.rows = align256(mla_staged_pool_bytes(batch, topk));
  l.list = align256(static_cast<size_t>(batch) * topk * sizeof(int32_t));
  l.table = align256(static_cast<size_t>(batch) * nblk * sizeof(int32_t));
  l.ctx = align256(static_cast<size_t>(batch) * sizeof(int32_t));
  l.decode = align256(plan_sparse_decode(batch, num_heads, topk).workspace);
  l.total = l.rows + l.list + l.table + l.ctx + l.decode;
  return l;
}
}  // namespace

size_t mla_sparse_decode_staged_workspace_size(int batch, int num_heads, int topk) {
  if (batch <= 0 || num_heads < 16 || num_heads % 16 != 0 || topk < 1) return 0;
  return staged_layout(batch, num_heads, topk).total;
}

mla_status_t mla_sparse_decode_staged(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                      int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                      int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                      int batch, int num_heads, int block_size, int topk, float softmax_scale,
                                      uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                      mla_stream_t stream) {
  mla_status_t s = check_decode_args(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table,
                                     max_blocks_per_req, context_lens, topk_idx, batch, num_heads, block_size, topk,
                                     softmax_scale, out, MLA_KV_NVFP4);
  if (s != MLA_OK || batch == 0) return s;
  if (lse && !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
  const StagedLayout l = staged_layout(batch, num_heads, topk);
  if (workspace_bytes < l.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* rows = ws;
  int32_t* list = reinterpret_cast<int32_t*>(ws + l.rows);
  int32_t* table = reinterpret_cast<int32_t*>(ws + l.rows + l.list);
  int32_t* ctx = reinterpret_cast<int32_t*>(ws + l.rows + l.list + l.table);
  void* dec_ws = ws + l.rows + l.list + l.table + l.ctx;
  const int nblk = (topk + kBlock - 1) / kBlock;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_stage_rows_fp8(kv_pool, kv_block_stride, num_blocks, block_table, max_blocks_per_req,
                                        context_lens, topk_idx, batch, topk, rows, list, table, ctx, st);
  if (e != cudaSuccess) return cuda_status(e);
  const DecodePlan plan = plan_sparse_decode(batch, num_heads, topk);
  return cuda_status(launch_sparse_decode(MLA_KV_FP8, q_nope, q_rope, rows, static_cast<int64_t>(kBlock) * kRowFp8,
                                          static_cast<int64_t>(batch) * nblk, table, nblk, ctx, list, batch, 1,
                                          num_heads, topk, softmax_scale, out, lse, dec_ws, plan, st));
}

size_t mla_sparse_decode_mtp_workspace_size(int batch, int q_len, int num_heads, int topk) {
  if (batch <= 0 || q_len < 1 || q_len > kMaxQueryTokens || num_heads < 16 || num_heads % 16 != 0 || topk < 1)
    return 0;
  return plan_sparse_decode(batch * q_len, num_heads, topk).workspace;
}

mla_status_t mla_sparse_decode_mtp(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                   int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                   int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                   int batch, int q_len, int num_heads, int block_size, int topk, float softmax_scale,
                                   mla_kv_format_t fmt, uint16_t* out, float* lse, void* workspace,
                                   size_t workspace_bytes, mla_stream_t stream) {
  if (fmt != MLA_KV_NVFP4 && fmt != MLA_KV_FP8) return MLA_ERR_INVALID_ARG;
  return decode_impl(fmt, q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, max_blocks_per_req,
                     context_lens, topk_idx, batch, q_len, num_heads, block_size, topk, softmax_scale, out, lse,
                     workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t mla_topk_workspace_size(int batch, int max_context_len, int topk) {
  if (batch <= 0 || max_context_len < 0 || topk < 1) return 0;
  return topk_workspace_bytes(batch, max_context_len, topk);
}

mla_status_t mla_topk(const float* scores, int64_t score_row_stride, const int32_t* context_lens, int batch,
                      int topk, int max_context_len, int32_t* topk_out, void* workspace, size_t workspace_bytes,
                      mla_stream_t stream) {
  if (batch < 0 || topk < 1 || topk > 2048 || max_context_len < 0) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!scores || !context_lens || !topk_out) return MLA_ERR_INVALID_ARG;
  if (score_row_stride < max_context_len || !aligned(scores, 4) || !aligned(topk_out, 4)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < topk_workspace_bytes(batch, max_context_len, topk)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_topk(scores, score_row_stride, context_lens, batch, topk, max_context_len, topk_out,
                                 workspace, reinterpret_cast<cudaStream_t>(stream)));
}

size_t mla_indexer_topk_workspace_size(int batch, int max_context_len, int topk) {
  if (batch <= 0 || max_context_len <= 0 || topk < 1) return 0;
  const size_t scores = align256(static_cast<size_t>(batch) * max_context_len * sizeof(float));
  return scores + align256(topk_workspace_bytes(batch, max_context_len, topk));
}

mla_status_t mla_indexer_topk(const uint16_t* q_idx, const float* head_w, const void* idx_key_pool,
                              int64_t idx_block_stride, int64_t num_blocks, const int32_t* block_table,
                              int max_blocks_per_req, const int32_t* context_lens, int batch, int n_idx_heads,
                              int block_size, int topk, int32_t* topk_out, float* scores_out, int max_context_len,
                              void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (batch < 0 || topk < 1 || topk > 2048 || max_context_len < 0) return MLA_ERR_INVALID_ARG;
  mla_status_t s = check_block_size(block_size);
  if (s != MLA_OK) return s;
  if (n_idx_heads != 8 && n_idx_heads != 16 && n_idx_heads != 32 && n_idx_heads != 64) {
    return (n_idx_heads > 0 && n_idx_heads % 8 == 0 && n_idx_heads <= 64) ? MLA_ERR_UNSUPPORTED
                                                                          : MLA_ERR_INVALID_ARG;
  }
  if (batch == 0) return MLA_OK;
  if (!q_idx || !head_w || !idx_key_pool || !block_table || !context_lens || !topk_out) return MLA_ERR_INVALID_ARG;
  if (!aligned(q_idx, 16) || !aligned(head_w, 4) || !aligned(idx_key_pool, 16)) return MLA_ERR_INVALID_ARG;
  if (idx_block_stride % 16 != 0 || idx_block_stride < static_cast<int64_t>(block_size) * (kIdxDim + 4))
    return MLA_ERR_INVALID_ARG;
  if (num_blocks < 0 || max_blocks_per_req < 1) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_indexer_topk_workspace_size(batch, max_context_len, topk);
  float* scores = scores_out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (need > 0) {
    if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
    if (!workspace || !aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  }
  if (scores == nullptr) scores = reinterpret_cast<float*>(ws);
  else if (!aligned(scores, 4)) return MLA_ERR_INVALID_ARG;
  const size_t scores_bytes = align256(static_cast<size_t>(batch) * max_context_len * sizeof(float));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_indexer_scores(q_idx, head_w, idx_key_pool, idx_block_stride, num_blocks, block_table,
                                        max_blocks_per_req, context_lens, batch, n_idx_heads, max_context_len, scores,
                                        max_context_len, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_topk(scores, max_context_len, context_lens, batch, topk, max_context_len, topk_out,
                                 ws ? ws + scores_bytes : nullptr, st));
}

}  // extern "C"
