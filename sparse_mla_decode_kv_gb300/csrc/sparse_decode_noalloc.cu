// mla_sparse_decode_noalloc: the NVFP4 sparse decode for callers that cannot
// hand the library a workspace.  Its split-K scratch is a fixed, file-scope
// device array instead of caller memory; nothing here allocates.
//
// Some callers cannot allocate device memory at call time: a serving process
// that reserves its whole device-memory budget at start-up and must not grow
// it afterwards, or a plain C host that embeds the library without any device
// allocator of its own.  They still own and pass every input and output
// buffer; only the scratch moves into the library.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mla_nvfp4.h"
#include "mla_device.cuh"
#include "mla_internal.h"

namespace {

// Split-K partials: per request-head and split, 512 f16 values of the
// normalised partial output plus one float log-sum-exp.
// Every GPU that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = MLA_SPARSE_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The array's name is only a host-side stand-in: its device address has to be
// looked up once per device, with that device current.  The cache is not
// invalidated by cudaDeviceReset; the header says so.
mla_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_sparse_decode_noalloc(const uint16_t* q_nope, const uint16_t* q_rope,
                                                  const void* kv_pool, int64_t kv_block_stride, int64_t num_blocks,
                                                  const int32_t* block_table, int max_blocks_per_req,
                                                  const int32_t* context_lens, const int32_t* topk_idx, int batch,
                                                  int num_heads, int block_size, int topk, float softmax_scale,
                                                  uint16_t* out, float* lse, mla_stream_t stream) {
  // Same validation and plan as mla_sparse_decode; the scratch must fit the array.
  const size_t need = mla_sparse_decode_workspace_size(batch, num_heads, topk);
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (batch > 0) {
    const mla_status_t s = scratch_for_current_device(&scratch);
    if (s != MLA_OK) return s;
  }
  return mla_sparse_decode(q_nope, q_rope, kv_pool, kv_block_stride, num_blocks, block_table, max_blocks_per_req,
                           context_lens, topk_idx, batch, num_heads, block_size, topk, softmax_scale, out, lse,
                           scratch, kScratchBytes, stream);
}
