// Host-side declarations shared between the C-ABI layer (mla_api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mla {

// Multiprocessor count of the current device (cached per device).
int device_sm_count();
// Device address of the library's fault word on the current device.
unsigned int* fault_word_ptr();
// Raises a kernel's dynamic shared-memory limit to `bytes` once per device:
// bit d of `*done` records device d (devices past 63 are configured on every
// call).  Safe when host threads drive different devices at once.
cudaError_t set_smem_limit_once(const void* kernel, int bytes, std::atomic<uint64_t>* done);
// True when the driver's tensor-map encoder is available (TMA paths need it).
bool tensor_maps_available();
// A 2-D TMA tensor map (no interleave, zero fill out of bounds) over `rows`
// rows of `inner` elements, rows `row_stride` bytes apart; box
// {box_inner, box_rows}.  False when the driver entry point is unavailable
// or the description is rejected.
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
                          uint64_t rows, uint64_t row_stride, uint32_t box_inner, uint32_t box_rows,
                          CUtensorMapSwizzle swizzle);

cudaError_t launch_quantize_append(const uint16_t* latent, const uint16_t* rope, const int64_t* slot_mapping,
                                   int64_t n_tokens, void* pool, int64_t num_blocks, int64_t block_stride, int fmt,
                                   cudaStream_t stream);

cudaError_t launch_index_key_append(const uint16_t* keys, const int64_t* slot_mapping, int64_t n_tokens, void* pool,
                                    int64_t num_blocks, int64_t block_stride, cudaStream_t stream);

// Staged path: NVFP4 rows re-stored as FP8 rows (staged_bt / staged_ctx may be
// null; when given, the identity block table and context lengths are written).
cudaError_t launch_stage_rows_fp8(const void* pool, int64_t block_stride, int64_t num_blocks,
                                  const int32_t* block_table, int max_blocks_per_req, const int32_t* context_lens,
                                  const int32_t* topk_idx, int batch, int topk, void* staged, int32_t* staged_topk,
                                  int32_t* staged_bt, int32_t* staged_ctx, cudaStream_t stream);

// Sparse decode: split plan and launch.  The plan is made for the number of
// (request, query token) pairs; q_len query tokens per request share its
// block table and context (token i sees t < ctx - (q_len - 1 - i)).
struct DecodePlan {
  int splits;          // CTAs per (request, 16-head group) along the top-k list
  int rows_per_split;  // multiple of 16
  bool cluster;        // the splits form a thread-block cluster and merge through DSMEM
  size_t workspace;    // bytes of split partials in global memory (0 for one split or a cluster merge)
};
DecodePlan plan_sparse_decode(int batch, int num_heads, int topk);
cudaError_t launch_sparse_decode(int fmt, const uint16_t* q_nope, const uint16_t* q_rope, const void* pool,
                                 int64_t block_stride, int64_t num_blocks, const int32_t* block_table,
                                 int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                 int batch, int q_len, int num_heads, int topk, float softmax_scale, uint16_t* out,
                                 float* lse, void* workspace, const DecodePlan& plan, cudaStream_t stream);

// Tensor-memory decode for 64-head blocks of NVFP4 rows in a pool TMA can
// gather from (sparse_decode_tc.cu).  Split partials use the workspace
// layout of the 16-head kernel.
struct TcDecodeParams {
  const uint16_t* q_nope;
  const uint16_t* q_rope;
  int64_t block_stride;
  int64_t num_blocks;
  const int32_t* block_table;
  int max_blocks_per_req;
  const int32_t* context_lens;
  const int32_t* topk_idx;
  int pairs;
  int q_len;
  int num_heads;
  int topk;
  int splits;
  float softmax_scale;
  uint16_t* out;
  float* lse;
  void* part_o;
  float* part_lse;
  unsigned int* fault_word;
};
bool sparse_decode_tc_supported(int fmt, int num_heads);
// The call runs the tensor-memory kernel (format, head count and a pool TMA
// can describe as a tensor of 352-byte rows; the pool base must also be
// 16-byte aligned, which every entry point already requires).
bool sparse_decode_uses_tc(int fmt, int num_heads, int64_t block_stride, int64_t num_blocks);
int plan_sparse_decode_tc(int pairs, int num_heads, int topk, int max_splits);
cudaError_t launch_sparse_decode_tc(const TcDecodeParams& p, const CUtensorMap& map, cudaStream_t stream);

// Indexer and top-k.
size_t topk_workspace_bytes(int batch, int max_context_len, int topk);
cudaError_t launch_topk(const float* scores, int64_t row_stride, const int32_t* context_lens, int batch, int topk,
                        int max_context_len, int32_t* out, void* workspace, cudaStream_t stream);
cudaError_t launch_indexer_scores(const uint16_t* q_idx, const float* head_w, const void* key_pool,
                                  int64_t block_stride, int64_t num_blocks, const int32_t* block_table,
                                  int max_blocks_per_req, const int32_t* context_lens, int batch, int n_heads,
                                  int max_context_len, float* scores, int64_t scores_stride, cudaStream_t stream);

}  // namespace mla
