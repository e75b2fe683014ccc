/*
 * mla_nvfp4.h -- C ABI of libmla_nvfp4.so: sparse multi-head latent attention
 * (MLA) decode over a paged latent KV cache stored as NVFP4 (352-byte rows)
 * or FP8 (576-byte rows), for NVIDIA GB300 (sm_103a).
 *
 * What the operations are, and where they are defined:
 *
 *  - The cached row.  A token's cache entry is a 512-value latent and a
 *    64-value rotary key shared by all heads (no head axis); every attention head reads the
 *    same row ("Prime Inference: serving GLM-5.3 to agents is a KV-cache
 *    problem", section "Prefill topology").  Stored as NVFP4 it is 256 bytes
 *    of 4-bit e2m1 codes, 32 one-byte e4m3 scales (one per 16 latent values)
 *    and 64 one-byte e4m3 rope values = 352 bytes; stored as FP8 it is 512 +
 *    64 e4m3 bytes = 576 bytes (same page, section "Four bits per latent
 *    value: where 352 comes from", row table).
 *  - Sparse selection.  The indexer rates all preceding tokens and attention
 *    reads at most top-k = 2,048 of them ("GLM-5.3 PCP/DCP long-context on
 *    H200", section 1; "Prime Inference", section "Decode: TP4, and the
 *    copies it keeps", index_topk 2048).  An indexer key is 128 e4m3 bytes
 *    and a float scale (PCP/DCP page, section 3).
 *  - Decode.  The selected rows are gathered through the block table,
 *    unpacked on chip, scored against every head's absorbed query, soft-maxed
 *    and blended, with no FP8 or BF16 copy written to memory ("Prime
 *    Inference", section "A kernel that reads four bits directly", figure
 *    "staged vs native decode"); when a context is shorter than top-k the
 *    list carries -1 entries, which are skipped (same section).
 *
 * Row layout inside the 352 bytes (the pages give only the totals):
 *   [0,256)   latent codes, element 2i in the low nibble of byte i
 *   [256,288) e4m3 scale g for latent elements [16g, 16g+16)
 *   [288,352) rope, e4m3
 * FP8 row: [0,512) latent e4m3, [512,576) rope e4m3.
 * Quantization: S_g = e4m3_rn_satfinite(max_i |x_i| / 6) (IEEE float32
 * division), code_i = e2m1_rn_satfinite(x_i / S_g), ties to even, the sign
 * bit copies the sign of x_i; a group whose S_g encodes to 0 stores sixteen
 * 0x0 codes; rope and FP8 latent values are e4m3_rn_satfinite(x).
 *
 * Conventions for every entry point:
 *  - All pointers marked "device" are CUDA device pointers on the current
 *    device; the caller owns every buffer.  The library allocates nothing and
 *    keeps no per-call state; scratch memory comes in through `workspace`.
 *  - Work is enqueued on `stream` and returns immediately (asynchronous).
 *  - Host-side argument errors return MLA_ERR_INVALID_ARG or
 *    MLA_ERR_UNSUPPORTED synchronously, before any launch; a launch failure
 *    returns MLA_ERR_CUDA and mla_last_cuda_error() gives the CUDA code.
 *  - Device data is never trusted: a top-k entry outside [0, context_len)
 *    (including -1), a logical block past max_blocks_per_req and a physical
 *    block id outside [0, num_blocks) are skipped (no load, no weight), and
 *    an out-of-range slot in mla_kv_quantize_append is not written.
 *  - bf16 arguments are passed as uint16_t bit patterns.
 *  - Every bounded device wait that runs out sets a bit in a library-wide
 *    device fault word (see mla_device_fault) instead of hanging; it never
 *    traps.
 */
#ifndef MLA_NVFP4_H
#define MLA_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* the same type as cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,        /* null pointer, bad size, misalignment */
  MLA_ERR_UNSUPPORTED = 2,        /* a valid value this build does not handle */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,
  MLA_ERR_CUDA = 4                /* a CUDA call or launch failed */
} mla_status_t;

typedef enum {
  MLA_KV_NVFP4 = 0, /* 352-byte rows */
  MLA_KV_FP8 = 1    /* 576-byte rows */
} mla_kv_format_t;

/* Bytes of one cached row: 352 (NVFP4), 576 (FP8), 0 for an unknown format. */
size_t mla_kv_row_bytes(mla_kv_format_t fmt);

/* A static, human-readable name of a status code. */
const char* mla_status_string(mla_status_t s);

/* The CUDA error code behind this thread's last MLA_ERR_CUDA (0 if none).
 * Thread-local; returns MLA_ERR_INVALID_ARG if cuda_err is NULL. */
mla_status_t mla_last_cuda_error(int* cuda_err);

/* Reads (and, if `clear` is nonzero, resets) the device fault word of the
 * current device: bit 0 = a decode wait ran out, bit 1 = an indexer or top-k
 * wait ran out.  Synchronises `stream`.  A nonzero word means some output of
 * an earlier call is incomplete. */
mla_status_t mla_device_fault(unsigned int* word, int clear, mla_stream_t stream);

/*
 * Quantize-on-write ("Prime Inference", section "Four bits per latent
 * value"; Prime Intellect's post: NVFP4 is the storage format).
 *
 *   latent        device bf16 [n_tokens, 512], row stride 512
 *   rope          device bf16 [n_tokens, 64], row stride 64
 *   slot_mapping  device int64 [n_tokens]; token n is written to block
 *                 slot / block_size, row slot % block_size; a negative slot
 *                 or one at or past num_blocks * block_size is skipped
 *   kv_pool       device, 16-byte aligned; block b starts at
 *                 kv_pool + b * kv_block_stride
 *   kv_block_stride  bytes, a multiple of 16, >= block_size * row bytes
 *   block_size    64 (other powers of two: MLA_ERR_UNSUPPORTED)
 * n_tokens == 0 is a no-op.  Two tokens with the same slot race.
 */
mla_status_t mla_kv_quantize_append(const uint16_t* latent, const uint16_t* rope, const int64_t* slot_mapping,
                                    int64_t n_tokens, void* kv_pool, int64_t num_blocks, int block_size,
                                    int64_t kv_block_stride, mla_kv_format_t fmt, mla_stream_t stream);

/*
 * Quantize-on-write of the indexer's keys ("GLM-5.3 PCP/DCP long-context on
 * H200", section 3: a key is 128 e4m3 bytes and a float scale).  Per
 * token: s = max_d |k_d| / 448 and code_d = e4m3_rn_satfinite(k_d / s), both
 * divisions IEEE float32; a key whose values are all zero stores s = 0 and
 * 128 zero codes.  Block layout (the layout mla_indexer_topk reads): block b
 * at idx_key_pool + b * idx_block_stride holds block_size x 128 code bytes,
 * then block_size float scales.
 *
 *   keys          device bf16 [n_tokens, 128], 16-byte aligned
 *   slot_mapping  device int64 [n_tokens]; as for mla_kv_quantize_append
 *                 (a negative or out-of-pool slot is skipped)
 *   idx_key_pool  device, 16-byte aligned
 *   idx_block_stride  bytes, a multiple of 16, >= block_size * 132
 *   block_size    64
 * n_tokens == 0 is a no-op.  Two tokens with the same slot race.
 */
mla_status_t mla_index_key_quantize_append(const uint16_t* keys, const int64_t* slot_mapping, int64_t n_tokens,
                                           void* idx_key_pool, int64_t num_blocks, int block_size,
                                           int64_t idx_block_stride, mla_stream_t stream);

/*
 * Absorbed-form sparse MLA decode over the NVFP4 cache ("Prime Inference",
 * section "A kernel that reads four bits directly").  For request b and head
 * h, with V_b = { t in topk_idx[b, :] : 0 <= t < context_lens[b] } (counted
 * with multiplicity) and c_t, r_t the dequantized latent and rope of token t
 * (logical block t / 64 through block_table[b, :]):
 *
 *   z[h,t]   = softmax_scale * (q_nope[b,h] . c_t + q_rope[b,h] . r_t)
 *   out[b,h] = sum_t softmax_t(z[h,.]) * c_t           (bf16, 512 values)
 *   lse[b,h] = log sum_t exp(z[h,t])                   (natural log, float)
 *
 * An empty V_b gives out = 0 and lse = -inf.  Arithmetic: FP16 tensor-core
 * operands (the dequantized values are exact in FP16; each head's q is
 * scaled by a power of two into [2^14, 2^15) before its bf16 -> FP16
 * conversion, the inverse folded into that head's softmax scale, so any
 * finite bf16 query is accepted) and FP32 accumulation and softmax; when
 * the list is split over several CTAs (mla_sparse_decode_plan), each split's
 * normalised partial output is rounded to FP16 in the workspace before the
 * FP32 LSE-weighted merge.
 *
 *   q_nope        device bf16 [batch, num_heads, 512] (W_UK already absorbed)
 *   q_rope        device bf16 [batch, num_heads, 64]
 *   kv_pool, kv_block_stride, num_blocks   as for mla_kv_quantize_append
 *   block_table   device int32 [batch, max_blocks_per_req]
 *   context_lens  device int32 [batch]
 *   topk_idx      device int32 [batch, topk], logical positions; any order
 *   num_heads     16, 32, 48, ..., 128
 *   topk          1..2048
 *   out           device bf16 [batch, num_heads, 512]
 *   lse           device float [batch, num_heads], or NULL
 *   workspace     device, 256-byte aligned, at least
 *                 mla_sparse_decode_workspace_size(batch, num_heads, topk)
 *                 bytes (that size depends on the current device and may be
 *                 0); contents on entry do not matter
 * batch == 0 is a no-op.
 */
size_t mla_sparse_decode_workspace_size(int batch, int num_heads, int topk);

/*
 * How mla_sparse_decode (and the FP8, no-alloc and draft-token variants, the
 * latter with batch = requests x query tokens) divides one call's work on the
 * current device.  Each (request, 16-head group) is split along its top-k
 * list into *splits CTAs of *rows_per_split entries (a multiple of 16); the
 * splits' partial outputs are combined by their LSEs.  *kernels is the number
 * of kernels the call launches: 1 for one split, or for 2..8 splits, which
 * form a thread-block cluster and merge inside the decode kernel; 2 for more
 * splits, merged by a second kernel.  Output pointers may be NULL.
 * MLA_ERR_INVALID_ARG for batch < 1, num_heads not a positive multiple of
 * 16, or topk < 1.
 *
 * The plan describes the 16-head kernel.  An NVFP4 call whose num_heads is a
 * multiple of 64 and whose pool stride is a whole number of 352-byte rows
 * runs the tensor-memory kernel instead: one CTA per (request, 64-head
 * block) and split, min(SMs / blocks, ceil(topk / 128), *splits) splits of
 * equal length (at least 1), merged by a second kernel when there are
 * several.  The workspace size covers both.
 */
mla_status_t mla_sparse_decode_plan(int batch, int num_heads, int topk, int* splits, int* rows_per_split,
                                    int* kernels);

/*
 * The division a call with this cache format and pool geometry actually
 * uses: as mla_sparse_decode_plan, and *tensor_memory = 1 when the call runs
 * the tensor-memory kernel (fmt MLA_KV_NVFP4, num_heads a multiple of 64,
 * kv_block_stride a whole number of 352-byte rows, num_blocks > 0 and fewer
 * than 2^31 pool rows; the pool base 16-byte aligned, as every call
 * requires).  Its splits are then per (request, 64-head block) with
 * ceil(topk / splits) rows each, and *kernels is 2 when a merge follows.
 * Output pointers may be NULL.  MLA_ERR_INVALID_ARG for an unknown fmt or
 * the arguments mla_sparse_decode_plan rejects.
 */
mla_status_t mla_sparse_decode_plan_fmt(int fmt, int batch, int num_heads, int topk, int64_t kv_block_stride,
                                        int64_t num_blocks, int* splits, int* rows_per_split, int* kernels,
                                        int* tensor_memory);
mla_status_t mla_sparse_decode(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                               int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                               int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                               int batch, int num_heads, int block_size, int topk, float softmax_scale,
                               uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                               mla_stream_t stream);

/*
 * Allocation-free variant of mla_sparse_decode (NVFP4 cache).  The pages
 * describe no such entry point; it exists for callers that cannot allocate
 * device memory when they call the decode: a serving process that reserves
 * its whole device-memory budget at start-up and may not grow it afterwards,
 * or a plain C host that embeds this library without a device allocator of
 * its own.  Those callers still own and pass every input and output buffer;
 * only the split-K scratch moves into the library.
 *
 *  - Arguments, results and errors are those of mla_sparse_decode, without
 *    the workspace pair.
 *  - The scratch is one file-scope device array of
 *    MLA_SPARSE_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which
 *    loads the library holds until the process exits.  A call whose
 *    mla_sparse_decode_workspace_size(batch, num_heads, topk) exceeds it
 *    returns MLA_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *  - The first call on a device looks up that device's address of the array
 *    (with the device current) and caches it; make that first call before any
 *    stream capture.  The call itself never calls cudaMalloc or cudaFree.
 *    The cached address does not survive cudaDeviceReset (the array may be
 *    placed elsewhere when the library's module is loaded again): a process
 *    that resets a device must not call this entry point on it afterwards.
 *  - Every call on a device shares the same array, which keeps whatever the
 *    last call left there (nothing in it needs to start at zero).  Calls that
 *    overlap on the GPU -- on different streams, or from different host
 *    threads -- race on it and must be serialised by the caller.
 */
#define MLA_SPARSE_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
mla_status_t mla_sparse_decode_noalloc(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                       int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                       int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                       int batch, int num_heads, int block_size, int topk, float softmax_scale,
                                       uint16_t* out, float* lse, mla_stream_t stream);

/* The same decode over the 576-byte FP8 cache: c_t and r_t are the e4m3
 * bytes themselves.  This is the in-library comparison path ("Prime
 * Inference", figure "staged vs native decode": FP8 attention on a real FP8
 * cache).  Identical arguments and workspace size. */
mla_status_t mla_sparse_decode_fp8(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                   int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                   int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                   int batch, int num_heads, int block_size, int topk, float softmax_scale,
                                   uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                   mla_stream_t stream);

/*
 * Several query tokens per request, decoded in one launch (speculative draft
 * tokens: "Prime Inference", section "A kernel that reads four bits
 * directly" -- the native kernel handles 15 query tokens in one launch).  Each
 * query token has its own top-k list; the q_len tokens of request b are the
 * last q_len positions of its context_lens[b] tokens, so token i sees only
 * t < context_lens[b] - (q_len - 1 - i) (entries at or past that bound are
 * masked like any out-of-context entry).  Otherwise the decode of each token
 * is exactly that of mla_sparse_decode (fmt MLA_KV_NVFP4) or
 * mla_sparse_decode_fp8 (fmt MLA_KV_FP8).
 *
 *   q_nope        device bf16 [batch, q_len, num_heads, 512]
 *   q_rope        device bf16 [batch, q_len, num_heads, 64]
 *   topk_idx      device int32 [batch, q_len, topk]
 *   q_len         1..64
 *   out           device bf16 [batch, q_len, num_heads, 512]
 *   lse           device float [batch, q_len, num_heads], or NULL
 *   workspace     at least mla_sparse_decode_mtp_workspace_size(batch,
 *                 q_len, num_heads, topk) bytes, 256-byte aligned
 * All other arguments as for mla_sparse_decode.
 */
size_t mla_sparse_decode_mtp_workspace_size(int batch, int q_len, int num_heads, int topk);
mla_status_t mla_sparse_decode_mtp(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                   int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                   int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                   int batch, int q_len, int num_heads, int block_size, int topk, float softmax_scale,
                                   mla_kv_format_t fmt, uint16_t* out, float* lse, void* workspace,
                                   size_t workspace_bytes, mla_stream_t stream);

/*
 * Staged path, kept as an ablation of the native decode ("Prime Inference",
 * section "A kernel that reads four bits directly", figure "staged vs native
 * decode": the first version gathered the selected NVFP4 rows, wrote an FP8
 * copy of each to GPU memory and ran the FP8 attention kernel on the copy,
 * moving 352 + 576 + 576 bytes per selected row instead of 352).
 *
 * mla_stage_rows_fp8 is the gather step.  For request b and list entry j
 * with token t = topk_idx[b, j], valid exactly when mla_sparse_decode would
 * use it, the 576-byte FP8 row holding e4m3_rn_satfinite(e2m1 x S) for each
 * latent value and the row's 64 rope bytes unchanged is written at
 *   staged_pool + (b * nblk * 64 + j) * 576,   nblk = ceil(topk / 64),
 * and staged_topk[b, j] = j; a masked entry writes staged_topk[b, j] = -1
 * and no row.  With block table [b, i] = b * nblk + i and context length
 * nblk * 64, the staged pool is an ordinary FP8 pool (block stride
 * 64 * 576) for mla_sparse_decode_fp8 with staged_topk as its list.
 *
 *   kv_pool ... topk   as for mla_sparse_decode (NVFP4 pool)
 *   staged_pool   device, 16-byte aligned, mla_staged_pool_bytes(batch, topk)
 *   staged_topk   device int32 [batch, topk]
 *
 * mla_sparse_decode_staged runs both steps (the gather, then the FP8 decode)
 * with every intermediate in `workspace`; its arguments and results are those
 * of mla_sparse_decode, and its outputs differ from the native decode's only
 * by the e4m3 rounding of the staged copy.
 */
size_t mla_staged_pool_bytes(int batch, int topk);
mla_status_t mla_stage_rows_fp8(const void* kv_pool, int64_t kv_block_stride, int64_t num_blocks,
                                const int32_t* block_table, int max_blocks_per_req, const int32_t* context_lens,
                                const int32_t* topk_idx, int batch, int block_size, int topk, void* staged_pool,
                                int32_t* staged_topk, mla_stream_t stream);
size_t mla_sparse_decode_staged_workspace_size(int batch, int num_heads, int topk);
mla_status_t mla_sparse_decode_staged(const uint16_t* q_nope, const uint16_t* q_rope, const void* kv_pool,
                                      int64_t kv_block_stride, int64_t num_blocks, const int32_t* block_table,
                                      int max_blocks_per_req, const int32_t* context_lens, const int32_t* topk_idx,
                                      int batch, int num_heads, int block_size, int topk, float softmax_scale,
                                      uint16_t* out, float* lse, void* workspace, size_t workspace_bytes,
                                      mla_stream_t stream);

/*
 * Exact top-k over float scores ("GLM-5.3 PCP/DCP long-context on H200",
 * section 1: attention reads only the 2,048 tokens the indexer rates best).
 * For request b the candidates are t in [0, min(context_lens[b],
 * max_context_len)), ordered by (score descending, t ascending), with -0.0
 * equal to +0.0; the first min(k, n) are written to topk_out[b, :] in
 * ascending t, and the rest of the row is -1.  NaN scores are not supported.
 *
 *   scores        device float, request b at scores + b * score_row_stride
 *   topk_out      device int32 [batch, topk]
 *   topk          1..2048
 *   workspace     device, 256-byte aligned, at least
 *                 mla_topk_workspace_size(...) bytes (candidate lists of
 *                 the parallel collection pass); contents on entry do not
 *                 matter
 */
size_t mla_topk_workspace_size(int batch, int max_context_len, int topk);
mla_status_t mla_topk(const float* scores, int64_t score_row_stride, const int32_t* context_lens, int batch,
                      int topk, int max_context_len, int32_t* topk_out, void* workspace, size_t workspace_bytes,
                      mla_stream_t stream);

/*
 * Indexer score plus exact top-k.  For request b and t < context_lens[b]:
 *
 *   score[b,t] = sum_h head_w[b,h] * max(0, s_t * (q_idx[b,h] . k_t))
 *
 * where k_t is the token's 128 e4m3 key values and s_t its float scale
 * ("GLM-5.3 PCP/DCP long-context on H200", section 3: a key is 128 e4m3
 * bytes and a float scale); then topk_out = mla_topk(score).  The products
 * run on the tensor cores with FP32 accumulation.  Each head's query is
 * first scaled by a power of two 2^k_h and its weight by 2^-k_h (exact:
 * relu is positively homogeneous), so any finite bf16 query is accepted.
 * With 32 or 64 index heads and a block stride that is a multiple of 128
 * bytes the operands are e4m3: the keys as stored, the query scaled into
 * [128, 256) and split into two e4m3 parts (an element is represented to
 * within max|q_h| 2^-17).  Otherwise they are FP16: the keys exact, the
 * query scaled into [2^14, 2^15) (exact for elements above 2^-10 of the
 * head's largest, FP16 subnormals below that).
 *
 *   q_idx         device bf16 [batch, n_idx_heads, 128]
 *   head_w        device float [batch, n_idx_heads]
 *   idx_key_pool  device, 16-byte aligned; block b at idx_key_pool +
 *                 b * idx_block_stride holds block_size x 128 key bytes
 *                 followed by block_size float scales
 *   idx_block_stride  bytes, a multiple of 16, >= block_size * 132
 *   n_idx_heads   8, 16, 32 or 64 (other multiples of 8 up to 64 return
 *                 MLA_ERR_UNSUPPORTED, anything else MLA_ERR_INVALID_ARG)
 *   topk_out      device int32 [batch, topk]
 *   scores_out    device float [batch, max_context_len] (entries past a
 *                 request's context are left untouched), or NULL to keep
 *                 the scores in the workspace only
 *   max_context_len  >= every context_lens[b] that should be fully scored;
 *                 longer contexts are cut to it
 */
size_t mla_indexer_topk_workspace_size(int batch, int max_context_len, int topk);
mla_status_t mla_indexer_topk(const uint16_t* q_idx, const float* head_w, const void* idx_key_pool,
                              int64_t idx_block_stride, int64_t num_blocks, const int32_t* block_table,
                              int max_blocks_per_req, const int32_t* context_lens, int batch, int n_idx_heads,
                              int block_size, int topk, int32_t* topk_out, float* scores_out, int max_context_len,
                              void* workspace, size_t workspace_bytes, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_NVFP4_H */
