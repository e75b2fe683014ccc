/*
 * mla_oracle.c -- plain, slow, float64 CPU oracle for sparse MLA decode over
 * an NVFP4 (or FP8) paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load or call this code.  The
 * product path (the CUDA library) never does, and shares no code with it: no
 * headers, tables, constants or helpers.  Everything here is written from the
 * definitions, in the order they are stated, with no blocking or fusion.
 *
 * Sources (page titles; sections / tables / figures on them):
 *  [P1] "Prime Inference: serving GLM-5.3 to agents is a KV-cache problem"
 *       (ai.thesatyajit.com): section "Four bits per latent value: where 352
 *       comes from" (row table: FP8 row 576 B, NVFP4 row 256 + 32 + 64 B);
 *       section "A kernel that reads four bits directly" (on-chip unpack,
 *       FP16 operands with FP32 accumulation, -1 entries zero-filled);
 *       section "Decode: TP4, and the copies it keeps" (index_topk 2048);
 *       section "Prefill topology" (512-value latent + 64-value rotary key,
 *       all heads up-project from the same latent).
 *  [P3] Prime Intellect's own post (aioga.com copy), paragraphs on NVFP4:
 *       the latent is stored as 4-bit values with one FP8 scale per 16 of
 *       them, and the 64 positional values are kept in FP8.
 *  [P5] "GLM-5.3 PCP/DCP long-context on H200", section 1 (the indexer
 *       rates all preceding tokens and attention reads only the 2,048 best)
 *       and section 3 (an indexer key is 128 e4m3 bytes and a float scale).
 *  Number formats the pages name but do not print: OCP 8-bit floating point
 *  specification (E4M3, "fn" variant: no infinities, S.1111.111 = NaN, max
 *  448) and OCP Microscaling Formats (MX) v1.0 (FP4 E2M1: values 0, 0.5, 1,
 *  1.5, 2, 3, 4, 6 and a sign bit).
 *
 * Readings where the pages are silent (the CUDA path implements the same ones):
 *  R-layout   NVFP4 row = [0,256) packed e2m1 codes, element 2i in the LOW
 *             nibble of byte i; [256,288) 32 e4m3 scales, scale g covering
 *             latent elements [16g,16g+16); [288,352) 64 rope values e4m3.
 *             FP8 row = [0,512) latent e4m3, [512,576) rope e4m3.
 *  R-scale    S_g = e4m3_rn_satfinite(amax_g / 6); no per-row or per-tensor
 *             second-level scale (the 352-byte total leaves no room for one).
 *  R-round    round-to-nearest-even everywhere; satfinite (clamp to the
 *             largest finite magnitude, never NaN).
 *  R-sign     the sign bit of every code copies the sign of the input, also
 *             when the magnitude rounds to zero (IEEE conversion semantics).
 *  R-zero     when S_g encodes to 0x00, all 16 codes of the group are 0x0.
 *  R-mask     a top-k entry outside [0, context_len) (including -1) is
 *             masked: no load and no weight (it does not enter the softmax).
 *  R-empty    a request with no valid entry outputs zeros and lse = -inf.
 *  R-keys     indexer key block = bs x 128 e4m3 bytes, then bs fp32 scales.
 *  R-causal  with Q query tokens per request, token i is the (Q-1-i)-th
 *             last position: it sees t < context_len - (Q - 1 - i).
 *  R-stage   the staged path's FP8 copy of an NVFP4 row holds
 *             e4m3_rn_satfinite(e2m1 * S) per latent value, rope bytes copied.
 *  R-keyscale indexer key scale s = amax / 448, codes e4m3(k / s), both
 *             divisions in IEEE single precision; amax = 0 -> s = 0, codes 0.
 *  R-topk     order by (score descending, token index ascending), take the
 *             first min(k, ctx), emit them in ascending index order, pad -1.
 *             -0.0 compares equal to +0.0.
 *
 * Build: gcc -std=c11 -O2 -fPIC -shared (no -ffast-math: the rounding
 * decisions below rely on IEEE double arithmetic and nearbyint()).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                           */
/* ------------------------------------------------------------------------ */

/* bfloat16 bit pattern -> double (bf16 is the upper half of an IEEE float). */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn"): bias 7, 3 mantissa bits, exponent field 0 is
 * subnormal (m/8 * 2^-6), S.1111.111 is NaN, no infinities. */
double oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* OCP MX FP4 E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: m * 0.5. */
double oracle_e2m1_to_double(uint8_t code) {
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 0x3;
  int m = code & 0x1;
  double v;
  if (e == 0)
    v = 0.5 * (double)m;
  else
    v = ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -v : v;
}

/* Round a finite double to E4M3, nearest-even, saturating to +-448.
 * The sign bit copies signbit(x) (R-sign). */
uint8_t oracle_e4m3_from_double(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  int e;        /* unbiased exponent of a in [1, 2) form */
  double q;     /* mantissa steps, rounded to nearest even */
  if (a >= 448.0) return sign | 0x7E; /* largest finite: 1.75 * 2^8 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9 */
    q = nearbyint(a * 512.0);
    if (q >= 8.0) return sign | 0x08; /* rounded up to the smallest normal */
    return sign | (uint8_t)q;
  }
  (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;             /* a = (1 + frac) * 2^e */
  q = nearbyint((ldexp(a, -e) - 1.0) * 8.0);
  if (q >= 8.0) { q = 0.0; e += 1; }
  if (e > 8 || (e == 8 && q > 6.0)) return sign | 0x7E; /* saturate */
  return sign | (uint8_t)(((e + 7) << 3) | (int)q);
}

/* Round a finite double to E2M1, nearest-even, saturating to +-6.
 * The grid is 0, 0.5, 1, 1.5 (step 0.5), 2, 3 (step 1), 4, 6 (step 2). */
uint8_t oracle_e2m1_from_double(double v) {
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  double a = fabs(v);
  double q;
  uint8_t mag;
  if (a < 2.0) {
    q = nearbyint(a * 2.0);          /* 0..4 halves */
    mag = (uint8_t)q;                /* codes 0..4 are 0, .5, 1, 1.5, 2 */
  } else if (a < 4.0) {
    q = nearbyint(a);                /* 2, 3 or 4 */
    mag = (q == 2.0) ? 4 : (q == 3.0) ? 5 : 6;
  } else {
    q = 2.0 * nearbyint(a / 2.0);    /* 4, 6, 8, ... */
    mag = (q <= 4.0) ? 6 : 7;        /* anything rounding past 6 saturates */
  }
  return sign | mag;
}

/* Array forms of the two encoders (used by the exhaustive self-tests). */
void oracle_e4m3_from_double_array(const double* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_from_double(x[i]);
}

void oracle_e2m1_from_double_array(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_e2m1_from_double(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Row formats                                                              */
/* ------------------------------------------------------------------------ */

#define ORACLE_LATENT 512
#define ORACLE_ROPE 64
#define ORACLE_GROUP 16
#define ORACLE_NVFP4_ROW 352 /* 256 codes + 32 scales + 64 rope */
#define ORACLE_FP8_ROW 576   /* 512 latent + 64 rope */
#define ORACLE_SCALES_OFF 256
#define ORACLE_ROPE_OFF_NVFP4 288
#define ORACLE_ROPE_OFF_FP8 512

size_t oracle_row_bytes(int fmt) { return fmt == 0 ? ORACLE_NVFP4_ROW : fmt == 1 ? ORACLE_FP8_ROW : 0; }

/* One 576-value latent row (bf16 bits) -> one 352-byte NVFP4 row.
 * [P1 "Four bits per latent value"], [P3 NVFP4 paragraph]; readings
 * R-layout, R-scale, R-round, R-sign, R-zero. */
void oracle_quantize_row_nvfp4(const uint16_t* latent, const uint16_t* rope, uint8_t* row) {
  memset(row, 0, ORACLE_NVFP4_ROW);
  for (int g = 0; g < ORACLE_LATENT / ORACLE_GROUP; g++) {
    double amax = 0.0;
    for (int i = 0; i < ORACLE_GROUP; i++) {
      double x = oracle_bf16_to_double(latent[g * ORACLE_GROUP + i]);
      if (fabs(x) > amax) amax = fabs(x);
    }
    uint8_t s_code = oracle_e4m3_from_double(amax / 6.0);
    double s = oracle_e4m3_to_double(s_code);
    row[ORACLE_SCALES_OFF + g] = s_code;
    for (int i = 0; i < ORACLE_GROUP; i++) {
      int idx = g * ORACLE_GROUP + i;
      uint8_t code = 0;
      if (s_code != 0) code = oracle_e2m1_from_double(oracle_bf16_to_double(latent[idx]) / s);
      if (idx & 1)
        row[idx >> 1] |= (uint8_t)(code << 4);
      else
        row[idx >> 1] |= code;
    }
  }
  for (int j = 0; j < ORACLE_ROPE; j++)
    row[ORACLE_ROPE_OFF_NVFP4 + j] = oracle_e4m3_from_double(oracle_bf16_to_double(rope[j]));
}

/* One latent row -> one 576-byte FP8 row: every value e4m3, no scale
 * [P1 row table, "FP8 row"]. */
void oracle_quantize_row_fp8(const uint16_t* latent, const uint16_t* rope, uint8_t* row) {
  for (int i = 0; i < ORACLE_LATENT; i++) row[i] = oracle_e4m3_from_double(oracle_bf16_to_double(latent[i]));
  for (int j = 0; j < ORACLE_ROPE; j++)
    row[ORACLE_ROPE_OFF_FP8 + j] = oracle_e4m3_from_double(oracle_bf16_to_double(rope[j]));
}

/* Stored bytes -> latent c[512] and rope r[64] as exact doubles. */
void oracle_dequant_row(const uint8_t* row, int fmt, double* c, double* r) {
  if (fmt == 0) {
    for (int i = 0; i < ORACLE_LATENT; i++) {
      uint8_t byte = row[i >> 1];
      uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
      double s = oracle_e4m3_to_double(row[ORACLE_SCALES_OFF + i / ORACLE_GROUP]);
      c[i] = oracle_e2m1_to_double(code) * s;
    }
    for (int j = 0; j < ORACLE_ROPE; j++) r[j] = oracle_e4m3_to_double(row[ORACLE_ROPE_OFF_NVFP4 + j]);
  } else {
    for (int i = 0; i < ORACLE_LATENT; i++) c[i] = oracle_e4m3_to_double(row[i]);
    for (int j = 0; j < ORACLE_ROPE; j++) r[j] = oracle_e4m3_to_double(row[ORACLE_ROPE_OFF_FP8 + j]);
  }
}

/* Quantize-on-write of n_tokens rows into a paged pool: token n goes to
 * slot = slot_mapping[n] (block = slot / block_size, offset = slot %
 * block_size).  A negative slot, or one whose block is outside
 * [0, num_blocks), is skipped.  Returns the number of skipped tokens. */
int64_t oracle_kv_quantize_append(const uint16_t* latent, const uint16_t* rope, const int64_t* slot_mapping,
                                  int64_t n_tokens, uint8_t* kv_pool, int64_t num_blocks, int block_size,
                                  int64_t kv_block_stride, int fmt) {
  size_t rb = oracle_row_bytes(fmt);
  int64_t skipped = 0;
  for (int64_t n = 0; n < n_tokens; n++) {
    int64_t slot = slot_mapping[n];
    if (slot < 0 || slot / block_size >= num_blocks) {
      skipped++;
      continue;
    }
    uint8_t* row = kv_pool + (slot / block_size) * kv_block_stride + (slot % block_size) * (int64_t)rb;
    if (fmt == 0)
      oracle_quantize_row_nvfp4(latent + n * ORACLE_LATENT, rope + n * ORACLE_ROPE, row);
    else
      oracle_quantize_row_fp8(latent + n * ORACLE_LATENT, rope + n * ORACLE_ROPE, row);
  }
  return skipped;
}

/* ------------------------------------------------------------------------ */
/* Staged path: NVFP4 rows re-stored as FP8 rows (ablation)                  */
/* ------------------------------------------------------------------------ */

/* One stored NVFP4 row -> the 576-byte FP8 row written by the staged path of
 * [P1 "A kernel that reads four bits directly", figure "staged vs native
 * decode": a gather kernel reads the 352-byte rows and writes a 576-byte FP8
 * copy, which an FP8 attention kernel then reads].  R-stage: every latent
 * value c_i = e2m1_i * S_g is re-encoded as e4m3 (nearest-even, satfinite,
 * sign kept); the 64 rope bytes are e4m3 already and are copied. */
void oracle_stage_row_fp8(const uint8_t* row, uint8_t* out) {
  double c[ORACLE_LATENT], r[ORACLE_ROPE];
  oracle_dequant_row(row, 0, c, r);
  for (int i = 0; i < ORACLE_LATENT; i++) out[i] = oracle_e4m3_from_double(c[i]);
  memcpy(out + ORACLE_ROPE_OFF_FP8, row + ORACLE_ROPE_OFF_NVFP4, ORACLE_ROPE);
}

/* Staged gather of a batch.  Entry j of request b, token t = topk_idx[b,j],
 * is valid when 0 <= t < context_lens[b], t / bs < max_blocks_per_req and the
 * physical block block_table[b, t / bs] lies in [0, num_blocks) (R-mask).  A
 * valid entry writes the staged row of t at
 *   staged_pool + ((b * nblk + j / bs) * bs + j % bs) * 576,  nblk = ceil(topk / bs)
 * and staged_topk[b,j] = j; a masked entry writes staged_topk[b,j] = -1 and
 * no row.  With staged block table [b,i] = b * nblk + i and staged context
 * length nblk * bs the staged pool is an ordinary 576-byte paged pool. */
void oracle_stage_rows_fp8(const uint8_t* kv_pool, int64_t kv_block_stride, int64_t num_blocks,
                           const int32_t* block_table, int max_blocks_per_req, const int32_t* context_lens,
                           const int32_t* topk_idx, int batch, int block_size, int topk, uint8_t* staged_pool,
                           int32_t* staged_topk) {
  int64_t nblk = (topk + block_size - 1) / block_size;
  for (int b = 0; b < batch; b++) {
    for (int j = 0; j < topk; j++) {
      int t = topk_idx[(int64_t)b * topk + j];
      int ok = t >= 0 && t < context_lens[b] && t / block_size < max_blocks_per_req;
      int64_t blk = ok ? block_table[(int64_t)b * max_blocks_per_req + t / block_size] : -1;
      ok = ok && blk >= 0 && blk < num_blocks;
      staged_topk[(int64_t)b * topk + j] = ok ? j : -1;
      if (!ok) continue;
      const uint8_t* row = kv_pool + blk * kv_block_stride + (int64_t)(t % block_size) * ORACLE_NVFP4_ROW;
      uint8_t* dst = staged_pool + (((int64_t)b * nblk + j / block_size) * block_size + j % block_size) *
                                       (int64_t)ORACLE_FP8_ROW;
      oracle_stage_row_fp8(row, dst);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Absorbed-form sparse MLA decode, one request                              */
/* ------------------------------------------------------------------------ */

/* For one request with H heads:
 *   V      = { t in topk : 0 <= t < context_len }        (R-mask)
 *   c_t,r_t = dequantized latent / rope of token t, found through the
 *            block table: block = block_table[t / bs], row = t % bs
 *   z[h,t] = scale * (q_nope[h] . c_t + q_rope[h] . r_t)
 *   p      = softmax over t of z[h, .]
 *   out[h] = sum_t p[h,t] c_t,   lse[h] = log sum_t exp(z[h,t])
 * [P1 "A kernel that reads four bits directly": every selected row is
 * unpacked and scored for all heads; the value vector is the latent itself
 * (absorbed form, [P5] section 6, sparse_mla_force_mqa: every KV row serves
 * all heads)].  Empty V gives out = 0, lse = -inf (R-empty). */
void oracle_sparse_decode_request(const uint16_t* q_nope, const uint16_t* q_rope, const uint8_t* kv_pool,
                                  int64_t kv_block_stride, const int32_t* block_table_row, int context_len,
                                  const int32_t* topk_row, int topk, int num_heads, int block_size,
                                  double softmax_scale, int fmt, double* out, double* lse) {
  size_t rb = oracle_row_bytes(fmt);
  int nv = 0;
  int* valid = (int*)malloc(sizeof(int) * (size_t)(topk > 0 ? topk : 1));
  double* c = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * ORACLE_LATENT);
  double* r = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1) * ORACLE_ROPE);
  double* z = (double*)malloc(sizeof(double) * (size_t)(topk > 0 ? topk : 1));
  for (int j = 0; j < topk; j++) {
    int t = topk_row[j];
    if (t < 0 || t >= context_len) continue;
    const uint8_t* row = kv_pool + (int64_t)block_table_row[t / block_size] * kv_block_stride +
                         (int64_t)(t % block_size) * (int64_t)rb;
    oracle_dequant_row(row, fmt, c + (size_t)nv * ORACLE_LATENT, r + (size_t)nv * ORACLE_ROPE);
    valid[nv++] = t;
  }
  for (int h = 0; h < num_heads; h++) {
    double* o = out + (size_t)h * ORACLE_LATENT;
    for (int i = 0; i < ORACLE_LATENT; i++) o[i] = 0.0;
    if (nv == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int v = 0; v < nv; v++) {
      double dot = 0.0;
      for (int i = 0; i < ORACLE_LATENT; i++)
        dot += oracle_bf16_to_double(q_nope[(size_t)h * ORACLE_LATENT + i]) * c[(size_t)v * ORACLE_LATENT + i];
      for (int j = 0; j < ORACLE_ROPE; j++)
        dot += oracle_bf16_to_double(q_rope[(size_t)h * ORACLE_ROPE + j]) * r[(size_t)v * ORACLE_ROPE + j];
      z[v] = softmax_scale * dot;
      if (z[v] > m) m = z[v];
    }
    double l = 0.0;
    for (int v = 0; v < nv; v++) l += exp(z[v] - m);
    for (int v = 0; v < nv; v++) {
      double p = exp(z[v] - m) / l;
      for (int i = 0; i < ORACLE_LATENT; i++) o[i] += p * c[(size_t)v * ORACLE_LATENT + i];
    }
    lse[h] = m + log(l);
  }
  (void)valid;
  free(valid);
  free(c);
  free(r);
  free(z);
}

/* Whole batch: q_nope [B,H,512], q_rope [B,H,64], block_table [B,max_blocks],
 * context_lens [B], topk_idx [B,topk] -> out [B,H,512], lse [B,H]. */
void oracle_sparse_decode(const uint16_t* q_nope, const uint16_t* q_rope, const uint8_t* kv_pool,
                          int64_t kv_block_stride, const int32_t* block_table, int max_blocks_per_req,
                          const int32_t* context_lens, const int32_t* topk_idx, int batch, int num_heads,
                          int block_size, int topk, double softmax_scale, int fmt, double* out, double* lse) {
  for (int b = 0; b < batch; b++)
    oracle_sparse_decode_request(q_nope + (size_t)b * num_heads * ORACLE_LATENT,
                                 q_rope + (size_t)b * num_heads * ORACLE_ROPE, kv_pool, kv_block_stride,
                                 block_table + (size_t)b * max_blocks_per_req, context_lens[b],
                                 topk_idx + (size_t)b * topk, topk, num_heads, block_size, softmax_scale, fmt,
                                 out + (size_t)b * num_heads * ORACLE_LATENT, lse + (size_t)b * num_heads);
}

/* Several query tokens per request (speculative drafts decoded together):
 * q_nope [B,Q,H,512], q_rope [B,Q,H,64], topk_idx [B,Q,k], out [B,Q,H,512],
 * lse [B,Q,H].  Every query token has its own top-k list ([P1] "A kernel
 * that reads four bits directly": the native kernel runs 15 query tokens per
 * launch).  R-causal: the Q tokens are the last Q positions of the request's
 * context_lens[b] tokens, so token i sees positions t < context_lens[b] -
 * (Q - 1 - i); list entries at or past that bound are masked (R-mask). */
void oracle_sparse_decode_mtp(const uint16_t* q_nope, const uint16_t* q_rope, const uint8_t* kv_pool,
                              int64_t kv_block_stride, const int32_t* block_table, int max_blocks_per_req,
                              const int32_t* context_lens, const int32_t* topk_idx, int batch, int q_len,
                              int num_heads, int block_size, int topk, double softmax_scale, int fmt, double* out,
                              double* lse) {
  for (int b = 0; b < batch; b++) {
    for (int i = 0; i < q_len; i++) {
      int64_t v = (int64_t)b * q_len + i;
      int ctx_i = context_lens[b] - (q_len - 1 - i);
      oracle_sparse_decode_request(q_nope + v * num_heads * ORACLE_LATENT, q_rope + v * num_heads * ORACLE_ROPE,
                                   kv_pool, kv_block_stride, block_table + (int64_t)b * max_blocks_per_req,
                                   ctx_i, topk_idx + v * topk, topk, num_heads, block_size, softmax_scale, fmt,
                                   out + v * num_heads * ORACLE_LATENT, lse + v * num_heads);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Indexer score and exact top-k                                             */
/* ------------------------------------------------------------------------ */

#define ORACLE_IDX_DIM 128

/* score[t] = sum_h w[h] * max(0, s_t * (q[h] . k_t)) for t in [0, ctx), where
 * k_t are 128 e4m3 values and s_t a float scale, found through the block
 * table (R-keys).  [P5 section 1: the indexer rates every preceding token;
 * section 3: a key is 128 e4m3 bytes and a float scale]. */
void oracle_indexer_scores_request(const uint16_t* q_idx, const float* head_w, int n_idx_heads,
                                   const uint8_t* idx_key_pool, int64_t idx_block_stride,
                                   const int32_t* block_table_row, int context_len, int block_size,
                                   double* scores) {
  for (int t = 0; t < context_len; t++) {
    const uint8_t* blk = idx_key_pool + (int64_t)block_table_row[t / block_size] * idx_block_stride;
    const uint8_t* key = blk + (int64_t)(t % block_size) * ORACLE_IDX_DIM;
    float s_f;
    memcpy(&s_f, blk + (int64_t)block_size * ORACLE_IDX_DIM + (int64_t)(t % block_size) * 4, 4);
    double s_t = (double)s_f;
    double score = 0.0;
    for (int h = 0; h < n_idx_heads; h++) {
      double dot = 0.0;
      for (int d = 0; d < ORACLE_IDX_DIM; d++)
        dot += oracle_bf16_to_double(q_idx[(size_t)h * ORACLE_IDX_DIM + d]) * oracle_e4m3_to_double(key[d]);
      double a = s_t * dot;
      score += (double)head_w[h] * (a > 0.0 ? a : 0.0);
    }
    scores[t] = score;
  }
}

/* One token's 128 bf16 indexer-key values -> 128 e4m3 codes and a float
 * scale [P5 section 3: a key is 128 e4m3 bytes and a float scale].
 * R-keyscale: s = amax / 448 and code_d = e4m3_rn_satfinite(k_d / s), both
 * divisions in IEEE single precision (the precision of the stored scale, so
 * every rounding decision is taken on a float).  amax = 0 stores s = 0 and
 * 128 zero codes. */
void oracle_quantize_index_key(const uint16_t* key, uint8_t* codes, float* scale) {
  float amax = 0.0f;
  for (int d = 0; d < ORACLE_IDX_DIM; d++) {
    float x = (float)oracle_bf16_to_double(key[d]);
    if (fabsf(x) > amax) amax = fabsf(x);
  }
  if (amax == 0.0f) {
    memset(codes, 0, ORACLE_IDX_DIM);
    *scale = 0.0f;
    return;
  }
  float s = amax / 448.0f;
  for (int d = 0; d < ORACLE_IDX_DIM; d++) {
    float q = (float)oracle_bf16_to_double(key[d]) / s;
    codes[d] = oracle_e4m3_from_double((double)q);
  }
  *scale = s;
}

/* Indexer-key quantize-on-write: token n's key goes to slot_mapping[n]
 * (block = slot / bs, offset o = slot % bs): codes at block + o * 128, scale
 * at block + bs * 128 + o * 4 (R-keys).  Slots that are negative or past the
 * pool are skipped; returns their number. */
int64_t oracle_index_key_quantize_append(const uint16_t* keys, const int64_t* slot_mapping, int64_t n_tokens,
                                         uint8_t* key_pool, int64_t num_blocks, int block_size,
                                         int64_t key_block_stride) {
  int64_t skipped = 0;
  for (int64_t n = 0; n < n_tokens; n++) {
    int64_t slot = slot_mapping[n];
    if (slot < 0 || slot / block_size >= num_blocks) {
      skipped++;
      continue;
    }
    uint8_t* blk = key_pool + (slot / block_size) * key_block_stride;
    int64_t o = slot % block_size;
    float s;
    oracle_quantize_index_key(keys + n * ORACLE_IDX_DIM, blk + o * ORACLE_IDX_DIM, &s);
    memcpy(blk + (int64_t)block_size * ORACLE_IDX_DIM + o * 4, &s, 4);
  }
  return skipped;
}

typedef struct {
  double score;
  int32_t t;
} oracle_scored_t;

static int cmp_score_desc_idx_asc(const void* pa, const void* pb) {
  const oracle_scored_t* a = (const oracle_scored_t*)pa;
  const oracle_scored_t* b = (const oracle_scored_t*)pb;
  if (a->score > b->score) return -1;
  if (a->score < b->score) return 1;
  return (a->t < b->t) ? -1 : (a->t > b->t) ? 1 : 0;
}

static int cmp_int_asc(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/* Exact top-k of scores[0..ctx) (R-topk).  -0.0 and +0.0 compare equal under
 * the C comparison operators, as R-topk wants. */
void oracle_topk_request(const double* scores, int context_len, int topk, int32_t* out) {
  int n = context_len < topk ? context_len : topk;
  oracle_scored_t* all = (oracle_scored_t*)malloc(sizeof(oracle_scored_t) * (size_t)(context_len > 0 ? context_len : 1));
  for (int t = 0; t < context_len; t++) {
    all[t].score = scores[t];
    all[t].t = t;
  }
  qsort(all, (size_t)context_len, sizeof(oracle_scored_t), cmp_score_desc_idx_asc);
  for (int j = 0; j < n; j++) out[j] = all[j].t;
  qsort(out, (size_t)n, sizeof(int32_t), cmp_int_asc);
  for (int j = n; j < topk; j++) out[j] = -1;
  free(all);
}

/* Same selection on single-precision scores (the GPU's own fp32 scores):
 * each float widens exactly to double, so the order is the float order. */
void oracle_topk_request_f32(const float* scores, int context_len, int topk, int32_t* out) {
  double* d = (double*)malloc(sizeof(double) * (size_t)(context_len > 0 ? context_len : 1));
  for (int t = 0; t < context_len; t++) d[t] = (double)scores[t];
  oracle_topk_request(d, context_len, topk, out);
  free(d);
}
