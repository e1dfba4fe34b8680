/*
 * pkv_oracle.h - the oracle for paged decode attention: a plain, slow,
 * obviously correct CPU restatement in float64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call it.  It shares no code, header,
 * table or helper with the CUDA library; it reads the same input bytes.
 *
 * Layouts (bf16 passed as uint16 bit patterns):
 *   q            [B][N][H]
 *   k/v cache    [num_blocks][bs][K][H]   row (block*bs + off)*K + kvh holds H values
 *   block_tables [B][max_nb]               int32 physical block ids
 *   context_lens [B]                       tokens attended, including the new one
 *   out          [B][N][H] double,  lse [B][N] double (natural log)
 * Query head n reads KV head n / (N/K)  (contiguous query groups).
 */
#ifndef PKV_ORACLE_H
#define PKV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* KV cache bytes = 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem. */
uint64_t oracle_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                         int64_t bytes_per_elem);

/* slot of each sequence's newest token (logical position ctx-1); -1 when ctx <= 0. */
void oracle_slot_mapping(const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                         int32_t B, int32_t bs, int64_t *slots);

/* copy k_new[i], v_new[i] ([T][K][H]) into cache slot slots[i]; negative slots are skipped. */
void oracle_append(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots, int32_t T,
                   uint16_t *k_cache, uint16_t *v_cache, int32_t K, int32_t H);

/* contiguous copy of each sequence's K/V rows: out[(cu_seqlens[b] + t)][K][H] for t < ctx_b. */
void oracle_gather(const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *block_tables,
                   int32_t max_nb, const int32_t *context_lens, const int64_t *cu_seqlens,
                   int32_t B, int32_t bs, int32_t K, int32_t H, uint16_t *k_out, uint16_t *v_out);

/* decode attention for every (b, n); nthreads <= 0 means all online cores. */
void oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                   int32_t B, int32_t N, int32_t K, int32_t H, int32_t bs, double scale,
                   double *out, double *lse, int nthreads);

/* the same attention restricted to each partition of partition_tokens logical tokens:
   part_out [B][N][max_parts][H], part_lse [B][N][max_parts]; an empty partition has
   out 0 and lse -inf. */
void oracle_decode_partitions(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_tables, int32_t max_nb,
                              const int32_t *context_lens, int32_t B, int32_t N, int32_t K,
                              int32_t H, int32_t bs, double scale, int32_t partition_tokens,
                              int32_t max_parts, double *part_out, double *part_lse, int nthreads);

/* combine partitions: lse = log sum_p exp(lse_p); out = sum_p exp(lse_p - lse) out_p. */
void oracle_lse_merge(const double *part_out, const double *part_lse, int32_t B, int32_t N,
                      int32_t H, int32_t max_parts, double *out, double *lse);

/* ---- several query tokens per sequence (speculative verification) ------------------
   The last T of each sequence's ctx tokens are new: query token t ([B][T][N][H]) sits at
   logical position ctx - T + t and attends to the tokens [0, ctx - T + t] -- the whole cache
   and the new tokens up to itself.  out [B][T][N][H], lse [B][T][N]. */
void oracle_slot_mapping_multi(const int32_t *block_tables, int32_t max_nb,
                               const int32_t *context_lens, int32_t B, int32_t T, int32_t bs,
                               int64_t *slots);
void oracle_decode_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                         int32_t B, int32_t T, int32_t N, int32_t K, int32_t H, int32_t bs,
                         double scale, double *out, double *lse, int nthreads);

/* ---- copy-on-write -----------------------------------------------------------------
   For each pair i: physical block src_dst[2i+1] of both pools becomes a byte copy of block
   src_dst[2i] (block_bytes = 16 * K * H * element bytes), in pair order. */
void oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *src_dst, int32_t n,
                        int64_t block_bytes);

/* ---- FP8 (e4m3) KV cache ----------------------------------------------------------
   Codes: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 holds
   subnormals m * 2^-9; S.1111.111 is NaN; no infinities; largest finite 448.
   Quantization of a value x of KV head kvh: code = e4m3(x / scale[kvh]) with the division
   in float (round to nearest) and round-to-nearest-even onto the e4m3 grid, saturating at
   +-448; dequantization: decode(code) * scale[kvh].  With scale_block_stride > 0 the scales
   are per (physical block, KV head): value x of a row in block blk uses
   scale[blk * scale_block_stride + kvh] instead (scale_block_stride = K for [num_blocks][K]). */
uint8_t oracle_e4m3_encode(float x);
double oracle_e4m3_decode(uint8_t code);

/* dst[r][kvh][h] = e4m3(src[r][kvh][h] / scale[kvh]) for rows [rows][K][H] (bf16 in); with
   scale_block_stride > 0, row r lies in block r / bs and uses that block's scales. */
void oracle_quantize_fp8(const uint16_t *src, int64_t rows, int32_t K, int32_t H,
                         const float *scale, int32_t scale_block_stride, int32_t bs, uint8_t *dst);

/* append: quantize k_new/v_new rows [T][K][H] into their slots (with the scales of the block
   a slot lies in, slot / bs); negative slots skipped. */
void oracle_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const float *k_scale,
                       const float *v_scale, int32_t scale_block_stride, int32_t bs,
                       const int64_t *slots, int32_t T, uint8_t *k_cache, uint8_t *v_cache, int32_t K,
                       int32_t H);

/* decode attention over an e4m3 cache [num_blocks][bs][K][H] dequantized with the per-head
   (or per (block, head)) scales; same outputs as oracle_decode. */
void oracle_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                       const float *k_scale, const float *v_scale, int32_t scale_block_stride,
                       const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                       int32_t B, int32_t N, int32_t K, int32_t H, int32_t bs, double scale, double *out,
                       double *lse, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
