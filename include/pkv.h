/*
 * pkv.h - libpagedkv: decode-step attention over a paged KV cache, for one
 * NVIDIA GB300 (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA
 * stream; no framework types.
 *
 * The method.  In a continuously batched decode step each sequence b has one
 * new query token with N query heads that share K KV heads (GQA; query head
 * n reads KV head n / (N/K)).  The token's own key and value are first
 * appended to the cache, then it attends to its whole history:
 *     s_t      = scale * q[b,n,:] . K[b,t,kvh,:]       t in [0, ctx_b)
 *     out[b,n] = sum_t softmax(s)_t V[b,t,kvh,:],      lse[b,n] = ln sum_t e^{s_t}
 * Sources: "Optimización de la inferencia" (aiengineeringfromscratch.com),
 * sections "Cache de KV" (append only the new token's K/V), "Página
 * Atención" (fixed-size pages anywhere in GPU memory, a page table from
 * logical positions to physical pages) and "Construye el mismo", Step 2
 * (max-subtracted scaled dot-product attention); CS336 Lecture 10 notes
 * "注意力层的算术强度分析" (decode attention intensity S/(S+1) < 1) and
 * "分页注意力（PagedAttention）" ("融合块读取和注意力的内核", FlashDecoding).
 *
 * Layouts (row-major, bf16 passed as 16-bit storage):
 *   k_cache, v_cache  [num_blocks][block_size=16][K][H]   separate K and V pools
 *   block_tables      [num_seqs][max_blocks_per_seq] int32; entry j of sequence b is
 *                     the physical block of its logical tokens 16j .. 16j+15
 *   context_lens      [num_seqs] int32: tokens attended, INCLUDING the token
 *                     appended this step (its logical position is ctx-1)
 *   q, out            [num_seqs][N][H] bf16;   lse [num_seqs][N] float (natural log)
 *   k_new, v_new      [num_tokens][K][H] bf16; slot_mapping [num_tokens] int64,
 *                     slot = block * 16 + offset, negative = skip the token
 * Supported shapes: block_size 16, H in {64, 128}, G = N/K in {1, 2, 4, 8}.
 *
 * Ownership: every pointer is caller-owned memory the current device can address: the KV
 * pools (read by TMA) and the workspaces must be device memory; every other buffer (q, out,
 * lse, k_new, v_new, block tables, context lengths, slot mappings) may also be pinned
 * (page-locked) host memory, which the kernels read and write in place -- on a GB300 over
 * NVLink-C2C, so a step's inputs and outputs need no separate copies.  The library allocates
 * nothing and keeps no state between calls besides cached device attributes (and the static
 * scratch of pkv_decode_attn_splitk_noalloc, described there).  Calls are asynchronous on the
 * given stream (0 = the legacy default stream).  Those caches are per device and live as long as
 * the process: resetting a device (cudaDeviceReset) while the library is loaded is not supported.
 *
 * Errors: each call returns a pkv_status.  Host-side validation happens
 * before anything is launched.  Bad values that only the device sees (a
 * block id outside [0, num_blocks), a slot beyond the pool, ctx beyond the
 * table width) set bits in the caller's err_flag (a device int32, nullable,
 * sticky: the caller zeroes it, synchronises and reads it, e.g. with
 * pkv_read_err_flag); the offending work is skipped, never a fault.  Every
 * wait inside a kernel is bounded; an expired wait sets PKV_FLAG_TIMEOUT.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;                   /* bf16 bit pattern */
typedef struct CUstream_st *pkv_stream_t;   /* identical to cudaStream_t */

enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = -1,        /* a required pointer is NULL */
    PKV_ERR_SHAPE = -2,       /* inconsistent sizes (N % K != 0, partitions too few, ...) */
    PKV_ERR_UNSUPPORTED = -3, /* H not in {64,128}, G not in {1,2,4,8}, block_size != 16 */
    PKV_ERR_RANGE = -4,       /* device-detected out-of-range value (err_flag non-zero) */
    PKV_ERR_CUDA = -5,        /* a CUDA call failed; pkv_last_error() has the text */
    PKV_ERR_ALIGN = -6,       /* a pointer lacks the alignment the layout needs */
    PKV_ERR_WORKSPACE = -7    /* workspace missing or smaller than required */
};

/* err_flag bits */
#define PKV_FLAG_BLOCK_RANGE 1 /* a block table entry outside [0, num_blocks) */
#define PKV_FLAG_SLOT_RANGE 2  /* a slot >= num_blocks * 16 */
#define PKV_FLAG_CTX_RANGE 4   /* context_len < 0 or > max_blocks_per_seq * 16 */
#define PKV_FLAG_TIMEOUT 8     /* a bounded in-kernel wait expired; the unit's result is void */
#define PKV_FLAG_OUT_RANGE 16  /* pkv_gather: a row beyond out_rows */
#define PKV_FLAG_GROUP_RANGE 32 /* pkv_decode_attn_prefix: a group or prefix beyond its declared
                                   bound, or a member shorter than its group's prefix */

typedef struct {
    int32_t num_blocks;   /* physical blocks in each pool */
    int32_t block_size;   /* tokens per block; must be 16 */
    int32_t num_kv_heads; /* K */
    int32_t head_dim;     /* H */
} pkv_cache_desc;

/*
 * KV cache bytes = 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem
 * ("Optimización de la inferencia", section "Cache de KV", memory formula;
 * Week 11 "Inference", Step 2).  Host only.
 */
uint64_t pkv_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                      int64_t bytes_per_elem);

/*
 * Slot mapping: slot_mapping[b] = block_tables[b][p / 16] * 16 + p % 16 for the
 * newest token p = context_lens[b] - 1 (the page table maps logical positions
 * to physical pages: "Optimización de la inferencia", "Página Atención").
 * ctx <= 0 gives -1.  num_blocks bounds the ids (out of range: flag, slot -1).
 */
int pkv_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *context_lens, int32_t num_seqs, int32_t num_blocks,
                     int64_t *slot_mapping, int32_t *err_flag, pkv_stream_t stream);

/*
 * Append: k_cache[slot / 16][slot % 16][:][:] = k_new[i] (and v), bit for bit,
 * for each token i with slot_mapping[i] >= 0 ("Optimización de la
 * inferencia", "Cache de KV": only the new token's key and value are computed
 * and joined to the cache).  Slots within one call must be distinct.
 * k_new/v_new/k_cache/v_cache must be 16-byte aligned.
 */
int pkv_append(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int64_t *slot_mapping,
               int32_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache, pkv_cache_desc cache,
               int32_t *err_flag, pkv_stream_t stream);

/*
 * Single-pass decode attention: one CTA per (sequence, KV head) reads each
 * K/V block once through the block table and serves the whole query group
 * from it (CS336 Lecture 10 notes: fused block-read + attention kernel).
 * out [num_seqs][N][H] bf16 (round-to-nearest-even of an fp32 result);
 * lse_out [num_seqs][N] float, nullable.  ctx = 0 gives out 0, lse -inf.
 * k_cache/v_cache 16-byte aligned; q and out 4-byte aligned.
 */
int pkv_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                    float scale, pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                    int32_t *err_flag, pkv_stream_t stream);

/*
 * Workspace for pkv_decode_attn_splitk (and the partitioned forms of pkv_decode_step,
 * pkv_decode_attn_fp8, pkv_decode_step_fp8): part_out float [num_seqs][N][max_partitions][H],
 * then (256-byte aligned) part_lse float [num_seqs][N][max_partitions], then (256-byte aligned)
 * merge counters int32 [num_seqs][N].  ZERO THE WORKSPACE ONCE before its first use: each call
 * leaves the counters at zero again, so a workspace can be reused (and captured in a CUDA graph)
 * without clearing it.  Calls that share a workspace must not overlap on the GPU.
 */
size_t pkv_splitk_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                  int32_t max_partitions);

/*
 * Split-KV decode attention (FlashDecoding, named in CS336 Lecture 10 notes,
 * "其他优化"): sequence b's table is cut into partitions of partition_blocks
 * blocks, partition p covering blocks [p * partition_blocks, (p+1) *
 * partition_blocks).  When num_seqs * num_kv_heads >= the device's SM count
 * (the grid runs in several waves) and max_partitions >= 1 + ceil((max_nb -
 * partition_blocks / 2) / partition_blocks) (partition_blocks >= 2), the
 * partitions taper instead: partition 0, launched last, covers the first
 * partition_blocks / 2 blocks and partition p >= 1 the partition_blocks blocks
 * after them, so that the grid's final wave is made of half-length CTAs.  The
 * partials are internal; the result is the same up to rounding.  One CTA per (partition, KV head, sequence), highest partition first, in one launch: a
 * sequence that fits in one partition is written to out directly; the others
 * leave normalised partial outputs and lse in the workspace, and the last CTA of
 * each (sequence, KV head) to finish merges them by log-sum-exp (the same
 * arithmetic as pkv_lse_merge, bit for bit).  max_partitions must be >=
 * ceil(max_blocks_per_seq / partition_blocks).  The workspace is caller-owned
 * device memory of at least pkv_splitk_workspace_bytes(...) bytes, 256-byte
 * aligned and zeroed before its first use.
 */
int pkv_decode_attn_splitk(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                           float scale, pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                           int32_t partition_blocks, int32_t max_partitions, void *workspace,
                           size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream);

/*
 * One whole decode step in one launch: for each sequence the new token's
 * K and V (k_new/v_new [num_seqs][K][H]) are written into the slot of its logical position
 * ctx-1 (slot_mapping_out[b] = that slot, or -1 for ctx 0; nullable) and the token attends to
 * its context including itself -- pkv_slot_mapping + pkv_append + pkv_decode_attn (or
 * pkv_decode_attn_splitk) fused.  The kernel that reads a sequence's last block replaces that
 * block's row ctx-1 with the new K/V on chip and writes it to the pools, so no separate append
 * pass runs ("Optimización de la inferencia", "Cache de KV": only the new token's K/V is
 * computed and joined to the cache; CUDA graphs / fused kernels: CS336 Lecture 10 notes,
 * "其他优化").  partition_blocks 0 = single pass (workspace unused, may be NULL); > 0 =
 * partitions laid out as in pkv_decode_attn_splitk (tapered under the same conditions), with
 * its workspace.  k_new/v_new 16-byte aligned.  Results are bit-identical to the three separate
 * calls.
 */
int pkv_decode_step(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                    pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                    int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                    int64_t *slot_mapping_out, pkv_cache_desc cache, int32_t partition_blocks,
                    int32_t max_partitions, void *workspace, size_t workspace_bytes,
                    int32_t *err_flag, pkv_stream_t stream);

/*
 * ---- FP8 (e4m3) KV cache -----------------------------------------------------------------
 * Cache quantization halves the bytes a decode step reads ("Week 11. Inference", Step 2:
 * storing K and V in 8 bits instead of 16; "Optimización de la inferencia", exercise on KV
 * cache quantization).  Pools hold e4m3 codes [num_blocks][16][K][H] (1 byte each; H = 128);
 * value = decode(code) * scale.  Scales (positive, finite floats; one array for K, one for V)
 * come in one of two granularities, chosen by scale_block_stride:
 *   0  one scale per KV head, float [K] (calibrated once for the whole pool);
 *   K  one scale per (physical block, KV head), float [num_blocks][K]: element (blk, kvh) scales
 *      every value of that head in that block (the block's 16 tokens).
 * Quantizing x: code = e4m3(x / scale) with the division rounded to nearest in fp32 and
 * round-to-nearest-even onto the e4m3 grid, saturating at +-448 (e4m3: 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities).  Attention reads the codes, widens them exactly to f16
 * for the tensor-core contractions and applies the scales (K's to the logits, V's to the weights
 * of each block relative to one V scale per partition, which multiplies the output); results
 * otherwise as pkv_decode_attn.  The per-block scales of the blocks a step writes into must be
 * set before the step (an append quantizes with them).
 */

/* dst[r][kvh][h] = e4m3(src[r][kvh][h] / scale[kvh]) for src bf16 [rows][K][H] (16-byte aligned);
   with scale_block_stride = K, src is a pool (rows a multiple of 16, row r in block r / 16) and
   the scale is scale[(r / 16) * K + kvh]. */
int pkv_quantize_fp8(const pkv_bf16 *src, int64_t rows, int32_t num_kv_heads, int32_t head_dim,
                     const float *scale, int32_t scale_block_stride, uint8_t *dst, pkv_stream_t stream);

/* pkv_append for an e4m3 pool: each token's K/V row quantized into its slot (with the scales of
   the slot's block, slot / 16, when scale_block_stride = K). */
int pkv_append_fp8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const float *k_scale,
                   const float *v_scale, int32_t scale_block_stride, const int64_t *slot_mapping,
                   int32_t num_tokens, uint8_t *k_cache, uint8_t *v_cache, pkv_cache_desc cache,
                   int32_t *err_flag, pkv_stream_t stream);

/* Decode attention over e4m3 pools: partition_blocks 0 = single pass (workspace unused),
   > 0 = partitions as in pkv_decode_attn_splitk (tapered under the same conditions) + log-sum-exp
   merge, with its workspace.
   q 8-byte aligned. */
int pkv_decode_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                        const float *k_scale, const float *v_scale, int32_t scale_block_stride,
                        const int32_t *block_tables,
                        int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                        int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                        pkv_cache_desc cache, int32_t partition_blocks, int32_t max_partitions,
                        void *workspace, size_t workspace_bytes, int32_t *err_flag,
                        pkv_stream_t stream);

/* pkv_decode_step for e4m3 pools: the new token is quantized into its slot and attended in
   the same launch; bit-identical to pkv_append_fp8 followed by pkv_decode_attn_fp8. */
int pkv_decode_step_fp8(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                        uint8_t *k_cache, uint8_t *v_cache, const float *k_scale,
                        const float *v_scale, int32_t scale_block_stride, const int32_t *block_tables,
                        int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                        int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                        int64_t *slot_mapping_out, pkv_cache_desc cache, int32_t partition_blocks,
                        int32_t max_partitions, void *workspace, size_t workspace_bytes,
                        int32_t *err_flag, pkv_stream_t stream);

/*
 * Size of the static scratch used by pkv_decode_attn_splitk_noalloc (8 MiB).
 */
#define PKV_STATIC_SCRATCH_BYTES (8u << 20)

/*
 * Split-KV decode attention that allocates nothing and takes no workspace.  The pages have
 * no counterpart: this entry point exists for callers that cannot call cudaMalloc where they
 * run attention (while a CUDA graph is being captured, inside an allocator's own callback, or
 * under a framework that owns the whole device heap).  Same arguments and result as
 * pkv_decode_attn_splitk without workspace/workspace_bytes; the partial outputs go to a
 * PKV_STATIC_SCRATCH_BYTES array built into the library, which every GPU that loads the
 * library holds until the process exits.
 *  - If pkv_splitk_workspace_bytes(num_seqs, N, H, max_partitions) exceeds
 *    PKV_STATIC_SCRATCH_BYTES the call returns PKV_ERR_WORKSPACE (pkv_last_error() says
 *    how much was needed) and launches nothing; so does every other refusal (max_partitions
 *    beyond 12288: PKV_ERR_UNSUPPORTED; partitions that do not cover the table: PKV_ERR_SHAPE).
 *  - The first call on a device looks up the scratch's device address with that device
 *    current (cudaGetSymbolAddress); make that first call before any stream capture.  A call
 *    with num_seqs = 0 (all pointers may then be any non-NULL, suitably aligned values) launches
 *    nothing but does that lookup, so a caller can prepare each device before its first real
 *    call.  The address stays valid until the process exits (see the note on device resets
 *    above).
 *  - All calls share the one array and it keeps the last call's contents; nothing in it has
 *    to start at zero.  Calls that overlap on the GPU (e.g. on two streams) race on it: order
 *    them on one stream or with events.
 */
int pkv_decode_attn_splitk_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                   const pkv_bf16 *v_cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens,
                                   int32_t num_seqs, int32_t num_q_heads, float scale,
                                   pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                                   int32_t partition_blocks, int32_t max_partitions,
                                   int32_t *err_flag, pkv_stream_t stream);

/*
 * The partition step alone: writes part_out [num_seqs][N][max_partitions][H] and
 * part_lse [num_seqs][N][max_partitions] (float, natural log) for the partitions
 * that hold tokens; partitions past a sequence's last block are not written.
 * Partition p always covers blocks [p * partition_blocks, (p+1) *
 * partition_blocks) here (never the tapered layout: the partials are the caller's).
 */
int pkv_decode_attn_partitions(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                               const pkv_bf16 *v_cache, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, float scale,
                               pkv_cache_desc cache, int32_t partition_blocks,
                               int32_t max_partitions, float *part_out, float *part_lse,
                               int32_t *err_flag, pkv_stream_t stream);

/*
 * Log-sum-exp merge of disjoint partitions (softmax over a union of disjoint
 * key sets):  lse = ln sum_p e^{lse_p};  out = sum_p e^{lse_p - lse} out_p.
 * Sequence b has ceil(ceil(ctx_b / 16) / partition_blocks) partitions; only
 * those are read.  out bf16 [num_seqs][N][H]; lse_out nullable.
 */
int pkv_lse_merge(const float *part_out, const float *part_lse, const int32_t *context_lens,
                  int32_t num_seqs, int32_t num_q_heads, int32_t head_dim, int32_t max_partitions,
                  int32_t partition_blocks, pkv_bf16 *out, float *lse_out, pkv_stream_t stream);

/*
 * Block-table gather (test and debug export): k_out[(cu_seqlens[b] + t)][K][H] =
 * k_cache[table[b][t / 16]][t % 16][K][H] for t < ctx_b (and v).  out_rows bounds
 * the output (rows beyond it: flag, skipped).  All buffers 16-byte aligned.
 */
int pkv_gather(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const int32_t *block_tables,
               int32_t max_blocks_per_seq, const int32_t *context_lens, const int64_t *cu_seqlens,
               int32_t num_seqs, pkv_bf16 *k_out, pkv_bf16 *v_out, int64_t out_rows,
               pkv_cache_desc cache, int32_t *err_flag, pkv_stream_t stream);

/*
 * ---- several new tokens per sequence (speculative verification) ---------------------------
 * The target model checks gamma + 1 drafted tokens in one pass ("Week 11. Inference", Step 3):
 * each sequence carries T = num_new new tokens, the last T of its ctx tokens (context_lens
 * counts them).  Token t sits at logical position ctx - T + t and attends to the tokens
 * [0, ctx - T + t]: the whole cache and the new tokens up to itself.  The causal mask lines up
 * with the end of the keys, not with their start (Week 11, "Common mistakes"; the masked
 * softmax of "Optimización de la inferencia", Step 2).  A token with no visible key (ctx < T)
 * gets out 0 and lse -inf.
 */

/* Slots of the last T logical positions of each sequence: slot_mapping int64 [num_seqs][T],
   -1 below position 0; a block id outside [0, num_blocks) or a context beyond the table sets a
   flag and gives -1.  Feed it to pkv_append with num_tokens = num_seqs * T and the new rows
   [num_seqs][T][K][H]. */
int pkv_slot_mapping_multi(const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs, int32_t num_new,
                           int32_t num_blocks, int64_t *slot_mapping, int32_t *err_flag,
                           pkv_stream_t stream);

/* Attention of T = num_new (1..64) query tokens per sequence after they were appended.
   q bf16 [num_seqs][T][N][H] (4-byte aligned), out bf16 [num_seqs][T][N][H], lse_out fp32
   [num_seqs][T][N] (nullable).  partition_blocks 0: one pass (no workspace); > 0: fixed
   partitions of that many blocks and a log-sum-exp merge, with max_partitions as for
   pkv_decode_attn_splitk and a workspace of pkv_splitk_workspace_bytes(num_seqs * T, N, H,
   max_partitions) bytes, 256-byte aligned and ZEROED BEFORE ITS FIRST USE.  On the mma.sync
   column kernel the partitions taper as in pkv_decode_attn_splitk, with num_seqs * chunks of
   32 rows * num_kv_heads in place of num_seqs * num_kv_heads; the tcgen05 kernel keeps them
   uniform.  On the mma.sync column kernel with 32 * max_partitions <= 8192 the merge runs in the same launch: a sequence
   held by one partition is written out directly, and the last CTA of each (sequence, KV head,
   chunk of 32 rows) to finish merges the chunk's partials (the arithmetic of pkv_lse_merge, bit
   for bit) and leaves its counter (in the workspace's counter area) at zero again, so the
   workspace can be reused and captured in a CUDA graph.  The tcgen05 kernel and larger splits
   merge in a second launch (pkv_lse_merge).  Calls that share a workspace must not overlap on
   the GPU.  Each CTA loads a K/V tile once for up to 32 of a sequence's (token, head) rows of
   one KV head (128 on the tensor cores when T * G > 32).  H in {64, 128}; G in {1, 2, 4, 8}.
   With more than 16 rows per CTA (min(T * G, 32) > 16) and H = 128 the contraction runs on the
   tcgen05 tensor cores (accumulators in tensor memory), otherwise on warp-level mma.sync; both
   compute the same definition (results agree within rounding, not bit for bit).  The tcgen05
   kernel's separate merge is launched with programmatic stream serialization (it may start while
   the attention grid's last CTAs run and waits for that grid in the kernel); the call is ordered
   on the stream as usual. */
int pkv_decode_attn_multi(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t num_new,
                          int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                          pkv_cache_desc cache, int32_t partition_blocks, int32_t max_partitions,
                          void *workspace, size_t workspace_bytes, int32_t *err_flag,
                          pkv_stream_t stream);

/* The whole verification step in one launch (two with the tcgen05 kernel's separate merge):
   pkv_slot_mapping_multi + pkv_append + pkv_decode_attn_multi fused.  k_new, v_new bf16
   [num_seqs][T][K][H] (16-byte aligned) are the T new tokens' keys and values; token t goes to the
   slot of position ctx - T + t (none below position 0) and slot_mapping_out int64 [num_seqs][T]
   (nullable, 8-byte aligned) receives those slots, -1 below position 0 or for a block id outside
   the pool (PKV_FLAG_BLOCK_RANGE).  The CTA that loads a block holding new positions first writes
   those rows into the pools (its KV head's part) and orders the writes before its own tile load,
   so attention reads them in the same pass ("Week 11. Inference", Step 3: gamma + 1 tokens checked
   in one pass; CS336 Lecture 10 notes, "其他优化": fused kernels).  Other arguments, the
   partition layout and the results are those of pkv_decode_attn_multi, bit for bit; the pools
   afterwards equal what pkv_append leaves. */
int pkv_decode_step_multi(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                          pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                          int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                          int32_t num_new, int32_t num_q_heads, float scale, pkv_bf16 *out,
                          float *lse_out, int64_t *slot_mapping_out, pkv_cache_desc cache,
                          int32_t partition_blocks, int32_t max_partitions, void *workspace,
                          size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream);

/* Limit (ns, default 2e9) of every bounded wait inside the attention kernels, for the calls
   launched after it is set (process-wide); returns the previous limit (0 sets 1 ns).  An
   expired wait sets PKV_FLAG_TIMEOUT and voids the unit's result: the kernel stops issuing,
   drains the copies it started, releases what it holds and returns, and a later call with the
   default limit runs normally.  Lowering it is a way to exercise those paths. */
uint64_t pkv_set_wait_limit_ns(uint64_t limit_ns);

/* Self-test of the bounded waits: one warp waits, with the attention kernels' bounded wait, on
   an mbarrier that nothing ever completes; after the current wait limit it gives up and sets
   PKV_FLAG_TIMEOUT in err_flag (device or pinned host int32, required).  No fault, no hang. */
int pkv_check_wait_expiry(int32_t *err_flag, pkv_stream_t stream);

/* 1 if pkv_decode_attn_multi with these sizes runs its tcgen05 column kernel, 0 if the mma.sync
   one (no GPU work; the answer assumes the half-major tensor-map layout, which the driver
   accepted on every GB300 here -- if it were refused the call would fall back to mma.sync). */
int pkv_multi_uses_tcgen05(int32_t num_new, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim);

/*
 * ---- shared prefixes and copy-on-write ------------------------------------------------------
 * Requests that share a prompt reference the same physical blocks; a request that diverges gets
 * its own copy of the block it writes into ("Optimización de la inferencia", "Página Atención",
 * copy-on-write; CS336 Lecture 10 transcript 01:21:58-01:23:17: share the prompt's KV cache,
 * split the block when the samples differ).
 */

/* Copy-on-write: for each pair i, physical block src_dst[2i+1] of both pools becomes a byte copy
   of block src_dst[2i] (whole blocks of 16 x K x H elements of elem_bytes, 1 for e4m3 pools or 2
   for bf16).  src_dst int32 [num_pairs][2] (device).  Pairs run concurrently: no destination
   may be another pair's source or destination.  An id outside [0, num_blocks) sets
   PKV_FLAG_BLOCK_RANGE and that pair is skipped.  Pools 16-byte aligned. */
int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_dst, int32_t num_pairs,
                    pkv_cache_desc cache, int32_t elem_bytes, int32_t *err_flag, pkv_stream_t stream);

/* Workspace bytes of pkv_decode_attn_prefix. */
size_t pkv_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                  int32_t max_blocks_per_seq, int32_t max_prefix_blocks,
                                  int32_t partition_blocks, int32_t prefix_partition_blocks);

/* Decode attention (one token per sequence, the result of pkv_decode_attn) for a batch whose
   sequences form groups that share their leading blocks.  group_starts int32 [num_groups + 1]
   (device, non-decreasing, within [0, num_seqs]): group g = sequences [group_starts[g],
   group_starts[g+1]); prefix_blocks int32 [num_groups] (device): the number of leading logical
   blocks that every member's table shares with the group's first member (full blocks: a partly
   filled prefix block is copied on write and belongs to each member).  Sequences outside every
   group have no shared prefix.  The shared blocks are attended once per KV head for all the
   group's queries (32 query rows per loaded tile; 128 on the tensor cores when a group holds more
   than 32 rows) in partitions of prefix_partition_blocks (0: partition_blocks), each sequence's
   own blocks separately in partitions of partition_blocks, and the partials are merged by their
   log-sum-exp.  With the tensor-core prefix pass the two passes are two launches that may run
   at the same time on the GPU (the second is launched with programmatic stream serialization);
   the merge after them is ordered behind both, so the call is ordered on the stream as usual.
   Host-side bounds: every group has at most max_group_size members and at most
   max_prefix_blocks (<= max_blocks_per_seq) shared blocks; a group beyond them, or a member
   shorter than its prefix, sets PKV_FLAG_GROUP_RANGE (that member's result is then void).  The
   members' tables are not compared: if they do not share the prefix, the result is attention
   over the first member's prefix blocks followed by the member's own blocks.  workspace of
   pkv_prefix_workspace_bytes(...) bytes, 256-byte aligned. */
int pkv_decode_attn_prefix(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                           float scale, const int32_t *group_starts, const int32_t *prefix_blocks,
                           int32_t num_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                           pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                           int32_t partition_blocks, int32_t prefix_partition_blocks, void *workspace,
                           size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream);

/* A whole shared-prefix decode step: pkv_slot_mapping + pkv_append + pkv_decode_attn_prefix, with
   the append done by the attention launch itself (copy-on-write sharing, "Optimización de la
   inferencia", "Página Atención"; the fused block-read + attention kernel of CS336 Lecture 10
   notes).  Each sequence's new K/V row (k_new / v_new [num_seqs][K][H], 16-byte aligned) is
   written into the slot of its position ctx - 1 by the suffix-pass CTA that loads that block,
   before it loads it; slot_mapping_out [num_seqs] (nullable, 8-byte aligned) receives the slots
   (-1 for ctx 0 or an out-of-range block id, as pkv_slot_mapping).  The new token must lie in the
   sequence's own blocks: a member whose context ends inside its group's shared blocks
   (ctx = 16 * prefix_blocks[g]) would write into a block every member reads, so its row is not
   written (slot -1) and PKV_FLAG_GROUP_RANGE is set.  Otherwise arguments and results as
   pkv_decode_attn_prefix, bit for bit equal to the three separate calls (outputs, lse, slots,
   pools, flags). */
int pkv_decode_step_prefix(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                           pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                           int32_t num_q_heads, float scale, const int32_t *group_starts,
                           const int32_t *prefix_blocks, int32_t num_groups, int32_t max_group_size,
                           int32_t max_prefix_blocks, pkv_bf16 *out, float *lse_out,
                           int64_t *slot_mapping_out, pkv_cache_desc cache, int32_t partition_blocks,
                           int32_t prefix_partition_blocks, void *workspace, size_t workspace_bytes,
                           int32_t *err_flag, pkv_stream_t stream);

/* Synchronise the stream, copy *err_flag to *host_value; PKV_ERR_RANGE if it is non-zero. */
int pkv_read_err_flag(const int32_t *err_flag, int32_t *host_value, pkv_stream_t stream);

/* Static text for a status code. */
const char *pkv_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
