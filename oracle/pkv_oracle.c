/*
 * pkv_oracle.c - the oracle: decode-step attention over a paged KV cache,
 * restated plainly in float64 on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
 * CPU-baseline leg call it; the product path never does.  It shares no code
 * with the CUDA library.
 *
 * What it follows:
 *  - KV cache size: "Optimización de la inferencia", section "Cache de KV",
 *    memory formula 2 * num_layers * num_kv_heads * head_dim * seq_len *
 *    bytes; also Week 11 "Inference", Step 2 (2 * B * S * L * K * H * bytes).
 *  - Paged layout: "Optimización de la inferencia", section "Página Atención"
 *    (fixed 16-token pages anywhere in memory, a page table mapping logical
 *    positions to physical pages); CS336 Lecture 10 notes, "分页注意力".
 *  - Appending the new token's K/V: "Optimización de la inferencia", section
 *    "Cache de KV" (compute K, V only for token N and join it to the cache),
 *    and Step 1 (KVCache.update writes the new keys/values after the cached
 *    ones and returns the cache up to and including them).
 *  - Attention: Step 2, scaled_dot_product_attention: scores = q . k / sqrt(d)
 *    (here an explicit scale), subtract the row maximum, exponentiate,
 *    normalise by the sum, multiply by V.  With one query token no mask
 *    applies (the mask there is built only when there is more than one query
 *    row; Week 11 "Inference", Common mistakes, warns against a causal mask
 *    at T = 1).
 *  - GQA: each KV head serves N/K query heads (CS336 Lecture 10 notes,
 *    "分组查询注意力"); query head n uses KV head n / (N/K).
 *  - Several query tokens per sequence: Week 11 "Inference", Step 3 (the target
 *    model verifies gamma + 1 tokens in one pass) and Common mistakes (the causal
 *    mask of the new tokens must line up with the end of the cached keys, not
 *    its start); Step 2 of "Optimización de la inferencia" masks future
 *    positions when there is more than one query row.
 *  - Copy-on-write: "Optimización de la inferencia", "Página Atención" (shared
 *    pages are stored once; a request that diverges gets its own pages);
 *    CS336 Lecture 10 transcript 01:21:58-01:23:17 (share the prompt's blocks,
 *    split a block when the samples differ).
 */
#include "pkv_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double bf16_to_double(uint16_t bits16)
{
    uint32_t bits = (uint32_t)bits16 << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

uint64_t oracle_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                         int64_t bytes_per_elem)
{
    return 2u * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim * (uint64_t)tokens *
           (uint64_t)bytes_per_elem;
}

/* Physical slot of logical token t of sequence b: the block table entry of
   block t / bs, and offset t % bs inside it. */
static int64_t physical_slot(const int32_t *block_tables, int32_t max_nb, int32_t b, int64_t t,
                             int32_t bs)
{
    int64_t block = block_tables[(int64_t)b * max_nb + t / bs];
    return block * bs + t % bs;
}

void oracle_slot_mapping(const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                         int32_t B, int32_t bs, int64_t *slots)
{
    for (int32_t b = 0; b < B; ++b) {
        int64_t pos = (int64_t)context_lens[b] - 1; /* the newest token */
        slots[b] = pos < 0 ? -1 : physical_slot(block_tables, max_nb, b, pos, bs);
    }
}

void oracle_append(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots, int32_t T,
                   uint16_t *k_cache, uint16_t *v_cache, int32_t K, int32_t H)
{
    size_t row = (size_t)K * (size_t)H; /* all KV heads of one token */
    for (int32_t i = 0; i < T; ++i) {
        if (slots[i] < 0) continue;
        memcpy(k_cache + (size_t)slots[i] * row, k_new + (size_t)i * row, row * sizeof(uint16_t));
        memcpy(v_cache + (size_t)slots[i] * row, v_new + (size_t)i * row, row * sizeof(uint16_t));
    }
}

void oracle_gather(const uint16_t *k_cache, const uint16_t *v_cache, const int32_t *block_tables,
                   int32_t max_nb, const int32_t *context_lens, const int64_t *cu_seqlens,
                   int32_t B, int32_t bs, int32_t K, int32_t H, uint16_t *k_out, uint16_t *v_out)
{
    size_t row = (size_t)K * (size_t)H;
    for (int32_t b = 0; b < B; ++b) {
        for (int64_t t = 0; t < context_lens[b]; ++t) {
            int64_t slot = physical_slot(block_tables, max_nb, b, t, bs);
            memcpy(k_out + (size_t)(cu_seqlens[b] + t) * row, k_cache + (size_t)slot * row,
                   row * sizeof(uint16_t));
            memcpy(v_out + (size_t)(cu_seqlens[b] + t) * row, v_cache + (size_t)slot * row,
                   row * sizeof(uint16_t));
        }
    }
}

/* Attention of one query vector over ntok contiguous keys/values [ntok][H]. */
static void attend(const double *q, const double *keys, const double *values, int64_t ntok,
                   int32_t H, double scale, double *scores, double *out, double *lse)
{
    if (ntok <= 0) { /* nothing to attend to: empty sum */
        for (int32_t h = 0; h < H; ++h) out[h] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int64_t t = 0; t < ntok; ++t) { /* scores = scale * q . k_t */
        double dot = 0.0;
        for (int32_t h = 0; h < H; ++h) dot += q[h] * keys[t * H + h];
        scores[t] = scale * dot;
    }
    double mx = scores[0]; /* subtract the maximum before exponentiating */
    for (int64_t t = 1; t < ntok; ++t)
        if (scores[t] > mx) mx = scores[t];
    double sum = 0.0;
    for (int64_t t = 0; t < ntok; ++t) {
        scores[t] = exp(scores[t] - mx);
        sum += scores[t];
    }
    for (int64_t t = 0; t < ntok; ++t) scores[t] /= sum; /* attention weights */
    for (int32_t h = 0; h < H; ++h) {                    /* weights times V */
        double acc = 0.0;
        for (int64_t t = 0; t < ntok; ++t) acc += scores[t] * values[t * H + h];
        out[h] = acc;
    }
    *lse = mx + log(sum);
}

typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const uint8_t *k8, *v8;             /* e4m3 pools instead of bf16 ones, when set */
    const float *k_scale, *v_scale;
    const int32_t *block_tables, *context_lens;
    int32_t max_nb, B, N, K, H, bs;
    double scale;
    int32_t partition_tokens, max_parts; /* partition_tokens <= 0: whole sequence */
    double *out, *lse;
    int nthreads, tid;
    int32_t T; /* query tokens per sequence (0 means 1) */
    int32_t scale_block_stride; /* e4m3: 0 = one scale per KV head, else per (block, head) */
} decode_job;

/* One (sequence, KV head) unit: gather its K/V rows through the block table into
   contiguous float64 arrays, then attend for each query head of the group.  With T > 1
   query tokens per sequence (the last T of its ctx tokens), query token t sits at logical
   position ctx - T + t and attends to tokens [0, ctx - T + t]: the whole cache and the new
   tokens up to itself (the causal mask aligned to the end of the keys, not to their start). */
static void decode_unit(const decode_job *j, int32_t b, int32_t kvh)
{
    const int32_t H = j->H, G = j->N / j->K;
    const int64_t ctx = j->context_lens[b] > 0 ? j->context_lens[b] : 0;
    double *keys = malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * (size_t)H);
    double *values = malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1) * (size_t)H);
    double *scores = malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
    double *qv = malloc(sizeof(double) * (size_t)H);
    for (int64_t t = 0; t < ctx; ++t) {
        int64_t slot = physical_slot(j->block_tables, j->max_nb, b, t, j->bs);
        const size_t row = ((size_t)slot * j->K + kvh) * H;
        for (int32_t h = 0; h < H; ++h) {
            if (j->k8) { /* dequantize: decode(code) * the scale of (physical block, head) */
                const size_t si = (j->scale_block_stride ? (size_t)(slot / j->bs) * (size_t)j->scale_block_stride : 0) + kvh;
                keys[t * H + h] = oracle_e4m3_decode(j->k8[row + h]) * (double)j->k_scale[si];
                values[t * H + h] = oracle_e4m3_decode(j->v8[row + h]) * (double)j->v_scale[si];
            } else {
                keys[t * H + h] = bf16_to_double(j->k_cache[row + h]);
                values[t * H + h] = bf16_to_double(j->v_cache[row + h]);
            }
        }
    }
    const int32_t T = j->T > 0 ? j->T : 1;
    for (int32_t t = 0; t < T; ++t)
    for (int32_t g = 0; g < G; ++g) {
        int32_t n = kvh * G + g;
        size_t bn = ((size_t)b * T + t) * j->N + n;
        const uint16_t *qrow = j->q + bn * H;
        for (int32_t h = 0; h < H; ++h) qv[h] = bf16_to_double(qrow[h]);
        int64_t visible = ctx - T + t + 1; /* keys this query token may see */
        if (visible < 0) visible = 0;
        if (visible > ctx) visible = ctx;
        if (j->partition_tokens <= 0) {
            attend(qv, keys, values, visible, H, j->scale, scores, j->out + bn * H, j->lse + bn);
        } else {
            for (int32_t p = 0; p < j->max_parts; ++p) {
                int64_t t0 = (int64_t)p * j->partition_tokens;
                int64_t t1 = t0 + j->partition_tokens;
                if (t1 > visible) t1 = visible;
                if (t0 > visible) t0 = visible;
                size_t bnp = bn * j->max_parts + p;
                attend(qv, keys + t0 * H, values + t0 * H, t1 - t0, H, j->scale, scores,
                       j->out + bnp * H, j->lse + bnp);
            }
        }
    }
    free(keys);
    free(values);
    free(scores);
    free(qv);
}

static void *decode_worker(void *arg)
{
    const decode_job *j = (const decode_job *)arg;
    int64_t units = (int64_t)j->B * j->K;
    for (int64_t u = j->tid; u < units; u += j->nthreads)
        decode_unit(j, (int32_t)(u / j->K), (int32_t)(u % j->K));
    return 0;
}

static void run_decode(decode_job proto)
{
    int nt = proto.nthreads;
    if (nt <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nt = c > 0 ? (int)c : 1;
    }
    if (nt > 512) nt = 512;
    if (nt > proto.B * proto.K) nt = proto.B * proto.K > 0 ? proto.B * proto.K : 1;
    decode_job jobs[512];
    pthread_t tids[512];
    int started[512];
    for (int t = 0; t < nt; ++t) {
        jobs[t] = proto;
        jobs[t].nthreads = nt;
        jobs[t].tid = t;
        started[t] = t > 0 && pthread_create(&tids[t], 0, decode_worker, &jobs[t]) == 0;
    }
    decode_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) {
        if (started[t])
            pthread_join(tids[t], 0);
        else
            decode_worker(&jobs[t]);
    }
}

void oracle_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                   const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                   int32_t B, int32_t N, int32_t K, int32_t H, int32_t bs, double scale,
                   double *out, double *lse, int nthreads)
{
    decode_job j = {q, k_cache, v_cache, 0, 0, 0, 0, block_tables, context_lens, max_nb, B, N, K,
                    H, bs, scale, 0, 1, out, lse, nthreads, 0};
    run_decode(j);
}

void oracle_decode_partitions(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                              const int32_t *block_tables, int32_t max_nb,
                              const int32_t *context_lens, int32_t B, int32_t N, int32_t K,
                              int32_t H, int32_t bs, double scale, int32_t partition_tokens,
                              int32_t max_parts, double *part_out, double *part_lse, int nthreads)
{
    decode_job j = {q, k_cache, v_cache, 0, 0, 0, 0, block_tables, context_lens, max_nb, B, N, K,
                    H, bs, scale, partition_tokens, max_parts, part_out, part_lse, nthreads, 0};
    run_decode(j);
}

void oracle_slot_mapping_multi(const int32_t *block_tables, int32_t max_nb,
                               const int32_t *context_lens, int32_t B, int32_t T, int32_t bs,
                               int64_t *slots)
{
    for (int32_t b = 0; b < B; ++b)
        for (int32_t t = 0; t < T; ++t) {
            int64_t pos = (int64_t)context_lens[b] - T + t;
            slots[(size_t)b * T + t] = pos >= 0 ? physical_slot(block_tables, max_nb, b, pos, bs) : -1;
        }
}

void oracle_decode_multi(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                         int32_t B, int32_t T, int32_t N, int32_t K, int32_t H, int32_t bs,
                         double scale, double *out, double *lse, int nthreads)
{
    decode_job j = {q, k_cache, v_cache, 0, 0, 0, 0, block_tables, context_lens, max_nb, B, N, K,
                    H, bs, scale, 0, 1, out, lse, nthreads, 0, T};
    run_decode(j);
}

void oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *src_dst, int32_t n,
                        int64_t block_bytes)
{
    for (int32_t i = 0; i < n; ++i) {
        const int64_t src = src_dst[2 * i], dst = src_dst[2 * i + 1];
        for (int64_t x = 0; x < block_bytes; ++x) {
            k_cache[dst * block_bytes + x] = k_cache[src * block_bytes + x];
            v_cache[dst * block_bytes + x] = v_cache[src * block_bytes + x];
        }
    }
}

/* Softmax over a union of disjoint key sets: each part's (out_p, lse_p) is its own
   normalised attention; the whole is the lse-weighted combination. */
void oracle_lse_merge(const double *part_out, const double *part_lse, int32_t B, int32_t N,
                      int32_t H, int32_t max_parts, double *out, double *lse)
{
    for (int64_t bn = 0; bn < (int64_t)B * N; ++bn) {
        const double *pl = part_lse + bn * max_parts;
        double mx = -INFINITY;
        for (int32_t p = 0; p < max_parts; ++p)
            if (pl[p] > mx) mx = pl[p];
        if (mx == -INFINITY) { /* no tokens at all */
            for (int32_t h = 0; h < H; ++h) out[bn * H + h] = 0.0;
            lse[bn] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int32_t p = 0; p < max_parts; ++p) sum += exp(pl[p] - mx);
        double total = mx + log(sum);
        for (int32_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t p = 0; p < max_parts; ++p)
                acc += exp(pl[p] - total) * part_out[(bn * max_parts + p) * H + h];
            out[bn * H + h] = acc;
        }
        lse[bn] = total;
    }
}

/* ---- FP8 (e4m3) -------------------------------------------------------------------------
   The format as the OCP 8-bit floating point specification defines E4M3: exponent bias 7,
   normal values (1 + m/8) * 2^(e-7) for exponent fields 1..15 (except S.1111.111, NaN),
   subnormals (m/8) * 2^-6, no infinities. */
double oracle_e4m3_decode(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 value (ties to the even code), saturating at +-448. */
uint8_t oracle_e4m3_encode(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* binade of a (exponents below -6 share the subnormal spacing 2^-9) */
    int e = -6;
    if (a >= ldexp(1.0, -6)) {
        int ex;
        frexp(a, &ex);       /* a = f * 2^ex, f in [0.5, 1) */
        e = ex - 1;
    }
    const double quantum = ldexp(1.0, e - 3);
    double r = nearbyint(a / quantum); /* a / quantum is exact; ties to even */
    if (e == -6 && r < 8.0) return (uint8_t)(sign | (uint8_t)r); /* subnormal (or zero) */
    if (r >= 16.0) {         /* rounded up into the next binade */
        r = 8.0;
        e += 1;
    }
    return (uint8_t)(sign | ((e + 7) << 3) | ((int)r - 8));
}

void oracle_quantize_fp8(const uint16_t *src, int64_t rows, int32_t K, int32_t H,
                         const float *scale, int32_t scale_block_stride, int32_t bs, uint8_t *dst)
{
    for (int64_t r = 0; r < rows; ++r) {
        /* row r of a pool belongs to physical block r / bs */
        const float *sc = scale + (scale_block_stride ? (size_t)(r / bs) * (size_t)scale_block_stride : 0);
        for (int32_t kvh = 0; kvh < K; ++kvh)
            for (int32_t h = 0; h < H; ++h) {
                size_t i = ((size_t)r * K + kvh) * H + h;
                float x = (float)bf16_to_double(src[i]);
                dst[i] = oracle_e4m3_encode(x / sc[kvh]);
            }
    }
}

void oracle_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const float *k_scale,
                       const float *v_scale, int32_t scale_block_stride, int32_t bs,
                       const int64_t *slots, int32_t T, uint8_t *k_cache, uint8_t *v_cache, int32_t K,
                       int32_t H)
{
    size_t row = (size_t)K * (size_t)H;
    for (int32_t i = 0; i < T; ++i) {
        if (slots[i] < 0) continue;
        /* the scales of the physical block the slot lies in */
        const size_t off = scale_block_stride ? (size_t)(slots[i] / bs) * (size_t)scale_block_stride : 0;
        oracle_quantize_fp8(k_new + (size_t)i * row, 1, K, H, k_scale + off, 0, 1, k_cache + (size_t)slots[i] * row);
        oracle_quantize_fp8(v_new + (size_t)i * row, 1, K, H, v_scale + off, 0, 1, v_cache + (size_t)slots[i] * row);
    }
}

void oracle_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                       const float *k_scale, const float *v_scale, int32_t scale_block_stride,
                       const int32_t *block_tables, int32_t max_nb, const int32_t *context_lens,
                       int32_t B, int32_t N, int32_t K, int32_t H, int32_t bs, double scale, double *out,
                       double *lse, int nthreads)
{
    decode_job j = {q, 0, 0, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, max_nb,
                    B, N, K, H, bs, scale, 0, 1, out, lse, nthreads, 0};
    j.scale_block_stride = scale_block_stride;
    run_decode(j);
}
