// pkv_api.cu - the C ABI of libpagedkv: host-side validation, TMA descriptor encoding and
// kernel launches.  Every entry point validates its arguments before launching anything and
// returns a pkv_status; device-detected errors go to the caller's err_flag.
#include <algorithm>
#include <atomic>
#include <cudaTypedefs.h>

#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_internal.h"

#define PKV_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_last_error;

int cuda_fail(cudaError_t e, const char *where)
{
    g_last_error = std::string(where) + ": " + cudaGetErrorName(e) + ": " + cudaGetErrorString(e);
    return PKV_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_attn_desc(const pkv_cache_desc &d, int32_t num_q_heads)
{
    if (d.block_size != 16) return PKV_ERR_UNSUPPORTED;
    if (d.num_blocks <= 0 || d.num_kv_heads <= 0 || num_q_heads <= 0) return PKV_ERR_SHAPE;
    if (d.head_dim != 64 && d.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % d.num_kv_heads != 0) return PKV_ERR_SHAPE;
    const int G = num_q_heads / d.num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int check_copy_desc(const pkv_cache_desc &d)
{
    if (d.block_size != 16) return PKV_ERR_UNSUPPORTED;
    if (d.num_blocks <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0) return PKV_ERR_SHAPE;
    if (d.head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;  // rows move as 16-byte vectors
    return PKV_OK;
}

// SM count of the current device (cached per device).
int sm_count(int *sms)
{
    static int cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
    if (!cache[dev]) {
        e = cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    *sms = cache[dev];
    return PKV_OK;
}

// ---- TMA descriptors for the K and V pools -----------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The box of one (physical block, KV head) tile: 16 token rows x H elements, split into
// 64-element (128-byte) rows so the 128-byte swizzle applies.  Half-major order
// (dims h_lo, token, half, head, block) lands in shared memory as [half][token][64], which
// makes the MMA fragment loads bank-conflict free; token-major order (h_lo, half, head,
// token, block) is the fallback with monotone strides.  With half_box the half-major box is one
// 64-element half (16 x 128 bytes): the tcgen05 column kernel lands the two halves of a K tile in
// separate regions, so consecutive tiles form one operand of uniform row stride.
CUresult encode_kv_map(CUtensorMap *map, const void *base, const pkv_cache_desc &d, int tok_major,
                       int half_box = 0)
{
    const cuuint64_t H = (cuuint64_t)d.head_dim, K = (cuuint64_t)d.num_kv_heads;
    const cuuint64_t halves = H / 64;
    const cuuint64_t tok_stride = K * H * 2, half_stride = 128, head_stride = H * 2;
    const cuuint64_t blk_stride = 16 * K * H * 2;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5];
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (!tok_major) {
        const cuuint64_t d5[5] = {64, 16, halves, K, (cuuint64_t)d.num_blocks};
        const cuuint64_t s4[4] = {tok_stride, half_stride, head_stride, blk_stride};
        const cuuint32_t b5[5] = {64, 16, half_box ? 1u : (cuuint32_t)halves, 1, 1};
        for (int i = 0; i < 5; ++i) dims[i] = d5[i], box[i] = b5[i];
        for (int i = 0; i < 4; ++i) strides[i] = s4[i];
    } else {
        const cuuint64_t d5[5] = {64, halves, K, 16, (cuuint64_t)d.num_blocks};
        const cuuint64_t s4[4] = {half_stride, head_stride, tok_stride, blk_stride};
        const cuuint32_t b5[5] = {64, (cuuint32_t)halves, 1, 16, 1};
        for (int i = 0; i < 5; ++i) dims[i] = d5[i], box[i] = b5[i];
        for (int i = 0; i < 4; ++i) strides[i] = s4[i];
    }
    return encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                       strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

int g_tok_major = -1;  // layout the driver accepted first (-1: not yet known)
std::mutex g_layout_mu;
// limit of every bounded wait inside the attention kernels (pkv_set_wait_limit_ns)
std::atomic<uint64_t> g_wait_ns{pkv::kWaitLimitNs};
#ifdef PKV_TEST_HOOKS
// test builds only: a tile index that the attention kernels' producers skip (-1: none)
std::atomic<int64_t> g_withhold_tile{-1};
#endif

int make_kv_maps(CUtensorMap *tk, CUtensorMap *tv, const void *k, const void *v,
                 const pkv_cache_desc &d, int *tok_major)
{
    if (!encode_fn()) {
        g_last_error = "cuTensorMapEncodeTiled is unavailable from the driver";
        return PKV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_layout_mu);
    const int first = g_tok_major < 0 ? 0 : g_tok_major;
    for (int attempt = 0; attempt < 2; ++attempt) {
        const int mode = attempt == 0 ? first : 1 - first;
        CUresult rk = encode_kv_map(tk, k, d, mode);
        CUresult rv = rk == CUDA_SUCCESS ? encode_kv_map(tv, v, d, mode) : rk;
        if (rk == CUDA_SUCCESS && rv == CUDA_SUCCESS) {
            g_tok_major = mode;
            *tok_major = mode;
            return PKV_OK;
        }
        if (g_tok_major >= 0) break;  // a layout worked before: this failure is the arguments'
        g_last_error = "cuTensorMapEncodeTiled failed (CUresult " + std::to_string((int)rk) + "/" +
                       std::to_string((int)rv) + ")";
    }
    return PKV_ERR_CUDA;
}

struct AttnArgs {
    const pkv_bf16 *q, *k_cache, *v_cache;
    const int32_t *block_tables;
    int32_t max_nb;
    const int32_t *context_lens;
    int32_t B, N;
    float scale;
    pkv_cache_desc d;
    int32_t *err_flag;
};

int validate_attn(const AttnArgs &a)
{
    if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens) return PKV_ERR_NULL;
    if (a.B < 0 || a.max_nb <= 0) return PKV_ERR_SHAPE;
    int st = check_attn_desc(a.d, a.N);
    if (st != PKV_OK) return st;
    if (a.B > 65535 || a.d.num_kv_heads > 65535) return PKV_ERR_SHAPE;  // grid limits
    if ((int64_t)a.max_nb * 16 > INT32_MAX) return PKV_ERR_SHAPE;
    if (!aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) || !aligned(a.q, 4)) return PKV_ERR_ALIGN;
    return PKV_OK;
}

pkv::AttnParams params_of(const AttnArgs &a, int tok_major)
{
    pkv::AttnParams p{};
    p.q = a.q;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.max_nb = a.max_nb;
    p.B = a.B;
    p.N = a.N;
    p.K = a.d.num_kv_heads;
    p.G = a.N / a.d.num_kv_heads;
    p.num_blocks = a.d.num_blocks;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.tok_major = tok_major;
    p.err_flag = a.err_flag;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
#ifdef PKV_TEST_HOOKS
    p.withhold_tile = g_withhold_tile.load(std::memory_order_relaxed);
#endif
    return p;
}

int64_t splitk_lse_offset(int32_t B, int32_t N, int32_t H, int32_t P)
{
    const int64_t out_bytes = (int64_t)B * N * P * H * 4;
    return (out_bytes + 255) / 256 * 256;
}

// Split-KV workspace: part_out fp32 [B][N][P][H], part_lse fp32 [B][N][P], then the merge counters
// int32 [B][N] (one per (sequence, KV head) is used; zero between calls).
int64_t splitk_counter_offset(int32_t B, int32_t N, int32_t H, int32_t P)
{
    const int64_t lse_end = splitk_lse_offset(B, N, H, P) + (int64_t)B * N * P * 4;
    return (lse_end + 255) / 256 * 256;
}

struct SplitWs {
    float *part_out, *part_lse;
    int32_t *counters;
};

// The in-kernel merge keeps G x max_parts weights in the attention kernel's drained ring (32 KiB
// at least); larger splits merge in pkv_lse_merge.  pkv_lse_merge keeps max_parts weights.
constexpr int64_t kInKernelMergeWeights = pkv::kInKernelMergeWeights;
constexpr int32_t kMaxMergeParts = 12288;

bool merge_in_kernel(int32_t N, int32_t K, int32_t max_parts)
{
    return (int64_t)(N / K) * max_parts <= kInKernelMergeWeights;
}

SplitWs split_ws(void *ws, int32_t B, int32_t N, int32_t H, int32_t P)
{
    char *base = static_cast<char *>(ws);
    return {reinterpret_cast<float *>(base), reinterpret_cast<float *>(base + splitk_lse_offset(B, N, H, P)),
            reinterpret_cast<int32_t *>(base + splitk_counter_offset(B, N, H, P))};
}

// Tapered partitions (partition_range in the kernels: partition 0, launched last, half as long)
// where the split grid runs in several waves -- at least one (sequence, KV head) unit per SM --,
// the caller's max_parts leaves room for the one extra partition, and the partials stay inside
// the library.  The grid's final wave is then made of half-length CTAs and its tail shrinks
// (Llama-3-8B batch of 64, 128-block partitions: bf16 180.2 -> 178.1 us, e4m3 118.8 -> 114.7).
// A single wave (fewer units than SMs: long contexts over few sequences) keeps uniform
// partitions: there the longest CTA sets the time.
bool taper_partitions(const AttnArgs &a, int32_t part_blocks, int32_t max_parts)
{
    int sms = 0;
    if (part_blocks < 2 || sm_count(&sms) != PKV_OK) return false;
    const int64_t h = part_blocks / 2;
    const int64_t need = a.max_nb <= h ? 1 : 1 + (a.max_nb - h + part_blocks - 1) / part_blocks;
    return (int64_t)a.B * a.d.num_kv_heads >= sms && max_parts >= need;
}

// counters != nullptr: the merge runs in the attention kernel (out, lse_out written there);
// otherwise every partition's partial is written for a separate merge.  taper: partition_range's
// tapered layout (the partials are the library's own), else partition p covers blocks
// [p * part_blocks, (p + 1) * part_blocks).
int run_partitions(const AttnArgs &a, int32_t part_blocks, int32_t max_parts, float *part_out,
                   float *part_lse, int32_t *counters, pkv_bf16 *out, float *lse_out, bool taper, cudaStream_t s)
{
    if (part_blocks <= 0 || max_parts <= 0) return PKV_ERR_SHAPE;
    if ((int64_t)max_parts * part_blocks < a.max_nb) return PKV_ERR_SHAPE;
    if (!aligned(part_out, 16) || !aligned(part_lse, 4)) return PKV_ERR_ALIGN;
    CUtensorMap tk, tv;
    int tok_major = 0;
    int st = make_kv_maps(&tk, &tv, a.k_cache, a.v_cache, a.d, &tok_major);
    if (st != PKV_OK) return st;
    pkv::AttnParams p = params_of(a, tok_major);
    p.part_blocks = part_blocks;
    p.taper = taper ? 1 : 0;
    p.max_parts = max_parts;
    p.part_out = part_out;
    p.part_lse = part_lse;
    p.counters = counters;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    cudaError_t e = pkv::launch_attn(a.d.head_dim, true, tk, tv, p, s);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "attn partitions launch");
}

}  // namespace

PKV_EXPORT uint64_t pkv_kv_bytes(int64_t layers, int64_t kv_heads, int64_t head_dim, int64_t tokens,
                                 int64_t bytes_per_elem)
{
    return 2ull * (uint64_t)layers * (uint64_t)kv_heads * (uint64_t)head_dim * (uint64_t)tokens *
           (uint64_t)bytes_per_elem;
}

PKV_EXPORT int pkv_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, int32_t num_seqs, int32_t num_blocks,
                                int64_t *slot_mapping, int32_t *err_flag, pkv_stream_t stream)
{
    if (!block_tables || !context_lens || !slot_mapping) return PKV_ERR_NULL;
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
    if ((int64_t)max_blocks_per_seq * 16 > INT32_MAX) return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    cudaError_t e = pkv::launch_slot_mapping(block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                             num_blocks, slot_mapping, err_flag, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "slot mapping launch");
}

PKV_EXPORT int pkv_append(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int64_t *slot_mapping,
                          int32_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                          pkv_cache_desc cache, int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
    if (num_tokens < 0) return PKV_ERR_SHAPE;
    int st = check_copy_desc(cache);
    if (st != PKV_OK) return st;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PKV_ERR_ALIGN;
    if (num_tokens == 0) return PKV_OK;
    if ((int64_t)num_tokens * cache.num_kv_heads * cache.head_dim / 8 > ((int64_t)1 << 40))
        return PKV_ERR_SHAPE;
    cudaError_t e = pkv::launch_append(k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache,
                                       cache.num_blocks, cache.num_kv_heads, cache.head_dim, err_flag,
                                       stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "append launch");
}

PKV_EXPORT int pkv_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                               float scale, pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                               int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    if (!out) return PKV_ERR_NULL;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (!aligned(out, 4) || !aligned(lse_out, 4)) return PKV_ERR_ALIGN;
    if (num_seqs == 0) return PKV_OK;
    CUtensorMap tk, tv;
    int tok_major = 0;
    st = make_kv_maps(&tk, &tv, k_cache, v_cache, cache, &tok_major);
    if (st != PKV_OK) return st;
    pkv::AttnParams p = params_of(a, tok_major);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    cudaError_t e = pkv::launch_attn(cache.head_dim, false, tk, tv, p, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "decode attention launch");
}

PKV_EXPORT size_t pkv_splitk_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                             int32_t max_partitions)
{
    if (num_seqs < 0 || num_q_heads < 0 || head_dim < 0 || max_partitions < 0) return 0;
    return (size_t)(splitk_counter_offset(num_seqs, num_q_heads, head_dim, max_partitions) +
                    (int64_t)num_seqs * num_q_heads * 4);
}

PKV_EXPORT int pkv_decode_attn_partitions(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                          const pkv_bf16 *v_cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                                          int32_t num_seqs, int32_t num_q_heads, float scale,
                                          pkv_cache_desc cache, int32_t partition_blocks,
                                          int32_t max_partitions, float *part_out, float *part_lse,
                                          int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    if (!part_out || !part_lse) return PKV_ERR_NULL;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    return run_partitions(a, partition_blocks, max_partitions, part_out, part_lse, nullptr, nullptr,
                          nullptr, false, stream);
}

namespace {

// pkv_lse_merge, for partials in the uniform (taper false) or the tapered partition layout.
// pdl: the partials come from the launch just before on the stream, which lets the merge be
// scheduled early (griddepcontrol.launch_dependents); the merge waits for it in the kernel.
int lse_merge_impl(const float *part_out, const float *part_lse, const int32_t *context_lens, int32_t num_seqs,
                   int32_t num_q_heads, int32_t head_dim, int32_t max_partitions, int32_t partition_blocks,
                   pkv_bf16 *out, float *lse_out, bool taper, cudaStream_t stream, bool pdl = false)
{
    if (!part_out || !part_lse || !context_lens || !out) return PKV_ERR_NULL;
    if (num_seqs < 0 || num_q_heads <= 0 || max_partitions <= 0 || partition_blocks <= 0)
        return PKV_ERR_SHAPE;
    if (head_dim <= 0 || head_dim > 1024 || max_partitions > kMaxMergeParts) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_q_heads > INT32_MAX / 2) return PKV_ERR_SHAPE;
    if (!aligned(part_out, 4) || !aligned(part_lse, 4) || !aligned(out, 2) || !aligned(lse_out, 4))
        return PKV_ERR_ALIGN;
    if (num_seqs == 0) return PKV_OK;
    cudaError_t e = pkv::launch_lse_merge(part_out, part_lse, context_lens, num_seqs, num_q_heads,
                                          head_dim, max_partitions, partition_blocks, taper, out, lse_out,
                                          stream, pdl);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "lse merge launch");
}

}  // namespace

PKV_EXPORT int pkv_lse_merge(const float *part_out, const float *part_lse, const int32_t *context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                             int32_t max_partitions, int32_t partition_blocks, pkv_bf16 *out,
                             float *lse_out, pkv_stream_t stream)
{
    return lse_merge_impl(part_out, part_lse, context_lens, num_seqs, num_q_heads, head_dim, max_partitions,
                          partition_blocks, out, lse_out, false, stream);
}

PKV_EXPORT int pkv_decode_attn_splitk(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                      const pkv_bf16 *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t num_q_heads, float scale,
                                      pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                                      int32_t partition_blocks, int32_t max_partitions,
                                      void *workspace, size_t workspace_bytes, int32_t *err_flag,
                                      pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    if (!out) return PKV_ERR_NULL;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (partition_blocks <= 0 || max_partitions <= 0) return PKV_ERR_SHAPE;
    if (!workspace) return PKV_ERR_WORKSPACE;
    if (workspace_bytes < pkv_splitk_workspace_bytes(num_seqs, num_q_heads, cache.head_dim,
                                                     max_partitions))
        return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
    if (!aligned(out, 4) || !aligned(lse_out, 4)) return PKV_ERR_ALIGN;
    if (num_seqs == 0) return PKV_OK;
    const SplitWs w = split_ws(workspace, num_seqs, num_q_heads, cache.head_dim, max_partitions);
    const bool taper = taper_partitions(a, partition_blocks, max_partitions);
    if (merge_in_kernel(num_q_heads, cache.num_kv_heads, max_partitions))
        return run_partitions(a, partition_blocks, max_partitions, w.part_out, w.part_lse, w.counters, out,
                              lse_out, taper, stream);
    st = run_partitions(a, partition_blocks, max_partitions, w.part_out, w.part_lse, nullptr, nullptr,
                        nullptr, taper, stream);
    if (st != PKV_OK) return st;
    return lse_merge_impl(w.part_out, w.part_lse, context_lens, num_seqs, num_q_heads, cache.head_dim,
                          max_partitions, partition_blocks, out, lse_out, taper, stream);
}

// ---- fused decode step: slot mapping + append + attention -----------------------------------
PKV_EXPORT int pkv_decode_step(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                               pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, float scale, pkv_bf16 *out,
                               float *lse_out, int64_t *slot_mapping_out, pkv_cache_desc cache,
                               int32_t partition_blocks, int32_t max_partitions, void *workspace,
                               size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    if (!out || !k_new || !v_new) return PKV_ERR_NULL;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (!aligned(out, 4) || !aligned(lse_out, 4) || !aligned(k_new, 16) || !aligned(v_new, 16) ||
        !aligned(slot_mapping_out, 8))
        return PKV_ERR_ALIGN;
    const bool split = partition_blocks > 0;
    SplitWs sw{nullptr, nullptr, nullptr};
    if (split) {
        if (max_partitions <= 0 || (int64_t)max_partitions * partition_blocks < max_blocks_per_seq)
            return PKV_ERR_SHAPE;
        if (!workspace) return PKV_ERR_WORKSPACE;
        if (workspace_bytes < pkv_splitk_workspace_bytes(num_seqs, num_q_heads, cache.head_dim,
                                                         max_partitions))
            return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
        sw = split_ws(workspace, num_seqs, num_q_heads, cache.head_dim, max_partitions);
    } else if (partition_blocks < 0) {
        return PKV_ERR_SHAPE;
    }
    if (num_seqs == 0) return PKV_OK;
    CUtensorMap tk, tv;
    int tok_major = 0;
    st = make_kv_maps(&tk, &tv, k_cache, v_cache, cache, &tok_major);
    if (st != PKV_OK) return st;
    pkv::AttnParams p = params_of(a, tok_major);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache_w = k_cache;
    p.v_cache_w = v_cache;
    p.slot_out = slot_mapping_out;
    if (split) {
        p.part_blocks = partition_blocks;
        p.taper = taper_partitions(a, partition_blocks, max_partitions) ? 1 : 0;
        p.max_parts = max_partitions;
        p.part_out = sw.part_out;
        p.part_lse = sw.part_lse;
        p.counters = merge_in_kernel(num_q_heads, cache.num_kv_heads, max_partitions) ? sw.counters : nullptr;
    }
    cudaError_t e = pkv::launch_attn(cache.head_dim, split, tk, tv, p, stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode step launch");
    if (!split || p.counters) return PKV_OK;
    return lse_merge_impl(sw.part_out, sw.part_lse, context_lens, num_seqs, num_q_heads, cache.head_dim,
                          max_partitions, partition_blocks, out, lse_out, p.taper != 0, stream);
}

// ---- FP8 (e4m3) pools with per-KV-head scales --------------------------------------------
namespace {

// e4m3 pool [num_blocks][16][K][H] bytes, H = 128: dims (h, head, token, block) with monotone
// strides; the box is one (block, head) tile, 16 rows of 128 bytes, 128B-swizzled.
int make_kv_maps_fp8(CUtensorMap *tk, CUtensorMap *tv, const void *k, const void *v,
                     const pkv_cache_desc &d)
{
    if (!encode_fn()) {
        g_last_error = "cuTensorMapEncodeTiled is unavailable from the driver";
        return PKV_ERR_CUDA;
    }
    const cuuint64_t H = (cuuint64_t)d.head_dim, K = (cuuint64_t)d.num_kv_heads;
    const cuuint64_t dims[4] = {H, K, 16, (cuuint64_t)d.num_blocks};
    const cuuint64_t strides[3] = {H, K * H, 16 * K * H};
    const cuuint32_t box[4] = {(cuuint32_t)H, 1, 16, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    for (int t = 0; t < 2; ++t) {
        CUresult r = encode_fn()(t ? tv : tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                                 const_cast<void *>(t ? v : k), dims, strides, box, es,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            g_last_error = "cuTensorMapEncodeTiled failed for the e4m3 pool (CUresult " +
                           std::to_string((int)r) + ")";
            return PKV_ERR_CUDA;
        }
    }
    return PKV_OK;
}

int check_fp8_desc(const pkv_cache_desc &d)
{
    if (d.block_size != 16) return PKV_ERR_UNSUPPORTED;
    if (d.num_blocks <= 0 || d.num_kv_heads <= 0) return PKV_ERR_SHAPE;
    if (d.head_dim != 128) return PKV_ERR_UNSUPPORTED;  // one 128-byte swizzle row per token
    return PKV_OK;
}

int fp8_attention(const AttnArgs &a, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                  const float *k_scale, const float *v_scale, int32_t scale_block_stride,
                  pkv_bf16 *out, float *lse_out,
                  int64_t *slot_out, int32_t partition_blocks, int32_t max_partitions,
                  void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (!out || !k_scale || !v_scale) return PKV_ERR_NULL;
    if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.context_lens) return PKV_ERR_NULL;
    if (a.B < 0 || a.max_nb <= 0 || a.N <= 0) return PKV_ERR_SHAPE;
    int st = check_fp8_desc(a.d);
    if (st != PKV_OK) return st;
    if (scale_block_stride != 0 && scale_block_stride != a.d.num_kv_heads) return PKV_ERR_SHAPE;
    if (a.N % a.d.num_kv_heads != 0) return PKV_ERR_SHAPE;
    const int G = a.N / a.d.num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (a.B > 65535 || a.d.num_kv_heads > 65535 || (int64_t)a.max_nb * 16 > INT32_MAX)
        return PKV_ERR_SHAPE;
    if (!aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) || !aligned(a.q, 8) || !aligned(out, 4) ||
        !aligned(lse_out, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(slot_out, 8))
        return PKV_ERR_ALIGN;
    const bool split = partition_blocks > 0;
    SplitWs sw{nullptr, nullptr, nullptr};
    if (split) {
        if (max_partitions <= 0 || (int64_t)max_partitions * partition_blocks < a.max_nb)
            return PKV_ERR_SHAPE;
        if (!workspace ||
            workspace_bytes < pkv_splitk_workspace_bytes(a.B, a.N, a.d.head_dim, max_partitions))
            return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
        sw = split_ws(workspace, a.B, a.N, a.d.head_dim, max_partitions);
    } else if (partition_blocks < 0) {
        return PKV_ERR_SHAPE;
    }
    if (a.B == 0) return PKV_OK;
    CUtensorMap tk, tv;
    st = make_kv_maps_fp8(&tk, &tv, a.k_cache, a.v_cache, a.d);
    if (st != PKV_OK) return st;
    pkv::AttnParams p = params_of(a, 0);
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.scale_stride = scale_block_stride;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache_w = const_cast<pkv_bf16 *>(a.k_cache);
    p.v_cache_w = const_cast<pkv_bf16 *>(a.v_cache);
    p.slot_out = slot_out;
    if (split) {
        p.part_blocks = partition_blocks;
        p.taper = taper_partitions(a, partition_blocks, max_partitions) ? 1 : 0;
        p.max_parts = max_partitions;
        p.part_out = sw.part_out;
        p.part_lse = sw.part_lse;
        p.counters = merge_in_kernel(a.N, a.d.num_kv_heads, max_partitions) ? sw.counters : nullptr;
    }
    int sms = 0;
    st = sm_count(&sms);
    if (st != PKV_OK) return st;
    const bool pairs = (int64_t)a.B * a.d.num_kv_heads < sms;
    cudaError_t e = pkv::launch_attn(a.d.head_dim, split, tk, tv, p, stream, true, pairs);
    if (e != cudaSuccess) return cuda_fail(e, "e4m3 attention launch");
    if (!split || p.counters) return PKV_OK;
    return lse_merge_impl(sw.part_out, sw.part_lse, a.context_lens, a.B, a.N, a.d.head_dim, max_partitions,
                          partition_blocks, out, lse_out, p.taper != 0, stream);
}

}  // namespace

PKV_EXPORT int pkv_quantize_fp8(const pkv_bf16 *src, int64_t rows, int32_t num_kv_heads,
                                int32_t head_dim, const float *scale, int32_t scale_block_stride,
                                uint8_t *dst, pkv_stream_t stream)
{
    if (!src || !scale || !dst) return PKV_ERR_NULL;
    if (rows < 0 || num_kv_heads <= 0 || head_dim <= 0) return PKV_ERR_SHAPE;
    if (scale_block_stride != 0 && (scale_block_stride != num_kv_heads || rows % 16 != 0)) return PKV_ERR_SHAPE;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (!aligned(src, 16) || !aligned(dst, 8) || !aligned(scale, 4)) return PKV_ERR_ALIGN;
    if (rows == 0) return PKV_OK;
    cudaError_t e = pkv::launch_quantize_fp8(src, rows, num_kv_heads, head_dim, scale, scale_block_stride, dst,
                                             stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "e4m3 quantize launch");
}

PKV_EXPORT int pkv_append_fp8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const float *k_scale,
                              const float *v_scale, int32_t scale_block_stride, const int64_t *slot_mapping,
                              int32_t num_tokens, uint8_t *k_cache, uint8_t *v_cache, pkv_cache_desc cache,
                              int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_new || !v_new || !k_scale || !v_scale || !slot_mapping || !k_cache || !v_cache)
        return PKV_ERR_NULL;
    if (num_tokens < 0) return PKV_ERR_SHAPE;
    int st = check_copy_desc(cache);
    if (st != PKV_OK) return st;
    if (scale_block_stride != 0 && scale_block_stride != cache.num_kv_heads) return PKV_ERR_SHAPE;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8))
        return PKV_ERR_ALIGN;
    if (num_tokens == 0) return PKV_OK;
    cudaError_t e = pkv::launch_append_fp8(k_new, v_new, k_scale, v_scale, scale_block_stride, slot_mapping,
                                           num_tokens,
                                           k_cache, v_cache, cache.num_blocks, cache.num_kv_heads,
                                           cache.head_dim, err_flag, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "e4m3 append launch");
}

PKV_EXPORT int pkv_decode_attn_fp8(const pkv_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                   const float *k_scale, const float *v_scale, int32_t scale_block_stride,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                                   pkv_cache_desc cache, int32_t partition_blocks,
                                   int32_t max_partitions, void *workspace, size_t workspace_bytes,
                                   int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, reinterpret_cast<const pkv_bf16 *>(k_cache), reinterpret_cast<const pkv_bf16 *>(v_cache),
               block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale, cache,
               err_flag};
    return fp8_attention(a, nullptr, nullptr, k_scale, v_scale, scale_block_stride, out, lse_out, nullptr,
                         partition_blocks, max_partitions, workspace, workspace_bytes, stream);
}

PKV_EXPORT int pkv_decode_step_fp8(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                   uint8_t *k_cache, uint8_t *v_cache, const float *k_scale,
                                   const float *v_scale, int32_t scale_block_stride, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens,
                                   int32_t num_seqs, int32_t num_q_heads, float scale, pkv_bf16 *out,
                                   float *lse_out, int64_t *slot_mapping_out, pkv_cache_desc cache,
                                   int32_t partition_blocks, int32_t max_partitions, void *workspace,
                                   size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_new || !v_new) return PKV_ERR_NULL;
    AttnArgs a{q, reinterpret_cast<const pkv_bf16 *>(k_cache), reinterpret_cast<const pkv_bf16 *>(v_cache),
               block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads, scale, cache,
               err_flag};
    return fp8_attention(a, k_new, v_new, k_scale, v_scale, scale_block_stride, out, lse_out, slot_mapping_out,
                         partition_blocks, max_partitions, workspace, workspace_bytes, stream);
}

PKV_EXPORT int pkv_gather(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, const int64_t *cu_seqlens, int32_t num_seqs,
                          pkv_bf16 *k_out, pkv_bf16 *v_out, int64_t out_rows, pkv_cache_desc cache,
                          int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_cache || !v_cache || !block_tables || !context_lens || !cu_seqlens || !k_out || !v_out)
        return PKV_ERR_NULL;
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || out_rows < 0) return PKV_ERR_SHAPE;
    int st = check_copy_desc(cache);
    if (st != PKV_OK) return st;
    if (num_seqs > 65535) return PKV_ERR_SHAPE;
    if ((int64_t)max_blocks_per_seq * 16 > INT32_MAX) return PKV_ERR_SHAPE;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_out, 16) || !aligned(v_out, 16))
        return PKV_ERR_ALIGN;
    if (num_seqs == 0) return PKV_OK;
    cudaError_t e = pkv::launch_gather(k_cache, v_cache, block_tables, max_blocks_per_seq,
                                       context_lens, cu_seqlens, num_seqs, cache.num_blocks,
                                       cache.num_kv_heads, cache.head_dim, k_out, v_out, out_rows,
                                       err_flag, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "gather launch");
}

PKV_EXPORT int pkv_read_err_flag(const int32_t *err_flag, int32_t *host_value, pkv_stream_t stream)
{
    if (!err_flag || !host_value) return PKV_ERR_NULL;
    cudaError_t e = cudaMemcpyAsync(host_value, err_flag, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                    stream);
    if (e != cudaSuccess) return cuda_fail(e, "err_flag copy");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "err_flag sync");
    return *host_value != 0 ? PKV_ERR_RANGE : PKV_OK;
}

PKV_EXPORT const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape (H in {64,128}, G in {1,2,4,8}, block_size 16)";
    case PKV_ERR_RANGE: return "device-detected out-of-range value (see err_flag bits)";
    case PKV_ERR_CUDA: return "CUDA error (see pkv_last_error)";
    case PKV_ERR_ALIGN: return "pointer misaligned for the layout";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

PKV_EXPORT const char *pkv_last_error(void) { return g_last_error.c_str(); }

// ---- split-KV attention for callers that cannot allocate device memory ---------------------
//
// Some callers cannot call cudaMalloc at the point where they run attention: code running
// while a CUDA graph is being captured, inside a custom allocator's own callback, or under a
// serving framework that owns every byte of the device heap and forbids allocations on the
// decode path.  For them, pkv_decode_attn_splitk_noalloc keeps its partial results in the
// file-scope array below instead of a caller-provided workspace.  The array is part of this
// library's device image: every GPU that loads it holds PKV_STATIC_SCRATCH_BYTES of device
// memory until the process exits.  All calls share it, and it keeps the previous call's
// contents; calls that overlap on the GPU (for example on two streams) race on it.
static __device__ __align__(256) unsigned char g_splitk_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
void *g_scratch_addr[kMaxScratchDevices] = {};
std::mutex g_scratch_mu;

// Host code cannot use g_splitk_scratch's name as a device address (on the host it names a
// stand-in).  The device address is looked up once per device, with that device current.
int scratch_address(void **addr)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxScratchDevices) {
        g_last_error = "device ordinal beyond the static scratch table";
        return PKV_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_splitk_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static split-KV scratch)");
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

PKV_EXPORT int pkv_decode_attn_splitk_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                              const pkv_bf16 *v_cache, const int32_t *block_tables,
                                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                                              int32_t num_seqs, int32_t num_q_heads, float scale,
                                              pkv_bf16 *out, float *lse_out, pkv_cache_desc cache,
                                              int32_t partition_blocks, int32_t max_partitions,
                                              int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    if (!out) return PKV_ERR_NULL;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (partition_blocks <= 0 || max_partitions <= 0) return PKV_ERR_SHAPE;
    if (!aligned(out, 4) || !aligned(lse_out, 4)) return PKV_ERR_ALIGN;
    // every refusal comes before anything is launched: the separate merge's own limit included
    if (max_partitions > kMaxMergeParts) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_partitions * partition_blocks < max_blocks_per_seq) return PKV_ERR_SHAPE;
    const size_t need = pkv_splitk_workspace_bytes(num_seqs, num_q_heads, cache.head_dim,
                                                   max_partitions);
    if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) {
        g_last_error = "split-KV partials need " + std::to_string(need) +
                       " bytes; the static scratch holds " +
                       std::to_string((size_t)PKV_STATIC_SCRATCH_BYTES) +
                       " (use pkv_decode_attn_splitk with a workspace, or fewer partitions)";
        return PKV_ERR_WORKSPACE;
    }
    // the per-device address lookup comes first: a call with no sequences does it and nothing else
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != PKV_OK) return st;
    if (num_seqs == 0) return PKV_OK;
    // Nothing in the scratch has to start at zero: the partition step writes every partial
    // output and lse that the merge then reads, within this call.
    float *part_out = static_cast<float *>(scratch);
    float *part_lse = reinterpret_cast<float *>(
        static_cast<char *>(scratch) +
        splitk_lse_offset(num_seqs, num_q_heads, cache.head_dim, max_partitions));
    const bool taper = taper_partitions(a, partition_blocks, max_partitions);
    st = run_partitions(a, partition_blocks, max_partitions, part_out, part_lse, nullptr, nullptr, nullptr, taper,
                        stream);
    if (st != PKV_OK) return st;
    return lse_merge_impl(part_out, part_lse, context_lens, num_seqs, num_q_heads, cache.head_dim,
                          max_partitions, partition_blocks, out, lse_out, taper, stream);
}

// ---- several new tokens per sequence, shared prefixes, copy-on-write ------------------------
namespace {

pkv::ColsParams cols_params_of(const AttnArgs &a, int tok_major)
{
    pkv::ColsParams p{};
    p.q = a.q;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.max_nb = a.max_nb;
    p.B = a.B;
    p.N = a.N;
    p.K = a.d.num_kv_heads;
    p.G = a.N / a.d.num_kv_heads;
    p.T = 1;
    p.num_blocks = a.d.num_blocks;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.tok_major = tok_major;
    p.err_flag = a.err_flag;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
#ifdef PKV_TEST_HOOKS
    p.withhold_tile = g_withhold_tile.load(std::memory_order_relaxed);
#endif
    p.chunk_rows = 32;
    return p;
}

constexpr int kColsPerCta = 32;   // query rows per CTA of the column-parallel kernel
constexpr int kColsPerCtaTc = 128;  // of the 128-row tcgen05 form, for rows beyond 32
// Query rows per CTA from which the tcgen05 column kernel does the work.  Its time per 64-token
// group is set by its MMA instructions (8 QK^T + 4 PV whatever the row count), the mma.sync
// kernel's by its per-warp tile updates (one per 8 rows): with 32 rows the tensor cores are 1.5x
// faster (Llama-3-8B batch of 64, 8 new tokens: 252 vs 377 us per step), with 16 rows the warps
// are (222 vs 238 us).
#ifndef PKV_COLS_TC_MIN_ROWS
#define PKV_COLS_TC_MIN_ROWS 17
#endif
constexpr int kColsTcMinRows = PKV_COLS_TC_MIN_ROWS;

int32_t prefix_parts_for(int32_t max_prefix_blocks, int32_t partition_blocks)
{
    const int32_t n = (max_prefix_blocks + partition_blocks - 1) / partition_blocks;
    return n > 0 ? n : 1;
}

}  // namespace

PKV_EXPORT int pkv_slot_mapping_multi(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_seqs, int32_t num_new,
                                      int32_t num_blocks, int64_t *slot_mapping, int32_t *err_flag,
                                      pkv_stream_t stream)
{
    if (!block_tables || !context_lens || !slot_mapping) return PKV_ERR_NULL;
    if (num_seqs < 0 || num_new <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
    if ((int64_t)max_blocks_per_seq * 16 > INT32_MAX || (int64_t)num_seqs * num_new > INT32_MAX)
        return PKV_ERR_SHAPE;
    if (!aligned(slot_mapping, 8)) return PKV_ERR_ALIGN;
    if (num_seqs == 0) return PKV_OK;
    cudaError_t e = pkv::launch_slot_mapping_multi(block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                                   num_new, num_blocks, slot_mapping, err_flag, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "multi-token slot mapping launch");
}

PKV_EXPORT int pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_dst, int32_t num_pairs,
                               pkv_cache_desc cache, int32_t elem_bytes, int32_t *err_flag,
                               pkv_stream_t stream)
{
    if (!k_cache || !v_cache || (num_pairs > 0 && !src_dst)) return PKV_ERR_NULL;
    if (num_pairs < 0) return PKV_ERR_SHAPE;
    if (elem_bytes != 1 && elem_bytes != 2) return PKV_ERR_UNSUPPORTED;
    int st = check_copy_desc(cache);
    if (st != PKV_OK) return st;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst, 4)) return PKV_ERR_ALIGN;
    if (num_pairs == 0) return PKV_OK;
    const int64_t block_bytes = (int64_t)cache.block_size * cache.num_kv_heads * cache.head_dim * elem_bytes;
    cudaError_t e = pkv::launch_copy_blocks(static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
                                            src_dst, num_pairs, cache.num_blocks, block_bytes, err_flag,
                                            stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "copy-blocks launch");
}

namespace {

// pkv_decode_attn_multi, and with k_new != nullptr the fused step pkv_decode_step_multi (the
// producers write the new rows into the pools before loading their blocks).
int multi_attention(const AttnArgs &a, int32_t num_new, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                    pkv_bf16 *k_cache_w, pkv_bf16 *v_cache_w, int64_t *slot_out, pkv_bf16 *out, float *lse_out,
                    int32_t partition_blocks, int32_t max_partitions, void *workspace, size_t workspace_bytes,
                    cudaStream_t stream)
{
    const pkv_cache_desc &cache = a.d;
    const int32_t num_seqs = a.B, num_q_heads = a.N, max_blocks_per_seq = a.max_nb;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (!out) return PKV_ERR_NULL;
    if (num_new <= 0 || num_new > 64) return PKV_ERR_SHAPE;
    if (!aligned(out, 4) || !aligned(lse_out, 4)) return PKV_ERR_ALIGN;
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_out, 8))) return PKV_ERR_ALIGN;
    if ((int64_t)num_seqs * num_new > INT32_MAX) return PKV_ERR_SHAPE;
    const int32_t G = num_q_heads / cache.num_kv_heads;
    const int32_t chunks = (num_new * G + kColsPerCta - 1) / kColsPerCta;
    const bool split = partition_blocks > 0;
    int32_t parts = 1, pb = max_blocks_per_seq;
    float *part_out = nullptr, *part_lse = nullptr;
    if (split) {
        if (max_partitions <= 0 || (int64_t)max_partitions * partition_blocks < max_blocks_per_seq)
            return PKV_ERR_SHAPE;
        const int64_t rows = (int64_t)num_seqs * num_new;
        if (!workspace || workspace_bytes < pkv_splitk_workspace_bytes((int32_t)rows, num_q_heads,
                                                                       cache.head_dim, max_partitions))
            return PKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
        parts = max_partitions;
        pb = partition_blocks;
        part_out = static_cast<float *>(workspace);
        part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             splitk_lse_offset((int32_t)rows, num_q_heads, cache.head_dim,
                                                               max_partitions));
    } else if (partition_blocks < 0) {
        return PKV_ERR_SHAPE;
    }
    const int64_t grid = (int64_t)cache.num_kv_heads * num_seqs * chunks * parts;
    if (grid > INT32_MAX) return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    CUtensorMap tk, tv;
    int tok_major = 0;
    st = make_kv_maps(&tk, &tv, a.k_cache, a.v_cache, cache, &tok_major);
    if (st != PKV_OK) return st;
    pkv::ColsParams p = cols_params_of(a, tok_major);
    p.T = num_new;
    p.part_blocks = pb;
    p.parts = parts;
    p.split = split ? 1 : 0;
    p.max_parts = split ? max_partitions : 1;
    p.chunks = chunks;
    p.out = reinterpret_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    p.part_out = part_out;
    p.part_lse = part_lse;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache_w = k_cache_w;
    p.v_cache_w = v_cache_w;
    p.slot_out = slot_out;
    // With more than 16 query rows per CTA the tensor-core (tcgen05) form of the column kernel does
    // the contraction.
    bool tc = std::min(num_new * G, kColsPerCta) >= kColsTcMinRows &&
              pkv::cols_tc_supported(cache.head_dim, tok_major);
    CUtensorMap tk_half;
    if (tc) tc = encode_kv_map(&tk_half, a.k_cache, cache, 0, 1) == CUDA_SUCCESS;
    int64_t grid_run = grid;
    if (tc && num_new * G > kColsPerCta) {
        // more than 32 rows: the 128-row tcgen05 form (a group's MMAs serve 128 rows for the cost
        // of 32), chunks of 128 rows
        p.chunk_rows = kColsPerCtaTc;
        p.chunks = (num_new * G + kColsPerCtaTc - 1) / kColsPerCtaTc;
        grid_run = (int64_t)cache.num_kv_heads * num_seqs * p.chunks * parts;
    }
    // The mma.sync kernel tapers its partitions as the one-token kernel does (partition_range) when
    // its grid runs in several waves and max_partitions has room: Llama-3-8B batch of 64, 4 new
    // tokens 222.5 -> 218.1 us, 2 new tokens 198.7 -> 196.8; the tcgen05 kernel gained nothing.
    if (split && !tc) {
        AttnArgs units = a;
        units.B = (int32_t)std::min<int64_t>((int64_t)num_seqs * chunks, INT32_MAX);
        p.taper = taper_partitions(units, partition_blocks, max_partitions) ? 1 : 0;
    }
    // The mma.sync kernel's last CTA of each (sequence, KV head, chunk of 32 rows) merges the chunk
    // in the same launch when the chunk's weights (32 x max_partitions) fit in its drained ring.
    // The tcgen05 kernel's partials go to pkv_lse_merge: its merging CTAs (the partition-0 CTAs,
    // which start last) would merge 32 rows with five warps at the end of the grid, measured
    // slower than the separate launch (Llama-3-8B batch of 64, 8 new tokens: 280 vs 262 us).
    if (split && !tc && (int64_t)kColsPerCta * max_partitions <= kInKernelMergeWeights)
        p.counters = split_ws(workspace, (int32_t)(num_seqs * (int64_t)num_new), num_q_heads, cache.head_dim,
                              max_partitions).counters;
    cudaError_t e = tc ? pkv::launch_attn_cols_tc(cache.head_dim, tk_half, tv, p, grid_run, stream)
                       : pkv::launch_attn_cols(cache.head_dim, tk, tv, p, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "multi-token attention launch");
    if (!split || p.counters) return PKV_OK;
    // rows of one sequence: its T tokens x N heads, all with the sequence's context length
    // (the tcgen05 kernel lets the merge be scheduled while its last CTAs run)
    return lse_merge_impl(part_out, part_lse, a.context_lens, num_seqs, num_new * num_q_heads,
                          cache.head_dim, max_partitions, partition_blocks, out, lse_out, p.taper != 0, stream, tc);
}

}  // namespace

PKV_EXPORT int pkv_decode_attn_multi(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *context_lens, int32_t num_seqs, int32_t num_new,
                                     int32_t num_q_heads, float scale, pkv_bf16 *out, float *lse_out,
                                     pkv_cache_desc cache, int32_t partition_blocks,
                                     int32_t max_partitions, void *workspace, size_t workspace_bytes,
                                     int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    return multi_attention(a, num_new, nullptr, nullptr, nullptr, nullptr, nullptr, out, lse_out, partition_blocks,
                           max_partitions, workspace, workspace_bytes, stream);
}

PKV_EXPORT int pkv_decode_step_multi(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                     pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                     int32_t num_new, int32_t num_q_heads, float scale, pkv_bf16 *out,
                                     float *lse_out, int64_t *slot_mapping_out, pkv_cache_desc cache,
                                     int32_t partition_blocks, int32_t max_partitions, void *workspace,
                                     size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_new || !v_new) return PKV_ERR_NULL;
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    return multi_attention(a, num_new, k_new, v_new, k_cache, v_cache, slot_mapping_out, out, lse_out,
                           partition_blocks, max_partitions, workspace, workspace_bytes, stream);
}

PKV_EXPORT uint64_t pkv_set_wait_limit_ns(uint64_t limit_ns)
{
    return g_wait_ns.exchange(limit_ns == 0 ? 1 : limit_ns);
}

#ifdef PKV_TEST_HOOKS
// Test builds only (-DPKV_TEST_HOOKS; declared in tests/pkv_test_hooks.h): every CTA's producer in
// the attention launches that follow skips its tile `tile`, so the consumers' bounded waits expire.
PKV_EXPORT int64_t pkv_debug_withhold_tile(int64_t tile)
{
    return g_withhold_tile.exchange(tile < 0 ? -1 : tile);
}
#endif

PKV_EXPORT int pkv_check_wait_expiry(int32_t *err_flag, pkv_stream_t stream)
{
    if (!err_flag) return PKV_ERR_NULL;
    cudaError_t e = pkv::launch_wait_expiry(g_wait_ns.load(std::memory_order_relaxed), err_flag, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "wait-expiry self-test launch");
}

PKV_EXPORT int pkv_multi_uses_tcgen05(int32_t num_new, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim)
{
    if (num_new <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    const int32_t G = num_q_heads / num_kv_heads;
    return std::min(num_new * G, kColsPerCta) >= kColsTcMinRows && pkv::cols_tc_supported(head_dim, 0) ? 1 : 0;
}

PKV_EXPORT size_t pkv_prefix_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                             int32_t max_blocks_per_seq, int32_t max_prefix_blocks,
                                             int32_t partition_blocks, int32_t prefix_partition_blocks)
{
    if (prefix_partition_blocks == 0) prefix_partition_blocks = partition_blocks;
    if (num_seqs < 0 || num_q_heads < 0 || head_dim < 0 || max_blocks_per_seq <= 0 ||
        max_prefix_blocks < 0 || partition_blocks <= 0 || prefix_partition_blocks <= 0)
        return 0;
    const int32_t parts = prefix_parts_for(max_prefix_blocks, prefix_partition_blocks) +
                          (max_blocks_per_seq + partition_blocks - 1) / partition_blocks;
    return pkv_splitk_workspace_bytes(num_seqs, num_q_heads, head_dim, parts);
}

namespace {

// pkv_decode_attn_prefix, and with k_new != nullptr the fused step pkv_decode_step_prefix (the
// suffix pass's producers write each sequence's new row into its slot before loading its block).
int prefix_attention(const AttnArgs &a, const int32_t *group_starts, const int32_t *prefix_blocks,
                     int32_t num_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                     const pkv_bf16 *k_new, const pkv_bf16 *v_new, pkv_bf16 *k_cache_w, pkv_bf16 *v_cache_w,
                     int64_t *slot_out, pkv_bf16 *out, float *lse_out, int32_t partition_blocks,
                     int32_t prefix_partition_blocks, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream)
{
    const pkv_cache_desc &cache = a.d;
    const int32_t num_seqs = a.B, num_q_heads = a.N, max_blocks_per_seq = a.max_nb;
    const pkv_bf16 *k_cache = a.k_cache, *v_cache = a.v_cache;
    if (prefix_partition_blocks == 0) prefix_partition_blocks = partition_blocks;
    int st = validate_attn(a);
    if (st != PKV_OK) return st;
    if (!out || !workspace) return PKV_ERR_NULL;
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_out, 8))) return PKV_ERR_ALIGN;
    if (num_groups < 0 || partition_blocks <= 0 || prefix_partition_blocks <= 0 || max_prefix_blocks < 0 ||
        max_prefix_blocks > max_blocks_per_seq)
        return PKV_ERR_SHAPE;
    if (num_groups > 0 && (!group_starts || !prefix_blocks)) return PKV_ERR_NULL;
    if (num_groups > 0 && (max_group_size <= 0 || max_group_size > num_seqs)) return PKV_ERR_SHAPE;
    if (!aligned(out, 4) || !aligned(lse_out, 4) || !aligned(workspace, 256)) return PKV_ERR_ALIGN;
    if (workspace_bytes < pkv_prefix_workspace_bytes(num_seqs, num_q_heads, cache.head_dim,
                                                     max_blocks_per_seq, max_prefix_blocks,
                                                     partition_blocks, prefix_partition_blocks))
        return PKV_ERR_WORKSPACE;
    const int32_t G = num_q_heads / cache.num_kv_heads;
    const int32_t prefix_parts = prefix_parts_for(max_prefix_blocks, prefix_partition_blocks);
    const int32_t suffix_parts = (max_blocks_per_seq + partition_blocks - 1) / partition_blocks;
    const int32_t max_parts = prefix_parts + suffix_parts;
    if (max_parts > kMaxMergeParts) return PKV_ERR_UNSUPPORTED;
    const int32_t chunks = num_groups > 0 ? (max_group_size * G + kColsPerCta - 1) / kColsPerCta : 1;
    const int64_t prefix_ctas = (int64_t)cache.num_kv_heads * num_groups * chunks * prefix_parts;
    const int64_t grid = prefix_ctas + (int64_t)cache.num_kv_heads * num_seqs * suffix_parts;
    if (grid > INT32_MAX) return PKV_ERR_SHAPE;
    if (num_seqs == 0) return PKV_OK;
    CUtensorMap tk, tv;
    int tok_major = 0;
    st = make_kv_maps(&tk, &tv, k_cache, v_cache, cache, &tok_major);
    if (st != PKV_OK) return st;
    pkv::ColsParams p = cols_params_of(a, tok_major);
    p.part_blocks = partition_blocks;
    p.prefix_part_blocks = prefix_partition_blocks;
    p.parts = max_parts;
    p.split = 1;
    p.max_parts = max_parts;
    p.chunks = chunks;
    p.part_out = static_cast<float *>(workspace);
    p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                           splitk_lse_offset(num_seqs, num_q_heads, cache.head_dim, max_parts));
    p.group_starts = group_starts;
    p.prefix_blocks = prefix_blocks;
    p.num_groups = num_groups;
    p.max_group = max_group_size;
    p.prefix_parts = prefix_parts;
    p.prefix_ctas = (int32_t)prefix_ctas;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache_w = k_cache_w;
    p.v_cache_w = v_cache_w;
    p.slot_out = slot_out;
    // With more than 16 rows per chunk (the group's members x G) the prefix pass runs on the
    // tcgen05 column kernel, whose time per 64-token group is set by its MMA count, not its rows;
    // the suffix pass (G rows) stays on mma.sync, in a second launch over the rest of the work.
    bool tc = prefix_ctas > 0 && std::min(max_group_size * G, kColsPerCta) >= kColsTcMinRows &&
              pkv::cols_tc_supported(cache.head_dim, tok_major);
    CUtensorMap tk_half;
    if (tc) tc = encode_kv_map(&tk_half, k_cache, cache, 0, 1) == CUDA_SUCCESS;
    cudaError_t e;
    if (tc) {
        // more than 32 rows a group: the 128-row tcgen05 form, chunks of 128 rows
        int64_t pctas = prefix_ctas;
        if (max_group_size * G > kColsPerCta) {
            p.chunk_rows = kColsPerCtaTc;
            p.chunks = (max_group_size * G + kColsPerCtaTc - 1) / kColsPerCtaTc;
            pctas = (int64_t)cache.num_kv_heads * num_groups * p.chunks * prefix_parts;
            p.prefix_ctas = (int32_t)pctas;
        }
        e = pkv::launch_attn_cols_tc(cache.head_dim, tk_half, tv, p, pctas, stream);
        if (e != cudaSuccess) return cuda_fail(e, "shared-prefix pass launch");
        // the suffix pass alone: with no prefix CTAs in its grid, its CTAs number the suffix work
        // from 0 (the partial slots and the merge do not depend on the prefix CTA count)
        // It shares no data with the prefix pass (only the merge reads both), so it is launched
        // with programmatic serialization: its CTAs start on the SMs the prefix pass leaves free
        // once every prefix CTA is running, and its last CTA waits for the prefix grid before it
        // exits, so the merge after it sees both passes.
        pkv::ColsParams ps = p;
        ps.prefix_ctas = 0;
        ps.chunk_rows = kColsPerCta;
        ps.pdl_wait = 1;
        e = pkv::launch_attn_cols(cache.head_dim, tk, tv, ps, grid - prefix_ctas, stream, true);
    } else {
        e = pkv::launch_attn_cols(cache.head_dim, tk, tv, p, grid, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "shared-prefix attention launch");
    e = pkv::launch_cascade_merge(p, cache.head_dim, reinterpret_cast<__nv_bfloat16 *>(out), lse_out, stream);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e, "shared-prefix merge launch");
}

}  // namespace

PKV_EXPORT int pkv_decode_attn_prefix(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      float scale, const int32_t *group_starts,
                                      const int32_t *prefix_blocks, int32_t num_groups,
                                      int32_t max_group_size, int32_t max_prefix_blocks, pkv_bf16 *out,
                                      float *lse_out, pkv_cache_desc cache, int32_t partition_blocks,
                                      int32_t prefix_partition_blocks, void *workspace,
                                      size_t workspace_bytes, int32_t *err_flag, pkv_stream_t stream)
{
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    return prefix_attention(a, group_starts, prefix_blocks, num_groups, max_group_size, max_prefix_blocks,
                            nullptr, nullptr, nullptr, nullptr, nullptr, out, lse_out, partition_blocks,
                            prefix_partition_blocks, workspace, workspace_bytes, stream);
}

PKV_EXPORT int pkv_decode_step_prefix(const pkv_bf16 *q, const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                                      pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t num_q_heads, float scale,
                                      const int32_t *group_starts, const int32_t *prefix_blocks,
                                      int32_t num_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                                      pkv_bf16 *out, float *lse_out, int64_t *slot_mapping_out,
                                      pkv_cache_desc cache, int32_t partition_blocks,
                                      int32_t prefix_partition_blocks, void *workspace, size_t workspace_bytes,
                                      int32_t *err_flag, pkv_stream_t stream)
{
    if (!k_new || !v_new) return PKV_ERR_NULL;
    AttnArgs a{q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
               num_q_heads, scale, cache, err_flag};
    return prefix_attention(a, group_starts, prefix_blocks, num_groups, max_group_size, max_prefix_blocks,
                            k_new, v_new, k_cache, v_cache, slot_mapping_out, out, lse_out, partition_blocks,
                            prefix_partition_blocks, workspace, workspace_bytes, stream);
}
