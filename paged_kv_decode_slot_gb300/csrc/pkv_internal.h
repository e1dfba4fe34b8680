// pkv_internal.h - kernel parameter blocks and launchers shared by the libpagedkv
// translation units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pkv {

// Launch `kernel`; with pdl, with programmatic stream serialization: its CTAs may be scheduled once
// every CTA of the grid ahead of it on the stream has executed griddepcontrol.launch_dependents
// (or exited), so the kernel must execute griddepcontrol.wait before it reads that grid's results.
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, Args &&...args)
{
    if (!pdl) {
        kernel<<<grid, block, smem, stream>>>(std::forward<Args>(args)...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The log-sum-exp merge of a row's partitions (merge_rows): kMergeWarps warps split the
// partitions; the last partition CTA of a split runs it inside the attention kernel when the
// G * parts weights fit in kInKernelMergeWeights floats, otherwise lse_merge_kernel does.
constexpr int kMergeWarps = 6;
// Default bound on the in-kernel waits; expiry sets PKV_FLAG_TIMEOUT and the kernel returns.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kInKernelMergeWeights = 8192;

// Test builds (-DPKV_TEST_HOOKS) can make every CTA's producer skip one of its tiles -- no load,
// no barrier arrival -- so that the consumers' bounded waits on it expire; product builds carry
// neither the parameter nor the check.
#ifdef PKV_TEST_HOOKS
#define PKV_TILE_WITHHELD(p, i) ((i) == (p).withhold_tile)
#else
#define PKV_TILE_WITHHELD(p, i) false
#endif

struct AttnParams {
    const uint16_t *q;             // [B][N][H] bf16
    const int32_t *block_tables;   // [B][max_nb]
    const int32_t *context_lens;   // [B]
    int32_t max_nb;
    int32_t B, N, K, G;
    int32_t num_blocks;
    float scale_log2;              // scale * log2(e)
    int32_t tok_major;             // smem tile layout chosen by the tensor map (see pkv_attn.cu)
    int32_t part_blocks;           // split-KV: blocks per partition
    int32_t taper;                 // split-KV: tapered partitions (partition_range), else uniform
    int32_t max_parts;             // split-KV: partition stride of part_out / part_lse
    __nv_bfloat16 *out;            // single pass: [B][N][H]
    float *lse_out;                // single pass: [B][N] (nullable)
    float *part_out;               // split-KV: [B][N][max_parts][H]
    float *part_lse;               // split-KV: [B][N][max_parts]
    // fused decode step (single pass / partitions): append the new token while attending
    const uint16_t *k_new;         // [B][K][H], nullable: no append
    const uint16_t *v_new;
    void *k_cache_w;               // the pools (bf16 or e4m3), written at the newest slot
    void *v_cache_w;
    const float *k_scale;          // e4m3 pools: scales (value = code * scale), [K] or [num_blocks][K]
    const float *v_scale;
    int32_t scale_stride;          // e4m3: 0 = one scale per KV head; K = per (physical block, KV head)
    int64_t *slot_out;             // [B] slot of the newest token (-1 none), nullable
    int32_t *counters;             // split-KV with the merge in the kernel: [B][K], zero between
                                   // calls (nullptr: write every partial, merge separately)
    int32_t *err_flag;             // nullable
    uint64_t wait_ns;              // limit of every in-kernel wait (pkv_set_wait_limit_ns)
#ifdef PKV_TEST_HOOKS
    int64_t withhold_tile;         // pkv_debug_withhold_tile: -1, or a tile no CTA loads
#endif
};

// fp8: e4m3 pools (H = 128); pairs: e4m3 consumers take two tiles per step (for grids with
// fewer (sequence, KV head) units than SMs, where each CTA's dependency chains set the pace).
cudaError_t launch_attn(int H, bool split, const CUtensorMap &tk, const CUtensorMap &tv,
                        const AttnParams &p, cudaStream_t stream, bool fp8 = false, bool pairs = false);

// Column-parallel attention (pkv_attn_cols.cu): a CTA serves up to 32 query rows ("columns")
// of one KV head over one list of logical blocks; each consumer warp owns 8 columns, and every
// column has its own visibility limit.  Two uses:
//  * several new tokens per sequence (group_starts == nullptr): work unit = (sequence, KV head,
//    column chunk, partition); column j of a sequence is token t = j / G, head g = j % G, and
//    sees the tokens [0, ctx - T + t];
//  * shared prefixes (group_starts != nullptr): the first prefix_ctas CTAs run the prefix pass
//    (work unit = (group, KV head, column chunk, prefix partition); columns are the group's
//    members x G heads, blocks come from the group's first member's table), the rest run each
//    sequence's suffix (work unit = (sequence, KV head, suffix partition)).  All write partials.
struct ColsParams {
    const uint16_t *q;             // multi: [B][T][N][H]; prefix: [B][N][H]
    const int32_t *block_tables;   // [B][max_nb]
    const int32_t *context_lens;   // [B]
    int32_t max_nb;
    int32_t B, N, K, G, T;
    int32_t num_blocks;
    float scale_log2;
    int32_t tok_major;
    int32_t part_blocks;           // blocks per partition
    int32_t taper;                 // multi: tapered partitions (partition_range), else uniform
    int32_t parts;                 // multi: partitions per sequence
    int32_t split;                 // multi: write partials (1) or final outputs (0, parts == 1)
    int32_t max_parts;             // partition stride of part_out / part_lse
    int32_t chunks;                // column chunks of chunk_rows per work unit
    int32_t chunk_rows;            // query rows per CTA: 32, or 128 on the 128-row tcgen05 kernel
    __nv_bfloat16 *out;            // multi, one pass: [rows][H]
    float *lse_out;                // nullable
    float *part_out;               // [rows][max_parts][H]
    float *part_lse;               // [rows][max_parts]
    int32_t *counters;             // multi, split: [B][K][chunks] merge counts (zero between
                                   // calls; nullptr: the partials are merged by a separate launch)
    const int32_t *group_starts;   // prefix mode: [num_groups + 1]
    const int32_t *prefix_blocks;  // prefix mode: [num_groups] shared leading blocks per group
    int32_t num_groups;
    int32_t max_group;             // prefix mode: declared bound on the members of a group
    int32_t prefix_part_blocks;    // prefix mode: blocks per prefix-pass partition
    int32_t prefix_parts;          // prefix mode: partitions of the prefix pass (grid)
    int32_t prefix_ctas;           // prefix mode: CTAs of the prefix pass
    int32_t pdl_wait;              // launched behind the prefix pass with programmatic
                                   // serialization: the last CTA waits for that grid before it exits
    // multi, fused step: the T new tokens' K/V rows [B][T][K][H] (nullable: no append) are written
    // into their slots by the producer that loads their block, before it loads it
    const uint16_t *k_new;
    const uint16_t *v_new;
    uint16_t *k_cache_w;           // the pools, written at the new tokens' slots
    uint16_t *v_cache_w;
    int64_t *slot_out;             // [B][T] slots of the new tokens (-1 below position 0), nullable
    int32_t *err_flag;
    uint64_t wait_ns;              // limit of every in-kernel wait (pkv_set_wait_limit_ns)
#ifdef PKV_TEST_HOOKS
    int64_t withhold_tile;         // pkv_debug_withhold_tile: -1, or a tile no CTA loads
#endif
};

// pdl: launch with programmatic stream serialization, so that the grid may start while the grid
// before it on the stream still runs (p.pdl_wait must then be set: the grid's last CTA waits for
// that grid at its end, so the next plain launch sees both grids' writes).
cudaError_t launch_attn_cols(int H, const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                             int64_t grid, cudaStream_t stream, bool pdl = false);
// tcgen05 form of the same column kernel (H = 128, half-major tensor maps only; the K map's box
// is one 64-element half of a tile, the V map's the whole tile).
bool cols_tc_supported(int H, int tok_major);
cudaError_t launch_attn_cols_tc(int H, const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                                int64_t grid, cudaStream_t stream);
cudaError_t launch_cascade_merge(const ColsParams &p, int H, __nv_bfloat16 *out, float *lse_out,
                                 cudaStream_t stream);
cudaError_t launch_slot_mapping_multi(const int32_t *block_tables, int max_nb,
                                      const int32_t *context_lens, int B, int T, int num_blocks,
                                      int64_t *slots, int32_t *err_flag, cudaStream_t stream);
cudaError_t launch_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *src_dst, int n,
                               int num_blocks, int64_t block_bytes, int32_t *err_flag,
                               cudaStream_t stream);

cudaError_t launch_wait_expiry(uint64_t limit_ns, int32_t *err_flag, cudaStream_t stream);

cudaError_t launch_quantize_fp8(const uint16_t *src, int64_t rows, int K, int H, const float *scale,
                                int scale_stride, uint8_t *dst, cudaStream_t stream);

cudaError_t launch_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const float *k_scale,
                              const float *v_scale, int scale_stride, const int64_t *slots, int T,
                              uint8_t *k_cache,
                              uint8_t *v_cache, int num_blocks, int K, int H, int32_t *err_flag,
                              cudaStream_t stream);

// taper: the partials come from partition_range's tapered layout (partition_count partitions).
// pdl: launched with programmatic stream serialization behind the kernel that wrote the partials
// (which executes griddepcontrol.launch_dependents); the merge waits for it in the kernel.
cudaError_t launch_lse_merge(const float *part_out, const float *part_lse,
                             const int32_t *context_lens, int B, int N, int H, int max_parts,
                             int part_blocks, bool taper, uint16_t *out, float *lse_out, cudaStream_t stream,
                             bool pdl = false);

cudaError_t launch_slot_mapping(const int32_t *block_tables, int max_nb, const int32_t *context_lens,
                                int B, int num_blocks, int64_t *slots, int32_t *err_flag,
                                cudaStream_t stream);

cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots, int T,
                          uint16_t *k_cache, uint16_t *v_cache, int num_blocks, int K, int H,
                          int32_t *err_flag, cudaStream_t stream);

cudaError_t launch_gather(const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, int max_nb, const int32_t *context_lens,
                          const int64_t *cu_seqlens, int B, int num_blocks, int K, int H,
                          uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *err_flag,
                          cudaStream_t stream);

}  // namespace pkv
