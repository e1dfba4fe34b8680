// pkv_cache_ops.cu - byte-moving kernels of the paged KV cache: slot mapping, append of the
// new token's K/V into its slot, and the block-table gather to a contiguous copy.
//
// The cache is [num_blocks][16][K][H] bf16, so all K heads of one token form one contiguous
// row of K*H elements and the 16 rows of a block are contiguous too.  Both copies therefore
// move whole 16-byte vectors with coalesced loads and stores.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// slot[b] = table[b][p / 16] * 16 + p % 16 for the newest token p = ctx_b - 1
// ("Optimización de la inferencia", "Página Atención": the page table maps logical positions
// to physical pages).
__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_tables, int max_nb,
                                    const int32_t *__restrict__ context_lens, int B, int num_blocks,
                                    int64_t *__restrict__ slots, int32_t *err_flag)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int ctx = context_lens[b];
    int64_t slot = -1;
    if (ctx > max_nb * kBlockSize) {
        set_flag(err_flag, PKV_FLAG_CTX_RANGE);
    } else if (ctx > 0) {
        const int pos = ctx - 1;
        const int blk = block_tables[(size_t)b * max_nb + pos / kBlockSize];
        if (blk < 0 || blk >= num_blocks)
            set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
        else
            slot = (int64_t)blk * kBlockSize + pos % kBlockSize;
    }
    slots[b] = slot;
}

// One thread per 16-byte vector of one token's [K][H] row: k_cache row `slot` <- k_new row i.
__global__ void append_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                              const int64_t *__restrict__ slots, int T, uint4 *__restrict__ k_cache,
                              uint4 *__restrict__ v_cache, int64_t capacity, int vec_per_row,
                              int32_t *err_flag)
{
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)T * vec_per_row) return;
    const int i = (int)(idx / vec_per_row);
    const int r = (int)(idx - (int64_t)i * vec_per_row);
    const int64_t slot = slots[i];
    if (slot < 0) return;  // skipped token
    if (slot >= capacity) {
        if (r == 0) set_flag(err_flag, PKV_FLAG_SLOT_RANGE);
        return;
    }
    const int64_t src = (int64_t)i * vec_per_row + r;
    const int64_t dst = slot * vec_per_row + r;
    k_cache[dst] = __ldg(k_new + src);
    v_cache[dst] = __ldg(v_new + src);
}

// One CTA per (logical block j, sequence b): its tokens are one contiguous run of rows in
// the pool and one contiguous run in the output.
__global__ void gather_kernel(const uint4 *__restrict__ k_cache, const uint4 *__restrict__ v_cache,
                              const int32_t *__restrict__ block_tables, int max_nb,
                              const int32_t *__restrict__ context_lens,
                              const int64_t *__restrict__ cu_seqlens, int num_blocks, int vec_per_row,
                              uint4 *__restrict__ k_out, uint4 *__restrict__ v_out, int64_t out_rows,
                              int32_t *err_flag)
{
    const int j = blockIdx.x, b = blockIdx.y;
    const int ctx = context_lens[b];
    if (ctx > max_nb * kBlockSize) {
        if (j == 0 && threadIdx.x == 0) set_flag(err_flag, PKV_FLAG_CTX_RANGE);
        return;
    }
    const int t0 = j * kBlockSize;
    if (t0 >= ctx) return;
    const int ntok = min(kBlockSize, ctx - t0);
    const int blk = block_tables[(size_t)b * max_nb + j];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
        return;
    }
    const int64_t row0 = cu_seqlens[b] + t0;
    if (row0 < 0 || row0 + ntok > out_rows) {
        if (threadIdx.x == 0) set_flag(err_flag, PKV_FLAG_OUT_RANGE);
        return;
    }
    const int64_t n = (int64_t)ntok * vec_per_row;
    const uint4 *ks = k_cache + (int64_t)blk * kBlockSize * vec_per_row;
    const uint4 *vs = v_cache + (int64_t)blk * kBlockSize * vec_per_row;
    uint4 *kd = k_out + row0 * vec_per_row;
    uint4 *vd = v_out + row0 * vec_per_row;
    for (int64_t x = threadIdx.x; x < n; x += blockDim.x) {
        kd[x] = __ldg(ks + x);
        vd[x] = __ldg(vs + x);
    }
}

// Slots of the last T logical positions of each sequence (several new tokens per step):
// slot[b][t] for position ctx_b - T + t; -1 below position 0.
__global__ void slot_mapping_multi_kernel(const int32_t *__restrict__ block_tables, int max_nb,
                                          const int32_t *__restrict__ context_lens, int B, int T,
                                          int num_blocks, int64_t *__restrict__ slots, int32_t *err_flag)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * T) return;
    const int b = (int)(i / T), t = (int)(i - (int64_t)b * T);
    const int ctx = context_lens[b];
    int64_t slot = -1;
    if (ctx > max_nb * kBlockSize) {
        if (t == 0) set_flag(err_flag, PKV_FLAG_CTX_RANGE);
    } else {
        const int pos = ctx - T + t;
        if (pos >= 0) {
            const int blk = block_tables[(size_t)b * max_nb + pos / kBlockSize];
            if (blk < 0 || blk >= num_blocks)
                set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
            else
                slot = (int64_t)blk * kBlockSize + pos % kBlockSize;
        }
    }
    slots[i] = slot;
}

// Copy-on-write: block dst of both pools becomes a byte copy of block src, one CTA per pair
// ("Optimización de la inferencia", "Página Atención": a request that diverges from a shared
// prefix gets its own pages; CS336 Lecture 10 transcript 01:23:17: split the block).
__global__ void copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                   const int32_t *__restrict__ src_dst, int num_blocks,
                                   int64_t vec_per_block, int32_t *err_flag)
{
    const int i = blockIdx.x;
    const int src = src_dst[2 * i], dst = src_dst[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0) set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
        return;
    }
    if (src == dst) return;
    const uint4 *ks = k_cache + (int64_t)src * vec_per_block, *vs = v_cache + (int64_t)src * vec_per_block;
    uint4 *kd = k_cache + (int64_t)dst * vec_per_block, *vd = v_cache + (int64_t)dst * vec_per_block;
    for (int64_t x = threadIdx.x; x < vec_per_block; x += blockDim.x) {
        kd[x] = ks[x];
        vd[x] = vs[x];
    }
}

cudaError_t launch_slot_mapping_multi(const int32_t *block_tables, int max_nb,
                                      const int32_t *context_lens, int B, int T, int num_blocks,
                                      int64_t *slots, int32_t *err_flag, cudaStream_t stream)
{
    const int threads = 128;
    const int64_t n = (int64_t)B * T;
    slot_mapping_multi_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, stream>>>(
        block_tables, max_nb, context_lens, B, T, num_blocks, slots, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *src_dst, int n,
                               int num_blocks, int64_t block_bytes, int32_t *err_flag,
                               cudaStream_t stream)
{
    copy_blocks_kernel<<<n, 256, 0, stream>>>(reinterpret_cast<uint4 *>(k_cache),
                                              reinterpret_cast<uint4 *>(v_cache), src_dst, num_blocks,
                                              block_bytes / 16, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t *block_tables, int max_nb, const int32_t *context_lens,
                                int B, int num_blocks, int64_t *slots, int32_t *err_flag,
                                cudaStream_t stream)
{
    const int threads = 128;
    slot_mapping_kernel<<<(B + threads - 1) / threads, threads, 0, stream>>>(
        block_tables, max_nb, context_lens, B, num_blocks, slots, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_append(const uint16_t *k_new, const uint16_t *v_new, const int64_t *slots, int T,
                          uint16_t *k_cache, uint16_t *v_cache, int num_blocks, int K, int H,
                          int32_t *err_flag, cudaStream_t stream)
{
    const int vec_per_row = K * H / 8;
    const int64_t total = (int64_t)T * vec_per_row;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    append_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), slots, T,
        reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
        (int64_t)num_blocks * kBlockSize, vec_per_row, err_flag);
    return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, int max_nb, const int32_t *context_lens,
                          const int64_t *cu_seqlens, int B, int num_blocks, int K, int H,
                          uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *err_flag,
                          cudaStream_t stream)
{
    gather_kernel<<<dim3(max_nb, B), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_cache), reinterpret_cast<const uint4 *>(v_cache),
        block_tables, max_nb, context_lens, cu_seqlens, num_blocks, K * H / 8,
        reinterpret_cast<uint4 *>(k_out), reinterpret_cast<uint4 *>(v_out), out_rows, err_flag);
    return cudaGetLastError();
}

}  // namespace pkv

// ------------------------------ bounded-wait self-test ------------------------------------
// One warp waits, with the same bounded wait the attention kernels use, on an mbarrier that no
// thread ever arrives at: the wait expires after limit_ns and the kernel sets PKV_FLAG_TIMEOUT.
namespace pkv {

__global__ void wait_expiry_kernel(uint64_t limit_ns, int32_t *err_flag)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(b, 0u, nullptr, limit_ns);
    if (!ok && threadIdx.x == 0) set_flag(err_flag, PKV_FLAG_TIMEOUT);
}

cudaError_t launch_wait_expiry(uint64_t limit_ns, int32_t *err_flag, cudaStream_t stream)
{
    wait_expiry_kernel<<<1, 32, 0, stream>>>(limit_ns, err_flag);
    return cudaGetLastError();
}

}  // namespace pkv

// ---------------------------------- FP8 (e4m3) cache ----------------------------------------
// code = e4m3(x / scale[kvh]): the division rounded to nearest in fp32, then round-to-nearest-
// even onto the e4m3 grid with saturation at +-448 (cvt.rn.satfinite).  One thread per 8 values.
// With scale_stride > 0 the scales are per (physical block, KV head): a value in block blk uses
// scale[blk * scale_stride + kvh].
namespace pkv {

__device__ __forceinline__ uint2 quantize8(const uint4 x, float sc)
{
    auto q2 = [&](uint32_t pair) -> uint32_t {
        return f32x2_to_e4m3x2(__fdiv_rn(bf16_to_f32((uint16_t)(pair & 0xFFFFu)), sc),
                               __fdiv_rn(bf16_to_f32((uint16_t)(pair >> 16)), sc));
    };
    return make_uint2(q2(x.x) | (q2(x.y) << 16), q2(x.z) | (q2(x.w) << 16));
}

__global__ void quantize_fp8_kernel(const uint4 *__restrict__ src, int64_t n8, int K, int H,
                                    const float *__restrict__ scale, int scale_stride,
                                    uint2 *__restrict__ dst)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const int64_t row = (i * 8) / H;  // [rows][K] of H-element head rows
    const int kvh = (int)(row % K);
    const int64_t blk = row / ((int64_t)K * kBlockSize);
    dst[i] = quantize8(__ldg(src + i), __ldg(scale + blk * scale_stride + kvh));
}

__global__ void append_fp8_kernel(const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                  const float *__restrict__ k_scale, const float *__restrict__ v_scale,
                                  int scale_stride, const int64_t *__restrict__ slots, int T,
                                  uint2 *__restrict__ k_cache,
                                  uint2 *__restrict__ v_cache, int64_t capacity, int K, int H,
                                  int32_t *err_flag)
{
    const int vec_per_row = K * H / 8;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)T * vec_per_row) return;
    const int i = (int)(idx / vec_per_row);
    const int r = (int)(idx - (int64_t)i * vec_per_row);
    const int64_t slot = slots[i];
    if (slot < 0) return;
    if (slot >= capacity) {
        if (r == 0) set_flag(err_flag, PKV_FLAG_SLOT_RANGE);
        return;
    }
    const int kvh = r * 8 / H;
    const int64_t src = (int64_t)i * vec_per_row + r, dst = slot * vec_per_row + r;
    const int64_t si = (slot / kBlockSize) * scale_stride + kvh;  // scales of the slot's block
    k_cache[dst] = quantize8(__ldg(k_new + src), __ldg(k_scale + si));
    v_cache[dst] = quantize8(__ldg(v_new + src), __ldg(v_scale + si));
}

cudaError_t launch_quantize_fp8(const uint16_t *src, int64_t rows, int K, int H, const float *scale,
                                int scale_stride, uint8_t *dst, cudaStream_t stream)
{
    const int64_t n8 = rows * K * H / 8;
    const int threads = 256;
    quantize_fp8_kernel<<<(unsigned)((n8 + threads - 1) / threads), threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(src), n8, K, H, scale, scale_stride, reinterpret_cast<uint2 *>(dst));
    return cudaGetLastError();
}

cudaError_t launch_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const float *k_scale,
                              const float *v_scale, int scale_stride, const int64_t *slots, int T,
                              uint8_t *k_cache,
                              uint8_t *v_cache, int num_blocks, int K, int H, int32_t *err_flag,
                              cudaStream_t stream)
{
    const int64_t total = (int64_t)T * K * H / 8;
    const int threads = 256;
    append_fp8_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k_new), reinterpret_cast<const uint4 *>(v_new), k_scale,
        v_scale, scale_stride, slots, T, reinterpret_cast<uint2 *>(k_cache), reinterpret_cast<uint2 *>(v_cache),
        (int64_t)num_blocks * kBlockSize, K, H, err_flag);
    return cudaGetLastError();
}

}  // namespace pkv
