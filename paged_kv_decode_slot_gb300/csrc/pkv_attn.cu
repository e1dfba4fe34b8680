// pkv_attn.cu - paged decode attention for sm_103a.
//
// One CTA per work unit (sequence b, KV head kvh[, partition p]).  A producer warp walks the
// unit's slice of the block table and streams each physical block's K and V tiles
// (16 tokens x H bf16 for head kvh) into a ring of shared-memory stages with TMA, one
// mbarrier pair per stage.  Four consumer warps take the stages round-robin; each keeps its
// own online-softmax state for the whole query group (the G = N/K query heads that share
// kvh), so every K/V byte fetched from HBM serves all G heads:
//     S^T[16 tok x 8] = K_tile[16 x H] . Q^T[H x 8]        (mma.sync m16n8k16, G padded to 8)
//     P^T            = exp2(S^T * scale*log2e - m)         (fp32, lazily rescaled running max)
//     O^T[H x 8]    += V_tile^T[H x 16] . P^T[16 x 8]      (P^T moved to the B operand with
//                                                          movmatrix; V^T via ldmatrix.trans)
// At the end the warps' partial states are merged in shared memory and the CTA writes the
// bf16 output and lse (single pass) or the fp32 normalised partial output and lse of its
// partition (split-KV, merged afterwards by lse_merge_kernel).
//
// This fuses the block-table gather with attention ("融合块读取和注意力的内核" and
// FlashDecoding in CS336 Lecture 10's notes) and computes, for one query token,
// softmax(q K^T * scale) V with the maximum subtracted ("Optimización de la inferencia",
// "Construye el mismo", Step 2).  The softmax is the online (running max / running sum)
// form of the same quantity; the LSE merge is exact for disjoint key sets.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kConsumerWarps = 4;
constexpr int kStages = 8;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
// Lazy rescaling: keep the running maximum until a new logit exceeds it by this much
// (log2 units), so exponentials stay <= 2^8 and the accumulator is rarely rescaled.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int H>
struct AttnLayout {
    static constexpr int kHalves = H / 64;                  // 128-byte rows per token row
    static constexpr int kTileBytes = kBlockSize * H * 2;   // one K or V tile
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile then V tile
    static constexpr int kPipeBytes = kStages * kStageBytes;
    static constexpr int kMergeBytes = kConsumerWarps * 8 * (H + 2) * 4;
    static constexpr int kDataBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
    static constexpr int kBarOffset = kDataBytes;           // full[kStages], empty[kStages]
    static constexpr int kMiscOffset = kBarOffset + 2 * kStages * 8;  // slot_ok[], abort, issued
    static constexpr int kBytes = kMiscOffset + (kStages + 4) * 4;
    static constexpr int kAlloc = kBytes + 1024;             // slack for 1024-byte alignment
};

template <int H>
int attn_smem_bytes() { return AttnLayout<H>::kAlloc; }

// Byte offset inside a TMA-written, 128B-swizzled tile of the 16-byte chunk holding
// elements h .. h+7 of token row tok.  Tile rows are 128 bytes; with half-major tiles the
// row of (tok, half) is half*16 + tok, with token-major tiles tok*kHalves + half.  The
// swizzle XORs the chunk index with the row index mod 8 (tile base 1024-byte aligned).
template <int H>
__device__ __forceinline__ uint32_t tile_chunk_offset(int tok, int h, int tok_major)
{
    constexpr int kHalves = AttnLayout<H>::kHalves;
    const int half = h >> 6;
    const int chunk = (h & 63) >> 3;
    const int row = tok_major ? tok * kHalves + half : half * kBlockSize + tok;
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int H, bool kSplit>
__global__ void __launch_bounds__(kAttnThreads)
attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
            const AttnParams p)
{
    using L = AttnLayout<H>;
    constexpr int kKSteps = H / 16;  // k-steps of the QK^T contraction, m-tiles of PV

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - raw_u32);

    const int kvh = kSplit ? blockIdx.y : blockIdx.x;
    const int b = kSplit ? blockIdx.z : blockIdx.y;
    const int part = kSplit ? blockIdx.x : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.G;

    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_nb * kBlockSize) {
        if (threadIdx.x == 0 && kvh == 0 && part == 0) set_flag(p.err_flag, PKV_FLAG_CTX_RANGE);
        ctx = 0;
    }
    const int nb = (ctx + kBlockSize - 1) / kBlockSize;
    const int blk_begin = kSplit ? part * p.part_blocks : 0;
    const int blk_end = kSplit ? min(nb, blk_begin + p.part_blocks) : nb;
    const int nblk = blk_end - blk_begin;

    if (nblk <= 0) {
        if (kSplit) return;  // an empty partition is never read by the merge
        for (int idx = threadIdx.x; idx < G * H; idx += kAttnThreads) {
            const int g = idx / H, h = idx - g * H;
            const size_t bn = (size_t)b * p.N + (size_t)kvh * G + g;
            p.out[bn * H + h] = __float2bfloat16_rn(0.0f);
            if (h == 0 && p.lse_out) p.lse_out[bn] = -INFINITY;
        }
        return;
    }

    const uint32_t bar_full = base_u32 + L::kBarOffset;
    const uint32_t bar_empty = bar_full + 8 * kStages;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(base + L::kMiscOffset);
    volatile int *abort_flag = slot_ok + kStages;
    volatile int *issued_count = abort_flag + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        *abort_flag = 0;
        *issued_count = 0;
        fence_barrier_init();
    }
    __syncthreads();

    float o[kKSteps][4];  // O^T fragments: rows h (16 per m-tile), cols g
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};

    if (warp == kConsumerWarps) {
        // ------------------------------ producer warp ------------------------------
        if (lane == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int32_t *tbl = p.block_tables + (size_t)b * p.max_nb + blk_begin;
        int cur = lane < nblk ? __ldg(tbl + lane) : 0;
        bool aborted = false;
        int issued = 0;
        for (int i0 = 0; i0 < nblk && !aborted; i0 += 32) {
            const int nxt = (i0 + 32 + lane < nblk) ? __ldg(tbl + i0 + 32 + lane) : 0;
            const int cnt = min(32, nblk - i0);
            const bool bad = lane < cnt && (cur < 0 || cur >= p.num_blocks);
            const unsigned badmask = __ballot_sync(0xFFFFFFFFu, bad);
            if (badmask && lane == 0) set_flag(p.err_flag, PKV_FLAG_BLOCK_RANGE);
            for (int k = 0; k < cnt; ++k) {
                const int bid = __shfl_sync(0xFFFFFFFFu, cur, k);
                int lane0_abort = 0;
                if (lane == 0) {
                    const int i = i0 + k;
                    const int s = i % kStages;
                    bool ok = true;
                    if (i >= kStages)
                        ok = mbar_wait_bounded(bar_empty + 8 * s, ((i / kStages) & 1) ^ 1,
                                               abort_flag, kWaitLimitNs);
                    if (!ok) {
                        if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                        *abort_flag = 1;
                        lane0_abort = 1;
                    } else if (!((badmask >> k) & 1u)) {
                        slot_ok[s] = 1;
                        const uint32_t dst = base_u32 + s * L::kStageBytes;
                        mbar_arrive_expect_tx(bar_full + 8 * s, L::kStageBytes);
                        if (p.tok_major) {
                            tma_load_5d(dst, &tm_k, bar_full + 8 * s, 0, 0, kvh, 0, bid);
                            tma_load_5d(dst + L::kTileBytes, &tm_v, bar_full + 8 * s, 0, 0, kvh, 0, bid);
                        } else {
                            tma_load_5d(dst, &tm_k, bar_full + 8 * s, 0, 0, 0, kvh, bid);
                            tma_load_5d(dst + L::kTileBytes, &tm_v, bar_full + 8 * s, 0, 0, 0, kvh, bid);
                        }
                        ++issued;
                    } else {
                        slot_ok[s] = 0;  // out-of-range block id: the tile is skipped
                        mbar_arrive(bar_full + 8 * s);
                        ++issued;
                    }
                }
                aborted = __shfl_sync(0xFFFFFFFFu, lane0_abort, 0) != 0;
                if (aborted) break;
            }
            cur = nxt;
        }
        if (lane == 0) *issued_count = issued;
    } else {
        // ------------------------------ consumer warps ------------------------------
        const int g_row = lane >> 2;        // Q^T column / fragment row owned by this lane
        const int c0 = (lane & 3) * 2;      // first of the two columns this lane accumulates
        uint32_t qf[kKSteps][2];            // Q^T as the B operand of S^T = K . Q^T
        {
            const bool live = g_row < G;
            const uint16_t *qrow = p.q + ((size_t)b * p.N + (size_t)kvh * G + (live ? g_row : 0)) * H;
#pragma unroll
            for (int kk = 0; kk < kKSteps; ++kk) {
                qf[kk][0] = live ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0)) : 0u;
                qf[kk][1] = live ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0 + 8)) : 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

        // ldmatrix source rows: lane l feeds matrix l/8, row l%8.
        const int mi = lane >> 3, ri = lane & 7;
        const int k_tok = ri + 8 * (mi & 1), k_hoff = 8 * (mi >> 1);  // K as A (non-trans)
        const int v_tok = ri + 8 * (mi >> 1), v_hoff = 8 * (mi & 1);  // V^T as A (trans)
        const float sl2 = p.scale_log2;

        for (int i = warp; i < nblk; i += kConsumerWarps) {
            const int s = i % kStages;
            if (!mbar_wait_bounded(bar_full + 8 * s, (i / kStages) & 1, abort_flag, kWaitLimitNs)) {
                if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            if (slot_ok[s]) {
                const int valid = min(kBlockSize, ctx - (blk_begin + i) * kBlockSize);
                const uint32_t kt = base_u32 + s * L::kStageBytes;
                const uint32_t vt = kt + L::kTileBytes;

                // S^T = K . Q^T, two independent accumulation chains
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < kKSteps; kk += 2) {
                    uint32_t a0[4], a1[4];
                    ldsm_x4(a0, kt + tile_chunk_offset<H>(k_tok, 16 * kk + k_hoff, p.tok_major));
                    ldsm_x4(a1, kt + tile_chunk_offset<H>(k_tok, 16 * kk + 16 + k_hoff, p.tok_major));
                    mma_bf16_16816(sa, a0, qf[kk][0], qf[kk][1]);
                    mma_bf16_16816(sb, a1, qf[kk + 1][0], qf[kk + 1][1]);
                }
                // rows: tokens t0 = lane/4 and t1 = t0 + 8; columns: g = c0, c0+1
                const int t0 = lane >> 2, t1 = t0 + 8;
                const float x0 = t0 < valid ? (sa[0] + sb[0]) * sl2 : -INFINITY;
                const float x1 = t0 < valid ? (sa[1] + sb[1]) * sl2 : -INFINITY;
                const float x2 = t1 < valid ? (sa[2] + sb[2]) * sl2 : -INFINITY;
                const float x3 = t1 < valid ? (sa[3] + sb[3]) * sl2 : -INFINITY;
                float mA = fmaxf(x0, x2), mB = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mA = fmaxf(mA, __shfl_xor_sync(0xFFFFFFFFu, mA, off));
                    mB = fmaxf(mB, __shfl_xor_sync(0xFFFFFFFFu, mB, off));
                }
                const bool needA = mA > m_run[0] + kRescaleThreshold;
                const bool needB = mB > m_run[1] + kRescaleThreshold;
                if (__any_sync(0xFFFFFFFFu, needA || needB)) {
                    const float alphaA = needA ? exp2f(m_run[0] - mA) : 1.f;
                    const float alphaB = needB ? exp2f(m_run[1] - mB) : 1.f;
                    if (needA) m_run[0] = mA;
                    if (needB) m_run[1] = mB;
                    l_run[0] *= alphaA;
                    l_run[1] *= alphaB;
#pragma unroll
                    for (int mt = 0; mt < kKSteps; ++mt) {
                        o[mt][0] *= alphaA;
                        o[mt][1] *= alphaB;
                        o[mt][2] *= alphaA;
                        o[mt][3] *= alphaB;
                    }
                }
                const uint32_t p01 = pack_bf16x2(exp2f(x0 - m_run[0]), exp2f(x1 - m_run[1]));
                const uint32_t p23 = pack_bf16x2(exp2f(x2 - m_run[0]), exp2f(x3 - m_run[1]));
                l_run[0] += bf16x2_lo(p01) + bf16x2_lo(p23);  // sums of the rounded weights
                l_run[1] += bf16x2_hi(p01) + bf16x2_hi(p23);
                const uint32_t pb0 = movmatrix_trans(p01);    // P^T rows tok 0-7 -> B frag
                const uint32_t pb1 = movmatrix_trans(p23);    // tok 8-15

                // O^T += V^T . P^T
                const bool partial = valid < kBlockSize;
                const int tc = (lane & 3) * 2;  // token columns of this lane's A fragment
#pragma unroll
                for (int mt = 0; mt < kKSteps; ++mt) {
                    uint32_t a[4];
                    ldsm_x4_trans(a, vt + tile_chunk_offset<H>(v_tok, 16 * mt + v_hoff, p.tok_major));
                    if (partial) {  // zero V of tokens past the context (they may be NaN poison)
                        const uint32_t lo0 = tc < valid ? 0x0000FFFFu : 0u;
                        const uint32_t hi0 = tc + 1 < valid ? 0xFFFF0000u : 0u;
                        const uint32_t lo1 = tc + 8 < valid ? 0x0000FFFFu : 0u;
                        const uint32_t hi1 = tc + 9 < valid ? 0xFFFF0000u : 0u;
                        a[0] &= lo0 | hi0;
                        a[1] &= lo0 | hi0;
                        a[2] &= lo1 | hi1;
                        a[3] &= lo1 | hi1;
                    }
                    mma_bf16_16816(o[mt], a, pb0, pb1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // Drain: wait (bounded) for copies that were issued and may still be landing.
        if (threadIdx.x == kConsumerWarps * 32) {
            const int issued = *issued_count;
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait_bounded(bar_full + 8 * (i % kStages), (i / kStages) & 1, nullptr,
                                  kDrainLimitNs);
        }
        __syncthreads();
        return;
    }

    // ------------------------- merge the consumer warps' states -------------------------
    float *mo = reinterpret_cast<float *>(base);              // [W][8][H]
    float *mm = mo + kConsumerWarps * 8 * H;                 // [W][8] running max (log2 units)
    float *ml = mm + kConsumerWarps * 8;                     // [W][8] running sum
    if (warp < kConsumerWarps) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_run[0] += __shfl_xor_sync(0xFFFFFFFFu, l_run[0], off);
            l_run[1] += __shfl_xor_sync(0xFFFFFFFFu, l_run[1], off);
        }
        const int c0 = (lane & 3) * 2;
        if (lane < 4) {
            mm[warp * 8 + c0] = m_run[0];
            mm[warp * 8 + c0 + 1] = m_run[1];
            ml[warp * 8 + c0] = l_run[0];
            ml[warp * 8 + c0 + 1] = l_run[1];
        }
        const int hr = lane >> 2;
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) {
            const int h = 16 * mt + hr;
            mo[(warp * 8 + c0) * H + h] = o[mt][0];
            mo[(warp * 8 + c0 + 1) * H + h] = o[mt][1];
            mo[(warp * 8 + c0) * H + h + 8] = o[mt][2];
            mo[(warp * 8 + c0 + 1) * H + h + 8] = o[mt][3];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * H; idx += kAttnThreads) {
        const int g = idx / H, h = idx - g * H;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * 8 + g]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float sc = exp2f(mm[w * 8 + g] - M);
                lsum += sc * ml[w * 8 + g];
                acc += sc * mo[(w * 8 + g) * H + h];
            }
        }
        const float val = lsum > 0.f ? acc / lsum : 0.f;
        const float lse = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
        const size_t bn = (size_t)b * p.N + (size_t)kvh * G + g;
        if (kSplit) {
            const size_t bnp = bn * p.max_parts + part;
            p.part_out[bnp * H + h] = val;
            if (h == 0) p.part_lse[bnp] = lse;
        } else {
            p.out[bn * H + h] = __float2bfloat16_rn(val);
            if (h == 0 && p.lse_out) p.lse_out[bn] = lse;
        }
    }
}

// ---------------------------------- LSE merge ----------------------------------------------
// One CTA per (query head n, sequence b), one thread per output element h.
__global__ void lse_merge_kernel(const float *__restrict__ part_out, const float *__restrict__ part_lse,
                                 const int32_t *__restrict__ context_lens, int N, int H, int max_parts,
                                 int part_blocks, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out)
{
    const int n = blockIdx.x, b = blockIdx.y, h = threadIdx.x;
    const size_t bn = (size_t)b * N + n;
    int ctx = context_lens[b];
    const int nb = ctx > 0 ? (ctx + kBlockSize - 1) / kBlockSize : 0;
    int np = (nb + part_blocks - 1) / part_blocks;
    if (np > max_parts) np = max_parts;
    const float *lp = part_lse + bn * max_parts;
    float M = -INFINITY;
    for (int q = 0; q < np; ++q) M = fmaxf(M, lp[q]);
    float total = -INFINITY, val = 0.f;
    if (M != -INFINITY) {
        float sum = 0.f;
        for (int q = 0; q < np; ++q) sum += expf(lp[q] - M);
        total = M + logf(sum);
        if (h < H) {
            const float *po = part_out + bn * max_parts * H + h;
            for (int q = 0; q < np; ++q) val += expf(lp[q] - total) * po[(size_t)q * H];
        }
    }
    if (h < H) out[bn * H + h] = __float2bfloat16_rn(val);
    if (h == 0 && lse_out) lse_out[bn] = total;
}

// ---------------------------------- launchers ----------------------------------------------
template <int H, bool kSplit>
static cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                                 dim3 grid, cudaStream_t stream)
{
    constexpr int smem = AttnLayout<H>::kAlloc;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attn_kernel<H, kSplit>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    attn_kernel<H, kSplit><<<grid, kAttnThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_attn(int H, bool split, const CUtensorMap &tk, const CUtensorMap &tv,
                        const AttnParams &p, cudaStream_t stream)
{
    dim3 grid = split ? dim3(p.max_parts, p.K, p.B) : dim3(p.K, p.B, 1);
    if (H == 128)
        return split ? launch_attn_t<128, true>(tk, tv, p, grid, stream)
                     : launch_attn_t<128, false>(tk, tv, p, grid, stream);
    return split ? launch_attn_t<64, true>(tk, tv, p, grid, stream)
                 : launch_attn_t<64, false>(tk, tv, p, grid, stream);
}

cudaError_t launch_lse_merge(const float *part_out, const float *part_lse, const int32_t *context_lens,
                             int B, int N, int H, int max_parts, int part_blocks, uint16_t *out,
                             float *lse_out, cudaStream_t stream)
{
    const int threads = H < 32 ? 32 : H;
    lse_merge_kernel<<<dim3(N, B), threads, 0, stream>>>(
        part_out, part_lse, context_lens, N, H, max_parts, part_blocks,
        reinterpret_cast<__nv_bfloat16 *>(out), lse_out);
    return cudaGetLastError();
}

}  // namespace pkv
