// pkv_attn_cols.cu - column-parallel decode attention: one CTA serves up to 32 query rows of one
// KV head over one list of logical blocks, so that each K/V tile it loads is used by every row.
//
// Two methods need more query rows per loaded tile than one decode token's G heads:
//  * verifying several new tokens per sequence at once (speculative decoding: the target model
//    checks gamma + 1 tokens in one pass -- "Week 11. Inference", Step 3).  Token t of the T new
//    ones sits at logical position ctx - T + t and sees the tokens [0, ctx - T + t]: the causal
//    mask of the new tokens lines up with the end of the keys, not with their start (Week 11,
//    "Common mistakes": a mask aligned to the top-left corner is the classic bug);
//  * sequences that share a prompt prefix through their block tables (copy-on-write sharing,
//    "Optimización de la inferencia", "Página Atención"; CS336 Lecture 10 transcript 01:21:58):
//    the shared blocks are attended once per KV head for all members' queries (the prefix pass),
//    each sequence's own blocks separately (the suffix pass), and the partials are merged by their
//    log-sum-exp, which is exact for disjoint key sets.
//
// CTA: 4 consumer warps + 2 producer warps, the same TMA ring as attn_kernel.  The CTA's ncols
// rows form ng = ceil(ncols / 8) groups of 8 (3 rounds up to 4); consumer warp w owns group
// w % ng and reads the tiles i = w / ng (mod 4 / ng), so each stage is consumed by ng warps and its
// empty barrier counts ng arrivals.  With ng < 4 the warps of one group split the tiles and their
// states are merged in shared memory, as in attn_kernel.
#include "pkv_cols.cuh"

namespace pkv {

// Q^T as the B operand for the warp's 8 columns: lane l holds row l/4 (qrow, or zeros).
template <int H>
__device__ __forceinline__ void load_q_frags_row(uint32_t (&qf)[H / 16][2], const uint16_t *qrow, int lane)
{
    const int c0 = (lane & 3) * 2;
#pragma unroll
    for (int kk = 0; kk < H / 16; ++kk) {
        qf[kk][0] = qrow ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0)) : 0u;
        qf[kk][1] = qrow ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0 + 8)) : 0u;
    }
}

// tile_update with a visibility limit per column: the lane's columns A (2(lane%4)) and B (+1) see
// the first va / vb tokens of the tile; tokens at or past `valid` may be poison and their V rows
// are zeroed.  A column that has seen no token yet keeps m = -inf and gets zero weights.
template <int H>
__device__ __forceinline__ void tile_update_cols(WarpAcc<H> &a, const uint32_t (&qf)[H / 16][2],
                                                 uint32_t kt, uint32_t vt, int va, int vb, int valid,
                                                 float sl2, int tok_major, int lane)
{
    constexpr int kKSteps = H / 16;
    const int mi = lane >> 3, ri = lane & 7;
    const int k_tok = ri + 8 * (mi & 1), k_hoff = 8 * (mi >> 1);
    const int v_tok = ri + 8 * (mi >> 1), v_hoff = 8 * (mi & 1);

    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kKSteps; kk += 2) {
        uint32_t a0[4], a1[4];
        ldsm_x4(a0, kt + tile_chunk_offset<H>(k_tok, 16 * kk + k_hoff, tok_major));
        ldsm_x4(a1, kt + tile_chunk_offset<H>(k_tok, 16 * kk + 16 + k_hoff, tok_major));
        mma_bf16_16816(sa, a0, qf[kk][0], qf[kk][1]);
        mma_bf16_16816(sb, a1, qf[kk + 1][0], qf[kk + 1][1]);
    }
    const int t0 = lane >> 2, t1 = t0 + 8;
    const float x0 = t0 < va ? (sa[0] + sb[0]) * sl2 : -INFINITY;
    const float x1 = t0 < vb ? (sa[1] + sb[1]) * sl2 : -INFINITY;
    const float x2 = t1 < va ? (sa[2] + sb[2]) * sl2 : -INFINITY;
    const float x3 = t1 < vb ? (sa[3] + sb[3]) * sl2 : -INFINITY;
    float mA = fmaxf(x0, x2), mB = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xFFFFFFFFu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xFFFFFFFFu, mB, off));
    }
    const bool needA = mA > a.m[0] + kRescaleThreshold;
    const bool needB = mB > a.m[1] + kRescaleThreshold;
    if (__any_sync(0xFFFFFFFFu, needA || needB)) {
        const float alphaA = needA ? exp2_sfu(a.m[0] - mA) : 1.f;
        const float alphaB = needB ? exp2_sfu(a.m[1] - mB) : 1.f;
        if (needA) a.m[0] = mA;
        if (needB) a.m[1] = mB;
        a.l[0] *= alphaA;
        a.l[1] *= alphaB;
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) {
            a.o[mt][0] *= alphaA;
            a.o[mt][1] *= alphaB;
            a.o[mt][2] *= alphaA;
            a.o[mt][3] *= alphaB;
        }
    }
    const float baseA = a.m[0] == -INFINITY ? 0.f : a.m[0];
    const float baseB = a.m[1] == -INFINITY ? 0.f : a.m[1];
    const uint32_t p01 = pack_bf16x2(exp2_sfu(x0 - baseA), exp2_sfu(x1 - baseB));
    const uint32_t p23 = pack_bf16x2(exp2_sfu(x2 - baseA), exp2_sfu(x3 - baseB));
    a.l[0] += bf16x2_lo(p01) + bf16x2_lo(p23);
    a.l[1] += bf16x2_hi(p01) + bf16x2_hi(p23);
    const uint32_t pb0 = movmatrix_trans(p01);
    const uint32_t pb1 = movmatrix_trans(p23);

    const bool partial = valid < kBlockSize;
    const int tc = (lane & 3) * 2;
#pragma unroll
    for (int mt = 0; mt < kKSteps; ++mt) {
        uint32_t av[4];
        ldsm_x4_trans(av, vt + tile_chunk_offset<H>(v_tok, 16 * mt + v_hoff, tok_major));
        if (partial) {
            const uint32_t lo0 = tc < valid ? 0x0000FFFFu : 0u;
            const uint32_t hi0 = tc + 1 < valid ? 0xFFFF0000u : 0u;
            const uint32_t lo1 = tc + 8 < valid ? 0x0000FFFFu : 0u;
            const uint32_t hi1 = tc + 9 < valid ? 0xFFFF0000u : 0u;
            av[0] &= lo0 | hi0;
            av[1] &= lo0 | hi0;
            av[2] &= lo1 | hi1;
            av[3] &= lo1 | hi1;
        }
        mma_bf16_16816(a.o[mt], av, pb0, pb1);
    }
}

template <int H>
__device__ __forceinline__ void attn_cols_body(const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                               const ColsParams &p)
{
    constexpr int S = kStages;
    using L = AttnLayout<H, S>;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - raw_u32);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    ColsWork wk;
    if (!cols_work(p, blockIdx.x, wk)) return;
    const int nblk = wk.blk_end - wk.blk_begin;
    // Split multi-token units merged in this launch: a sequence held by one partition is written
    // out directly, one held by several leaves partials for the last of its CTAs to merge.
    const bool merge_multi = p.counters != nullptr && wk.mode == kModeMulti && wk.slot >= 0;
    const int nparts = merge_multi ? cols_nparts(p, wk) : 0;
    const bool direct = wk.slot < 0 || (merge_multi && nparts <= 1);
    multi_slots_below_zero(p, wk);
    if (nblk <= 0) {
        // several new tokens, empty sequence (one pass, or partition 0 when merged here): 0, -inf
        if (wk.slot < 0 || (merge_multi && wk.slot == 0 && nparts == 0)) {
            for (int idx = threadIdx.x; idx < wk.ncols * H; idx += kAttnThreads) {
                const int j = idx / H, h = idx - j * H;
                int64_t row;
                int vis;
                col_of(p, wk, j, row, vis);
                p.out[row * H + h] = __float2bfloat16_rn(0.0f);
                if (h == 0 && p.lse_out) p.lse_out[row] = -INFINITY;
            }
        }
        return;
    }
    const int ng = wk.ncols <= 8 ? 1 : (wk.ncols <= 16 ? 2 : 4);  // column groups of 8
    const int R = kConsumerWarps / ng;                            // tile streams

    const uint32_t bar_full = base_u32 + L::kBarOffset;
    const uint32_t bar_empty = bar_full + 8 * S;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(base + L::kMiscOffset);
    volatile int *abort_flag = slot_ok + S;
    volatile int *issued_count = abort_flag + 1;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int q = 0; q < kProducers; ++q) issued_count[q] = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, ng);  // every consumer warp of the tile's stream
        }
        fence_barrier_init();
    }
    __syncthreads();

    WarpAcc<H> acc;
    if (warp >= kConsumerWarps) {
        const int pw = warp - kConsumerWarps;
        if (lane == 0 && pw == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int32_t *tbl = p.block_tables + (size_t)wk.table_row * p.max_nb + wk.blk_begin;
        const int64_t issued = run_producer<kProducers>(
            pw, lane, nblk, [&](int64_t i) { return __ldg(tbl + i); }, p.num_blocks, p.err_flag,
            [&](int64_t i, int bid, bool ok, float2) {
                if (PKV_TILE_WITHHELD(p, i)) return true;  // test builds: never loaded, never signalled
                return produce_tile<H, S>(i, wk.kvh, bid, ok, base_u32, bar_full, bar_empty, slot_ok,
                                          abort_flag, &tm_k, &tm_v, p.tok_major, p.err_flag, p.wait_ns);
            },
            NoAux(), false, 0, [&](int64_t i, int bid, bool ok) { append_multi_rows<H>(p, wk, i, bid, ok, lane); });
        if (lane == 0) issued_count[pw] = (int)issued;
    } else {
        const int cg = warp % ng, r = warp / ng;
        uint32_t qf[H / 16][2];
        {
            const int jq = kColsPerWarp * cg + (lane >> 2);
            const uint16_t *qrow = nullptr;
            if (jq < wk.ncols) {
                int64_t row;
                int vis;
                col_of(p, wk, jq, row, vis);
                qrow = p.q + row * H;
            }
            load_q_frags_row<H>(qf, qrow, lane);
        }
        int visA = 0, visB = 0;  // tokens visible to the lane's S columns
        {
            const int jA = kColsPerWarp * cg + 2 * (lane & 3);
            int64_t row;
            if (jA < wk.ncols) col_of(p, wk, jA, row, visA);
            if (jA + 1 < wk.ncols) col_of(p, wk, jA + 1, row, visB);
        }
        acc_reset<H>(acc);
        for (int i = r; i < nblk; i += R) {
            const int s = i % S;
            // lanes may differ at the deadline: the warp agrees before its collective MMA work
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_full + 8 * s, (i / S) & 1, abort_flag, p.wait_ns))) {
                if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            if (slot_ok[s]) {
                const int tok0 = (wk.blk_begin + i) * kBlockSize;
                const int valid = min(kBlockSize, wk.data_end - tok0);
                const int va = max(0, min(visA - tok0, valid));
                const int vb = max(0, min(visB - tok0, valid));
                const uint32_t kt = base_u32 + s * L::kStageBytes;
                tile_update_cols<H>(acc, qf, kt, kt + L::kTileBytes, va, vb, valid, p.scale_log2,
                                    p.tok_major, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }
    }

    __syncthreads();
    const bool aborted = *abort_flag != 0;
    const bool merge_here = merge_multi && nparts > 1;
    if (aborted) {
        if (warp >= kConsumerWarps && lane == 0)
            drain_ring<S, kProducers>(bar_full, warp - kConsumerWarps, issued_count[warp - kConsumerWarps]);
        __syncthreads();
        // the sequence's other partitions still count on this one: it leaves a void partial
        if (!merge_here) return;
    }

    // merge: column j (group j / 8, row j % 8) was seen by warps j/8 + ng * r, r < R
    float *mo = reinterpret_cast<float *>(base);
    float *mm = mo + kConsumerWarps * 8 * H;
    float *ml = mm + kConsumerWarps * 8;
    if (!aborted) {
        if (warp < kConsumerWarps) deposit<H>(acc, mo, mm, ml, warp, lane);
        __syncthreads();
    }
    for (int idx = threadIdx.x; idx < wk.ncols * H; idx += kAttnThreads) {
        const int j = idx / H, h = idx - j * H;
        float val = __int_as_float(0x7FC00000), lse = __int_as_float(0x7FC00000);  // NaN: void
        if (!aborted) {
            const int cg = j / kColsPerWarp, g8 = j - cg * kColsPerWarp;
            float M = -INFINITY;
            for (int rr = 0; rr < R; ++rr) M = fmaxf(M, mm[(cg + ng * rr) * 8 + g8]);
            float accv = 0.f, lsum = 0.f;
            if (M != -INFINITY) {
                for (int rr = 0; rr < R; ++rr) {
                    const int w = cg + ng * rr;
                    const float sc = exp2_sfu(mm[w * 8 + g8] - M);
                    lsum += sc * ml[w * 8 + g8];
                    accv += sc * mo[(w * 8 + g8) * H + h];
                }
            }
            val = M != -INFINITY ? accv / lsum : 0.f;
            lse = M != -INFINITY ? (M + log2f(lsum)) * kLn2 : -INFINITY;
        }
        int64_t row;
        int vis;
        col_of(p, wk, j, row, vis);
        if (direct) {
            p.out[row * H + h] = __float2bfloat16_rn(val);
            if (h == 0 && p.lse_out) p.lse_out[row] = lse;
        } else {
            const int64_t rp = row * p.max_parts + wk.slot;
            p.part_out[rp * H + h] = val;
            if (h == 0) p.part_lse[rp] = lse;
        }
    }
    if (merge_here) cols_merge_chunk<H>(p, wk, nparts, reinterpret_cast<float *>(base), kAttnThreads);
}

template <int H>
__global__ void __launch_bounds__(kAttnThreads, PKV_CTAS_PER_SM)
attn_cols_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const ColsParams p)
{
    // the merge launched behind this grid (programmatic serialization) may be scheduled once every
    // CTA of it runs; it waits for this grid's completion before it reads the partials
    pdl_launch_dependents();
    attn_cols_body<H>(tm_k, tm_v, p);
    // the suffix pass launched behind the tcgen05 prefix pass: its last CTA (scheduled last, so its
    // wait holds no slot another CTA of this grid needs) waits for that grid, so this one completes
    // only after it and the merge launched next reads both passes' partials
    if (p.pdl_wait && blockIdx.x == gridDim.x - 1) pdl_wait_primary();
}

// Merge of the prefix pass and the suffix pass of one (sequence, query head): slots
// [0, ceil(pnb / prefix PB)) hold the shared prefix, the next ceil((nb - pnb) / PB) the
// sequence's own blocks; one warp computes the log-sum-exp weights, every thread one element.
// Which slots hold data takes dependent reads (the length, the group, its prefix), so the row's
// partial lse of every slot and each thread's partial values of the first kCascadePrefetch slots
// are loaded before them, independently (the workspace holds max_parts slots a row; slots that
// hold no data are read but never used).
constexpr int kCascadePrefetch = 8;

__global__ void cascade_merge_kernel(const ColsParams p, __nv_bfloat16 *__restrict__ out,
                                     float *__restrict__ lse_out)
{
    extern __shared__ float wts[];  // [max_parts]
    __shared__ float row_lse;
    pdl_wait_primary();  // launched behind the attention launch (programmatic serialization)
    const int n = blockIdx.x, b = blockIdx.y, h = threadIdx.x;
    const int H = blockDim.x;
    const int64_t row = (int64_t)b * p.N + n;
    const float *po = p.part_out + row * p.max_parts * H + h;
    float v[kCascadePrefetch];
#pragma unroll
    for (int q = 0; q < kCascadePrefetch; ++q) v[q] = q < p.max_parts ? __ldcg(po + (size_t)q * H) : 0.f;
    for (int q = h; q < p.max_parts; q += H) wts[q] = __ldcg(p.part_lse + row * p.max_parts + q);
    const int ctx = p.context_lens[b];
    const int g = group_of(p, b);
    const int pnb = g >= 0 ? prefix_blocks_of(p, g) : 0;
    const bool ok = ctx >= 0 && ctx <= p.max_nb * kBlockSize && pnb * kBlockSize <= ctx;
    const int nb = ok ? (ctx + kBlockSize - 1) / kBlockSize : 0;
    const int np = ok ? (pnb + p.prefix_part_blocks - 1) / p.prefix_part_blocks +
                            (nb - pnb + p.part_blocks - 1) / p.part_blocks
                      : 0;
    __syncthreads();
    if (h < 32) {
        const float L = lse_merge_weights<true>(wts, np, wts, h);
        if (h == 0) row_lse = L;
    }
    __syncthreads();
    // sum_q w_q o_q in slot order (lse_merge_value's arithmetic), the first slots from registers
    float val = 0.f;
#pragma unroll
    for (int q = 0; q < kCascadePrefetch; ++q)
        if (q < np) val += wts[q] * v[q];
    for (int q = kCascadePrefetch; q < np; ++q) val += wts[q] * __ldcg(po + (size_t)q * H);
    out[row * H + h] = __float2bfloat16_rn(val);
    if (h == 0 && lse_out) lse_out[row] = row_lse;
}

template <typename Kern>
static cudaError_t ensure_cols_smem(Kern kern, int smem, int *cached)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cached[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) cached[dev] = 1;
    return e;
}

template <int H>
static cudaError_t launch_cols_t(const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                                 int64_t grid, cudaStream_t stream, bool pdl)
{
    constexpr int smem = AttnLayout<H>::kAlloc;
    static int cached[64] = {};
    cudaError_t e = ensure_cols_smem(attn_cols_kernel<H>, smem, cached);
    if (e != cudaSuccess) return e;
    return launch_kernel(attn_cols_kernel<H>, dim3((unsigned)grid), dim3(kAttnThreads), smem, stream, pdl, tk, tv, p);
}

cudaError_t launch_attn_cols(int H, const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                             int64_t grid, cudaStream_t stream, bool pdl)
{
    if (grid <= 0) return cudaSuccess;
    if (pdl && !p.pdl_wait) return cudaErrorInvalidValue;
    if (H == 64) return launch_cols_t<64>(tk, tv, p, grid, stream, pdl);
    if (H == 128) return launch_cols_t<128>(tk, tv, p, grid, stream, pdl);
    return cudaErrorInvalidValue;
}

cudaError_t launch_cascade_merge(const ColsParams &p, int H, __nv_bfloat16 *out, float *lse_out,
                                 cudaStream_t stream)
{
    if (p.B <= 0) return cudaSuccess;
    // behind the attention launch that wrote the partials (whose completion implies the prefix
    // pass's when the two passes are two launches)
    return launch_kernel(cascade_merge_kernel, dim3(p.N, p.B), dim3(H), (size_t)p.max_parts * sizeof(float),
                         stream, true, p, out, lse_out);
}

}  // namespace pkv
