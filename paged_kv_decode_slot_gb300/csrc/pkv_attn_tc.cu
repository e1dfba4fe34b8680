// pkv_attn_tc.cu - column-parallel decode attention on the 5th-generation tensor cores (tcgen05).
//
// Same work as attn_cols_kernel (one CTA: up to 32 query rows of one KV head over one list of
// logical blocks -- several new tokens per sequence, "Week 11. Inference", Step 3), but with 16+
// query rows per loaded K/V tile the contraction is dense enough for the tensor cores proper:
//     S[rows x 64 tok]  = Q[rows x H] . K_group^T              (tcgen05.mma, accumulator in TMEM)
//     P                 = exp2(S * scale*log2e - m)            (one thread per query row)
//     O[rows x H]      += P[rows x 64 tok] . V_group[64 x H]   (tcgen05.mma, P read from TMEM)
// computed over groups of four 16-token tiles with the online (running max / running sum) softmax
// ("Optimización de la inferencia", "Construye el mismo", Step 2), so every K/V byte fetched from
// HBM serves all rows of the CTA and no warp spends issue slots on the contraction itself.
//
// Two forms, by the number RW of row warps: 32 query rows a CTA (RW = 1, 5 warps, a 12-stage ring)
// and 128 (RW = 4, 8 warps, an 8-stage ring, so that two CTAs still fit an SM): the MMA has
// M = 128 rows whatever the form, and a group costs the same MMA instructions for 32 rows as for
// 128, so groups of rows wider than 32 (a shared prefix read for every member of its group, or many
// new tokens) take the 128-row form.  CTA = RW + 4 warps:
//  * warps RW+2, RW+3: TMA producers, the same full/empty mbarrier ring as the other attention
//    kernels (K and V tiles, 128-byte swizzled -- the layout the MMA reads directly).  The
//    two 64-element halves of a K tile land in two separate regions, so the K tiles of four
//    consecutive stages form one 64-token operand: one MMA per 16-element step covers a whole
//    group (a tcgen05.mma costs its issuing thread about the same time for N = 16 as for N = 256,
//    so the number of instructions, not their size, sets the pace);
//  * warp RW: allocates 256 TMEM columns (O: 128, two S/P buffers of 64) and issues, from one lane,
//    QK^T of group g (8 MMAs, N = 64) as soon as its tiles landed (and PV(g-2) freed the S buffer);
//  * warp RW+1: issues PV of group g (one MMA per tile) from one lane as soon as every row warp
//    wrote its part of P, and
//    one commit that releases the group's four stages.  Two issuing threads: an MMA costs its
//    issuer a fixed latency, and a PV no longer waits behind the next group's loads;
//  * warps 0 .. RW-1: one thread per query row (warp w: TMEM lanes 32w .. 32w+31): reads the row's
//    64 logits, masks tokens the row may not see, keeps the lazily rescaled running max and sum,
//    writes P (bf16) over the logits, and at the end reads O, normalises it and writes out / lse
//    (or the partials).
// The MMA has M = 128 rows; with RW = 1, rows 32..127 are padding whose results are never read.
#include "pkv_cols.cuh"
#include "pkv_tcgen05.cuh"

namespace pkv {

constexpr int kTcGroupTiles = 4;   // tiles per softmax step (64 tokens)
constexpr int kTcM = 128;          // MMA rows
constexpr int kTcProducers = 2;
constexpr uint32_t kTcCols = 256;  // TMEM columns: O [0, H), S/P buffers at H and H + 64

// Ring depths of the two forms (stages of one K and one V tile; a multiple of 4): 12 and 8 keep
// two CTAs per SM, which the tensor memory allows (256 columns each).
#ifndef PKV_TC_STAGES_32
#define PKV_TC_STAGES_32 12
#endif
#ifndef PKV_TC_STAGES_128
#define PKV_TC_STAGES_128 8
#endif

// RW row warps (32 rows each), then the QK^T warp, the PV warp and the two producers.
template <int RW>
struct TcRoles {
    static_assert(RW == 1 || RW == 4, "32 or 128 query rows a CTA");
    static constexpr int kRows = 32 * RW;
    static constexpr int kStages = RW == 1 ? PKV_TC_STAGES_32 : PKV_TC_STAGES_128;
    static constexpr int kQkWarp = RW, kPvWarp = RW + 1, kProd0 = RW + 2;
    static constexpr int kThreads = (RW + 4) * 32;
    static_assert(kStages % kTcProducers == 0, "pipeline depth must be a multiple of the producer warps");
    static_assert(kStages >= 2 * kTcGroupTiles, "two groups of tiles must fit in the ring");
};

template <int H, int RW>
struct TcLayout {
    static_assert(H == 128, "the tensor-core column kernel is built for H = 128");
    static constexpr int kStages = TcRoles<RW>::kStages;
    // Q: the CTA's rows as the K-major A operand, two 64-element halves of rows / 8 atoms each
    static constexpr int kQOffset = 0;
    static constexpr int kQHalfBytes = (TcRoles<RW>::kRows / 8) * 1024;
    // K: two regions (one per 64-element half) of [stage][16 tokens][128 bytes]
    static constexpr int kKHalfTile = kBlockSize * 128;
    static constexpr int kKOffset = kQOffset + (H / 64) * kQHalfBytes;
    static constexpr int kKRegion = kStages * kKHalfTile;
    // V: [stage][half][16 tokens][128 bytes]
    static constexpr int kVTile = kBlockSize * H * 2;
    static constexpr int kVOffset = kKOffset + (H / 64) * kKRegion;
    static constexpr int kStageBytes = 2 * kVTile;  // bytes one stage receives (K and V)
    static constexpr int kRingOffset = kKOffset;
    // barriers: full[S], group_free[S / 4], s_full[2], p_ready[2], o_done, fin
    static constexpr int kGroupSlots = kStages / kTcGroupTiles;
    static constexpr int kBarOffset = kVOffset + kStages * kVTile;
    static constexpr int kMiscOffset = kBarOffset + (kStages + kGroupSlots + 6) * 8;  // slot_ok[S], abort, issued[P], tmem
    static constexpr int kBytes = kMiscOffset + (kStages + 2 + kTcProducers) * 4;
    static constexpr int kAlloc = kBytes + 1024;
    // The A descriptor spans M = 128 rows: with 32 rows the padding rows read on into the ring (in
    // bounds).
    static_assert(kRingOffset + (H / 64 - 1) * kQHalfBytes + (kTcM / 8) * 1024 <= kBarOffset,
                  "the padding rows of the Q operand must stay inside the CTA's shared memory");
    static_assert(kKOffset % 1024 == 0 && kVOffset % 1024 == 0 && kKHalfTile % 1024 == 0 && kVTile % 1024 == 0,
                  "128B-swizzle atoms need 1024-byte alignment");
    static_assert(kStages % kTcGroupTiles == 0, "a group's K tiles must not wrap around the ring");
    static_assert(kAlloc + 1024 <= 228 * 1024 && 3 * (kAlloc + 1024) > 228 * 1024,
                  "at most two CTAs per SM (2 x 256 TMEM columns fill the SM's 512)");
};

// Producer side of one tile: wait until the previous group in the tile's group slot is released
// (one commit after that group's PV frees its four stages), then three TMA loads (the two K halves
// into their regions, the V tile) completing on the stage's full barrier; an out-of-range block
// id marks the stage skipped.  Returns false when the wait expired.
template <int H, int RW>
__device__ __forceinline__ bool produce_tile_tc(int64_t i, int kvh, int bid, bool ok, uint32_t kreg, uint32_t vreg,
                                                uint32_t bar_full, uint32_t bar_free, volatile int *slot_ok,
                                                volatile int *abort_flag, const CUtensorMap *tm_kh,
                                                const CUtensorMap *tm_v, int32_t *err_flag, uint64_t wait_ns)
{
    using L = TcLayout<H, RW>;
    constexpr int S = L::kStages;
    const int s = (int)(i % S);
    const int slot = (int)((i / kTcGroupTiles) % L::kGroupSlots);
    if (i >= S && !mbar_wait_bounded(bar_free + 8 * slot, (uint32_t)(((i / S) & 1) ^ 1), abort_flag, wait_ns)) {
        if (!*abort_flag) set_flag(err_flag, PKV_FLAG_TIMEOUT);
        *abort_flag = 1;
        return false;
    }
    const uint32_t bar = bar_full + 8 * s;
    if (ok) {
        slot_ok[s] = 1;
        mbar_arrive_expect_tx(bar, L::kStageBytes);
#pragma unroll
        for (int half = 0; half < H / 64; ++half)
            tma_load_5d(kreg + half * L::kKRegion + s * L::kKHalfTile, tm_kh, bar, 0, 0, half, kvh, bid);
        tma_load_5d(vreg + s * L::kVTile, tm_v, bar, 0, 0, 0, kvh, bid);
    } else {
        slot_ok[s] = 0;  // out-of-range block id: the tile is skipped
        mbar_arrive(bar);
    }
    return true;
}

template <int H, int RW>
__global__ void __launch_bounds__(TcRoles<RW>::kThreads, 2)
attn_cols_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const ColsParams p)
{
    using L = TcLayout<H, RW>;
    using R = TcRoles<RW>;
    constexpr int S = L::kStages;
    constexpr int kTcThreads = R::kThreads;
    constexpr int GT = kTcGroupTiles;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - raw_u32);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // a suffix pass launched behind this grid (programmatic serialization) may start as soon as
    // every CTA of this one is running: the two passes share no data until the merge
    pdl_launch_dependents();

    ColsWork wk;
    if (!cols_work<R::kRows>(p, blockIdx.x, wk)) return;
    const int nblk = wk.blk_end - wk.blk_begin;
    multi_slots_below_zero(p, wk);
    if (nblk <= 0) {
        // several new tokens, one pass, empty sequence: 0 and -inf
        if (wk.slot < 0) {
            for (int idx = threadIdx.x; idx < wk.ncols * H; idx += kTcThreads) {
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
    const int ngroups = (nblk + GT - 1) / GT;

    const uint32_t q_u32 = base_u32 + L::kQOffset;
    const uint32_t kreg = base_u32 + L::kKOffset;  // K halves: kreg, kreg + kKRegion
    const uint32_t vreg = base_u32 + L::kVOffset;
    const uint32_t bar_full = base_u32 + L::kBarOffset;
    const uint32_t bar_free = bar_full + 8 * S;                    // [slots]: a group's PV done
    const uint32_t bar_sfull = bar_free + 8 * L::kGroupSlots;      // [2]: QK^T of a group done
    const uint32_t bar_pready = bar_sfull + 16;                    // [2]: P of a group written to TMEM
    const uint32_t bar_odone = bar_pready + 16;                    // every MMA done
    const uint32_t bar_fin = bar_odone + 8;        // drain after an expired wait
    volatile int *slot_ok = reinterpret_cast<volatile int *>(base + L::kMiscOffset);
    volatile int *abort_flag = slot_ok + S;
    volatile int *issued_count = abort_flag + 1;  // [kTcProducers]
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(issued_count + kTcProducers);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int q = 0; q < kTcProducers; ++q) issued_count[q] = 0;
        for (int st = 0; st < S; ++st) mbar_init(bar_full + 8 * st, 1);
        for (int q = 0; q < L::kGroupSlots; ++q) mbar_init(bar_free + 8 * q, 1);
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sfull + 8, 1);
        mbar_init(bar_pready, RW);  // every row warp writes its rows of P
        mbar_init(bar_pready + 8, RW);
        mbar_init(bar_odone, 1);
        mbar_init(bar_fin, 2);  // one commit from each MMA-issuing warp
        fence_barrier_init();
    }
    __syncthreads();  // the barriers are ready: the producers start loading at once

    // Meanwhile the row warps and the two MMA warps put the CTA's q rows into the K-major,
    // 128B-swizzled A operand (rows past ncols are zero) and the QK^T warp allocates the tensor
    // memory; they meet at a named barrier.
    uint32_t tm_o = 0, tm_s = 0;  // O at tm_o (lane 0, first allocated column), S/P at tm_s, tm_s + 64
    constexpr int kQThreads = (RW + 2) * 32;
    if (warp < RW + 2) {
        // all of a thread's loads first (one round trip), then the stores
        constexpr int kUnits = R::kRows * (H / 8), kPer = (kUnits + kQThreads - 1) / kQThreads;
        uint4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + kQThreads * k;
            const int r = idx / (H / 8), u = idx - r * (H / 8);  // row, 16-byte unit of the row
            v[k] = make_uint4(0u, 0u, 0u, 0u);
            if (idx < kUnits && r < wk.ncols) {
                int64_t row;
                int vis;
                col_of(p, wk, r, row, vis);
                const uint32_t *src = reinterpret_cast<const uint32_t *>(p.q + row * H + 8 * u);
                v[k] = make_uint4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
            }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = threadIdx.x + kQThreads * k;
            if (idx < kUnits) {
                const int r = idx / (H / 8), u = idx - r * (H / 8);
                const int half = u >> 3, cu = u & 7;
                st_shared_v4(q_u32 + half * L::kQHalfBytes + (r >> 3) * 1024 + (r & 7) * 128 + ((cu ^ (r & 7)) << 4),
                             v[k]);
            }
        }
        fence_proxy_async_shared();
        if (warp == R::kQkWarp) {
            tmem_alloc(smem_u32((const void *)tmem_slot), kTcCols);
            tmem_relinquish();
        }
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"n"(kQThreads) : "memory");  // row warps and MMA warps
        tc_fence_after();
        tm_o = *tmem_slot;
        tm_s = tm_o + H;
    }

    if (warp >= R::kProd0) {
        // ------------------------------ producer warps ------------------------------
        const int pw = warp - R::kProd0;
        if (lane == 0 && pw == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int32_t *tbl = p.block_tables + (size_t)wk.table_row * p.max_nb + wk.blk_begin;
        const int64_t issued = run_producer<kTcProducers>(
            pw, lane, nblk, [&](int64_t i) { return __ldg(tbl + i); }, p.num_blocks, p.err_flag,
            [&](int64_t i, int bid, bool ok, float2) {
                if (PKV_TILE_WITHHELD(p, i)) return true;  // test builds: never loaded, never signalled
                return produce_tile_tc<H, RW>(i, wk.kvh, bid, ok, kreg, vreg, bar_full, bar_free, slot_ok, abort_flag,
                                          &tm_k, &tm_v, p.err_flag, p.wait_ns);
            },
            NoAux(), false, 0, [&](int64_t i, int bid, bool ok) { append_multi_rows<H>(p, wk, i, bid, ok, lane); });
        if (lane == 0) issued_count[pw] = (int)issued;
    } else if (warp == R::kQkWarp) {
        // ----------------------- QK^T warp (lane 0 issues) -----------------------
        bool ok = true;
        for (int g = 0; g < ngroups && ok; ++g) {
            const int i0 = g * GT, gt = min(GT, nblk - i0);
            for (int j = 0; j < gt && ok; ++j) {
                const int i = i0 + j;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_full + 8 * (i % S), (uint32_t)((i / S) & 1),
                                                               abort_flag, p.wait_ns));
            }
            // S buffer g % 2 holds P(g - 2) until PV(g - 2) has read it (the release of its slot)
            if (ok && g >= 2) {
                const int gq = g - 2;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_free + 8 * (gq % L::kGroupSlots),
                                                               (uint32_t)((gq / L::kGroupSlots) & 1), abort_flag,
                                                               p.wait_ns));
            }
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                // S[:, 0 .. 16 gt) = Q . K^T over the group's gt tiles (stages i0 % S ..,
                // contiguous in each K region); a skipped tile's stale rows are masked later
                const uint32_t sb = tm_s + 64 * (g & 1);
                const uint32_t idesc = idesc_bf16_f32(kTcM, kBlockSize * gt, 0, 0);
                const uint32_t kt = kreg + (i0 % S) * L::kKHalfTile;
#pragma unroll
                for (int kk = 0; kk < H / 16; ++kk) {
                    const uint32_t koff = (kk & 3) * 32;
                    tc_mma_ss(sb, smem_desc_sw128(q_u32 + (kk >> 2) * L::kQHalfBytes + koff, 16, 1024),
                              smem_desc_sw128(kt + (kk >> 2) * L::kKRegion + koff, 16, 1024), idesc, kk > 0);
                }
                tc_commit(bar_sfull + 8 * (g & 1));
            }
            __syncwarp();
        }
        if (!ok) {
            if (lane == 0 && !*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == R::kPvWarp) {
        // ------------------------- PV warp (lane 0 issues) -------------------------
        constexpr uint32_t kIdPV = idesc_bf16_f32(kTcM, H, 0, 1);  // O: N = H, V MN-major
        // The tile holding the end of the data may carry poison in its later rows: their V rows
        // are zeroed before PV reads them (their weights are zero, but 0 x NaN is NaN).
        const int tail_valid = wk.data_end % kBlockSize;
        const int tail_tile = tail_valid ? (wk.data_end - 1) / kBlockSize - wk.blk_begin : -1;
        bool ok = true;
        uint32_t o_acc = 0;
        for (int g = 0; g < ngroups && ok; ++g) {
            const int i0 = g * GT, gt = min(GT, nblk - i0);
            ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_pready + 8 * (g & 1), (uint32_t)((g >> 1) & 1),
                                                           abort_flag, p.wait_ns));
            if (!ok) break;
            if (tail_tile >= i0 && tail_tile < i0 + gt && slot_ok[tail_tile % S]) {
                const uint32_t vt = vreg + (tail_tile % S) * L::kVTile;
                const int nz = (kBlockSize - tail_valid) * (H / 8);  // 16-byte units of the rows
                for (int idx = lane; idx < nz; idx += 32) {
                    const int r = tail_valid + idx / (H / 8), u = idx % (H / 8);
                    st_shared_v4(vt + (u >> 3) * (kBlockSize * 128) + (r >> 3) * 1024 + (r & 7) * 128 + ((u & 7) << 4),
                                 make_uint4(0u, 0u, 0u, 0u));
                }
                fence_proxy_async_shared();
            }
            __syncwarp();
            tc_fence_after();
            if (lane == 0) {
                const uint32_t pb = tm_s + 64 * (g & 1);
                for (int j = 0; j < gt; ++j) {
                    const int s = (i0 + j) % S;
                    if (!slot_ok[s]) continue;
                    tc_mma_ts(tm_o, pb + (kBlockSize / 2) * j,
                              smem_desc_sw128(vreg + s * L::kVTile, kBlockSize * 128, 1024), kIdPV, o_acc);
                    o_acc = 1;
                }
                tc_commit(bar_free + 8 * (g % L::kGroupSlots));  // PV(g) done: its stages are free
            }
            __syncwarp();
        }
        if (ok) {
            if (lane == 0) tc_commit(bar_odone);  // after the last PV: every MMA has completed
        } else {
            if (lane == 0 && !*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // --------------------- row warps: one thread per query row ---------------------
        const int r = 32 * warp + lane;  // TMEM lane r = MMA row r = query row r of the CTA
        const uint32_t lq = (uint32_t)(32 * warp) << 16;  // the warp's TMEM lane quarter
        const bool real = r < wk.ncols;
        int64_t row = 0;
        int vis = 0;
        if (real) col_of(p, wk, r, row, vis);
        const int lim = min(vis, wk.data_end);  // the row counts the tokens [0, lim) of the list
        float m = -INFINITY, l = 0.f;           // running max (log2 units, lazily raised) and sum
        bool ok = true;
        for (int g = 0; g < ngroups && ok; ++g) {
            const int i0 = g * GT, gt = min(GT, nblk - i0);
            // the tiles' full barriers (already complete) order the producers' slot_ok writes
            for (int j = 0; j < gt && ok; ++j) {
                const int i = i0 + j;
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_full + 8 * (i % S), (uint32_t)((i / S) & 1),
                                                               abort_flag, p.wait_ns));
            }
            if (ok)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_sfull + 8 * (g & 1), (uint32_t)((g >> 1) & 1),
                                                               abort_flag, p.wait_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t sb = tm_s + 64 * (g & 1);
            uint32_t sr[GT][16];
#pragma unroll
            for (int t = 0; t < GT; ++t) tmem_ld16(lq + sb + 16 * t, sr[t]);
            tmem_ld_wait();
            const int tok0 = (wk.blk_begin + i0) * kBlockSize;
            float x[GT * 16];
            float mx = -INFINITY;
#pragma unroll
            for (int t = 0; t < GT; ++t) {
                const bool tile_ok = t < gt && slot_ok[(i0 + t) % S] != 0;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float v = __uint_as_float(sr[t][c]) * p.scale_log2;
                    x[16 * t + c] = (tile_ok && tok0 + 16 * t + c < lim) ? v : -INFINITY;
                    mx = fmaxf(mx, x[16 * t + c]);
                }
            }
            const bool need = mx > m + kRescaleThreshold;
            if (__any_sync(0xFFFFFFFFu, need)) {
                const float alpha = need ? exp2_sfu(m - mx) : 1.f;
                if (need) m = mx;
                l *= alpha;
                if (g > 0) {
                    // O holds the groups before g: rescale it once their PV has completed (the
                    // release of group g-1's slot)
                    const int gq = g - 1;
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_free + 8 * (gq % L::kGroupSlots),
                                                                   (uint32_t)((gq / L::kGroupSlots) & 1), abort_flag,
                                                                   p.wait_ns));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < H; c += 16) {
                        uint32_t o[16];
                        tmem_ld16(lq + tm_o + c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st16(lq + tm_o + c, o);
                    }
                    tmem_st_wait();
                }
            }
            // A row that has seen no key keeps m = -inf and weights exp2(-inf - 0) = 0.
            const float bm = m == -INFINITY ? 0.f : m;
            uint32_t pk[2][16];
#pragma unroll
            for (int c = 0; c < GT * 8; ++c) {
                const uint32_t v = pack_bf16x2(exp2_sfu(x[2 * c] - bm), exp2_sfu(x[2 * c + 1] - bm));
                pk[c >> 4][c & 15] = v;
                l += bf16x2_lo(v) + bf16x2_hi(v);  // the sum of the weights PV uses
            }
            tmem_st16(lq + sb, pk[0]);
            tmem_st16(lq + sb + 16, pk[1]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pready + 8 * (g & 1));
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_odone, 0u, abort_flag, p.wait_ns));
        if (!ok) {
            if (lane == 0 && !*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
            *abort_flag = 1;
        } else {
            tc_fence_after();
            const bool seen = m != -INFINITY;
            const float inv = seen ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 0; c < H; c += 16) {
                uint32_t o[16];
                tmem_ld16(lq + tm_o + c, o);
                tmem_ld_wait();
                if (!real) continue;
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = seen ? __uint_as_float(o[k]) * inv : 0.f;
                if (wk.slot < 0) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
                    // out rows are H bf16 = 256 bytes; 4-byte stores (out is only 4-byte aligned)
                    uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + row * H + c);
#pragma unroll
                    for (int k = 0; k < 8; ++k) dst[k] = w[k];
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(p.part_out + (row * p.max_parts + wk.slot) * H + c);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
            }
            if (real) {
                const float lse = seen ? (m + log2f(l)) * kLn2 : -INFINITY;
                if (wk.slot < 0) {
                    if (p.lse_out) p.lse_out[row] = lse;
                } else {
                    p.part_lse[row * p.max_parts + wk.slot] = lse;
                }
            }
        }
    }

    // ------------------------------------ teardown ------------------------------------
    __syncthreads();
    if (*abort_flag) {
        if (warp >= R::kProd0 && lane == 0)
            drain_ring<S, kTcProducers>(bar_full, warp - R::kProd0, issued_count[warp - R::kProd0]);
        if (warp == R::kQkWarp || warp == R::kPvWarp) {
            // every MMA this CTA issued completes before its TMEM is released
            if (lane == 0) tc_commit(bar_fin);
            __syncwarp();
            mbar_wait_bounded(bar_fin, 0u, nullptr, kDrainLimitNs);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == R::kQkWarp) {
        tc_fence_after();
        tmem_dealloc(tm_o, kTcCols);
    }
}

template <int H, int RW>
static cudaError_t launch_cols_tc_t(const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                                    int64_t grid, cudaStream_t stream)
{
    constexpr int smem = TcLayout<H, RW>::kAlloc;
    static int cached[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!cached[dev]) {
        cudaError_t e =
            cudaFuncSetAttribute(attn_cols_tc_kernel<H, RW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        cached[dev] = 1;
    }
    attn_cols_tc_kernel<H, RW><<<(unsigned)grid, TcRoles<RW>::kThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

bool cols_tc_supported(int H, int tok_major) { return H == 128 && !tok_major; }

cudaError_t launch_attn_cols_tc(int H, const CUtensorMap &tk, const CUtensorMap &tv, const ColsParams &p,
                                int64_t grid, cudaStream_t stream)
{
    if (grid <= 0) return cudaSuccess;
    if (!cols_tc_supported(H, p.tok_major)) return cudaErrorInvalidValue;
    if (p.chunk_rows == 128) return launch_cols_tc_t<128, 4>(tk, tv, p, grid, stream);
    if (p.chunk_rows == 32) return launch_cols_tc_t<128, 1>(tk, tv, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
