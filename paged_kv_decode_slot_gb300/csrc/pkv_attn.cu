// pkv_attn.cu - paged decode attention for sm_103a.
//
// Work is cut into tiles: one tile = one physical block (16 tokens) of one KV head.  A CTA has
// two producer warps and four consumer warps.  The producers walk the CTA's tiles, look each one
// up in the block table, and stream its K and V (16 x H bf16 each) into a ring of shared-memory
// stages with TMA, one mbarrier pair per stage.  The consumer warps take the stages round-robin;
// each keeps an online-softmax state for the whole query group (the G = N/K query heads that share
// the KV head), so every K/V byte fetched from HBM serves all G heads:
//     S^T[16 tok x 8] = K_tile[16 x H] . Q^T[H x 8]        (mma.sync m16n8k16, G padded to 8)
//     P^T            = exp2(S^T * scale*log2e - m)         (fp32, lazily rescaled running max)
//     O^T[H x 8]    += V_tile^T[H x 16] . P^T[16 x 8]      (P^T moved to the B operand with
//                                                          movmatrix; V^T via ldmatrix.trans)
// When a unit (sequence, KV head) ends, the four warps' states are merged in shared memory.
//
// Two ways to cut the work:
//  * attn_kernel<H, false>: one CTA per (KV head, sequence), whole sequence (single pass).
//  * attn_kernel<H, true>:  one CTA per (KV head, sequence, partition), partitions of a fixed
//    number of blocks (FlashDecoding), highest partition first.  A sequence that fits in one
//    partition is written out directly; the partial results of a longer one are merged by the
//    last of its CTAs to finish (a per-unit counter that the merger resets), or -- when the caller
//    asks for the partials themselves -- by lse_merge_kernel.
//
// This fuses the block-table gather with attention ("融合块读取和注意力的内核" and FlashDecoding
// in CS336 Lecture 10's notes) and computes, for one query token, softmax(q K^T * scale) V with
// the maximum subtracted ("Optimización de la inferencia", "Construye el mismo", Step 2), in its
// online (running max / running sum) form; the log-sum-exp merge of disjoint key sets is exact.
#include "pkv_attn_common.cuh"

namespace pkv {

// Fused decode step: the consumer warp that holds a sequence's last block writes the new token's
// K and V (k_new/v_new row of this KV head) into that tile's row ctx-1 in shared memory -- so
// attention sees it in the same pass -- and into its slot of the pools in global memory.  Lanes
// [0, H/8) move the K row, [H/8, H/4) the V row, 16 bytes each.  Each writer then fences its
// shared-memory stores against the TMA that later refills the stage.
template <int H>
__device__ __forceinline__ void append_new_token(const AttnParams &p, int b, int kvh, int ctx, int bid,
                                                 uint32_t kt, uint32_t vt, int lane)
{
    constexpr int kChunks = H / 8;
    if (lane >= 2 * kChunks) return;
    const int tok = (ctx - 1) % kBlockSize;
    const bool is_v = lane >= kChunks;
    const int c = is_v ? lane - kChunks : lane;
    const size_t row = ((size_t)b * p.K + kvh) * H + 8 * c;
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) + row));
    st_shared_v4((is_v ? vt : kt) + tile_chunk_offset<H>(tok, 8 * c, p.tok_major), v);
    uint16_t *dst = static_cast<uint16_t *>(is_v ? p.v_cache_w : p.k_cache_w) +
                    (((size_t)bid * kBlockSize + tok) * p.K + kvh) * H + 8 * c;
    *reinterpret_cast<uint4 *>(dst) = v;
    fence_proxy_async_shared();
}

// The same for an e4m3 cache: the new token's bf16 K/V rows are quantized with the head's scale
// (code = e4m3(x / scale), the division rounded to nearest) while being written.  Lanes
// [0, H/16) handle the K row, [H/16, H/8) the V row, 16 codes each.
template <int H>
__device__ __forceinline__ void append_new_token_fp8(const AttnParams &p, int b, int kvh, int ctx,
                                                     int bid, uint32_t kt, uint32_t vt, float k_sc,
                                                     float v_sc, int lane)
{
    constexpr int kChunks = H / 16;
    if (lane >= 2 * kChunks) return;
    const int tok = (ctx - 1) % kBlockSize;
    const bool is_v = lane >= kChunks;
    const int c = is_v ? lane - kChunks : lane;
    const float sc = is_v ? v_sc : k_sc;  // the scales of the block being written
    const uint4 *src = reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) +
                                                        ((size_t)b * p.K + kvh) * H + 16 * c);
    const uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
    auto q2 = [&](uint32_t pair) -> uint32_t {  // two bf16 -> two e4m3 codes (low first)
        return f32x2_to_e4m3x2(__fdiv_rn(bf16_to_f32((uint16_t)(pair & 0xFFFFu)), sc),
                               __fdiv_rn(bf16_to_f32((uint16_t)(pair >> 16)), sc));
    };
    uint4 v;
    v.x = q2(x0.x) | (q2(x0.y) << 16);
    v.y = q2(x0.z) | (q2(x0.w) << 16);
    v.z = q2(x1.x) | (q2(x1.y) << 16);
    v.w = q2(x1.z) | (q2(x1.w) << 16);
    st_shared_v4((is_v ? vt : kt) + fp8_chunk_offset(tok, c), v);
    uint8_t *dst = reinterpret_cast<uint8_t *>(is_v ? p.v_cache_w : p.k_cache_w) +
                   (((size_t)bid * kBlockSize + tok) * p.K + kvh) * H + 16 * c;
    *reinterpret_cast<uint4 *>(dst) = v;
    fence_proxy_async_shared();
}

// ------------------------ single pass and fixed partitions --------------------------------
// kFp8: the pools hold e4m3 codes with per-KV-head scales (H = 128); the K scale is folded into
// the logit multiplier, the V scale into the final normalisation.
template <int H, bool kSplit, bool kFp8 = false, bool kPairs = false, bool kBScale = false, bool kDeep = false>
__global__ void __launch_bounds__(kAttnThreads, kDeep ? 2 : PKV_CTAS_PER_SM)
attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
            const AttnParams p)
{
    constexpr int S = kFp8 ? kStagesFp8 : (kDeep ? kStagesDeep : kStages);
    using L = AttnLayout<H, S, kConsumerWarps, kProducers, kFp8 ? 1 : 2>;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - raw_u32);

    // Split grid (K, B, P): partitions are the slowest dimension and the highest runs first, so
    // the extra partitions of the longest sequences start before the rest (longest-first).
    const int kvh = blockIdx.x;
    const int b = blockIdx.y;
    const int part = kSplit ? (int)gridDim.z - 1 - (int)blockIdx.z : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.G;

    // The producers' first block-table entries do not depend on the context length: loaded
    // before it (within the table row), their round trip overlaps its round trip.
    const int first_blk = kSplit ? partition_first_block(part, p.part_blocks, p.taper != 0) : 0;
    int tbl_first = 0;
    if (warp >= kConsumerWarps) {
        const int64_t j = first_blk + (warp - kConsumerWarps) + (int64_t)kProducers * lane;
        if (j < p.max_nb) tbl_first = __ldg(p.block_tables + (size_t)b * p.max_nb + j);
    }
    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_nb * kBlockSize) {
        if (threadIdx.x == 0 && kvh == 0 && part == 0) set_flag(p.err_flag, PKV_FLAG_CTX_RANGE);
        ctx = 0;
    }
    const int nb = (ctx + kBlockSize - 1) / kBlockSize;
    const int nparts = kSplit ? partition_count(nb, p.part_blocks, p.taper != 0) : 1;
    int blk_begin = 0, blk_end = nb;
    if (kSplit) partition_range(part, nparts, nb, p.part_blocks, p.taper != 0, blk_begin, blk_end);
    const int nblk = blk_end - blk_begin;
    // In-kernel merge (split with counters): a sequence held by one partition is written out
    // directly; one held by several leaves partials, and the last of its CTAs to finish (per KV
    // head, counted in p.counters) merges them and resets the count to zero.
    const bool merge_here = kSplit && p.counters != nullptr;
    const bool direct = !kSplit || (merge_here && nparts <= 1);

    if (nblk <= 0) {
        // A single pass over an empty sequence writes 0 / -inf (so does partition 0 of an empty
        // sequence when the merge runs in the kernel); an empty partition is never read by the
        // merge and writes nothing.  An empty sequence appends nothing.
        if (p.slot_out && nb == 0 && kvh == 0 && part == 0 && threadIdx.x == 0) p.slot_out[b] = -1;
        if (!kSplit || (merge_here && nb == 0 && part == 0)) {
            for (int idx = threadIdx.x; idx < G * H; idx += kAttnThreads) {
                const int g = idx / H, h = idx - g * H;
                const size_t bn = (size_t)b * p.N + (size_t)kvh * G + g;
                p.out[bn * H + h] = __float2bfloat16_rn(0.0f);
                if (h == 0 && p.lse_out) p.lse_out[bn] = -INFINITY;
            }
        }
        return;
    }

    const uint32_t bar_full = base_u32 + L::kBarOffset;
    const uint32_t bar_empty = bar_full + 8 * S;
    volatile int *slot_ok = reinterpret_cast<volatile int *>(base + L::kMiscOffset);
    volatile int *abort_flag = slot_ok + S;
    volatile int *issued_count = abort_flag + 1;  // [kProducers]
    // e4m3 with per-(block, head) scales: the producers store each stage's (K, V) scales; each
    // consumer warp takes its tiles' weights relative to the largest V scale it has seen so far
    // (VScaleRef), which multiplies its state before the warps' states are merged.  With per-head
    // scales the head's V scale multiplies the output at the end.
    volatile float2 *stage_sc = reinterpret_cast<volatile float2 *>(base + L::kScaleOffset);
    constexpr bool bscale = kFp8 && kBScale;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int q = 0; q < kProducers; ++q) issued_count[q] = 0;
        init_ring<S>(bar_full, bar_empty);
    }
    __syncthreads();

    WarpAcc<H> acc;
    VScaleRef vr{0.f, 0.f};  // e4m3 with per-(block, head) scales only

    if (warp >= kConsumerWarps) {
        // ------------------------------ producer warps ------------------------------
        const int pw = warp - kConsumerWarps;
        if (lane == 0 && pw == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int32_t *tbl = p.block_tables + (size_t)b * p.max_nb + blk_begin;
        const int64_t issued = run_producer<kProducers, bscale>(
            pw, lane, nblk, [&](int64_t i) { return __ldg(tbl + i); }, p.num_blocks, p.err_flag,
            [&](int64_t i, int bid, bool ok, float2 sc) {
                if (PKV_TILE_WITHHELD(p, i)) return true;  // test builds: never loaded, never signalled
                return produce_tile<H, S, kFp8>(i, kvh, bid, ok, base_u32, bar_full, bar_empty,
                                                slot_ok, abort_flag, &tm_k, &tm_v, p.tok_major,
                                                p.err_flag, p.wait_ns, bscale ? stage_sc : nullptr, sc);
            },
            [&](int bid) {
                if (!bscale) return make_float2(0.f, 0.f);
                const size_t si = (size_t)bid * p.scale_stride + kvh;
                return make_float2(__ldg(p.k_scale + si), __ldg(p.v_scale + si));
            },
            true, tbl_first);
        if (lane == 0) issued_count[pw] = (int)issued;
    } else {
        // ------------------------------ consumer warps ------------------------------
        uint32_t qf[H / 16][2];
        if constexpr (kFp8)
            load_q_frags_fp8<H>(qf, p.q, p.N, b, kvh, G, lane);
        else
            load_q_frags<H>(qf, p.q, p.N, b, kvh, G, lane);
        acc_reset<H>(acc);
        const float sl2 = kFp8 ? p.scale_log2 * p.k_scale[kvh] : p.scale_log2;
        // fused append: the warp that will hold the last block warms the new K/V rows in L2
        if (p.k_new && blk_end == nb && warp == (nb - 1 - blk_begin) % kConsumerWarps && lane < 2) {
            const size_t row = ((size_t)b * p.K + kvh) * H;
            prefetch_l2((lane ? p.v_new : p.k_new) + row);
        }
        if constexpr (kPairs) {
            // e4m3, few CTAs per SM: each warp takes its next two tiles (i and i + W) in one step
            // (two independent chains in flight); the ring holds S >= 2W stages, so the producer
            // can always fill the second one.
            static_assert(S >= 2 * kConsumerWarps, "pairs of tiles need two stages per warp");
            for (int i = warp; i < nblk; i += 2 * kConsumerWarps) {
                const int i2 = i + kConsumerWarps;
                const bool has2 = i2 < nblk;
                const int s1 = i % S, s2 = i2 % S;
                bool ok = mbar_wait_bounded(bar_full + 8 * s1, (i / S) & 1, abort_flag, p.wait_ns);
                if (ok && has2) ok = mbar_wait_bounded(bar_full + 8 * s2, (i2 / S) & 1, abort_flag, p.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok);  // lanes may differ at the deadline: the warp agrees
                if (!ok) {
                    if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                uint32_t kts[2], vts[2];
                int valid[2];
                float sl2s[2] = {sl2, sl2}, vss[2] = {0.f, 0.f};
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int it = t ? i2 : i, st = t ? s2 : s1;
                    const bool here = t == 0 || has2;
                    kts[t] = base_u32 + (here ? st : s1) * L::kStageBytes;
                    vts[t] = kts[t] + L::kTileBytes;
                    valid[t] = here && slot_ok[st] ? min(kBlockSize, ctx - (blk_begin + it) * kBlockSize) : 0;
                    if (bscale && valid[t] > 0) {
                        sl2s[t] = p.scale_log2 * stage_sc[st].x;
                        vss[t] = stage_sc[st].y;
                    }
                    // fused append: the tile of the sequence's last block holds the new token
                    const bool newest = here && p.k_new && blk_begin + it == nb - 1;
                    if (newest) {
                        const int last_bid = __ldg(p.block_tables + (size_t)b * p.max_nb + nb - 1);
                        if (slot_ok[st]) {
                            append_new_token_fp8<H>(p, b, kvh, ctx, last_bid, kts[t], vts[t],
                                                    bscale ? stage_sc[st].x : p.k_scale[kvh],
                                                    bscale ? stage_sc[st].y : p.v_scale[kvh], lane);
                            __syncwarp();
                        }
                        if (p.slot_out && kvh == 0 && lane == 0)
                            p.slot_out[b] = slot_ok[st] ? (int64_t)last_bid * kBlockSize + (ctx - 1) % kBlockSize : -1;
                    }
                }
                if (valid[0] > 0 || valid[1] > 0) tile_update_fp8_n<H, 2, bscale>(acc, qf, kts, vts, valid, sl2s, vss, vr, lane);
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar_empty + 8 * s1);
                    if (has2) mbar_arrive(bar_empty + 8 * s2);
                }
            }
        } else
        for (int i = warp; i < nblk; i += kConsumerWarps) {
            const int s = i % S;
            // lanes may differ at the deadline: the warp agrees before its collective MMA work
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar_full + 8 * s, (i / S) & 1, abort_flag, p.wait_ns))) {
                if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            // fused append: the tile of the sequence's last block holds the new token
            const bool newest = p.k_new && blk_begin + i == nb - 1;
            const int last_bid = newest ? __ldg(p.block_tables + (size_t)b * p.max_nb + nb - 1) : -1;
            if (slot_ok[s]) {
                const int valid = min(kBlockSize, ctx - (blk_begin + i) * kBlockSize);
                const uint32_t kt = base_u32 + s * L::kStageBytes;
                float sl2_t = sl2, vs_t = 0.f;  // this tile's logit multiplier and V scale
                if constexpr (bscale) {
                    sl2_t = p.scale_log2 * stage_sc[s].x;
                    vs_t = stage_sc[s].y;
                }
                if (newest) {
                    if constexpr (kFp8)
                        append_new_token_fp8<H>(p, b, kvh, ctx, last_bid, kt, kt + L::kTileBytes,
                                                bscale ? stage_sc[s].x : p.k_scale[kvh],
                                                bscale ? stage_sc[s].y : p.v_scale[kvh], lane);
                    else
                        append_new_token<H>(p, b, kvh, ctx, last_bid, kt, kt + L::kTileBytes, lane);
                    __syncwarp();
                }
                if constexpr (kFp8)
                    tile_update_fp8<H, bscale>(acc, qf, kt, kt + L::kTileBytes, valid, sl2_t, vs_t, vr, lane);
                else
                    tile_update<H>(acc, qf, kt, kt + L::kTileBytes, valid, sl2, p.tok_major, lane);
            }
            if (newest && p.slot_out && kvh == 0 && lane == 0)
                p.slot_out[b] = slot_ok[s] ? (int64_t)last_bid * kBlockSize + (ctx - 1) % kBlockSize : -1;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * s);
        }
    }

    __syncthreads();
    const bool aborted = *abort_flag != 0;
    if (aborted) {
        if (warp >= kConsumerWarps && lane == 0)
            drain_ring<S, kProducers>(bar_full, warp - kConsumerWarps,
                                            issued_count[warp - kConsumerWarps]);
        __syncthreads();
        // the sequence's other partitions still count on this one: it leaves a void partial
        if (!(merge_here && nparts > 1)) return;
    }

    // ------------------------- merge the consumer warps' states -------------------------
    float *mo = reinterpret_cast<float *>(base);              // [W][8][H]
    float *mm = mo + kConsumerWarps * 8 * H;                 // [W][8]
    float *ml = mm + kConsumerWarps * 8;                     // [W][8]
    if (!aborted) {
        if (warp < kConsumerWarps) {
            if constexpr (bscale) acc_scale_o<H>(acc, vr.v);  // each warp's O in value units
            deposit<H, kFp8>(acc, mo, mm, ml, warp, lane);
        }
        __syncthreads();
    }
    const float vscale = kFp8 && !bscale ? p.v_scale[kvh] : 1.f;
    for (int idx = threadIdx.x; idx < G * H; idx += kAttnThreads) {
        const int g = idx / H, h = idx - g * H;
        float val = __int_as_float(0x7FC00000), lse = __int_as_float(0x7FC00000);  // NaN: void
        if (!aborted) {
            combine<H>(mo, mm, ml, g, h, val, lse);
            val *= vscale;
        }
        const size_t bn = (size_t)b * p.N + (size_t)kvh * G + g;
        if (!direct) {
            const size_t bnp = bn * p.max_parts + part;
            p.part_out[bnp * H + h] = val;
            if (h == 0) p.part_lse[bnp] = lse;
        } else {
            p.out[bn * H + h] = __float2bfloat16_rn(val);
            if (h == 0 && p.lse_out) p.lse_out[bn] = lse;
        }
    }
    if (!merge_here || nparts <= 1) return;

    // ----------------- in-kernel log-sum-exp merge by the last partition -----------------
    // The host only asks for it when G * max_parts weights fit in the (drained) ring.
    __shared__ int last_one;
    __syncthreads();  // every partial of this CTA is written
    int32_t *count = p.counters + (size_t)b * p.K + kvh;
    if (threadIdx.x == 0) last_one = atomic_add_acq_rel_gpu(count, 1) == nparts - 1;
    __syncthreads();
    if (!last_one) return;
    float *wts = reinterpret_cast<float *>(base);                          // [G][nparts]
    float *red = reinterpret_cast<float *>(base) + kInKernelMergeWeights;  // [kMergeWarps][8][H]
    const size_t bn0 = (size_t)b * p.N + (size_t)kvh * G;
    // the rows' partial lse first, all loads independent (one round trip), then each row's weights
    // from that copy, in place
    for (int idx = threadIdx.x; idx < G * nparts; idx += kAttnThreads) {
        const int g = idx / nparts, q = idx - g * nparts;
        wts[idx] = __ldcg(p.part_lse + (bn0 + g) * p.max_parts + q);
    }
    __syncthreads();
    for (int g = warp; g < G; g += kAttnThreads / 32) {
        const float L = lse_merge_weights<true>(wts + g * nparts, nparts, wts + g * nparts, lane);
        if (lane == 0 && p.lse_out) p.lse_out[bn0 + g] = L;
    }
    __syncthreads();
    merge_rows<H, 8>(wts, nparts, G, p.part_out + bn0 * p.max_parts * H, (size_t)p.max_parts * H, red, p.out + bn0 * H,
                     H, threadIdx.x, kAttnThreads);
    if (threadIdx.x == 0) *count = 0;  // ready for the next call
}

// ---------------------------------- LSE merge ----------------------------------------------
// One CTA per (query head n, sequence b), one thread per output element h.
// One CTA merges R consecutive rows (query heads) of one sequence: R = 8 when their weights fit in
// shared memory, else 1.  Each row's bits do not depend on R (merge_rows).
template <int H, int R>
__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_kernel(const float *__restrict__ part_out, const float *__restrict__ part_lse,
                 const int32_t *__restrict__ context_lens, int N, int max_parts, int part_blocks, int taper,
                 __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out)
{
    extern __shared__ float smem_f[];  // weights [R][np], then the warps' sums [kMergeWarps][R][H]
    pdl_wait_primary();  // launched behind the attention grid (programmatic serialization): its partials
    const int n0 = blockIdx.x * R, b = blockIdx.y, t = threadIdx.x;
    const int nrows = min(R, N - n0);
    const size_t bn0 = (size_t)b * N + n0;
    int ctx = context_lens[b];
    const int nb = ctx > 0 ? (ctx + kBlockSize - 1) / kBlockSize : 0;
    int np = partition_count(nb, part_blocks, taper != 0);
    if (np > max_parts) np = max_parts;
    float *wts = smem_f;
    float *red = smem_f + ((size_t)R * max_parts + 3) / 4 * 4;
    // the rows' partial lse first, all loads independent (one round trip), then each row's weights
    // from that copy, in place
    for (int idx = t; idx < nrows * np; idx += blockDim.x) {
        const int g = idx / np, q = idx - g * np;
        wts[g * np + q] = __ldcg(part_lse + (bn0 + g) * max_parts + q);
    }
    __syncthreads();
    for (int g = t >> 5; g < nrows; g += kMergeWarps) {
        const float L = lse_merge_weights<true>(wts + g * np, np, wts + g * np, t & 31);
        if ((t & 31) == 0 && lse_out) lse_out[bn0 + g] = L;
    }
    __syncthreads();
    merge_rows<H, R>(wts, np, nrows, part_out + bn0 * max_parts * H, (size_t)max_parts * H, red, out + bn0 * H, H, t,
                     blockDim.x);
}

// ---------------------------------- launchers ----------------------------------------------
template <typename Kern>
static cudaError_t ensure_smem(Kern kern, int smem, int *cached)
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cached[dev] >= smem) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) cached[dev] = smem;
    return e;
}

template <int H, bool kSplit, bool kFp8, bool kPairs = false, bool kBScale = false, bool kDeep = false>
static cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                                 dim3 grid, cudaStream_t stream)
{
    constexpr int smem = AttnLayout<H, kFp8 ? kStagesFp8 : (kDeep ? kStagesDeep : kStages), kConsumerWarps,
                                    kProducers, kFp8 ? 1 : 2>::kAlloc;
    static int cached[64] = {};
    cudaError_t e = ensure_smem(attn_kernel<H, kSplit, kFp8, kPairs, kBScale, kDeep>, smem, cached);
    if (e != cudaSuccess) return e;
    attn_kernel<H, kSplit, kFp8, kPairs, kBScale, kDeep><<<grid, kAttnThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

// SMs of the current device (cached per device).
static int device_sms()
{
    static int sms[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 0;
    if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms[dev];
}

cudaError_t launch_attn(int H, bool split, const CUtensorMap &tk, const CUtensorMap &tv,
                        const AttnParams &p, cudaStream_t stream, bool fp8, bool pairs)
{
    dim3 grid = split ? dim3(p.K, p.B, p.max_parts) : dim3(p.K, p.B, 1);
    if (fp8) {  // e4m3 pools: H = 128 only; tile pairs for grids with few CTAs per SM
        if (p.scale_stride) {  // per-(block, head) scales
            if (pairs)
                return split ? launch_attn_t<128, true, true, true, true>(tk, tv, p, grid, stream)
                             : launch_attn_t<128, false, true, true, true>(tk, tv, p, grid, stream);
            return split ? launch_attn_t<128, true, true, false, true>(tk, tv, p, grid, stream)
                         : launch_attn_t<128, false, true, false, true>(tk, tv, p, grid, stream);
        }
        if (pairs)
            return split ? launch_attn_t<128, true, true, true>(tk, tv, p, grid, stream)
                         : launch_attn_t<128, false, true, true>(tk, tv, p, grid, stream);
        return split ? launch_attn_t<128, true, true>(tk, tv, p, grid, stream)
                     : launch_attn_t<128, false, true>(tk, tv, p, grid, stream);
    }
    // bf16: a grid that fits in one wave at two CTAs per SM takes the deeper ring (kStagesDeep)
    const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
    const int sms = device_sms();
    if (sms > 0 && ctas <= 2 * (int64_t)sms) {
        if (H == 128)
            return split ? launch_attn_t<128, true, false, false, false, true>(tk, tv, p, grid, stream)
                         : launch_attn_t<128, false, false, false, false, true>(tk, tv, p, grid, stream);
        return split ? launch_attn_t<64, true, false, false, false, true>(tk, tv, p, grid, stream)
                     : launch_attn_t<64, false, false, false, false, true>(tk, tv, p, grid, stream);
    }
    if (H == 128)
        return split ? launch_attn_t<128, true, false>(tk, tv, p, grid, stream)
                     : launch_attn_t<128, false, false>(tk, tv, p, grid, stream);
    return split ? launch_attn_t<64, true, false>(tk, tv, p, grid, stream)
                 : launch_attn_t<64, false, false>(tk, tv, p, grid, stream);
}

// pkv_lse_merge for rows of at most kFewParts partition slots (max_parts <= kFewParts): one warp per
// row, six rows a CTA.  Every load -- the length, the row's partial lse and partials of every slot
// -- is issued at once (slots past the row's partitions are read and never used), then the weights
// (lse_merge_weights, on the warp's copy of the lse) and the sum in merge_rows' order: merge slot s
// adds partitions s, s + kMergeWarps, ... with fused multiply-adds, the slots' sums are added in slot
// order -- the same bits as merge_rows and the in-kernel merges.  Few registers, so many CTAs per SM
// (merge_rows keeps eight rows a warp in flight: 96 registers, three 192-thread CTAs per SM; eight
// new tokens on the Llama-3-8B batch of 64 merge 16,384 rows).
constexpr int kFewParts = 8;

template <int H>
__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_few_kernel(const float *__restrict__ part_out, const float *__restrict__ part_lse,
                     const int32_t *__restrict__ context_lens, int N, int max_parts, int part_blocks, int taper,
                     __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out)
{
    constexpr int E = H / 32;
    static_assert(E == 2 || E == 4, "H = 64 or 128");
    __shared__ float wsm[kMergeWarps][kFewParts];
    pdl_wait_primary();  // launched behind the attention grid (programmatic serialization): its partials
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kMergeWarps + warp, b = blockIdx.y;
    if (n >= N) return;  // the whole warp
    const size_t row = (size_t)b * N + n;
    const float *po = part_out + row * max_parts * H + lane * E;
    float v[kFewParts][E];
#pragma unroll
    for (int q = 0; q < kFewParts; ++q) {
        if (q < max_parts) {
            if constexpr (E == 4) {
                const float4 x = __ldcg(reinterpret_cast<const float4 *>(po + (size_t)q * H));
                v[q][0] = x.x, v[q][1] = x.y, v[q][2] = x.z, v[q][3] = x.w;
            } else {
                const float2 x = __ldcg(reinterpret_cast<const float2 *>(po + (size_t)q * H));
                v[q][0] = x.x, v[q][1] = x.y;
            }
        }
    }
    const float lp = lane < max_parts ? __ldcg(part_lse + row * max_parts + lane) : 0.f;
    const int ctx = context_lens[b];
    const int nb = ctx > 0 ? (ctx + kBlockSize - 1) / kBlockSize : 0;
    const int np = min(partition_count(nb, part_blocks, taper != 0), max_parts);
    float *w = wsm[warp];
    if (lane < kFewParts) w[lane] = lp;
    __syncwarp();
    const float L = lse_merge_weights<true>(w, np, w, lane);
    if (lane == 0 && lse_out) lse_out[row] = L;
    float sum[E];
#pragma unroll
    for (int e = 0; e < E; ++e) sum[e] = 0.f;
#pragma unroll
    for (int s = 0; s < kMergeWarps; ++s) {
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
        for (int q = s; q < kFewParts; q += kMergeWarps) {
            if (q < np) {
                const float wq = w[q];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(wq, v[q][e], acc[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) sum[e] += acc[e];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) out[row * H + lane * E + e] = __float2bfloat16_rn(sum[e]);
}

template <int H, int R>
static cudaError_t launch_lse_merge_t(const float *part_out, const float *part_lse, const int32_t *context_lens,
                                      int B, int N, int max_parts, int part_blocks, int taper, uint16_t *out,
                                      float *lse_out, cudaStream_t stream, bool pdl)
{
    const size_t smem = (((size_t)R * max_parts + 3) / 4 * 4 + (size_t)kMergeWarps * R * H) * sizeof(float);
    static int cached[64] = {};
    cudaError_t e = ensure_smem(lse_merge_kernel<H, R>, (int)smem, cached);
    if (e != cudaSuccess) return e;
    return launch_kernel(lse_merge_kernel<H, R>, dim3((N + R - 1) / R, B), dim3(kMergeWarps * 32), smem, stream,
                         pdl, part_out, part_lse, context_lens, N, max_parts, part_blocks, taper,
                         reinterpret_cast<__nv_bfloat16 *>(out), lse_out);
}

cudaError_t launch_lse_merge(const float *part_out, const float *part_lse, const int32_t *context_lens,
                             int B, int N, int H, int max_parts, int part_blocks, bool taper, uint16_t *out,
                             float *lse_out, cudaStream_t stream, bool pdl)
{
    const int tp = taper ? 1 : 0;
    if (max_parts <= kFewParts && (H == 128 || H == 64)) {
        const dim3 grid((N + kMergeWarps - 1) / kMergeWarps, B);
        __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out);
        return H == 128 ? launch_kernel(lse_merge_few_kernel<128>, grid, dim3(kMergeWarps * 32), 0, stream, pdl,
                                        part_out, part_lse, context_lens, N, max_parts, part_blocks, tp, o, lse_out)
                        : launch_kernel(lse_merge_few_kernel<64>, grid, dim3(kMergeWarps * 32), 0, stream, pdl,
                                        part_out, part_lse, context_lens, N, max_parts, part_blocks, tp, o, lse_out);
    }
    // eight rows per CTA while their weights stay within 32 KB
    const bool eight = (int64_t)8 * max_parts <= 8192;
    if (H == 128)
        return eight ? launch_lse_merge_t<128, 8>(part_out, part_lse, context_lens, B, N, max_parts, part_blocks, tp, out, lse_out, stream, pdl)
                     : launch_lse_merge_t<128, 1>(part_out, part_lse, context_lens, B, N, max_parts, part_blocks, tp, out, lse_out, stream, pdl);
    if (H == 64)
        return eight ? launch_lse_merge_t<64, 8>(part_out, part_lse, context_lens, B, N, max_parts, part_blocks, tp, out, lse_out, stream, pdl)
                     : launch_lse_merge_t<64, 1>(part_out, part_lse, context_lens, B, N, max_parts, part_blocks, tp, out, lse_out, stream, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
