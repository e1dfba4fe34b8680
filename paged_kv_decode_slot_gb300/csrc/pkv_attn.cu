// pkv_attn.cu - paged decode attention for sm_103a.
//
// Work is cut into tiles: one tile = one physical block (16 tokens) of one KV head.  A CTA has
// a producer warp and four consumer warps.  The producer walks the CTA's tiles, looks each one
// up in the block table, and streams its K and V (16 x H bf16 each) into a ring of shared-memory
// stages with TMA, one mbarrier pair per stage.  The consumer warps take the stages round-robin;
// each keeps an online-softmax state for the whole query group (the G = N/K query heads that share
// the KV head), so every K/V byte fetched from HBM serves all G heads:
//     S^T[16 tok x 8] = K_tile[16 x H] . Q^T[H x 8]        (mma.sync m16n8k16, G padded to 8)
//     P^T            = exp2(S^T * scale*log2e - m)         (fp32, lazily rescaled running max)
//     O^T[H x 8]    += V_tile^T[H x 16] . P^T[16 x 8]      (P^T moved to the B operand with
//                                                          movmatrix; V^T via ldmatrix.trans)
// When a unit (sequence, KV head) ends, the four warps' states are merged in shared memory.
//
// Three ways to cut the work:
//  * attn_kernel<H, false>: one CTA per (KV head, sequence), whole sequence (single pass).
//  * attn_kernel<H, true>:  one CTA per (KV head, sequence, partition), partitions of a fixed
//    number of blocks (FlashDecoding), highest partition first; partial results are merged by
//    lse_merge_kernel.
//  * attn_balanced_kernel<H>: a persistent grid (about two CTAs per SM, a multiple of K) in which
//    CTA c serves KV head c % K and takes the (c / K)-th equal share of that head's tiles in
//    (sequence, block) order, keeping its TMA ring streaming across unit boundaries.  The K CTAs
//    of one share read the same physical blocks at the same time (one per head), as the K CTAs of
//    a sequence do in the single pass.  Units that lie inside one share are finished in place;
//    units cut by a share boundary leave fp32 partials (at most two per CTA) for
//    balanced_merge_kernel.
//
// This fuses the block-table gather with attention ("融合块读取和注意力的内核" and FlashDecoding
// in CS336 Lecture 10's notes) and computes, for one query token, softmax(q K^T * scale) V with
// the maximum subtracted ("Optimización de la inferencia", "Construye el mismo", Step 2), in its
// online (running max / running sum) form; the log-sum-exp merge of disjoint key sets is exact.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

// Pipeline depth (K+V tile pairs in flight per CTA), CTAs per SM and producer warps per CTA.  The
// bytes in flight per SM (stages x 8 KiB x CTAs at H = 128) must cover HBM latency under full
// load, and one producer warp issues only about 2.6 M tiles/s (two TMA tile loads each), so a CTA
// needs more than one to keep its ring full.
#ifndef PKV_STAGES
#define PKV_STAGES 8
#endif
#ifndef PKV_CTAS_PER_SM
#define PKV_CTAS_PER_SM 3
#endif
#ifndef PKV_BAL_STAGES
#define PKV_BAL_STAGES 8
#endif
#ifndef PKV_BAL_WARPS
#define PKV_BAL_WARPS 4
#endif
#ifndef PKV_BAL_CTAS_PER_SM
#define PKV_BAL_CTAS_PER_SM 2
#endif

#ifndef PKV_PRODUCERS
#define PKV_PRODUCERS 2
#endif
#ifndef PKV_BAL_PRODUCERS
#define PKV_BAL_PRODUCERS 2
#endif

#ifndef PKV_FP8_STAGES
#define PKV_FP8_STAGES 16
#endif

constexpr int kConsumerWarps = 4;
constexpr int kStages = PKV_STAGES;
constexpr int kStagesFp8 = PKV_FP8_STAGES;  // e4m3 tiles are half the bytes: twice the depth
constexpr int kProducers = PKV_PRODUCERS;
constexpr int kAttnThreads = (kConsumerWarps + kProducers) * 32;
constexpr int kBalStages = PKV_BAL_STAGES;
constexpr int kBalWarps = PKV_BAL_WARPS;
constexpr int kBalProducers = PKV_BAL_PRODUCERS;
constexpr int kBalThreads = (kBalWarps + kBalProducers) * 32;
// Stage s is reused by tiles s, s+S, s+2S, ... and tile i goes to consumer warp i % W.  With
// S a multiple of W every use of a stage belongs to the same warp, so a warp only waits for a
// stage's next phase after it consumed the previous one and mbarrier parities cannot alias.
// The same holds for the producer warps (producer p issues tiles i = p mod P).
static_assert(kStages % kConsumerWarps == 0, "pipeline depth must be a multiple of the consumer warps");
static_assert(kBalStages % kBalWarps == 0, "pipeline depth must be a multiple of the consumer warps");
static_assert(kStages % kProducers == 0, "pipeline depth must be a multiple of the producer warps");
static_assert(kStagesFp8 % kConsumerWarps == 0 && kStagesFp8 % kProducers == 0,
              "pipeline depth must be a multiple of the consumer and producer warps");
static_assert(kBalStages % kBalProducers == 0, "pipeline depth must be a multiple of the producer warps");

int balanced_ctas_per_sm() { return PKV_BAL_CTAS_PER_SM; }
// Lazy rescaling: keep the running maximum until a new logit exceeds it by this much
// (log2 units), so exponentials stay <= 2^8 and the accumulator is rarely rescaled.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;

template <int H, int S = kStages, int W = kConsumerWarps, int P = kProducers, int EB = 2>
struct AttnLayout {
    static constexpr int kHalves = H / 64;                  // 128-byte rows per bf16 token row
    static constexpr int kTileBytes = kBlockSize * H * EB;  // one K or V tile (EB bytes/element)
    static constexpr int kStageBytes = 2 * kTileBytes;      // K tile then V tile
    static constexpr int kPipeBytes = S * kStageBytes;
    static constexpr int kMergeBytes = W * 8 * (H + 2) * 4;
    // single-pass / partition kernel: the merge area reuses the drained pipeline
    static constexpr int kDataBytes = kPipeBytes > kMergeBytes ? kPipeBytes : kMergeBytes;
    static constexpr int kBarOffset = kDataBytes;           // full[S], empty[S]
    static constexpr int kMiscOffset = kBarOffset + 2 * S * 8;  // slot_ok[S], abort, issued[P]
    static constexpr int kBytes = kMiscOffset + (S + 1 + P) * 4;
    static constexpr int kAlloc = kBytes + 1024;             // slack for 1024-byte alignment
    // balanced kernel: pipeline, its own merge area, barriers, misc, then the block prefix
    static constexpr int kBalMergeOffset = kPipeBytes;
    static constexpr int kBalBarOffset = kBalMergeOffset + kMergeBytes;
    static constexpr int kBalMiscOffset = kBalBarOffset + 2 * S * 8;
    // misc: int64 issued[P], abort flag (padded to 8 bytes), slot_ok[S]
    static constexpr int kBalSeqOffset = (kBalMiscOffset + 8 * P + 8 + S * 4 + 15) / 16 * 16;
    static int balanced_alloc(int B) { return kBalSeqOffset + (B + 1) * 8 + 1024; }
    static_assert(kBalMiscOffset % 8 == 0, "the balanced kernel's int64 counter needs 8-byte alignment");
    static_assert(kBalSeqOffset % 16 == 0 && kPipeBytes % 1024 == 0, "shared-memory layout alignment");
    static_assert(kTileBytes % 1024 == 0, "TMA destinations with 128B swizzle need 1024-byte alignment");
};

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

// ----------------------------- per-warp online-softmax state -----------------------------
template <int H>
struct WarpAcc {
    float o[H / 16][4];  // O^T fragments: rows h (16 per m-tile), columns g = c0, c0+1
    float m[2];          // running max of columns c0, c0+1 (log2 units)
    float l[2];          // this lane's share of the running sums
};

template <int H>
__device__ __forceinline__ void acc_reset(WarpAcc<H> &a)
{
#pragma unroll
    for (int mt = 0; mt < H / 16; ++mt) a.o[mt][0] = a.o[mt][1] = a.o[mt][2] = a.o[mt][3] = 0.f;
    a.m[0] = a.m[1] = -INFINITY;
    a.l[0] = a.l[1] = 0.f;
}

// Q^T as the B operand of S^T = K . Q^T: lane l holds q[g = l/4][16kk + 2(l%4) + {0,1}] and
// the same +8; rows g >= G are zero.
template <int H>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[H / 16][2], const uint16_t *q, int N,
                                             int b, int kvh, int G, int lane)
{
    const int g_row = lane >> 2, c0 = (lane & 3) * 2;
    const bool live = g_row < G;
    const uint16_t *qrow = q + ((size_t)b * N + (size_t)kvh * G + (live ? g_row : 0)) * H;
#pragma unroll
    for (int kk = 0; kk < H / 16; ++kk) {
        qf[kk][0] = live ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0)) : 0u;
        qf[kk][1] = live ? __ldg(reinterpret_cast<const unsigned int *>(qrow + 16 * kk + c0 + 8)) : 0u;
    }
}

// One 16-token tile (the first `valid` tokens count) folded into a warp's state.
template <int H>
__device__ __forceinline__ void tile_update(WarpAcc<H> &a, const uint32_t (&qf)[H / 16][2],
                                            uint32_t kt, uint32_t vt, int valid, float sl2,
                                            int tok_major, int lane)
{
    constexpr int kKSteps = H / 16;
    const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: lane feeds matrix mi, row ri
    const int k_tok = ri + 8 * (mi & 1), k_hoff = 8 * (mi >> 1);  // K as A (non-trans)
    const int v_tok = ri + 8 * (mi >> 1), v_hoff = 8 * (mi & 1);  // V^T as A (trans)

    // S^T = K . Q^T, two independent accumulation chains
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kKSteps; kk += 2) {
        uint32_t a0[4], a1[4];
        ldsm_x4(a0, kt + tile_chunk_offset<H>(k_tok, 16 * kk + k_hoff, tok_major));
        ldsm_x4(a1, kt + tile_chunk_offset<H>(k_tok, 16 * kk + 16 + k_hoff, tok_major));
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
    const bool needA = mA > a.m[0] + kRescaleThreshold;
    const bool needB = mB > a.m[1] + kRescaleThreshold;
    if (__any_sync(0xFFFFFFFFu, needA || needB)) {
        const float alphaA = needA ? exp2f(a.m[0] - mA) : 1.f;
        const float alphaB = needB ? exp2f(a.m[1] - mB) : 1.f;
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
    const uint32_t p01 = pack_bf16x2(exp2f(x0 - a.m[0]), exp2f(x1 - a.m[1]));
    const uint32_t p23 = pack_bf16x2(exp2f(x2 - a.m[0]), exp2f(x3 - a.m[1]));
    a.l[0] += bf16x2_lo(p01) + bf16x2_lo(p23);  // sums of the rounded weights
    a.l[1] += bf16x2_hi(p01) + bf16x2_hi(p23);
    const uint32_t pb0 = movmatrix_trans(p01);    // P^T rows tok 0-7 -> B fragment
    const uint32_t pb1 = movmatrix_trans(p23);    // tok 8-15

    // O^T += V^T . P^T
    const bool partial = valid < kBlockSize;
    const int tc = (lane & 3) * 2;  // token columns of this lane's A fragment
#pragma unroll
    for (int mt = 0; mt < kKSteps; ++mt) {
        uint32_t av[4];
        ldsm_x4_trans(av, vt + tile_chunk_offset<H>(v_tok, 16 * mt + v_hoff, tok_major));
        if (partial) {  // zero V of tokens past the context (they may be NaN poison)
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

// ------------------------------------ FP8 (e4m3) tiles ------------------------------------
// An e4m3 tile is 16 token rows of H = 128 bytes (128B-swizzled).  ldmatrix reads it as b16
// pairs and cvt widens pairs to f16 exactly, so the contractions run as f16 mma.sync.  Reading
// b16 pairs permutes the head dimension inside each 16-element step; q (the other operand of
// QK^T) is loaded in the same order, and in P.V the accumulator rows come out as
// h = 16*mt + 2*(lane/4) (+1 for the upper 8 rows) instead of 16*mt + lane/4 (+8).
__device__ __forceinline__ uint32_t fp8_chunk_offset(int tok, int chunk)
{
    return static_cast<uint32_t>(tok * 128 + ((chunk ^ (tok & 7)) << 4));
}

// q as f16 B fragments: k-step kk, lane (g = lane/4, m = lane%4): b0 = q[16kk + 4m .. +1],
// b1 = q[16kk + 4m + 2 .. +3]; rows g >= G are zero.
template <int H>
__device__ __forceinline__ void load_q_frags_fp8(uint32_t (&qf)[H / 16][2], const uint16_t *q, int N,
                                                 int b, int kvh, int G, int lane)
{
    const int g_row = lane >> 2, m = lane & 3;
    const bool live = g_row < G;
    const uint16_t *qrow = q + ((size_t)b * N + (size_t)kvh * G + (live ? g_row : 0)) * H;
#pragma unroll
    for (int kk = 0; kk < H / 16; ++kk) {
        if (live) {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(qrow + 16 * kk + 4 * m));
            qf[kk][0] = pack_f16x2(bf16_to_f32((uint16_t)(v.x & 0xFFFFu)), bf16_to_f32((uint16_t)(v.x >> 16)));
            qf[kk][1] = pack_f16x2(bf16_to_f32((uint16_t)(v.y & 0xFFFFu)), bf16_to_f32((uint16_t)(v.y >> 16)));
        } else {
            qf[kk][0] = qf[kk][1] = 0u;
        }
    }
}

// One 16-token e4m3 tile folded into a warp's state (the codes only; the per-head scales are
// folded into sl2 and into the final normalisation).
template <int H>
__device__ __forceinline__ void tile_update_fp8(WarpAcc<H> &a, const uint32_t (&qf)[H / 16][2],
                                                uint32_t kt, uint32_t vt, int valid, float sl2, int lane)
{
    constexpr int kKSteps = H / 16;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi & 1), coff = mi >> 1;  // ldmatrix row address of this lane

    // S^T = K . Q^T
    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kKSteps; kk += 2) {
        uint32_t r[4];
        ldsm_x4(r, kt + fp8_chunk_offset(tok, kk + coff));
        uint32_t a0[4], a1[4];
        a0[0] = e4m3x2_to_f16x2((uint16_t)(r[0] & 0xFFFFu));
        a0[1] = e4m3x2_to_f16x2((uint16_t)(r[1] & 0xFFFFu));
        a0[2] = e4m3x2_to_f16x2((uint16_t)(r[0] >> 16));
        a0[3] = e4m3x2_to_f16x2((uint16_t)(r[1] >> 16));
        a1[0] = e4m3x2_to_f16x2((uint16_t)(r[2] & 0xFFFFu));
        a1[1] = e4m3x2_to_f16x2((uint16_t)(r[3] & 0xFFFFu));
        a1[2] = e4m3x2_to_f16x2((uint16_t)(r[2] >> 16));
        a1[3] = e4m3x2_to_f16x2((uint16_t)(r[3] >> 16));
        mma_f16_16816(sa, a0, qf[kk][0], qf[kk][1]);
        mma_f16_16816(sb, a1, qf[kk + 1][0], qf[kk + 1][1]);
    }
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
    const bool needA = mA > a.m[0] + kRescaleThreshold;
    const bool needB = mB > a.m[1] + kRescaleThreshold;
    if (__any_sync(0xFFFFFFFFu, needA || needB)) {
        const float alphaA = needA ? exp2f(a.m[0] - mA) : 1.f;
        const float alphaB = needB ? exp2f(a.m[1] - mB) : 1.f;
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
    const uint32_t p01 = pack_f16x2(exp2f(x0 - a.m[0]), exp2f(x1 - a.m[1]));
    const uint32_t p23 = pack_f16x2(exp2f(x2 - a.m[0]), exp2f(x3 - a.m[1]));
    a.l[0] += f16x2_lo(p01) + f16x2_lo(p23);
    a.l[1] += f16x2_hi(p01) + f16x2_hi(p23);
    const uint32_t pb0 = movmatrix_trans(p01);
    const uint32_t pb1 = movmatrix_trans(p23);

    // O^T += V^T . P^T: ldmatrix.trans gives lane bytes (tok 2m, h 2c'), (tok 2m, h 2c'+1),
    // (tok 2m+1, h 2c'), (tok 2m+1, h 2c'+1) with c' = lane/4; prmt regroups them per h.
    const bool partial = valid < kBlockSize;
    const int tc = (lane & 3) * 2;
#pragma unroll
    for (int mt = 0; mt < kKSteps; mt += 2) {
        uint32_t r[4];
        ldsm_x4_trans(r, vt + fp8_chunk_offset(tok, mt + coff));
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const uint32_t lo = byte_perm(r[2 * hf], 0u, 0x3120u);      // tokens 0-7 of the tile
            const uint32_t hi = byte_perm(r[2 * hf + 1], 0u, 0x3120u);  // tokens 8-15
            uint32_t av[4];
            av[0] = e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu));
            av[1] = e4m3x2_to_f16x2((uint16_t)(lo >> 16));
            av[2] = e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu));
            av[3] = e4m3x2_to_f16x2((uint16_t)(hi >> 16));
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
            mma_f16_16816(a.o[mt + hf], av, pb0, pb1);
        }
    }
}

// Finish a warp's sums (across the lanes that share a column) and store its state in the
// merge area: mo[W][8][H], mm[W][8] (running max), ml[W][8] (running sum).
template <int H, bool kFp8 = false>
__device__ __forceinline__ void deposit(WarpAcc<H> &a, float *mo, float *mm, float *ml, int warp,
                                        int lane)
{
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        a.l[0] += __shfl_xor_sync(0xFFFFFFFFu, a.l[0], off);
        a.l[1] += __shfl_xor_sync(0xFFFFFFFFu, a.l[1], off);
    }
    const int c0 = (lane & 3) * 2;
    if (lane < 4) {
        mm[warp * 8 + c0] = a.m[0];
        mm[warp * 8 + c0 + 1] = a.m[1];
        ml[warp * 8 + c0] = a.l[0];
        ml[warp * 8 + c0 + 1] = a.l[1];
    }
    const int hr = lane >> 2;
#pragma unroll
    for (int mt = 0; mt < H / 16; ++mt) {
        // rows of the accumulator: h0 for o[mt][0..1], h1 for o[mt][2..3]
        const int h0 = kFp8 ? 16 * mt + 2 * hr : 16 * mt + hr;
        const int h1 = kFp8 ? h0 + 1 : h0 + 8;
        mo[(warp * 8 + c0) * H + h0] = a.o[mt][0];
        mo[(warp * 8 + c0 + 1) * H + h0] = a.o[mt][1];
        mo[(warp * 8 + c0) * H + h1] = a.o[mt][2];
        mo[(warp * 8 + c0 + 1) * H + h1] = a.o[mt][3];
    }
}

// Combine the deposited states for column g, element h: normalised output and lse (natural).
template <int H, int W = kConsumerWarps>
__device__ __forceinline__ void combine(const float *mo, const float *mm, const float *ml, int g,
                                        int h, float &val, float &lse)
{
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, mm[w * 8 + g]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float sc = exp2f(mm[w * 8 + g] - M);
            lsum += sc * ml[w * 8 + g];
            acc += sc * mo[(w * 8 + g) * H + h];
        }
    }
    // No key at all (M = -inf) gives 0 and -inf; a NaN anywhere in the inputs stays NaN.
    val = M != -INFINITY ? acc / lsum : 0.f;
    lse = M != -INFINITY ? (M + log2f(lsum)) * kLn2 : -INFINITY;
}

template <int S>
__device__ __forceinline__ void init_ring(uint32_t bar_full, uint32_t bar_empty)
{
    for (int s = 0; s < S; ++s) {
        mbar_init(bar_full + 8 * s, 1);
        mbar_init(bar_empty + 8 * s, 1);
    }
    fence_barrier_init();
}

// Producer side of one tile: wait for the stage to be free, then load the tile (or mark it
// skipped).  Runs on one lane.  Returns false when the wait expired.  bf16 tiles come through
// 5-D maps (half-major or token-major), e4m3 tiles through a 4-D map (h, head, token, block).
template <int H, int S, bool kFp8 = false>
__device__ __forceinline__ bool produce_tile(int64_t i, int kvh, int bid, bool ok, uint32_t base_u32,
                                             uint32_t bar_full, uint32_t bar_empty,
                                             volatile int *slot_ok, volatile int *abort_flag,
                                             const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                                             int tok_major, int32_t *err_flag)
{
    using L = AttnLayout<H, S, kConsumerWarps, kProducers, kFp8 ? 1 : 2>;
    const int s = (int)(i % S);
    if (i >= S &&
        !mbar_wait_bounded(bar_empty + 8 * s, (uint32_t)(((i / S) & 1) ^ 1), abort_flag,
                           kWaitLimitNs)) {
        if (!*abort_flag) set_flag(err_flag, PKV_FLAG_TIMEOUT);
        *abort_flag = 1;
        return false;
    }
    if (ok) {
        slot_ok[s] = 1;
        const uint32_t dst = base_u32 + s * L::kStageBytes;
        const uint32_t bar = bar_full + 8 * s;
        mbar_arrive_expect_tx(bar, L::kStageBytes);
        if (kFp8) {
            tma_load_4d(dst, tm_k, bar, 0, kvh, 0, bid);
            tma_load_4d(dst + L::kTileBytes, tm_v, bar, 0, kvh, 0, bid);
        } else if (tok_major) {
            tma_load_5d(dst, tm_k, bar, 0, 0, kvh, 0, bid);
            tma_load_5d(dst + L::kTileBytes, tm_v, bar, 0, 0, kvh, 0, bid);
        } else {
            tma_load_5d(dst, tm_k, bar, 0, 0, 0, kvh, bid);
            tma_load_5d(dst + L::kTileBytes, tm_v, bar, 0, 0, 0, kvh, bid);
        }
    } else {
        slot_ok[s] = 0;  // out-of-range block id: the tile is skipped
        mbar_arrive(bar_full + 8 * s);
    }
    return true;
}

// Producer warp p of P issues the CTA's tiles i = p, p + P, p + 2P, ... in order: `lookup(i)`
// gives tile i's physical block id (lanes look up 32 tiles at a time, the next 32 while the
// current ones are issued) and `issue(i, bid, ok)` waits for the stage and loads it, returning
// false when its wait expired.  Returns the number of tiles this producer issued (on lane 0).
template <int P, typename Lookup, typename Issue>
__device__ __forceinline__ int64_t run_producer(int pw, int lane, int64_t n, Lookup lookup,
                                                int num_blocks, int32_t *err_flag, Issue issue)
{
    const int64_t mine = n > pw ? (n - pw + P - 1) / P : 0;
    int cur = lane < mine ? lookup(pw + (int64_t)P * lane) : 0;
    int64_t issued = 0;
    bool aborted = false;
    for (int64_t k0 = 0; k0 < mine && !aborted; k0 += 32) {
        const int nxt = (k0 + 32 + lane < mine) ? lookup(pw + (int64_t)P * (k0 + 32 + lane)) : 0;
        const int cnt = (int)min((int64_t)32, mine - k0);
        const bool bad = lane < cnt && (cur < 0 || cur >= num_blocks);
        const unsigned badmask = __ballot_sync(0xFFFFFFFFu, bad);
        if (badmask && lane == 0) set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
        for (int k = 0; k < cnt; ++k) {
            const int bid = __shfl_sync(0xFFFFFFFFu, cur, k);
            int lane0_abort = 0;
            if (lane == 0) {
                if (issue(pw + (int64_t)P * (k0 + k), bid, !((badmask >> k) & 1u)))
                    ++issued;
                else
                    lane0_abort = 1;
            }
            aborted = __shfl_sync(0xFFFFFFFFu, lane0_abort, 0) != 0;
            if (aborted) break;
        }
        cur = nxt;
    }
    return issued;
}

// Drain after an expired wait: producer pw waits (bounded) for its copies that may still land.
template <int S, int P>
__device__ __forceinline__ void drain_ring(uint32_t bar_full, int pw, int64_t issued)
{
    for (int64_t k = issued > S / P ? issued - S / P : 0; k < issued; ++k) {
        const int64_t i = pw + (int64_t)P * k;
        mbar_wait_bounded(bar_full + 8 * (int)(i % S), (uint32_t)((i / S) & 1), nullptr, kDrainLimitNs);
    }
}

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
                                                     int bid, uint32_t kt, uint32_t vt, int lane)
{
    constexpr int kChunks = H / 16;
    if (lane >= 2 * kChunks) return;
    const int tok = (ctx - 1) % kBlockSize;
    const bool is_v = lane >= kChunks;
    const int c = is_v ? lane - kChunks : lane;
    const float sc = (is_v ? p.v_scale : p.k_scale)[kvh];
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
template <int H, bool kSplit, bool kFp8 = false>
__global__ void __launch_bounds__(kAttnThreads, PKV_CTAS_PER_SM)
attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
            const AttnParams p)
{
    constexpr int S = kFp8 ? kStagesFp8 : kStages;
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
        // A single pass over an empty sequence writes 0 / -inf; an empty partition is never
        // read by the merge and writes nothing.  An empty sequence appends nothing.
        if (p.slot_out && nb == 0 && kvh == 0 && part == 0 && threadIdx.x == 0) p.slot_out[b] = -1;
        if (!kSplit) {
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

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int q = 0; q < kProducers; ++q) issued_count[q] = 0;
        init_ring<S>(bar_full, bar_empty);
    }
    __syncthreads();

    WarpAcc<H> acc;

    if (warp >= kConsumerWarps) {
        // ------------------------------ producer warps ------------------------------
        const int pw = warp - kConsumerWarps;
        if (lane == 0 && pw == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        const int32_t *tbl = p.block_tables + (size_t)b * p.max_nb + blk_begin;
        const int64_t issued = run_producer<kProducers>(
            pw, lane, nblk, [&](int64_t i) { return __ldg(tbl + i); }, p.num_blocks, p.err_flag,
            [&](int64_t i, int bid, bool ok) {
                return produce_tile<H, S, kFp8>(i, kvh, bid, ok, base_u32, bar_full, bar_empty,
                                                slot_ok, abort_flag, &tm_k, &tm_v, p.tok_major,
                                                p.err_flag);
            });
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
        for (int i = warp; i < nblk; i += kConsumerWarps) {
            const int s = i % S;
            if (!mbar_wait_bounded(bar_full + 8 * s, (i / S) & 1, abort_flag, kWaitLimitNs)) {
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
                if (newest) {
                    if constexpr (kFp8)
                        append_new_token_fp8<H>(p, b, kvh, ctx, last_bid, kt, kt + L::kTileBytes, lane);
                    else
                        append_new_token<H>(p, b, kvh, ctx, last_bid, kt, kt + L::kTileBytes, lane);
                    __syncwarp();
                }
                if constexpr (kFp8)
                    tile_update_fp8<H>(acc, qf, kt, kt + L::kTileBytes, valid, sl2, lane);
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
    if (*abort_flag) {
        if (warp >= kConsumerWarps && lane == 0)
            drain_ring<S, kProducers>(bar_full, warp - kConsumerWarps,
                                            issued_count[warp - kConsumerWarps]);
        __syncthreads();
        return;
    }

    // ------------------------- merge the consumer warps' states -------------------------
    float *mo = reinterpret_cast<float *>(base);              // [W][8][H]
    float *mm = mo + kConsumerWarps * 8 * H;                 // [W][8]
    float *ml = mm + kConsumerWarps * 8;                     // [W][8]
    if (warp < kConsumerWarps) deposit<H, kFp8>(acc, mo, mm, ml, warp, lane);
    __syncthreads();
    const float vscale = kFp8 ? p.v_scale[kvh] : 1.f;
    for (int idx = threadIdx.x; idx < G * H; idx += kAttnThreads) {
        const int g = idx / H, h = idx - g * H;
        float val, lse;
        combine<H>(mo, mm, ml, g, h, val, lse);
        val *= vscale;
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

// ------------------------------ balanced (stream-K) split ---------------------------------
// For each KV head the tiles are numbered in (sequence b, block j) order; sequence b owns
// tiles [pre[b], pre[b+1]) with pre[b+1] - pre[b] = nb_b.  Of the grid's S = gridDim.x / K
// shares per head, share s takes tiles [floor(T*s/S), floor(T*(s+1)/S)); CTA c = s*K + kvh.
struct TileLoc {
    int b, j, nb;
    int64_t unit_start;  // first tile of sequence b
};

__device__ __forceinline__ TileLoc locate_tile(const int64_t *pre, int B, int64_t t)
{
    int lo = 0, hi = B - 1;  // largest b with pre[b] <= t (it has tiles since pre[b+1] > t)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= t) lo = mid; else hi = mid - 1;
    }
    TileLoc L;
    L.b = lo;
    L.nb = (int)(pre[lo + 1] - pre[lo]);
    L.j = (int)(t - pre[lo]);
    L.unit_start = pre[lo];
    return L;
}

__device__ __forceinline__ int64_t share_start(int64_t T, int G, int c)
{
    return T * c / G;  // the host bounds T * grid below 2^62
}

template <int W>
__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
}

template <int H>
__global__ void __launch_bounds__(kBalThreads, PKV_BAL_CTAS_PER_SM)
attn_balanced_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const AttnParams p)
{
    constexpr int S = kBalStages, W = kBalWarps, P = kBalProducers;
    using L = AttnLayout<H, S, W, P>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_u32 - raw_u32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.B, K = p.K, G = p.G;
    int64_t *pre = reinterpret_cast<int64_t *>(base + L::kBalSeqOffset);   // [B + 1]

    // Per-sequence block counts and their prefix, by warp 0 (B <= 1024: 32 sequences a lane).
    // An out-of-range context length counts as empty (and is flagged once).
    auto blocks_of = [&](int s) {
        const int c = p.context_lens[s];
        return (c < 0 || c > p.max_nb * kBlockSize) ? 0 : (c + kBlockSize - 1) / kBlockSize;
    };
    if (warp == 0) {
        const int per = (B + 31) / 32;
        const int s0 = min(B, lane * per), s1 = min(B, s0 + per);
        int64_t local = 0;
        for (int s = s0; s < s1; ++s) {
            const int c = p.context_lens[s];
            if ((c < 0 || c > p.max_nb * kBlockSize) && blockIdx.x == 0)
                set_flag(p.err_flag, PKV_FLAG_CTX_RANGE);
            local += blocks_of(s);
        }
        int64_t incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
        }
        int64_t run = incl - local;
        for (int s = s0; s < s1; ++s) {
            pre[s] = run;
            run += blocks_of(s);
        }
        if (lane == 31) pre[B] = incl;
    }
    __syncthreads();
    const int64_t T = pre[B];
    const int c = blockIdx.x, kvh = c % K, shares = gridDim.x / K, sh = c / K;
    if (c == 0 && p.prefix_out)
        for (int s = threadIdx.x; s <= B; s += kBalThreads) p.prefix_out[s] = pre[s];
    const int64_t t0 = share_start(T, shares, sh), t1 = share_start(T, shares, sh + 1);
    if (t0 >= t1) return;
    const int64_t n = t1 - t0;

    const uint32_t bar_full = base_u32 + L::kBalBarOffset;
    const uint32_t bar_empty = bar_full + 8 * S;
    volatile int64_t *issued_count = reinterpret_cast<volatile int64_t *>(base + L::kBalMiscOffset);  // [P]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + L::kBalMiscOffset + 8 * P);
    volatile int *slot_ok = abort_flag + 2;
    float *mo = reinterpret_cast<float *>(base + L::kBalMergeOffset);
    float *mm = mo + W * 8 * H;
    float *ml = mm + W * 8;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int q = 0; q < P; ++q) issued_count[q] = 0;
        init_ring<S>(bar_full, bar_empty);
    }
    __syncthreads();

    if (warp >= W) {
        // ------------------------------ producer warps ------------------------------
        const int pw = warp - W;
        if (lane == 0 && pw == 0) {
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
        }
        auto lookup = [&](int64_t i) -> int {
            const TileLoc tl = locate_tile(pre, B, t0 + i);
            return __ldg(p.block_tables + (size_t)tl.b * p.max_nb + tl.j);
        };
        const int64_t issued = run_producer<P>(
            pw, lane, n, lookup, p.num_blocks, p.err_flag, [&](int64_t i, int bid, bool ok) {
                return produce_tile<H, S>(i, kvh, bid, ok, base_u32, bar_full, bar_empty, slot_ok,
                                          abort_flag, &tm_k, &tm_v, p.tok_major, p.err_flag);
            });
        if (lane == 0) issued_count[pw] = issued;
    } else {
        // ------------------------------ consumer warps ------------------------------
        // Every consumer warp walks the same units in order and meets the others at two
        // consumer-only barriers per unit (also after an expired wait, so nobody is stranded).
        WarpAcc<H> acc;
        uint32_t qf[H / 16][2];
        bool aborted = false;
        bool first_unit = true;
        int64_t t = t0;
        while (t < t1) {
            const TileLoc u = locate_tile(pre, B, t);
            const int64_t ue = min(t1, u.unit_start + u.nb);   // end of this unit's part here
            const bool whole = u.unit_start >= t0 && u.unit_start + u.nb <= t1;
            const int ctx = p.context_lens[u.b];
            load_q_frags<H>(qf, p.q, p.N, u.b, kvh, G, lane);
            acc_reset<H>(acc);
            const int64_t ibeg = t - t0, iend = ue - t0;
            int64_t i = ibeg + (int64_t)((warp - (int)(ibeg % W) + W) % W);
            for (; i < iend && !aborted; i += W) {
                const int s = (int)(i % S);
                if (!mbar_wait_bounded(bar_full + 8 * s, (uint32_t)((i / S) & 1), abort_flag,
                                       kWaitLimitNs)) {
                    if (!*abort_flag) set_flag(p.err_flag, PKV_FLAG_TIMEOUT);
                    *abort_flag = 1;
                    aborted = true;
                    break;
                }
                if (slot_ok[s]) {
                    const int j = u.j + (int)(i - ibeg);
                    const int valid = min(kBlockSize, ctx - j * kBlockSize);
                    const uint32_t kt = base_u32 + s * L::kStageBytes;
                    tile_update<H>(acc, qf, kt, kt + L::kTileBytes, valid, p.scale_log2, p.tok_major, lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_empty + 8 * s);
            }
            deposit<H>(acc, mo, mm, ml, warp, lane);
            consumer_bar<W>();
            if (!*abort_flag) {
                const int slot = first_unit ? 0 : 1;
                for (int idx = threadIdx.x; idx < G * H; idx += W * 32) {
                    const int g = idx / H, h = idx - g * H;
                    float val, lse;
                    combine<H, W>(mo, mm, ml, g, h, val, lse);
                    if (whole) {
                        const size_t bn = (size_t)u.b * p.N + (size_t)kvh * G + g;
                        p.out[bn * H + h] = __float2bfloat16_rn(val);
                        if (h == 0 && p.lse_out) p.lse_out[bn] = lse;
                    } else {
                        const size_t cs = ((size_t)c * 2 + slot) * 8 + g;
                        p.part_out[cs * H + h] = val;
                        if (h == 0) p.part_lse[cs] = lse;
                    }
                }
            }
            consumer_bar<W>();
            first_unit = false;
            t = ue;
        }
    }

    __syncthreads();
    if (*abort_flag) {
        if (warp >= W && lane == 0) drain_ring<S, P>(bar_full, warp - W, issued_count[warp - W]);
        __syncthreads();
    }
}

// Merge of the units the balanced kernel left split: one CTA per (KV head, sequence).  A unit
// whose tiles all fell into one share is already final.  The pieces' lse are loaded in
// parallel, their weights e^{lse_q - lse} computed once, then every (g, h) output element
// sums its pieces.
constexpr int kMergeThreads = 128;
constexpr int kMaxPieces = 512;  // pieces of one unit held in shared memory per pass

__global__ void __launch_bounds__(kMergeThreads)
balanced_merge_kernel(const float *__restrict__ part_out, const float *__restrict__ part_lse,
                      const int64_t *__restrict__ pre, int B, int N, int K, int H, int grid, int KG,
                      __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out)
{
    __shared__ int piece_cs[kMaxPieces];        // (CTA, slot) index of each non-empty piece
    __shared__ float wgt[kMaxPieces][8];        // lse of piece q, column g, then its weight
    __shared__ float tot[8];
    // Pieces come from CTA c = share * (K / KG) + kvh / KG, slot (first/last unit of its share),
    // head kvh % KG of its group: entry ((c * 2 + slot) * KG + kvh % KG) * 8 + g.
    const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int G = N / K, groups = K / KG, shares = grid / groups;
    const int grp = kvh / KG, kh = kvh - grp * KG;
    const int64_t T = pre[B];
    const int nb = (int)(pre[b + 1] - pre[b]);
    if (nb == 0) {  // empty sequence: no CTA touched it
        for (int idx = tid; idx < G * H; idx += kMergeThreads) {
            const int g = idx / H, h = idx - g * H;
            const size_t bn = (size_t)b * N + (size_t)kvh * G + g;
            out[bn * H + h] = __float2bfloat16_rn(0.f);
            if (h == 0 && lse_out) lse_out[bn] = -INFINITY;
        }
        return;
    }
    const int64_t s = pre[b], e = s + nb;
    auto share_of = [&](int64_t t) {
        int c = (int)(t * shares / T);
        while (c + 1 < shares && share_start(T, shares, c + 1) <= t) ++c;
        while (c > 0 && share_start(T, shares, c) > t) --c;
        return c;
    };
    const int q0 = share_of(s), q1 = share_of(e - 1);
    if (q0 == q1) return;
    const int slot0 = share_start(T, shares, q0) == s ? 0 : 1;
    // Non-empty shares between q0 and q1 hold one piece each (shares with no tiles wrote nothing).
    int np = 0;
    if (tid == 0) {
        for (int q = q0; q <= q1 && np < kMaxPieces; ++q)
            if (share_start(T, shares, q) != share_start(T, shares, q + 1))
                piece_cs[np++] = ((q * groups + grp) * 2 + (q == q0 ? slot0 : 0)) * KG + kh;
        tot[0] = __int_as_float(np);
    }
    __syncthreads();
    np = __float_as_int(tot[0]);
    __syncthreads();
    for (int idx = tid; idx < np * G; idx += kMergeThreads) {
        const int q = idx / G, g = idx - q * G;
        wgt[q][g] = part_lse[(size_t)piece_cs[q] * 8 + g];
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int q = 0; q < np; ++q) M = fmaxf(M, wgt[q][tid]);
        float total = -INFINITY;
        if (M != -INFINITY) {
            float sum = 0.f;
            for (int q = 0; q < np; ++q) sum += expf(wgt[q][tid] - M);
            total = M + logf(sum);
            for (int q = 0; q < np; ++q) wgt[q][tid] = expf(wgt[q][tid] - total);
        } else {
            for (int q = 0; q < np; ++q) wgt[q][tid] = 0.f;
        }
        tot[tid] = total;
    }
    __syncthreads();
    for (int idx = tid; idx < G * H; idx += kMergeThreads) {
        const int g = idx / H, h = idx - g * H;
        float val = 0.f;
#pragma unroll 4
        for (int q = 0; q < np; ++q)
            val += wgt[q][g] * part_out[((size_t)piece_cs[q] * 8 + g) * H + h];
        const size_t bn = (size_t)b * N + (size_t)kvh * G + g;
        out[bn * H + h] = __float2bfloat16_rn(val);
        if (h == 0 && lse_out) lse_out[bn] = tot[g];
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

template <int H, bool kSplit, bool kFp8>
static cudaError_t launch_attn_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                                 dim3 grid, cudaStream_t stream)
{
    constexpr int smem = AttnLayout<H, kFp8 ? kStagesFp8 : kStages, kConsumerWarps, kProducers,
                                    kFp8 ? 1 : 2>::kAlloc;
    static int cached[64] = {};
    cudaError_t e = ensure_smem(attn_kernel<H, kSplit, kFp8>, smem, cached);
    if (e != cudaSuccess) return e;
    attn_kernel<H, kSplit, kFp8><<<grid, kAttnThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_attn(int H, bool split, const CUtensorMap &tk, const CUtensorMap &tv,
                        const AttnParams &p, cudaStream_t stream, bool fp8)
{
    dim3 grid = split ? dim3(p.K, p.B, p.max_parts) : dim3(p.K, p.B, 1);
    if (fp8)  // e4m3 pools: H = 128 only
        return split ? launch_attn_t<128, true, true>(tk, tv, p, grid, stream)
                     : launch_attn_t<128, false, true>(tk, tv, p, grid, stream);
    if (H == 128)
        return split ? launch_attn_t<128, true, false>(tk, tv, p, grid, stream)
                     : launch_attn_t<128, false, false>(tk, tv, p, grid, stream);
    return split ? launch_attn_t<64, true, false>(tk, tv, p, grid, stream)
                 : launch_attn_t<64, false, false>(tk, tv, p, grid, stream);
}

template <int H>
static cudaError_t launch_balanced_t(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                                     int grid, cudaStream_t stream)
{
    using L = AttnLayout<H, kBalStages, kBalWarps, kBalProducers>;
    const int smem = L::balanced_alloc(p.B);
    static int cached[64] = {};
    cudaError_t e = ensure_smem(attn_balanced_kernel<H>, L::balanced_alloc(kMaxBalancedSeqs), cached);
    if (e != cudaSuccess) return e;
    attn_balanced_kernel<H><<<grid, kBalThreads, smem, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

cudaError_t launch_attn_balanced(int H, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, int grid, cudaStream_t stream)
{
    return H == 128 ? launch_balanced_t<128>(tk, tv, p, grid, stream)
                    : launch_balanced_t<64>(tk, tv, p, grid, stream);
}

cudaError_t launch_balanced_merge(const float *part_out, const float *part_lse, const int64_t *pre,
                                  int B, int N, int K, int H, int grid, int KG, uint16_t *out,
                                  float *lse_out, cudaStream_t stream)
{
    balanced_merge_kernel<<<dim3(K, B), kMergeThreads, 0, stream>>>(
        part_out, part_lse, pre, B, N, K, H, grid, KG, reinterpret_cast<__nv_bfloat16 *>(out), lse_out);
    return cudaGetLastError();
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
