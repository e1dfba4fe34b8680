// pkv_attn_common.cuh - building blocks shared by the attention kernels: ring and tile
// constants, the shared-memory layout, the swizzled tile addressing, the per-warp online-softmax
// state and its tile update (QK^T and PV with mma.sync), the merge of warp states, and the TMA
// producer side of the full/empty mbarrier ring.
#pragma once

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

#ifndef PKV_PRODUCERS
#define PKV_PRODUCERS 2
#endif

#ifndef PKV_FP8_STAGES
#define PKV_FP8_STAGES 16
#endif

#ifndef PKV_CONSUMERS
#define PKV_CONSUMERS 4
#endif
// A grid that fits in one wave at two CTAs per SM leaves the third CTA slot of every SM empty;
// there the bf16 kernel takes a deeper ring at two CTAs per SM instead (more bytes in flight per
// CTA for the same bytes per SM): the 20-sequence shared-prompt batch, 160 CTAs, 30.5 -> 26.6 us.
#ifndef PKV_STAGES_DEEP
#define PKV_STAGES_DEEP 12
#endif
constexpr int kConsumerWarps = PKV_CONSUMERS;
constexpr int kStages = PKV_STAGES;
constexpr int kStagesDeep = PKV_STAGES_DEEP;
constexpr int kStagesFp8 = PKV_FP8_STAGES;  // e4m3 tiles are half the bytes: twice the depth
constexpr int kProducers = PKV_PRODUCERS;
constexpr int kAttnThreads = (kConsumerWarps + kProducers) * 32;
// Stage s is reused by tiles s, s+S, s+2S, ... and tile i goes to consumer warp i % W.  With
// S a multiple of W every use of a stage belongs to the same warp, so a warp only waits for a
// stage's next phase after it consumed the previous one and mbarrier parities cannot alias.
// The same holds for the producer warps (producer p issues tiles i = p mod P).
static_assert(kStages % kConsumerWarps == 0, "pipeline depth must be a multiple of the consumer warps");
static_assert(kStages % kProducers == 0, "pipeline depth must be a multiple of the producer warps");
static_assert(kStagesFp8 % kConsumerWarps == 0 && kStagesFp8 % kProducers == 0,
              "pipeline depth must be a multiple of the consumer and producer warps");
static_assert(kStagesDeep % kConsumerWarps == 0 && kStagesDeep % kProducers == 0,
              "pipeline depth must be a multiple of the consumer and producer warps");

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
    // in-kernel partition merge: weights [G][parts] then the warps' sums [kMergeWarps][8][H]
    static constexpr int kLseMergeBytes = kInKernelMergeWeights * 4 + kMergeWarps * 8 * H * 4;
    // single-pass / partition kernel: the merge areas reuse the drained pipeline
    static constexpr int kMergeMax = kMergeBytes > kLseMergeBytes ? kMergeBytes : kLseMergeBytes;
    static constexpr int kDataBytes = kPipeBytes > kMergeMax ? kPipeBytes : kMergeMax;
    static constexpr int kBarOffset = kDataBytes;           // full[S], empty[S]
    static constexpr int kMiscOffset = kBarOffset + 2 * S * 8;  // slot_ok[S], abort, issued[P]
    // e4m3 with per-(block, head) scales: the (K, V) scales of each stage's tile, float2[S]
    static constexpr int kScaleOffset = (kMiscOffset + (S + 1 + P) * 4 + 7) / 8 * 8;
    static constexpr int kBytes = kScaleOffset + S * 8;
    static constexpr int kAlloc = kBytes + 1024;             // slack for 1024-byte alignment
    static_assert(kPipeBytes % 1024 == 0, "shared-memory layout alignment");
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
    const uint32_t p01 = pack_bf16x2(exp2_sfu(x0 - a.m[0]), exp2_sfu(x1 - a.m[1]));
    const uint32_t p23 = pack_bf16x2(exp2_sfu(x2 - a.m[0]), exp2_sfu(x3 - a.m[1]));
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

// Reference V scale of a warp's e4m3 tiles with one scale per (physical block, KV head).  The
// warp's O holds sum_t w_t (vs_t / v) code_t, so its output is O * v / l.  v is the largest V scale
// the warp has seen (0 before its first tile): when a tile's scale exceeds it, O is rescaled by
// v / vs_t and v moves up, as the running maximum of the logits does.  Every tile's ratio vs_t / v
// is then at most 1 and its f16 weights at most 2^8, whatever the spread of the caller's scales;
// the running sum l takes the unscaled fp32 weights, so a tiny ratio (weights that round to f16
// subnormals or zero) costs at most that tile's tiny V values, never the normaliser.
struct VScaleRef {
    float v;    // largest V scale seen so far (0: none yet)
    float inv;  // 1 / v (0 before the first tile)
};

// One 16-token e4m3 tile folded into a warp's state (the codes only: the tile's K scale is folded
// into sl2).  kBS: per-(block, head) scales -- the tile's V scale vs_t enters through vr (above);
// otherwise the head's V scale multiplies the output at the end and vs_t / vr are unused.
template <int H, bool kBS = false>
__device__ __forceinline__ void tile_update_fp8(WarpAcc<H> &a, const uint32_t (&qf)[H / 16][2],
                                                uint32_t kt, uint32_t vt, int valid, float sl2, float vs_t,
                                                VScaleRef &vr, int lane)
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
        if constexpr (kBS) {  // (per-half conversions: the register allocation measured faster here)
            a0[0] = e4m3x2_to_f16x2((uint16_t)(r[0] & 0xFFFFu));
            a0[1] = e4m3x2_to_f16x2((uint16_t)(r[1] & 0xFFFFu));
            a0[2] = e4m3x2_to_f16x2((uint16_t)(r[0] >> 16));
            a0[3] = e4m3x2_to_f16x2((uint16_t)(r[1] >> 16));
            a1[0] = e4m3x2_to_f16x2((uint16_t)(r[2] & 0xFFFFu));
            a1[1] = e4m3x2_to_f16x2((uint16_t)(r[3] & 0xFFFFu));
            a1[2] = e4m3x2_to_f16x2((uint16_t)(r[2] >> 16));
            a1[3] = e4m3x2_to_f16x2((uint16_t)(r[3] >> 16));
        } else {
            e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
            e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
            e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
            e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
        }
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
    const bool needV = kBS && vs_t > vr.v;  // one value per tile: warp-uniform
    if (__any_sync(0xFFFFFFFFu, needA || needB) || needV) {
        float alphaA = needA ? exp2_sfu(a.m[0] - mA) : 1.f;
        float alphaB = needB ? exp2_sfu(a.m[1] - mB) : 1.f;
        if (needA) a.m[0] = mA;
        if (needB) a.m[1] = mB;
        a.l[0] *= alphaA;
        a.l[1] *= alphaB;
        if (needV) {  // O moves to the new reference scale; l counts unscaled weights
            const float f = vr.v / vs_t;
            alphaA *= f;
            alphaB *= f;
            vr.v = vs_t;
            vr.inv = 1.f / vs_t;
        }
#pragma unroll
        for (int mt = 0; mt < kKSteps; ++mt) {
            a.o[mt][0] *= alphaA;
            a.o[mt][1] *= alphaB;
            a.o[mt][2] *= alphaA;
            a.o[mt][3] *= alphaB;
        }
    }
    const float w0 = exp2_sfu(x0 - a.m[0]), w1 = exp2_sfu(x1 - a.m[1]);
    const float w2 = exp2_sfu(x2 - a.m[0]), w3 = exp2_sfu(x3 - a.m[1]);
    const float vsr = kBS ? vs_t * vr.inv : 1.f;  // <= 1 (+ rounding)
    const uint32_t p01 = pack_f16x2(w0 * vsr, w1 * vsr);
    const uint32_t p23 = pack_f16x2(w2 * vsr, w3 * vsr);
    if constexpr (kBS) {
        a.l[0] += w0 + w2;
        a.l[1] += w1 + w3;
    } else {  // sums of the rounded weights: the weighted average is exactly normalised
        a.l[0] += f16x2_lo(p01) + f16x2_lo(p23);
        a.l[1] += f16x2_hi(p01) + f16x2_hi(p23);
    }
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
            if constexpr (kBS) {
                av[0] = e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu));
                av[1] = e4m3x2_to_f16x2((uint16_t)(lo >> 16));
                av[2] = e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu));
                av[3] = e4m3x2_to_f16x2((uint16_t)(hi >> 16));
            } else {
                e4m3x4_to_f16x2x2(lo, av[0], av[1]);
                e4m3x4_to_f16x2x2(hi, av[2], av[3]);
            }
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

// NT e4m3 tiles (each 16 tokens, the first valid[t] of them count) folded into a warp's state in
// one step: the NT QK^T chains are independent, one max / rescale covers all 16 NT tokens, then
// the NT PV products accumulate.  A warp that takes two of its tiles at once has two
// independent dependency chains in flight where one tile's chain would leave it waiting.  A
// column that has seen no key keeps m = -inf and gets zero weights.  The caller skips a step in
// which no tile has a valid token.
// kBS: per-tile logit multipliers sl2[t] and V scales vs[t] (0 for a tile without valid tokens),
// the V scales entering through vr as in tile_update_fp8; otherwise sl2[0] for every tile.
template <int H, int NT, bool kBS = false>
__device__ __forceinline__ void tile_update_fp8_n(WarpAcc<H> &a, const uint32_t (&qf)[H / 16][2],
                                                  const uint32_t (&kt)[NT], const uint32_t (&vt)[NT],
                                                  const int (&valid)[NT], const float (&sl2)[NT],
                                                  const float (&vs)[NT], VScaleRef &vr, int lane)
{
    constexpr int kKSteps = H / 16;
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = ri + 8 * (mi & 1), coff = mi >> 1;
    const int t0 = lane >> 2, t1 = t0 + 8;

    // S^T = K . Q^T for each tile
    float x[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < kKSteps; kk += 2) {
            uint32_t r[4];
            ldsm_x4(r, kt[t] + fp8_chunk_offset(tok, kk + coff));
            uint32_t a0[4], a1[4];
            if constexpr (kBS) {  // (as in tile_update_fp8)
                a0[0] = e4m3x2_to_f16x2((uint16_t)(r[0] & 0xFFFFu));
                a0[1] = e4m3x2_to_f16x2((uint16_t)(r[1] & 0xFFFFu));
                a0[2] = e4m3x2_to_f16x2((uint16_t)(r[0] >> 16));
                a0[3] = e4m3x2_to_f16x2((uint16_t)(r[1] >> 16));
                a1[0] = e4m3x2_to_f16x2((uint16_t)(r[2] & 0xFFFFu));
                a1[1] = e4m3x2_to_f16x2((uint16_t)(r[3] & 0xFFFFu));
                a1[2] = e4m3x2_to_f16x2((uint16_t)(r[2] >> 16));
                a1[3] = e4m3x2_to_f16x2((uint16_t)(r[3] >> 16));
            } else {
                e4m3x4_to_f16x2x2(r[0], a0[0], a0[2]);
                e4m3x4_to_f16x2x2(r[1], a0[1], a0[3]);
                e4m3x4_to_f16x2x2(r[2], a1[0], a1[2]);
                e4m3x4_to_f16x2x2(r[3], a1[1], a1[3]);
            }
            mma_f16_16816(sa, a0, qf[kk][0], qf[kk][1]);
            mma_f16_16816(sb, a1, qf[kk + 1][0], qf[kk + 1][1]);
        }
        const float m_t = sl2[kBS ? t : 0];
        x[t][0] = t0 < valid[t] ? (sa[0] + sb[0]) * m_t : -INFINITY;
        x[t][1] = t0 < valid[t] ? (sa[1] + sb[1]) * m_t : -INFINITY;
        x[t][2] = t1 < valid[t] ? (sa[2] + sb[2]) * m_t : -INFINITY;
        x[t][3] = t1 < valid[t] ? (sa[3] + sb[3]) * m_t : -INFINITY;
    }
    float mA = -INFINITY, mB = -INFINITY;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        mA = fmaxf(mA, fmaxf(x[t][0], x[t][2]));
        mB = fmaxf(mB, fmaxf(x[t][1], x[t][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(0xFFFFFFFFu, mA, off));
        mB = fmaxf(mB, __shfl_xor_sync(0xFFFFFFFFu, mB, off));
    }
    float vmax = 0.f;
    if constexpr (kBS) {
#pragma unroll
        for (int t = 0; t < NT; ++t) vmax = fmaxf(vmax, vs[t]);
    }
    const bool needA = mA > a.m[0] + kRescaleThreshold;
    const bool needB = mB > a.m[1] + kRescaleThreshold;
    const bool needV = kBS && vmax > vr.v;  // warp-uniform
    if (__any_sync(0xFFFFFFFFu, needA || needB) || needV) {
        float alphaA = needA ? exp2_sfu(a.m[0] - mA) : 1.f;
        float alphaB = needB ? exp2_sfu(a.m[1] - mB) : 1.f;
        if (needA) a.m[0] = mA;
        if (needB) a.m[1] = mB;
        a.l[0] *= alphaA;
        a.l[1] *= alphaB;
        if (needV) {
            const float f = vr.v / vmax;
            alphaA *= f;
            alphaB *= f;
            vr.v = vmax;
            vr.inv = 1.f / vmax;
        }
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
    uint32_t pb[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const float r_t = kBS ? vs[t] * vr.inv : 1.f;
        const float w0 = exp2_sfu(x[t][0] - baseA), w1 = exp2_sfu(x[t][1] - baseB);
        const float w2 = exp2_sfu(x[t][2] - baseA), w3 = exp2_sfu(x[t][3] - baseB);
        const uint32_t p01 = pack_f16x2(w0 * r_t, w1 * r_t);
        const uint32_t p23 = pack_f16x2(w2 * r_t, w3 * r_t);
        if constexpr (kBS) {
            a.l[0] += w0 + w2;
            a.l[1] += w1 + w3;
        } else {
            a.l[0] += f16x2_lo(p01) + f16x2_lo(p23);
            a.l[1] += f16x2_hi(p01) + f16x2_hi(p23);
        }
        pb[t][0] = movmatrix_trans(p01);
        pb[t][1] = movmatrix_trans(p23);
    }

    // O^T += V^T . P^T for each tile (see tile_update_fp8 for the byte regrouping)
    const int tc = (lane & 3) * 2;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const bool partial = valid[t] < kBlockSize;
#pragma unroll
        for (int mt = 0; mt < kKSteps; mt += 2) {
            uint32_t r[4];
            ldsm_x4_trans(r, vt[t] + fp8_chunk_offset(tok, mt + coff));
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t lo = byte_perm(r[2 * hf], 0u, 0x3120u);
                const uint32_t hi = byte_perm(r[2 * hf + 1], 0u, 0x3120u);
                uint32_t av[4];
                if constexpr (kBS) {
                    av[0] = e4m3x2_to_f16x2((uint16_t)(lo & 0xFFFFu));
                    av[1] = e4m3x2_to_f16x2((uint16_t)(lo >> 16));
                    av[2] = e4m3x2_to_f16x2((uint16_t)(hi & 0xFFFFu));
                    av[3] = e4m3x2_to_f16x2((uint16_t)(hi >> 16));
                } else {
                    e4m3x4_to_f16x2x2(lo, av[0], av[1]);
                    e4m3x4_to_f16x2x2(hi, av[2], av[3]);
                }
                if (partial) {
                    const uint32_t lo0 = tc < valid[t] ? 0x0000FFFFu : 0u;
                    const uint32_t hi0 = tc + 1 < valid[t] ? 0xFFFF0000u : 0u;
                    const uint32_t lo1 = tc + 8 < valid[t] ? 0x0000FFFFu : 0u;
                    const uint32_t hi1 = tc + 9 < valid[t] ? 0xFFFF0000u : 0u;
                    av[0] &= lo0 | hi0;
                    av[1] &= lo0 | hi0;
                    av[2] &= lo1 | hi1;
                    av[3] &= lo1 | hi1;
                }
                mma_f16_16816(a.o[mt + hf], av, pb[t][0], pb[t][1]);
            }
        }
    }
}

// O *= f (a warp's accumulator moved to other units, e.g. by its V-scale reference before the
// warps' states are merged).
template <int H>
__device__ __forceinline__ void acc_scale_o(WarpAcc<H> &a, float f)
{
#pragma unroll
    for (int mt = 0; mt < H / 16; ++mt) {
        a.o[mt][0] *= f;
        a.o[mt][1] *= f;
        a.o[mt][2] *= f;
        a.o[mt][3] *= f;
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
            const float sc = exp2_sfu(mm[w * 8 + g] - M);
            lsum += sc * ml[w * 8 + g];
            acc += sc * mo[(w * 8 + g) * H + h];
        }
    }
    // No key at all (M = -inf) gives 0 and -inf; a NaN anywhere in the inputs stays NaN.
    val = M != -INFINITY ? acc / lsum : 0.f;
    lse = M != -INFINITY ? (M + log2f(lsum)) * kLn2 : -INFINITY;
}

// Log-sum-exp weights of one output row's n partial results (natural-log lse_q; -inf for a part
// without keys): M = max_q lse_q, L = M + ln sum_q exp(lse_q - M), w_q = exp(lse_q - L), all
// zero and L = -inf when M = -inf.  Called by one whole warp (lanes stride the parts, shuffles
// reduce); writes w[0..n) and returns L on every lane.  The merged output is sum_q w_q o_q.
// kShared: lp is a copy in shared memory (plain loads; the arithmetic, hence the bits, are the
// same), and w may be lp itself (each lane reads its q's last before it writes them).
template <bool kShared = false>
__device__ __forceinline__ float lse_merge_weights(const float *lp, int n, float *w, int lane)
{
    auto ld = [&](int q) { return kShared ? lp[q] : __ldcg(lp + q); };
    float M = -INFINITY;
    for (int q = lane; q < n; q += 32) M = fmaxf(M, ld(q));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    float L = -INFINITY;
    if (M != -INFINITY) {
        float sum = 0.f;
        for (int q = lane; q < n; q += 32) sum += expf(ld(q) - M);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
        L = M + logf(sum);
    }
    for (int q = lane; q < n; q += 32) w[q] = L == -INFINITY ? 0.f : expf(ld(q) - L);
    __syncwarp();
    return L;
}

// sum_q w_q o_q for one element h of a row whose partials are po[q * stride] (independent loads).
__device__ __forceinline__ float lse_merge_value(const float *w, const float *po, int n, size_t stride)
{
    float val = 0.f;
#pragma unroll 4
    for (int q = 0; q < n; ++q) val += w[q] * __ldcg(po + (size_t)q * stride);
    return val;
}

// Partitions of a sequence of nb blocks, and the blocks [begin, end) of partition `part`.
// Uniform: ceil(nb / pb) partitions, partition p covering [p * pb, (p + 1) * pb) clipped to nb.
// Tapered (pb >= 2): partition 0, which the split grid launches last, covers [0, pb / 2) and
// partition p >= 1 covers [pb / 2 + (p - 1) * pb, pb / 2 + p * pb), clipped to nb -- one
// partition more than uniform at most, and the grid's final wave is made of half-length CTAs.
// Partitions at or past the count are empty.
__device__ __forceinline__ int partition_count(int nb, int pb, bool taper)
{
    if (nb <= 0) return 0;
    const int h = pb / 2;
    return !taper ? (nb + pb - 1) / pb : (nb <= h ? 1 : 1 + (nb - h + pb - 1) / pb);
}

// First block of partition `part` whatever the sequence's length (partition_range's begin for a
// partition that holds blocks).
__device__ __forceinline__ int partition_first_block(int part, int pb, bool taper)
{
    return !taper ? part * pb : (part == 0 ? 0 : pb / 2 + (part - 1) * pb);
}

__device__ __forceinline__ void partition_range(int part, int nparts, int nb, int pb, bool taper, int &begin,
                                                int &end)
{
    if (part >= nparts) {
        begin = end = nb;
        return;
    }
    const int h = pb / 2;
    begin = !taper ? part * pb : (part == 0 ? 0 : h + (part - 1) * pb);
    end = min(nb, !taper ? begin + pb : (part == 0 ? h : begin + pb));
}

// out[g][h] = sum_q w[g * n + q] * po[g * po_row + q * H + h] for nrows <= kMaxRows rows, in an
// order that depends on nothing but n: merge slot w (< kMergeWarps) adds the partitions q = w,
// w + kMergeWarps, ... in increasing q with fused multiply-adds, lane l holding the row's elements
// [l * H / 32, (l + 1) * H / 32) from one vector load per partition (all of a slot's loads are
// independent, so they are in flight together); the slots' sums, staged in red
// [kMergeWarps][kMaxRows][H], are then added in slot order.  Warp w takes the slots w, w + W, ...
// of the CTA's W warps, so a CTA merging one row and one merging eight, with five warps or six,
// give the same bits.  Ends with the rows written (bf16) and a __syncthreads between the two
// phases.
template <int H, int kMaxRows>
__device__ __forceinline__ void merge_rows(const float *w, int n, int nrows, const float *po, size_t po_row,
                                           float *red, __nv_bfloat16 *out, size_t out_row, int tid, int nthreads)
{
    constexpr int E = H / 32;
    static_assert(E == 2 || E == 4, "H = 64 or 128");
    const int warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
    for (int slot = warp; slot < kMergeWarps; slot += nwarps) {
        float acc[kMaxRows][E];
#pragma unroll
        for (int g = 0; g < kMaxRows; ++g)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
        for (int q = slot; q < n; q += kMergeWarps) {
#pragma unroll
            for (int g = 0; g < kMaxRows; ++g) {
                if (g < nrows) {
                    const float wq = w[g * n + q];
                    const float *src = po + g * po_row + (size_t)q * H + lane * E;
                    if constexpr (E == 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                        acc[g][0] = __fmaf_rn(wq, v.x, acc[g][0]);
                        acc[g][1] = __fmaf_rn(wq, v.y, acc[g][1]);
                        acc[g][2] = __fmaf_rn(wq, v.z, acc[g][2]);
                        acc[g][3] = __fmaf_rn(wq, v.w, acc[g][3]);
                    } else {
                        const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                        acc[g][0] = __fmaf_rn(wq, v.x, acc[g][0]);
                        acc[g][1] = __fmaf_rn(wq, v.y, acc[g][1]);
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < kMaxRows; ++g)
            if (g < nrows)
#pragma unroll
                for (int e = 0; e < E; ++e) red[(slot * kMaxRows + g) * H + lane * E + e] = acc[g][e];
    }
    __syncthreads();
    for (int idx = tid; idx < nrows * H; idx += nthreads) {
        const int g = idx / H, h = idx - g * H;
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < kMergeWarps; ++ww) v += red[(ww * kMaxRows + g) * H + h];
        out[g * out_row + h] = __float2bfloat16_rn(v);
    }
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
                                             int tok_major, int32_t *err_flag, uint64_t wait_ns,
                                             volatile float2 *stage_scale = nullptr, float2 scales = {})
{
    using L = AttnLayout<H, S, kConsumerWarps, kProducers, kFp8 ? 1 : 2>;
    const int s = (int)(i % S);
    if (i >= S &&
        !mbar_wait_bounded(bar_empty + 8 * s, (uint32_t)(((i / S) & 1) ^ 1), abort_flag, wait_ns)) {
        if (!*abort_flag) set_flag(err_flag, PKV_FLAG_TIMEOUT);
        *abort_flag = 1;
        return false;
    }
    // the tile's scales, once the stage is free and before its barrier can complete
    if (stage_scale) {
        stage_scale[s].x = scales.x;
        stage_scale[s].y = scales.y;
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
// current ones are issued), `aux(bid)` a per-block value fetched along with it (in-range ids
// only; e.g. the block's e4m3 scales), and `issue(i, bid, ok, aux)` waits for the stage and
// loads it, returning false when its wait expired.  Returns the number of tiles this producer
// issued (on lane 0).
struct NoAux {
    __device__ __forceinline__ float2 operator()(int) const { return make_float2(0.f, 0.f); }
};

struct NoBefore {
    __device__ __forceinline__ void operator()(int64_t, int, bool) const {}
};

// `first` (have_first): lookup(pw + P * lane) already loaded by the caller -- a caller that knows
// its table row before its tile count issues these loads early, overlapping their round trip with
// whatever the count waits for.  `before(i, bid, ok)` runs on the whole warp right before lane 0
// issues tile i (e.g. to write new rows into the block that tile i then loads).
template <int P, bool kAux = false, typename Lookup, typename Issue, typename Aux = NoAux,
          typename Before = NoBefore>
__device__ __forceinline__ int64_t run_producer(int pw, int lane, int64_t n, Lookup lookup,
                                                int num_blocks, int32_t *err_flag, Issue issue, Aux aux = Aux(),
                                                bool have_first = false, int first = 0, Before before = Before())
{
    const int64_t mine = n > pw ? (n - pw + P - 1) / P : 0;
    auto fetch = [&](int bid) {
        if constexpr (kAux) return bid >= 0 && bid < num_blocks ? aux(bid) : make_float2(0.f, 0.f);
        return make_float2(0.f, 0.f);
    };
    int cur = lane < mine ? (have_first ? first : lookup(pw + (int64_t)P * lane)) : 0;
    float2 cur_aux = lane < mine ? fetch(cur) : make_float2(0.f, 0.f);
    int64_t issued = 0;
    bool aborted = false;
    for (int64_t k0 = 0; k0 < mine && !aborted; k0 += 32) {
        const bool more = k0 + 32 + lane < mine;
        const int nxt = more ? lookup(pw + (int64_t)P * (k0 + 32 + lane)) : 0;
        const float2 nxt_aux = more ? fetch(nxt) : make_float2(0.f, 0.f);
        const int cnt = (int)min((int64_t)32, mine - k0);
        const bool bad = lane < cnt && (cur < 0 || cur >= num_blocks);
        const unsigned badmask = __ballot_sync(0xFFFFFFFFu, bad);
        if (badmask && lane == 0) set_flag(err_flag, PKV_FLAG_BLOCK_RANGE);
        for (int k = 0; k < cnt; ++k) {
            const int bid = __shfl_sync(0xFFFFFFFFu, cur, k);
            float2 a = make_float2(0.f, 0.f);
            if constexpr (kAux) a = make_float2(__shfl_sync(0xFFFFFFFFu, cur_aux.x, k), __shfl_sync(0xFFFFFFFFu, cur_aux.y, k));
            int lane0_abort = 0;
            before(pw + (int64_t)P * (k0 + k), bid, !((badmask >> k) & 1u));
            if (lane == 0) {
                if (issue(pw + (int64_t)P * (k0 + k), bid, !((badmask >> k) & 1u), a))
                    ++issued;
                else
                    lane0_abort = 1;
            }
            aborted = __shfl_sync(0xFFFFFFFFu, lane0_abort, 0) != 0;
            if (aborted) break;
        }
        cur = nxt;
        cur_aux = nxt_aux;
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

}  // namespace pkv
