// pkv_cols.cuh - the work of one column-parallel attention CTA (several new tokens per sequence,
// or the prefix / suffix passes of shared-prefix decode): which KV head, which block list, which
// query rows ("columns") and which visible-token limit each row has.  Shared by the mma.sync column
// kernel and the tcgen05 column kernel.
#pragma once

#include "pkv_attn_common.cuh"

namespace pkv {

constexpr int kColsPerWarp = 8;
constexpr int kColsPerCta = 32;  // at most 4 groups of 8 rows; the API sizes its chunks by this
static_assert(kConsumerWarps % 4 == 0, "column groups of a CTA must divide its consumer warps");

enum ColsMode { kModeMulti = 0, kModePrefix = 1, kModeSuffix = 2 };

// The work of one CTA (identical in every thread).
struct ColsWork {
    int mode;
    int kvh;
    int b;          // multi / suffix: the sequence; prefix: the group's first member
    int ctx;        // multi / suffix: the sequence's context length
    int vis;        // prefix / suffix: tokens every column sees
    int col_base;   // first column of this CTA's chunk
    int ncols;      // columns of this CTA (1 .. chunk_rows)
    int table_row;  // block-table row the blocks come from
    int blk_begin, blk_end;
    int data_end;   // tokens [0, data_end) of the block list hold data; later slots may be poison
    int slot;       // partition slot of the outputs, -1: final outputs (multi, one pass)
};

// Shared leading blocks of group g, clamped to what the prefix pass covers and the table holds.
__device__ __forceinline__ int prefix_blocks_of(const ColsParams &p, int g)
{
    return max(0, min(p.prefix_blocks[g], min(p.prefix_parts * p.prefix_part_blocks, p.max_nb)));
}

// Group of sequence b: the largest g with group_starts[g] <= b (b outside every group: -1).
__device__ __forceinline__ int group_of(const ColsParams &p, int b)
{
    if (p.num_groups <= 0 || b < p.group_starts[0] || b >= p.group_starts[p.num_groups]) return -1;
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.group_starts[mid] <= b) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Decode CTA c of the grid into its work (kChunkRows: the kernel's query rows per CTA, which the
// caller's p.chunk_rows matches).  Returns false when the CTA has nothing to do.
template <int kChunkRows = kColsPerCta>
__device__ __forceinline__ bool cols_work(const ColsParams &p, int64_t c, ColsWork &w)
{
    const bool first_thread = threadIdx.x == 0;
    w.kvh = (int)(c % p.K);
    c /= p.K;
    if (!p.group_starts) {
        // several new tokens: partitions slowest, highest first (the longest work starts first)
        const int64_t per_part = (int64_t)p.B * p.chunks;
        const int part = p.parts - 1 - (int)(c / per_part);
        c %= per_part;
        const int chunk = (int)(c % p.chunks);
        w.mode = kModeMulti;
        w.b = (int)(c / p.chunks);
        int ctx = p.context_lens[w.b];
        if (ctx < 0 || ctx > p.max_nb * kBlockSize) {
            if (first_thread && w.kvh == 0 && part == 0 && chunk == 0) set_flag(p.err_flag, PKV_FLAG_CTX_RANGE);
            ctx = 0;
        }
        w.ctx = ctx;
        w.vis = ctx;
        w.col_base = chunk * kChunkRows;
        w.ncols = min(kChunkRows, p.T * p.G - w.col_base);
        w.table_row = w.b;
        const int nb = (ctx + kBlockSize - 1) / kBlockSize;
        partition_range(part, partition_count(nb, p.part_blocks, p.taper != 0), nb, p.part_blocks, p.taper != 0,
                        w.blk_begin, w.blk_end);
        w.data_end = ctx;
        w.slot = p.split ? part : -1;
        return w.ncols > 0;
    }
    if (c < p.prefix_ctas / p.K) {
        // prefix pass: (group, prefix partition, chunk) -- the chunks of one partition next to each
        // other, so the CTAs that read the same prefix tiles run together (the tiles stay in L2)
        const int chunk = (int)(c % p.chunks);
        c /= p.chunks;
        const int ppart = (int)(c % p.prefix_parts);
        const int g = (int)(c / p.prefix_parts);
        const int gs_raw = p.group_starts[g], ge_raw = p.group_starts[g + 1];
        const int gs = max(0, min(gs_raw, p.B)), ge = max(gs, min(ge_raw, p.B));
        const int cols = (ge - gs) * p.G;
        int pnb = p.prefix_blocks[g];
        if (first_thread && w.kvh == 0 && ppart == 0 && chunk == p.chunks - 1 &&
            (ge - gs > p.max_group || pnb > p.prefix_parts * p.prefix_part_blocks || pnb < 0 ||
             gs != gs_raw || ge != ge_raw))
            set_flag(p.err_flag, PKV_FLAG_GROUP_RANGE);
        pnb = prefix_blocks_of(p, g);
        w.mode = kModePrefix;
        w.b = gs;
        w.vis = pnb * kBlockSize;
        w.col_base = chunk * kChunkRows;
        w.ncols = min(kChunkRows, cols - w.col_base);
        w.table_row = gs;
        w.blk_begin = ppart * p.prefix_part_blocks;
        w.blk_end = min(pnb, w.blk_begin + p.prefix_part_blocks);
        w.data_end = w.vis;
        w.slot = ppart;
        return w.ncols > 0 && w.blk_begin < w.blk_end;
    }
    // suffix pass: (suffix partition, sequence), partitions slowest and in ascending order: the
    // grid covers the table's whole width, so the partitions past the shorter suffixes (empty
    // CTAs that return at once) come after all the work
    c -= p.prefix_ctas / p.K;
    const int spart = (int)(c / p.B);
    w.mode = kModeSuffix;
    w.b = (int)(c % p.B);
    // the sequence's reporter: flags, and in the fused step the slot of a new token nobody writes
    const bool report = first_thread && w.kvh == 0 && spart == 0;
    int64_t *const no_slot = p.k_new ? p.slot_out : nullptr;
    int ctx = p.context_lens[w.b];
    if (ctx < 0 || ctx > p.max_nb * kBlockSize) {
        if (report) {
            set_flag(p.err_flag, PKV_FLAG_CTX_RANGE);
            if (no_slot) no_slot[w.b] = -1;
        }
        return false;
    }
    const int g = group_of(p, w.b);
    const int pnb = g >= 0 ? prefix_blocks_of(p, g) : 0;
    if (pnb * kBlockSize > ctx) {
        if (report) {
            set_flag(p.err_flag, PKV_FLAG_GROUP_RANGE);
            if (no_slot) no_slot[w.b] = -1;
        }
        return false;
    }
    // fused step: the new token (position ctx - 1) goes into the sequence's own blocks, past the
    // shared ones (writing it into a shared block would change every member's prefix)
    if (report && p.k_new && (ctx == 0 || pnb * kBlockSize == ctx)) {
        if (ctx > 0) set_flag(p.err_flag, PKV_FLAG_GROUP_RANGE);
        if (no_slot) no_slot[w.b] = -1;
    }
    const int nb = (ctx + kBlockSize - 1) / kBlockSize;
    w.ctx = ctx;
    w.vis = ctx;
    w.col_base = 0;
    w.ncols = p.G;
    w.table_row = w.b;
    w.blk_begin = pnb + spart * p.part_blocks;
    w.blk_end = min(nb, w.blk_begin + p.part_blocks);
    w.data_end = ctx;
    // a row's partials are contiguous: its prefix partitions, then its suffix partitions
    w.slot = (pnb + p.prefix_part_blocks - 1) / p.prefix_part_blocks + spart;
    return w.blk_begin < w.blk_end;
}

// Row (of q, out and the partials) and visible-token limit of column j of the CTA.
__device__ __forceinline__ void col_of(const ColsParams &p, const ColsWork &w, int j, int64_t &row,
                                       int &vis)
{
    const int cj = w.col_base + j;
    if (w.mode == kModeMulti) {
        const int t = cj / p.G, g = cj - t * p.G;
        row = ((int64_t)w.b * p.T + t) * p.N + (int64_t)w.kvh * p.G + g;
        vis = w.ctx - p.T + t + 1;
    } else if (w.mode == kModePrefix) {
        const int m = cj / p.G, g = cj - m * p.G;
        row = (int64_t)(w.b + m) * p.N + (int64_t)w.kvh * p.G + g;
        vis = w.vis;
    } else {
        row = (int64_t)w.b * p.N + (int64_t)w.kvh * p.G + cj;
        vis = w.vis;
    }
}

// Fused steps (several new tokens, or the suffix pass of shared-prefix decode with T = 1): right
// before the producer warp loads tile i (logical block blk_begin + i) of a multi-token or suffix
// unit, it writes the new tokens whose positions fall in that block -- token t of the last T sits
// at position ctx - T + t -- from k_new / v_new into their slots (this KV head's H elements of each
// row), fences those writes against the TMA load that follows, and (KV head 0, first chunk)
// records their slots.  The CTAs of the unit's other chunks write the same bytes.  A block id
// outside the pool (flagged by the producer) is not written and its slots are -1.  The same rows
// land where pkv_slot_mapping(_multi) + pkv_append put them.
template <int H>
__device__ __forceinline__ void append_multi_rows(const ColsParams &p, const ColsWork &wk, int64_t i, int bid,
                                                  bool ok, int lane)
{
    if (!p.k_new || wk.mode == kModePrefix) return;
    const int j = wk.blk_begin + (int)i;
    const int first = wk.ctx - p.T;
    const int lo = max(max(first, 0), j * kBlockSize), hi = min(wk.ctx, (j + 1) * kBlockSize);
    if (lo >= hi) return;  // the same on every lane
    if (ok) {
        constexpr int kVec = H / 8;  // 16-byte vectors per row
        const int per = (hi - lo) * kVec;
        for (int idx = lane; idx < 2 * per; idx += 32) {
            const bool is_v = idx >= per;
            const int r = is_v ? idx - per : idx;
            const int pos = lo + r / kVec, c = r % kVec;
            const size_t src = (((size_t)wk.b * p.T + (pos - first)) * p.K + wk.kvh) * H + 8 * c;
            const size_t dst = (((size_t)bid * kBlockSize + pos % kBlockSize) * p.K + wk.kvh) * H + 8 * c;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>((is_v ? p.v_new : p.k_new) + src));
            *reinterpret_cast<uint4 *>((is_v ? p.v_cache_w : p.k_cache_w) + dst) = v;
        }
        fence_proxy_async_global();
    }
    if (p.slot_out && wk.kvh == 0 && wk.col_base == 0)
        for (int pos = lo + lane; pos < hi; pos += 32)
            p.slot_out[(int64_t)wk.b * p.T + (pos - first)] = ok ? (int64_t)bid * kBlockSize + pos % kBlockSize : -1;
    __syncwarp();
}

// Fused multi-token step: slots of new tokens below position 0 (ctx < T) are -1, written by the
// CTAs of the unit's first partition (KV head 0, first chunk), which exist whatever the length.
__device__ __forceinline__ void multi_slots_below_zero(const ColsParams &p, const ColsWork &wk)
{
    if (!p.slot_out || !p.k_new || wk.mode != kModeMulti || wk.kvh != 0 || wk.col_base != 0 || wk.blk_begin != 0)
        return;
    for (int t = threadIdx.x; t < p.T && wk.ctx - p.T + t < 0; t += blockDim.x)
        p.slot_out[(int64_t)wk.b * p.T + t] = -1;
}

// Partitions of a multi-token unit's sequence that hold blocks (the CTAs its merge waits for).
__device__ __forceinline__ int cols_nparts(const ColsParams &p, const ColsWork &w)
{
    const int nb = (w.ctx + kBlockSize - 1) / kBlockSize;
    return partition_count(nb, p.part_blocks, p.taper != 0);
}

// In-kernel log-sum-exp merge of one chunk of a split multi-token unit.  Every CTA of the unit
// calls it once its partials are written (void NaN partials after an expired wait, so the count
// still completes); the last of the nparts CTAs of (sequence, KV head, chunk) to arrive merges the
// chunk's rows with the arithmetic of the separate merge (lse_merge_weights, merge_rows: the same
// bits) and resets the count to zero for the next call.  `smem` is kLseMergeBytes of the CTA's
// shared memory that nothing uses any more.  Rows of one head g are N rows apart from token to
// token, so each merge_rows call takes up to eight tokens of one head.
template <int H>
__device__ void cols_merge_chunk(const ColsParams &p, const ColsWork &wk, int nparts, float *smem, int nthreads)
{
    __shared__ int last_one;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;
    __syncthreads();  // every partial of this CTA is written
    // (the mma.sync column kernel, the only one merging here, always runs 32-row chunks)
    int32_t *count = p.counters + ((int64_t)wk.b * p.K + wk.kvh) * p.chunks + wk.col_base / kColsPerCta;
    if (tid == 0) last_one = atomic_add_acq_rel_gpu(count, 1) == nparts - 1;
    __syncthreads();
    if (!last_one) return;
    const int G = p.G;
    const int tcount = wk.ncols / G;            // tokens of the chunk (a chunk holds whole tokens)
    float *wts = smem;                          // [G][tcount][nparts]
    float *red = smem + kInKernelMergeWeights;  // [kMergeWarps][8][H]
    // the chunk's partial lse first, all loads independent (one round trip), then each row's
    // weights from that copy, in place
    for (int idx = tid; idx < wk.ncols * nparts; idx += nthreads) {
        const int j = idx / nparts, q = idx - j * nparts;
        int64_t row;
        int vis;
        col_of(p, wk, j, row, vis);
        const int tl = j / G, g = j - tl * G;
        wts[((size_t)g * tcount + tl) * nparts + q] = __ldcg(p.part_lse + row * p.max_parts + q);
    }
    __syncthreads();
    for (int j = warp; j < wk.ncols; j += nwarps) {
        int64_t row;
        int vis;
        col_of(p, wk, j, row, vis);
        const int tl = j / G, g = j - tl * G;
        float *wr = wts + ((size_t)g * tcount + tl) * nparts;
        const float L = lse_merge_weights<true>(wr, nparts, wr, lane);
        if (lane == 0 && p.lse_out) p.lse_out[row] = L;
    }
    __syncthreads();
    for (int g = 0; g < G; ++g) {
        for (int t0 = 0; t0 < tcount; t0 += 8) {
            int64_t row;
            int vis;
            col_of(p, wk, t0 * G + g, row, vis);
            merge_rows<H, 8>(wts + ((size_t)g * tcount + t0) * nparts, nparts, min(8, tcount - t0),
                             p.part_out + row * p.max_parts * H, (size_t)p.N * p.max_parts * H, red,
                             p.out + row * H, (size_t)p.N * H, tid, nthreads);
            __syncthreads();  // red is reused by the next rows
        }
    }
    if (tid == 0) *count = 0;  // ready for the next call
}

}  // namespace pkv
