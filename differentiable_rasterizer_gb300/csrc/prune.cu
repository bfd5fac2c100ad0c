// prune.cu -- gs_prune_tiles: hardware-aware pruning of the sorted per-tile
// lists (ByteSplat, English abstract: pruning that weighs rendering quality
// against the per-tile shared-memory budget).
//
// Rule: a tile list longer than the budget K keeps its K most opaque entries
// (opacity = the projected o, record float 5; equal opacities go to the entry
// earlier in the list, i.e. the nearer one) and stays in depth order.
//
// One CTA per (view, tile); tiles within the budget return at once.  A longer
// list needs the K-th largest opacity o* (positive floats order like their bit
// patterns), then keeps every entry with o > o* and the first K - #(o > o*)
// entries with o == o*, compacting the ids in place (an entry never moves to a
// later slot).  The range end becomes start + K.
//   Lists up to 4096 entries: each thread holds 16 consecutive entries in
//   registers; o* is built one bit at a time from block-wide counts, and the
//   kept entries are placed by two block scans (ties, then kept counts).
//   Longer lists: 8-bit radix select passes with shared-memory histograms, then
//   an ordered compaction 256 entries at a time (each chunk read completely
//   before any of it is written).
#include "gs_common.cuh"

namespace gs {

constexpr int kPruneThreads = 256;
constexpr int kPer = 16;                             // register path: entries per thread
constexpr int kRegMax = kPruneThreads * kPer;        // lists up to 4096 entries

// Block-wide sum / exclusive scan of one int per thread.  `buf` alternates
// between two shared arrays so consecutive calls need one barrier each.
__device__ __forceinline__ int block_sum(int v, int (*s_red)[kPruneThreads / 32], int& buf)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[buf][warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kPruneThreads / 32; ++w) t += s_red[buf][w];
    buf ^= 1;
    return t;
}

__device__ __forceinline__ int block_excl_scan(int v, int (*s_red)[kPruneThreads / 32], int& buf)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) s_red[buf][warp] = incl;
    __syncthreads();
    int off = 0;
#pragma unroll
    for (int w = 0; w < kPruneThreads / 32; ++w)
        if (w < warp) off += s_red[buf][w];
    buf ^= 1;
    return off + incl - v;
}

__global__ void __launch_bounds__(kPruneThreads) prune_tiles_kernel(const float4* __restrict__ rec, int64_t n,
                                                                   uint32_t* ids, uint2* ranges, int32_t budget)
{
    __shared__ int s_red[2][kPruneThreads / 32];
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_sel[2];   // selected prefix, entries still needed at it

    const size_t ri = (size_t)blockIdx.y * gridDim.x + blockIdx.x;   // ranges are [view][tile]
    const uint2 range = ranges[ri];
    const int64_t len = (int64_t)range.y - (int64_t)range.x;
    if (!GS_IN_RANGE(len, 1ll << 32, GS_CHECK_RANGE)) return;
    if (len <= budget) return;
    const int v = blockIdx.y;
    const size_t lo = range.x;
    const float4* __restrict__ recv = rec + (size_t)v * (size_t)n * 3;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int buf = 0;

    if (len <= kRegMax) {
        // Register path: thread t holds entries 16 t .. 16 t + 15 (ids and opacity bits).
        uint32_t g[kPer], b[kPer];
        const int64_t k0 = (int64_t)threadIdx.x * kPer;
        const int nv = (int)max((int64_t)0, min((int64_t)kPer, len - k0));   // valid entries of this thread
#pragma unroll
        for (int i = 0; i < kPer; ++i) g[i] = i < nv ? ids[lo + k0 + i] : 0u;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            b[i] = (i < nv && GS_IN_RANGE(g[i], n, GS_CHECK_PRUNE_ID)) ? __float_as_uint(__ldg(recv + (size_t)g[i] * 3 + 1).y)
                                                                     : 0u;
        // largest T with #(o >= T) >= budget, one bit at a time (bit 31, the sign, is 0): T = o*
        uint32_t T = 0;
        for (int bit = 30; bit >= 0; --bit) {
            const uint32_t cand = T | (1u << bit);
            int c = 0;
#pragma unroll
            for (int i = 0; i < kPer; ++i) c += (i < nv && b[i] >= cand) ? 1 : 0;
            if (block_sum(c, s_red, buf) >= budget) T = cand;
        }
        int gt = 0, ties = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            gt += (i < nv && b[i] > T) ? 1 : 0;
            ties += (i < nv && b[i] == T) ? 1 : 0;
        }
        const int need = budget - block_sum(gt, s_red, buf);   // ties kept, nearest first
        int tie_rank = block_excl_scan(ties, s_red, buf);
        uint32_t keep = 0;
        int nkeep = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            bool k = false;
            if (i < nv) {
                if (b[i] > T) k = true;
                else if (b[i] == T) k = tie_rank++ < need;
            }
            keep |= (k ? 1u : 0u) << i;
            nkeep += k ? 1 : 0;
        }
        int out = block_excl_scan(nkeep, s_red, buf);   // every read above precedes these writes
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if ((keep >> i) & 1u) ids[lo + out++] = g[i];
        if (threadIdx.x == 0) ranges[ri] = make_uint2(range.x, range.x + (uint32_t)budget);
        return;
    }

    // Long lists: radix select of the budget-th largest opacity bit pattern, 8 bits a
    // pass, gathering the opacities again each pass.
    auto obits = [&](int64_t k) -> uint32_t {
        const uint32_t gid = ids[lo + k];
        if (!GS_IN_RANGE(gid, n, GS_CHECK_PRUNE_ID)) return 0u;
        return __float_as_uint(__ldg(recv + (size_t)gid * 3 + 1).y);
    };
    uint32_t prefix = 0, need = (uint32_t)budget;
    for (int shift = 24; shift >= 0; shift -= 8) {
        s_hist[threadIdx.x] = 0u;
        __syncthreads();
        const uint32_t hi_mask = shift == 24 ? 0u : ~((1u << (shift + 8)) - 1u);
        for (int64_t base = 0; base < len; base += kPruneThreads) {
            const int64_t k = base + threadIdx.x;
            const uint32_t bb = k < len ? obits(k) : 0u;
            const bool m = k < len && (bb & hi_mask) == prefix;
            const uint32_t dig = (bb >> shift) & 0xffu;
            // opacities share their top bits: one atomic per distinct digit per warp
            const uint32_t peers = __match_any_sync(0xffffffffu, m ? dig : 0x100u + (uint32_t)lane);
            if (m && lane == __ffs(peers) - 1) atomicAdd(&s_hist[dig], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds digits 255 - 8 l .. 248 - 8 l; the lane whose running count
            // (from the top digit down) crosses `need` walks its eight
            uint32_t h[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = s_hist[255 - 8 * lane - i];
                sum += h[i];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += y;
            }
            const uint32_t excl = incl - sum;
            if (excl < need && need <= incl) {
                uint32_t cum = excl;
                int i = 0;
                for (; i < 7; ++i) {
                    if (cum + h[i] >= need) break;
                    cum += h[i];
                }
                s_sel[0] = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
                s_sel[1] = need - cum;
            }
        }
        __syncthreads();
        prefix = s_sel[0];
        need = s_sel[1];
        __syncthreads();   // s_sel and s_hist are rewritten by the next pass
    }
    const uint32_t othr = prefix;   // o*; `need` entries equal to it are kept

    // ordered compaction: ties ranked by position
    uint32_t ties_before = 0, kept_before = 0;
    for (int64_t base = 0; base < len; base += kPruneThreads) {
        const int64_t k = base + threadIdx.x;
        const bool valid = k < len;
        const uint32_t bb = valid ? obits(k) : 0u;
        const uint32_t gid = valid ? ids[lo + k] : 0u;
        const bool tie = valid && bb == othr;
        const uint32_t tb = __ballot_sync(0xffffffffu, tie);
        if (lane == 0) s_red[0][warp] = __popc(tb);
        __syncthreads();
        uint32_t tie_rank = ties_before + __popc(tb & ((1u << lane) - 1u)), tie_tot = 0;
        for (int w = 0; w < kPruneThreads / 32; ++w) {
            const uint32_t c = s_red[0][w];
            if (w < warp) tie_rank += c;
            tie_tot += c;
        }
        const bool keep = valid && (bb > othr || (tie && tie_rank < need));
        const uint32_t kb = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) s_red[1][warp] = __popc(kb);
        __syncthreads();
        uint32_t out = kept_before + __popc(kb & ((1u << lane) - 1u)), keep_tot = 0;
        for (int w = 0; w < kPruneThreads / 32; ++w) {
            const uint32_t c = s_red[1][w];
            if (w < warp) out += c;
            keep_tot += c;
        }
        if (keep) ids[lo + out] = gid;   // out <= k: this chunk was read above, later chunks are untouched
        ties_before += tie_tot;
        kept_before += keep_tot;
        __syncthreads();   // s_red reused by the next chunk
    }
    if (threadIdx.x == 0) ranges[ri] = make_uint2(range.x, range.x + (uint32_t)budget);
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_prune_tiles(const gs_proj* proj, int64_t n, int32_t n_views, int32_t width, int32_t height,
                                    int32_t budget, uint32_t* ids, uint32_t* tile_ranges, void* stream)
{
    GS_NVTX_RANGE("gs_prune_tiles");
    if (!proj || !tile_ranges || budget < 1 || n < 0 || n > INT32_MAX) return GS_ERR_INVALID_ARG;
    if (n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 || height < 1) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!proj->rec || !ids)) return GS_ERR_INVALID_ARG;
    if (!aligned16(proj->rec)) return GS_ERR_INVALID_ARG;
    const long long tiles = (long long)tiles_x_of(width) * tiles_y_of(height);
    if (tiles > INT32_MAX) return GS_ERR_INVALID_ARG;
    prune_tiles_kernel<<<dim3((unsigned)tiles, (unsigned)n_views), kPruneThreads, 0, (cudaStream_t)stream>>>(
        reinterpret_cast<const float4*>(proj->rec), n, ids, reinterpret_cast<uint2*>(tile_ranges), budget);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
