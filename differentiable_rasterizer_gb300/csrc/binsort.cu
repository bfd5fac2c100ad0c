// binsort.cu -- gs_bin_sort: 16x16 tile binning with (tile, depth) keys and a
// sort, then per-tile ranges of the sorted instance list.
//
// The sort by key = ((v * tiles + tile) << 32) | bits(depth), stable in the
// Gaussian index, is done as a counting sort on the high part followed by a
// sort of every (view, tile) bucket on (bits(depth), index):
//
//   1. count:   block b owns a contiguous range of Gaussians and, view after
//               view, counts their instances per tile in shared memory (native
//               integer atomics); the counts go out tile-major,
//               cnt[(v * tiles + tile) * B + b];
//   2. scan:    one exclusive scan of cnt gives, for every (tile, block), where
//               that block's instances of that tile start in the output;
//   3. stats:   tile ranges, the instance total, the largest bucket and the lists
//               of buckets too large for a warp sort; the totals go to the host
//               (the step's one host synchronisation: capacity check);
//   4. scatter: the same blocks append (bits(depth) << 32 | g) to their slice of
//               every bucket through shared-memory cursors (any order);
//   5. sort:    buckets of <= kWarpCap instances: one warp, bitonic in registers;
//               <= kRegCap: one CTA, bitonic in registers (long strides through
//               shared memory); <= kBigCap: one 1024-thread CTA, the same with
//               4-16 keys per thread;
//               larger: one CTA splits the bucket by key range into kSplit
//               sub-buckets (counting scatter), sorts the small ones as above and
//               splits the large ones again (depth first, at most seven levels).
// Every bucket ends sorted by (bits(depth), g), so the output equals a stable
// radix sort of instances emitted in (view, Gaussian) order.
#include "gs_common.cuh"
#include "scan.cuh"

namespace gs {

constexpr int kBinThreads = 1024;          // count / scatter block size
constexpr int kBinBlocks = 304;            // count / scatter blocks for several views (2 per SM) ...
constexpr int kBinBlocksOneView = 152;     // ... or for a single view (fewer count entries to scan)
constexpr int kBandTiles = 40960;          // shared-memory tile counters per block (160 KB)
constexpr int64_t kMaxCounts = 1 << 26;    // cap on (view, tile, block) count entries
constexpr int kWarpCap = 256;              // bucket sizes sorted by one warp (8 keys per lane)
constexpr int kRegCap = 2048;              // bucket sizes sorted by one 256-thread CTA in registers
constexpr int kRegThreads = 256;
constexpr int kMidThreads = 1024;          // mid-class sort: kMidThreads * 16 = kBigCap keys
constexpr int kBigCap = 16384;             // bucket sizes sorted by one CTA in shared memory
constexpr int kSplit = 1024;               // sub-buckets per split of a larger bucket
constexpr int kStack = 8 * kSplit;         // pending sub-buckets (<= 1023 per level, <= 7 levels)
constexpr int kSortWarps = 8;              // warps per block of the warp-sort kernel

// Partition of the (view, Gaussian) axis and of the tile rows for count/scatter.
struct BinGeom {
    int64_t n;           // Gaussians per view
    int64_t per_block;   // Gaussians per block
    int32_t B;           // blocks (each takes its Gaussian range in every view)
    int32_t views;
    int32_t tiles_x, tiles_y, tiles;
    int32_t band_rows;   // tile rows per block band
};

// -------------------------------------------------------------------- count / scatter
// Block (b, band): Gaussians [b * per_block, (b + 1) * per_block) in tile rows
// [band * band_rows, ...), view after view.  All blocks work on about the same
// view at a time, so the scatter's writes stay within one view's part of the
// output (a few L2-sized regions instead of all views' at once).
template <bool kScatter>
__global__ void __launch_bounds__(kBinThreads) bin_kernel(const uint32_t* __restrict__ touched_cnt,
                                                          const ushort4* __restrict__ rect,
                                                          const float* __restrict__ depth, BinGeom G,
                                                          uint32_t* __restrict__ cnt, uint64_t* __restrict__ tmp,
                                                          unsigned int* __restrict__ stats,
                                                          const unsigned long long* __restrict__ total,
                                                          unsigned long long capacity)
{
    extern __shared__ uint32_t s_cnt[];
    // the scatter runs before the host has seen the instance count: it writes
    // nothing when the count exceeds the caller's capacity
    if (kScatter && *total > capacity) return;
    const int b = blockIdx.x, band = blockIdx.y;
    if (!kScatter && b == 0 && band == 0 && threadIdx.x < 5) stats[threadIdx.x] = 0u;   // bucket_stats, error word
    const int row0 = band * G.band_rows;
    const int row1 = min(G.tiles_y, row0 + G.band_rows);
    const int nt = (row1 - row0) * G.tiles_x;
    const int64_t g0 = (int64_t)b * G.per_block;
    const int64_t g1 = min(G.n, g0 + G.per_block);
    for (int v = 0; v < G.views; ++v) {
        const size_t cbase =
            ((size_t)v * (size_t)G.tiles + (size_t)row0 * (size_t)G.tiles_x) * (size_t)G.B + (size_t)b;
        if (v > 0) __syncthreads();   // the previous view's counters are out of use
        // counters (count) or cursors = this block's start in every bucket (scatter)
        for (int i = threadIdx.x; i < nt; i += blockDim.x) s_cnt[i] = kScatter ? cnt[cbase + (size_t)i * G.B] : 0u;
        __syncthreads();
        const size_t vb = (size_t)v * (size_t)G.n;
        constexpr int U = 4;   // Gaussians in flight per thread
        for (int64_t gb = g0 + threadIdx.x; gb < g1; gb += (int64_t)U * blockDim.x) {
            uint32_t tc[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = gb + (int64_t)u * blockDim.x;
                tc[u] = g < g1 ? __ldg(touched_cnt + vb + g) : 0u;
            }
            ushort4 r[U];
            uint64_t key[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = gb + (int64_t)u * blockDim.x;
                r[u] = tc[u] ? __ldg(rect + vb + g) : make_ushort4(0, 0, 0, 0);
                if (kScatter)
                    key[u] = tc[u] ? (((uint64_t)__float_as_uint(__ldg(depth + vb + g)) << 32) | (uint64_t)g) : 0ull;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!tc[u]) continue;
                if (!(GS_IN_RANGE(r[u].x, r[u].z, GS_CHECK_BIN_RECT) && GS_IN_RANGE(r[u].z - 1, G.tiles_x, GS_CHECK_BIN_RECT) &&
                      GS_IN_RANGE(r[u].y, r[u].w, GS_CHECK_BIN_RECT) && GS_IN_RANGE(r[u].w - 1, G.tiles_y, GS_CHECK_BIN_RECT)))
                    continue;
                const int y0 = max((int)r[u].y, row0), y1 = min((int)r[u].w, row1);
                for (int ty = y0; ty < y1; ++ty) {
                    uint32_t* row = s_cnt + (ty - row0) * G.tiles_x;
                    for (int tx = r[u].x; tx < r[u].z; ++tx) {
                        const uint32_t pos = atomicAdd(row + tx, 1u);
                        if (kScatter && GS_IN_RANGE(pos, capacity, GS_CHECK_BIN_SLOT)) tmp[pos] = key[u];
                    }
                }
            }
        }
        if (!kScatter) {
            __syncthreads();
            for (int i = threadIdx.x; i < nt; i += blockDim.x) cnt[cbase + (size_t)i * G.B] = s_cnt[i];
        }
    }
}

// Per (view, tile): range [start, end) from the scanned counts; stats[0] =
// largest bucket, stats[1..3] = number of buckets listed in lists[0][...]
// (kWarpCap < size <= kRegCap), lists[1][...] (<= kBigCap) and lists[2][...]
// (larger), each list nb long.
__global__ void bucket_stats_kernel(const uint32_t* __restrict__ off, int32_t B, int64_t nb,
                                    const unsigned long long* __restrict__ total, uint2* __restrict__ ranges,
                                    unsigned int* __restrict__ stats, uint32_t* __restrict__ lists)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nb) return;
    const uint32_t s = off[(size_t)t * B];
    const uint32_t e = t + 1 < nb ? off[(size_t)(t + 1) * B] : (uint32_t)*total;
    ranges[t] = make_uint2(s, e);
    const uint32_t c = e - s;
    if (c <= (uint32_t)kWarpCap) return;
    atomicMax(stats, c);
    const int cls = c <= (uint32_t)kRegCap ? 0 : (c <= (uint32_t)kBigCap ? 1 : 2);
    lists[(size_t)cls * nb + atomicAdd(stats + 1 + cls, 1u)] = (uint32_t)t;
}

// -------------------------------------------------------------------- sorts
#ifdef GS_CHECKED
// Gaussian count and instance capacity of the running gs_bin_sort call, for the
// checks at the sorts' output (set by the host before the first launch).
__device__ long long g_sort_limits[2];
#endif

// Sorted keys leave as key = (tile_lin << 32) | bits(depth), value = g.
__device__ __forceinline__ void emit_sorted(uint64_t k, uint64_t hi, uint64_t* __restrict__ keys,
                                            uint32_t* __restrict__ ids, size_t pos)
{
#ifdef GS_CHECKED
    if (!GS_IN_RANGE(pos, g_sort_limits[1], GS_CHECK_SORT_SLOT)) return;
    (void)GS_IN_RANGE((uint32_t)k, g_sort_limits[0], GS_CHECK_SORT_ID);   // written all the same; the raster drops it
#endif
    keys[pos] = hi | (k >> 32);
    ids[pos] = (uint32_t)k;
}

// Bitonic sort of 32 * E keys held by one warp, lane l owning elements
// [l * E, (l + 1) * E): strides below E are register swaps, the others lane
// exchanges.
template <int E>
__device__ __forceinline__ void warp_bitonic(uint64_t (&x)[E])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= E) {
                const int lj = j / E;
                const bool lower = (lane & lj) == 0;
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    const bool up = (((lane * E + r) & k) == 0);
                    const uint64_t y = __shfl_xor_sync(0xffffffffu, x[r], lj);
                    x[r] = (lower == up) ? (y < x[r] ? y : x[r]) : (y > x[r] ? y : x[r]);
                }
            } else {
#pragma unroll
                for (int r = 0; r < E; ++r) {
                    if ((r & j) == 0) {
                        const bool up = (((lane * E + r) & k) == 0);
                        const uint64_t p = x[r], q = x[r | j];
                        if ((p > q) == up) {
                            x[r] = q;
                            x[r | j] = p;
                        }
                    }
                }
            }
        }
    }
}

template <int E>
__device__ __forceinline__ void warp_sort_e(const uint64_t* __restrict__ src, size_t o, int c, uint64_t hi,
                                            uint64_t* __restrict__ keys, uint32_t* __restrict__ ids)
{
    const int lane = threadIdx.x & 31;
    uint64_t x[E];
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int i = lane * E + r;
        x[r] = i < c ? src[o + i] : ~0ull;
    }
    warp_bitonic<E>(x);
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int i = lane * E + r;
        if (i < c) emit_sorted(x[r], hi, keys, ids, o + i);
    }
}

// One warp sorts src[o, o + c), 0 < c <= kWarpCap, into keys / ids at o.
__device__ __forceinline__ void warp_sort(const uint64_t* __restrict__ src, size_t o, int c, uint64_t hi,
                                          uint64_t* __restrict__ keys, uint32_t* __restrict__ ids)
{
    if (c <= 32) warp_sort_e<1>(src, o, c, hi, keys, ids);
    else if (c <= 64) warp_sort_e<2>(src, o, c, hi, keys, ids);
    else if (c <= 128) warp_sort_e<4>(src, o, c, hi, keys, ids);
    else warp_sort_e<8>(src, o, c, hi, keys, ids);
}

// Shared-memory slot of element i in a block-sorted array of E keys per thread
// (one pad word per E keys: blocked and striped accesses stay near conflict free).
template <int E>
__device__ __forceinline__ int pad_slot(int i) { return i + i / E; }

// A kT-thread CTA sorts src[o, o + c), c <= kT * E: thread t
// holds elements [t * E, (t + 1) * E) in registers; strides below E are register
// swaps, strides below 32 E lane exchanges, the rest go through shared memory s
// (kT * (E + 1) keys).
template <int kT, int E, bool kUnroll>
__device__ __forceinline__ void reg_sort(const uint64_t* __restrict__ src, size_t o, int c, uint64_t hi,
                                         uint64_t* __restrict__ keys, uint32_t* __restrict__ ids, uint64_t* s)
{
    constexpr int P = kT * E;
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < P; i += kT) s[pad_slot<E>(i)] = i < c ? src[o + i] : ~0ull;
    __syncthreads();
    uint64_t x[E];
#pragma unroll
    for (int r = 0; r < E; ++r) x[r] = s[pad_slot<E>(tid * E + r)];
    __syncthreads();
    // Small networks are unrolled whole; for large ones (kUnroll = false) the
    // stage loops run at run time and only the register-stride stages (j < E)
    // and the per-key loops are unrolled, so every index into x stays a
    // constant without unrolling thousands of stages.
#pragma unroll(kUnroll ? 16 : 1)
    for (int k = 2; k <= P; k <<= 1) {
        if ((k >> 1) >= 32 * E) {
#pragma unroll
            for (int r = 0; r < E; ++r) s[pad_slot<E>(tid * E + r)] = x[r];
            __syncthreads();
#pragma unroll(kUnroll ? 16 : 1)
            for (int j = k >> 1; j >= 32 * E; j >>= 1) {
                for (int i = tid; i < P; i += kT) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const uint64_t a = s[pad_slot<E>(i)], b = s[pad_slot<E>(ixj)];
                        if ((a > b) == ((i & k) == 0)) {
                            s[pad_slot<E>(i)] = b;
                            s[pad_slot<E>(ixj)] = a;
                        }
                    }
                }
                __syncthreads();
            }
#pragma unroll
            for (int r = 0; r < E; ++r) x[r] = s[pad_slot<E>(tid * E + r)];
            __syncthreads();
        }
#pragma unroll(kUnroll ? 16 : 1)
        for (int j = (k >> 1) < 32 * E ? (k >> 1) : 16 * E; j >= E; j >>= 1) {
            const int lj = j / E;
            const bool lower = (lane & lj) == 0;
#pragma unroll
            for (int r = 0; r < E; ++r) {
                const bool up = (((tid * E + r) & k) == 0);
                const uint64_t y = __shfl_xor_sync(0xffffffffu, x[r], lj);
                x[r] = (lower == up) ? (y < x[r] ? y : x[r]) : (y > x[r] ? y : x[r]);
            }
        }
#pragma unroll
        for (int j = E / 2; j > 0; j >>= 1) {
            if (j > (k >> 1)) continue;
#pragma unroll
            for (int r = 0; r < E; ++r) {
                if ((r & j) == 0) {
                    const bool up = (((tid * E + r) & k) == 0);
                    const uint64_t p = x[r], q = x[r | j];
                    if ((p > q) == up) {
                        x[r] = q;
                        x[r | j] = p;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < E; ++r) s[pad_slot<E>(tid * E + r)] = x[r];
    __syncthreads();
    for (int i = tid; i < c; i += kT) emit_sorted(s[pad_slot<E>(i)], hi, keys, ids, o + i);
}

// Bitonic sort of s[0, P) ascending (P a power of two), all threads of the block.
__device__ __forceinline__ void block_bitonic(uint64_t* s, int P)
{
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < P; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint64_t x = s[i], y = s[ixj];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) {
                        s[i] = y;
                        s[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// All threads of the block sort src[o, o + c), c <= kBigCap, through s.
__device__ __forceinline__ void cta_sort(uint64_t* s, const uint64_t* src, size_t o, int c, uint64_t hi,
                                         uint64_t* __restrict__ keys, uint32_t* __restrict__ ids)
{
    int P = 1;
    while (P < c) P <<= 1;
    for (int i = threadIdx.x; i < P; i += blockDim.x) s[i] = i < c ? src[o + i] : ~0ull;
    __syncthreads();
    block_bitonic(s, P);
    for (int i = threadIdx.x; i < c; i += blockDim.x) emit_sorted(s[i], hi, keys, ids, o + i);
    __syncthreads();
}

// Warp w of the block sorts bucket blockIdx.x * kSortWarps + w if it holds
// 1..kWarpCap instances.
__global__ void __launch_bounds__(kSortWarps * 32) sort_warp_kernel(const uint2* __restrict__ ranges, int64_t nb,
                                                                    const uint64_t* __restrict__ tmp,
                                                                    uint64_t* __restrict__ keys,
                                                                    uint32_t* __restrict__ ids,
                                                                    const unsigned long long* __restrict__ total,
                                                                    unsigned long long capacity)
{
    if (*total > capacity) return;   // launched before the host's capacity check, like the scatter
    const int64_t t = (int64_t)blockIdx.x * kSortWarps + (threadIdx.x >> 5);
    if (t >= nb) return;
    const uint2 r = ranges[t];
    const int c = (int)(r.y - r.x);
    if (c == 0 || c > kWarpCap) return;
    warp_sort(tmp, r.x, c, (uint64_t)t << 32, keys, ids);
}

// Sort of one bucket by key-range slices.  The bucket is split by uniform
// slices of its [min, max] key interval into kT sub-buckets (the monotone digit
// of the huge-bucket splitter below), a counting scatter through shared memory
// puts the sub-buckets in digit order, and each sub-bucket is sorted on its own:
// up to kThreadCap keys by one thread (insertion), larger ones by a warp
// (register bitonic, as for small buckets).  That is O(c) work plus small sorts
// where a bitonic network over the whole bucket needs O(c log^2 c).  Keys are
// unique within a bucket, so the result does not depend on the scatter's order.
constexpr int kThreadCap = 8;
constexpr int kSplitMidCap = 8192;   // mid-class buckets sorted by slices (larger: bitonic)

// One warp sorts s[0, c), c <= 32 E, in place (shared memory).
template <int E>
__device__ __forceinline__ void warp_sort_smem_e(uint64_t* s, int c)
{
    const int lane = threadIdx.x & 31;
    uint64_t x[E];
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int i = lane * E + r;
        x[r] = i < c ? s[i] : ~0ull;
    }
    warp_bitonic<E>(x);
#pragma unroll
    for (int r = 0; r < E; ++r) {
        const int i = lane * E + r;
        if (i < c) s[i] = x[r];
    }
}

__device__ __forceinline__ void warp_sort_smem(uint64_t* s, int c)
{
    if (c <= 32) warp_sort_smem_e<1>(s, c);
    else if (c <= 64) warp_sort_smem_e<2>(s, c);
    else if (c <= 128) warp_sort_smem_e<4>(s, c);
    else warp_sort_smem_e<8>(s, c);
}

template <int kT>
struct SplitSmem {
    uint32_t start[kT], cur[kT], big[kT];   // per slice: size, cursor / start, slices left to warps
    uint64_t red[2][kT / 32];
    uint32_t wsum[kT / 32], wmax[kT / 32];
    uint32_t nbig;
};

// A kT-thread block sorts tmp[o, o + c) into keys / ids at o through s_in and
// s_out (c keys each).  Returns false, having written nothing, when a slice
// holds more than kWarpCap keys (a tight cluster of depths): the caller sorts
// the bucket another way (after a barrier; s_in and s_out are free again).
template <int kT>
__device__ bool split_sort(const uint64_t* __restrict__ tmp, size_t o, int c, uint64_t hi,
                           uint64_t* __restrict__ keys, uint32_t* __restrict__ ids, uint64_t* s_in,
                           uint64_t* s_out, SplitSmem<kT>& S)
{
    constexpr int kW = kT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t kmin = ~0ull, kmax = 0ull;
    for (int i = tid; i < c; i += kT) {
        const uint64_t k = tmp[o + i];
        s_in[i] = k;
        kmin = k < kmin ? k : kmin;
        kmax = k > kmax ? k : kmax;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const uint64_t a = __shfl_xor_sync(0xffffffffu, kmin, d);
        const uint64_t b = __shfl_xor_sync(0xffffffffu, kmax, d);
        kmin = a < kmin ? a : kmin;
        kmax = b > kmax ? b : kmax;
    }
    if (lane == 0) {
        S.red[0][warp] = kmin;
        S.red[1][warp] = kmax;
    }
    S.start[tid] = 0u;
    if (tid == 0) S.nbig = 0u;
    __syncthreads();
    for (int w = 0; w < kW; ++w) {
        kmin = S.red[0][w] < kmin ? S.red[0][w] : kmin;
        kmax = S.red[1][w] > kmax ? S.red[1][w] : kmax;
    }
    // digit(k) = floor((k - kmin) * scale / 2^64): non-decreasing in k, below kT
    const uint64_t range = kmax - kmin;
    const bool direct = range < (uint64_t)kT;
    const uint64_t scale = direct ? 0ull : (~0ull / (range + 1ull)) * (uint64_t)kT;
    auto digit = [&](uint64_t k) -> uint32_t {
        const uint64_t d = k - kmin;
        return direct ? (uint32_t)d : (uint32_t)__umul64hi(d, scale);
    };
    for (int i = tid; i < c; i += kT) atomicAdd(&S.start[digit(s_in[i])], 1u);
    __syncthreads();
    // exclusive scan of the slice sizes, and the largest
    const uint32_t mine = S.start[tid];
    uint32_t incl = mine, mx = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    }
    if (lane == 31) S.wsum[warp] = incl;
    if (lane == 0) S.wmax[warp] = mx;
    __syncthreads();
    uint32_t wpre = 0, bmax = 0;
    for (int w = 0; w < kW; ++w) {
        wpre += w < warp ? S.wsum[w] : 0u;
        bmax = max(bmax, S.wmax[w]);
    }
    if (bmax > (uint32_t)kWarpCap) return false;   // block-uniform
    const uint32_t start = wpre + incl - mine;
    S.cur[tid] = start;
    __syncthreads();
    for (int i = tid; i < c; i += kT) {
        const uint64_t k = s_in[i];
        s_out[atomicAdd(&S.cur[digit(k)], 1u)] = k;
    }
    __syncthreads();
    if (mine > (uint32_t)kThreadCap) {
        S.big[atomicAdd(&S.nbig, 1u)] = tid;   // a slice for a warp
        S.cur[tid] = start;                    // its start (the cursor ended at its end)
    } else {
        // insertion sort of this thread's slice [start, start + mine)
        for (uint32_t a = start + 1; a < start + mine; ++a) {
            const uint64_t k = s_out[a];
            uint32_t b = a;
            while (b > start && s_out[b - 1] > k) {
                s_out[b] = s_out[b - 1];
                --b;
            }
            s_out[b] = k;
        }
    }
    __syncthreads();
    for (uint32_t b = warp; b < S.nbig; b += kW) {
        const uint32_t d = S.big[b];
        warp_sort_smem(s_out + S.cur[d], (int)S.start[d]);   // S.start[d]: the slice's size
    }
    __syncthreads();
    for (int i = tid; i < c; i += kT) emit_sorted(s_out[i], hi, keys, ids, o + i);
    return true;
}

// One kRegThreads-thread CTA per listed bucket of kWarpCap < size <= kRegCap,
// sorted by key-range slices (the block's register bitonic network when a slice
// is too large).  Launched before the host knows the class size: one block per
// possible bucket, the ones past the device-held count (or all, if the capacity
// is short) exit.
__global__ void __launch_bounds__(kRegThreads) sort_reg_kernel(const uint32_t* __restrict__ list,
                                                               const uint2* __restrict__ ranges,
                                                               const uint64_t* __restrict__ tmp,
                                                               uint64_t* __restrict__ keys, uint32_t* __restrict__ ids,
                                                               const unsigned int* __restrict__ count,
                                                               const unsigned long long* __restrict__ total,
                                                               unsigned long long capacity)
{
    __shared__ uint64_t s[kRegThreads * 9];
    __shared__ uint64_t s_out[kRegCap];
    __shared__ SplitSmem<kRegThreads> S;
    if (*total > capacity || blockIdx.x >= *count) return;
    const uint32_t t = list[blockIdx.x];
    const uint2 r = ranges[t];
    const int c = (int)(r.y - r.x);
    const uint64_t hi = (uint64_t)t << 32;
    if (split_sort<kRegThreads>(tmp, r.x, c, hi, keys, ids, s, s_out, S)) return;
    __syncthreads();
    if (c <= 2 * kRegThreads) reg_sort<kRegThreads, 2, true>(tmp, r.x, c, hi, keys, ids, s);
    else if (c <= 4 * kRegThreads) reg_sort<kRegThreads, 4, true>(tmp, r.x, c, hi, keys, ids, s);
    else reg_sort<kRegThreads, 8, true>(tmp, r.x, c, hi, keys, ids, s);
}

// One kMidThreads-thread CTA per listed bucket of kRegCap < size <= kBigCap:
// up to kSplitMidCap instances by key-range slices (the first 2 c keys of the
// dynamic buffer hold the keys and their slice order), otherwise --
// and when a slice is too large -- the register / shuffle / shared-memory
// bitonic with 4, 8 or 16 keys per thread (dynamic shared memory:
// kMidThreads * (E + 1) keys for the largest E).
__global__ void __launch_bounds__(kMidThreads) sort_mid_kernel(const uint32_t* __restrict__ list,
                                                               const uint2* __restrict__ ranges,
                                                               const uint64_t* __restrict__ tmp,
                                                               uint64_t* __restrict__ keys, uint32_t* __restrict__ ids)
{
    extern __shared__ uint64_t s_mid[];
    __shared__ SplitSmem<kMidThreads> S;
    const uint32_t t = list[blockIdx.x];
    const uint2 r = ranges[t];
    const int c = (int)(r.y - r.x);
    const uint64_t hi = (uint64_t)t << 32;
    if (c <= kSplitMidCap) {
        if (split_sort<kMidThreads>(tmp, r.x, c, hi, keys, ids, s_mid, s_mid + c, S)) return;
        __syncthreads();
    }
    if (c <= 4 * kMidThreads) reg_sort<kMidThreads, 4, false>(tmp, r.x, c, hi, keys, ids, s_mid);
    else if (c <= 8 * kMidThreads) reg_sort<kMidThreads, 8, false>(tmp, r.x, c, hi, keys, ids, s_mid);
    else reg_sort<kMidThreads, 16, false>(tmp, r.x, c, hi, keys, ids, s_mid);
}

// Block-wide min / max of 64-bit values (blockDim.x == 1024).
__device__ __forceinline__ void block_minmax(uint64_t& lo, uint64_t& hi, uint64_t* s_red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t a = __shfl_xor_sync(0xffffffffu, lo, o);
        const uint64_t b = __shfl_xor_sync(0xffffffffu, hi, o);
        lo = a < lo ? a : lo;
        hi = b > hi ? b : hi;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        s_red[warp] = lo;
        s_red[32 + warp] = hi;
    }
    __syncthreads();
    lo = s_red[0];
    hi = s_red[32];
    for (int w = 1; w < 32; ++w) {
        lo = s_red[w] < lo ? s_red[w] : lo;
        hi = s_red[32 + w] > hi ? s_red[32 + w] : hi;
    }
    __syncthreads();
}

// Exclusive scan of s[0, 1024) in place by a 1024-thread block.
__device__ __forceinline__ void block_scan_1024(uint32_t* s, uint32_t* s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t x = s[threadIdx.x];
    uint32_t incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t wpre = 0;
    for (int w = 0; w < warp; ++w) wpre += s_warp[w];
    __syncthreads();
    s[threadIdx.x] = wpre + incl - x;
    __syncthreads();
}

// Shared memory of the huge-bucket kernel (dynamic): the block sort area, the
// pending stack, the sub-bucket counters and cursors.
struct HugeSmem {
    uint64_t keys[kBigCap];
    uint2 stack[kStack];          // (offset, count | in_keys_buffer << 31)
    uint32_t hist[kSplit];
    uint32_t cur[kSplit];
    uint64_t red[64];
    uint32_t warp_sums[32];
    int sp;
};

// One 1024-thread CTA per listed bucket of more than kBigCap instances.  A
// range is split by uniform slices of its [min, max] key interval:
// digit(k) = floor((k - min) * s / 2^64) with s = floor((2^64 - 1) / (range + 1))
// * kSplit (or k - min when the range is below kSplit) is non-decreasing in k
// and below kSplit, so the sub-buckets in digit order are in key order.  Each
// level shrinks the key interval by a factor of at least kSplit / 2 and keys are
// unique within a bucket (below 2^63: depth is finite and positive), so at most
// seven levels are ever pending and the stack never holds more than
// 7 * (kSplit - 1) + 1 ranges.
__global__ void __launch_bounds__(1024) sort_huge_kernel(const uint32_t* __restrict__ list,
                                                         const uint2* __restrict__ ranges, uint64_t* tmp,
                                                         uint64_t* keys, uint32_t* __restrict__ ids,
                                                         unsigned int* __restrict__ error)
{
    extern __shared__ __align__(16) unsigned char s_raw[];
    HugeSmem& S = *reinterpret_cast<HugeSmem*>(s_raw);
    const uint32_t t = list[blockIdx.x];
    const uint2 r0 = ranges[t];
    const uint64_t hi_key = (uint64_t)t << 32;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        S.stack[0] = make_uint2(r0.x, r0.y - r0.x);
        S.sp = 1;
    }
    __syncthreads();
    while (S.sp > 0) {
        const uint2 top = S.stack[S.sp - 1];
        __syncthreads();
        if (threadIdx.x == 0) S.sp -= 1;
        const size_t o = top.x;
        const uint32_t c = top.y & 0x7fffffffu;
        const bool in_keys = (top.y >> 31) != 0;
        const uint64_t* src = in_keys ? keys : tmp;
        uint64_t* dst = in_keys ? tmp : keys;
        // key interval of the range
        uint64_t kmin = ~0ull, kmax = 0ull;
        for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
            const uint64_t k = src[o + i];
            kmin = k < kmin ? k : kmin;
            kmax = k > kmax ? k : kmax;
        }
        block_minmax(kmin, kmax, S.red);
        const uint64_t range = kmax - kmin;
        const bool direct = range < (uint64_t)kSplit;
        const uint64_t scale = direct ? 0ull : (~0ull / (range + 1ull)) * (uint64_t)kSplit;
        S.hist[threadIdx.x] = 0u;
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
            const uint64_t d = src[o + i] - kmin;
            atomicAdd(&S.hist[direct ? (uint32_t)d : (uint32_t)__umul64hi(d, scale)], 1u);
        }
        __syncthreads();
        const uint32_t my_cnt = S.hist[threadIdx.x];
        block_scan_1024(S.hist, S.warp_sums);   // hist = sub-bucket starts
        S.cur[threadIdx.x] = S.hist[threadIdx.x];
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < c; i += blockDim.x) {
            const uint64_t k = src[o + i];
            const uint64_t d = k - kmin;
            const uint32_t dig = direct ? (uint32_t)d : (uint32_t)__umul64hi(d, scale);
            dst[o + atomicAdd(&S.cur[dig], 1u)] = k;
        }
        __syncthreads();               // every cursor increment is done
        S.cur[threadIdx.x] = my_cnt;   // sub-bucket sizes
        __syncthreads();               // dst and the sizes are visible to the whole block
        // small sub-buckets: one warp each
        for (int d = warp; d < kSplit; d += 32) {
            const int sc = (int)S.cur[d];
            if (sc > 0 && sc <= kWarpCap) warp_sort(dst, o + S.hist[d], sc, hi_key, keys, ids);
        }
        // medium sub-buckets: the whole block; large ones are pushed
        for (int d = 0; d < kSplit; ++d) {
            const uint32_t sc = S.cur[d];
            if (sc <= (uint32_t)kWarpCap) continue;
            if (sc <= (uint32_t)kBigCap) {
                cta_sort(S.keys, dst, o + S.hist[d], (int)sc, hi_key, keys, ids);
            } else if (threadIdx.x == 0) {
                if (S.sp < kStack) {   // the bound above keeps sp < kStack
                    S.stack[S.sp] = make_uint2((uint32_t)(o + S.hist[d]), sc | (in_keys ? 0u : 0x80000000u));
                    S.sp += 1;
                } else {
                    atomicOr(error, 1u);   // a range left unsorted: reported, never silent
                }
            }
        }
        __syncthreads();
    }
}

// Aligned bump layout of the workspace.
struct WsLayout {
    size_t cnt, off, scan_sums, totals, stats, lists, tmp, bytes;
};

inline size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

inline BinGeom bin_geom(int64_t n, int n_views, int tiles_x, int tiles_y)
{
    BinGeom G;
    G.n = n;
    G.tiles_x = tiles_x;
    G.tiles_y = tiles_y;
    G.tiles = tiles_x * tiles_y;
    const int64_t ntile_ids = (int64_t)G.tiles * n_views;
    G.views = n_views;
    int64_t B = n_views == 1 ? kBinBlocksOneView : kBinBlocks;
    if (B * ntile_ids > kMaxCounts) B = kMaxCounts / ntile_ids;
    if (B > n) B = n;
    if (B < 1) B = 1;
    G.per_block = (n + B - 1) / B;
    if (G.per_block < 1) G.per_block = 1;
    G.B = (int32_t)((n + G.per_block - 1) / G.per_block);
    if (G.B < 1) G.B = 1;
    G.band_rows = kBandTiles / tiles_x;
    if (G.band_rows < 1) G.band_rows = 1;
    if (G.band_rows > tiles_y) G.band_rows = tiles_y;
    return G;
}

inline WsLayout ws_layout(const BinGeom& G, int64_t ntile_ids, int64_t capacity)
{
    const int64_t ncnt = ntile_ids * G.B;
    WsLayout L;
    size_t o = 0;
    L.cnt = o;       o = align_up(o + sizeof(uint32_t) * (size_t)ncnt);
    L.off = o;       o = align_up(o + sizeof(uint32_t) * (size_t)ncnt);
    L.scan_sums = o; o = align_up(o + scan_ws_bytes(ncnt));
    L.totals = o;    // instance total (u64) and the bucket stats (4 x u32), read back in one copy,
    L.stats = o + sizeof(unsigned long long);   // then the huge-bucket splitter's error word (u32)
    o = align_up(o + sizeof(unsigned long long) + 5 * sizeof(unsigned int));
    L.lists = o;     o = align_up(o + 3 * sizeof(uint32_t) * (size_t)ntile_ids);
    L.tmp = o;       o = align_up(o + sizeof(uint64_t) * (size_t)capacity);
    L.bytes = o;
    return L;
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_bin_sort(const gs_proj* proj, int64_t n, int32_t n_views, int32_t width, int32_t height,
                                 int64_t capacity, uint64_t* keys, uint32_t* ids, uint32_t* tile_ranges,
                                 int64_t* n_instances, void* ws, size_t* ws_bytes, void* stream)
{
    GS_NVTX_RANGE("gs_bin_sort");
    if (!ws_bytes || n < 0 || n > INT32_MAX || n_views < 1 || n_views > GS_MAX_VIEWS) return GS_ERR_INVALID_ARG;
    if (width <= 0 || height <= 0 || width > 65535 * kTile || height > 65535 * kTile) return GS_ERR_INVALID_ARG;
    if (capacity < 0 || capacity > (int64_t)UINT32_MAX) return GS_ERR_INVALID_ARG;
    const int tiles_x = tiles_x_of(width), tiles_y = tiles_y_of(height);
    const int64_t tiles = (int64_t)tiles_x * tiles_y;
    const int64_t ntile_ids = tiles * n_views;
    if (ntile_ids > (int64_t)INT32_MAX / 2 || tiles_x > kBandTiles) return GS_ERR_INVALID_ARG;
    const BinGeom G = bin_geom(n, n_views, tiles_x, tiles_y);
    const WsLayout L = ws_layout(G, ntile_ids, capacity);
    if (!ws) {
        *ws_bytes = L.bytes;
        return GS_OK;
    }
    if (*ws_bytes < L.bytes) return GS_ERR_INVALID_ARG;
    if (!proj || !tile_ranges || !n_instances) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!proj->depth || !proj->rect || !proj->tiles_touched)) return GS_ERR_INVALID_ARG;
    if (capacity > 0 && (!keys || !ids)) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
#ifdef GS_CHECKED
    {
        // pageable source: staged before the call returns; calls on two streams at once share it
        const long long lim[2] = {(long long)n, (long long)capacity};
        GS_CUDA_TRY(cudaMemcpyToSymbolAsync(g_sort_limits, lim, sizeof lim, 0, cudaMemcpyHostToDevice, s));
    }
#endif
    char* w = (char*)ws;
    uint32_t* cnt = (uint32_t*)(w + L.cnt);
    uint32_t* off = (uint32_t*)(w + L.off);
    unsigned long long* scan_sums = (unsigned long long*)(w + L.scan_sums);
    unsigned long long* totals = (unsigned long long*)(w + L.totals);
    unsigned int* stats = (unsigned int*)(w + L.stats);
    uint32_t* lists = (uint32_t*)(w + L.lists);
    uint64_t* tmp = (uint64_t*)(w + L.tmp);
    uint2* ranges = reinterpret_cast<uint2*>(tile_ranges);
    const ushort4* rect4 = reinterpret_cast<const ushort4*>(proj->rect);
    const int64_t ncnt = ntile_ids * G.B;
    const int bands = (tiles_y + G.band_rows - 1) / G.band_rows;
    const dim3 bin_grid((unsigned)G.B, (unsigned)bands, 1u);
    const size_t bin_smem = sizeof(uint32_t) * (size_t)G.band_rows * (size_t)tiles_x;

    if (n > 0) {
        GS_CUDA_TRY(cudaFuncSetAttribute(bin_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bin_smem));
        bin_kernel<false><<<bin_grid, kBinThreads, bin_smem, s>>>(proj->tiles_touched, rect4, proj->depth, G, cnt,
                                                                   nullptr, stats, nullptr, 0ull);
        GS_LAUNCH_CHECK();
    } else {
        GS_CUDA_TRY(cudaMemsetAsync(cnt, 0, sizeof(uint32_t) * (size_t)ncnt, s));
        GS_CUDA_TRY(cudaMemsetAsync(stats, 0, 5 * sizeof(unsigned int), s));
    }
    GS_CUDA_TRY((scan_launch<uint32_t, false>(cnt, ncnt, off, scan_sums, totals, s)));
    const int threads = 256;
    bucket_stats_kernel<<<(unsigned)((ntile_ids + threads - 1) / threads), threads, 0, s>>>(off, G.B, ntile_ids, totals,
                                                                                           ranges, stats, lists);
    GS_LAUNCH_CHECK();
    struct HostCounts {
        unsigned long long total;
        unsigned int st[4];
    };
    static_assert(sizeof(HostCounts) == sizeof(unsigned long long) + 4 * sizeof(unsigned int), "host copy layout");
    // Read back through one pinned host buffer per calling thread (allocated on the
    // first call, kept for the thread's life): a copy to pageable memory would
    // block this call until the GPU had drained the stream.
    static thread_local HostCounts* t_counts = nullptr;
    if (!t_counts) {
        void* p = nullptr;
        GS_CUDA_TRY(cudaHostAlloc(&p, sizeof(HostCounts), cudaHostAllocPortable));
        t_counts = static_cast<HostCounts*>(p);
    }
    HostCounts& host = *t_counts;
    GS_CUDA_TRY(cudaMemcpyAsync(&host, totals, sizeof(HostCounts), cudaMemcpyDeviceToHost, s));
    // The host waits for this copy only (an event), not for the stream: the
    // scatter and the sorts of buckets up to kRegCap instances, which need no
    // host-side count, are queued behind it and keep the GPU busy during the
    // round trip.  They check the device-held count against the capacity and do
    // nothing if it is short.
    cudaEvent_t copied;
    GS_CUDA_TRY(cudaEventCreateWithFlags(&copied, cudaEventDisableTiming));
    cudaError_t ce = cudaEventRecord(copied, s);
    if (ce == cudaSuccess && n > 0) {
        ce = cudaFuncSetAttribute(bin_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bin_smem);
        if (ce == cudaSuccess) {
            bin_kernel<true><<<bin_grid, kBinThreads, bin_smem, s>>>(proj->tiles_touched, rect4, proj->depth, G, off,
                                                                      tmp, nullptr, totals,
                                                                      (unsigned long long)capacity);
            ce = cudaGetLastError();
        }
        if (ce == cudaSuccess) {
            sort_warp_kernel<<<(unsigned)((ntile_ids + kSortWarps - 1) / kSortWarps), kSortWarps * 32, 0, s>>>(
                ranges, ntile_ids, tmp, keys, ids, totals, (unsigned long long)capacity);
            ce = cudaGetLastError();
        }
        if (ce == cudaSuccess) {
            // buckets of 257..2048 instances: at most one per (view, tile)
            sort_reg_kernel<<<(unsigned)ntile_ids, kRegThreads, 0, s>>>(lists, ranges, tmp, keys, ids, stats + 1,
                                                                        totals, (unsigned long long)capacity);
            ce = cudaGetLastError();
        }
    }
    if (ce == cudaSuccess) ce = cudaEventSynchronize(copied);
    cudaEventDestroy(copied);
    if (ce != cudaSuccess) return GS_ERR_CUDA;
    *n_instances = (int64_t)host.total;
    if ((int64_t)host.total > capacity) return GS_ERR_CAPACITY;
    if (host.total == 0) return GS_OK;
    if (host.st[2] > 0) {
        const int e = host.st[0] <= 4u * kMidThreads ? 4 : (host.st[0] <= 8u * kMidThreads ? 8 : 16);
        // the bitonic network's kMidThreads * (e + 1) keys, or the slice sort's 2 c
        const size_t split_keys = 2 * (size_t)(host.st[0] < (unsigned)kSplitMidCap ? host.st[0] : kSplitMidCap);
        const size_t bitonic_keys = (size_t)kMidThreads * (size_t)(e + 1);
        const size_t smem = sizeof(uint64_t) * (split_keys > bitonic_keys ? split_keys : bitonic_keys);
        GS_CUDA_TRY(cudaFuncSetAttribute(sort_mid_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sort_mid_kernel<<<host.st[2], kMidThreads, smem, s>>>(lists + ntile_ids, ranges, tmp, keys, ids);
        GS_LAUNCH_CHECK();
    }
    if (host.st[3] > 0) {
        const size_t smem = sizeof(HugeSmem);
        GS_CUDA_TRY(cudaFuncSetAttribute(sort_huge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
        sort_huge_kernel<<<host.st[3], 1024, smem, s>>>(lists + 2 * ntile_ids, ranges, tmp, keys, ids, stats + 4);
        GS_LAUNCH_CHECK();
        // the splitter's error word: a second read-back, only when a bucket of more
        // than kBigCap instances exists
        GS_CUDA_TRY(cudaMemcpyAsync(&host.st[0], stats + 4, sizeof(unsigned int), cudaMemcpyDeviceToHost, s));
        GS_CUDA_TRY(cudaStreamSynchronize(s));
        if (host.st[0] != 0u) return GS_ERR_DEVICE;
    }
    return GS_OK;
}
