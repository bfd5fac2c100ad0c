// binsort.cu -- gs_bin_sort: 16x16 tile binning with (tile, depth) keys and a
// sort, then per-tile ranges of the sorted instance list.
//
// Per-tile path (the normal case):
//   1. count instances per (view, tile) with atomics;
//   2. exclusive scan of the counts = the start of every tile's bucket;
//   3. one pass over the buckets: instance total, largest bucket, list of buckets
//      larger than a shared-memory block sort holds; scatter cursors;
//   4. the totals go to the host (the step's one host synchronisation);
//   5. scatter: every visible (view, Gaussian) appends (depth bits << 32 | index)
//      to the bucket of each tile of its rect (atomic cursor, any order);
//   6. one CTA per bucket sorts it by (depth bits, index) in shared memory
//      (bitonic) and writes key = ((v*tiles + tile) << 32) | depth bits, value =
//      index, and the tile's range.
// The result equals a stable sort by (tile, depth) of instances emitted in
// (view, Gaussian) order: within a bucket the index breaks depth ties.
// Buckets over kBigCap instances use the LSD radix path instead: scan of
// tiles_touched, emit, 8-bit LSD passes (block digit histograms -> scan ->
// stable scatter with ranks from __match_any_sync), ranges from the sorted keys.
#include "gs_common.cuh"
#include "scan.cuh"

namespace gs {

constexpr int kSortThreads = 256;
constexpr int kSortPerThread = 16;
constexpr int kSortItems = kSortThreads * kSortPerThread;   // one block's tile of keys
constexpr int kWarps = kSortThreads / 32;

__global__ void emit_kernel(const uint32_t* __restrict__ touched_cnt, const uint32_t* __restrict__ offsets,
                            const ushort4* __restrict__ rect, const float* __restrict__ depth, int64_t n,
                            int64_t total_vn, int tiles_x, int tiles, uint64_t* __restrict__ keys,
                            uint32_t* __restrict__ ids)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total_vn) return;
    const uint32_t cnt = touched_cnt[i];
    if (cnt == 0) return;
    const int64_t v = i / n;
    const uint32_t g = (uint32_t)(i - v * n);
    const ushort4 r = rect[i];
    const uint64_t dbits = (uint64_t)__float_as_uint(depth[i]);
    uint32_t off = offsets[i];
    const uint64_t vbase = (uint64_t)v * (uint64_t)tiles;
    for (int ty = r.y; ty < r.w; ++ty)
        for (int tx = r.x; tx < r.z; ++tx) {
            keys[off] = ((vbase + (uint64_t)(ty * tiles_x + tx)) << 32) | dbits;
            ids[off] = g;
            ++off;
        }
}

__device__ __forceinline__ int64_t sort_item(int it)
{
    // warp-striped: warp w owns [w*512, (w+1)*512) of the block tile, 32 consecutive per iteration
    return (int64_t)blockIdx.x * kSortItems + (int64_t)(threadIdx.x >> 5) * (32 * kSortPerThread) +
           (int64_t)it * 32 + (threadIdx.x & 31);
}

__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(const uint64_t* __restrict__ keys, int64_t N,
                                                                  int shift, uint32_t mask, uint32_t* __restrict__ hist,
                                                                  int64_t nb)
{
    __shared__ uint32_t s_h[256];
    s_h[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kSortPerThread; ++it) {
        const int64_t i = sort_item(it);
        if (i < N) atomicAdd(&s_h[(uint32_t)(keys[i] >> shift) & mask], 1u);
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * nb + blockIdx.x] = s_h[threadIdx.x];   // digit-major
}

__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(
    const uint64_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in, int64_t N, int shift, uint32_t mask,
    const uint32_t* __restrict__ offs, int64_t nb, uint64_t* __restrict__ keys_out, uint32_t* __restrict__ vals_out)
{
    __shared__ uint32_t s_cnt[kWarps][256];
    __shared__ uint32_t s_goff[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s_cnt[w][threadIdx.x] = 0;
    s_goff[threadIdx.x] = offs[(int64_t)threadIdx.x * nb + blockIdx.x];
    __syncthreads();
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint64_t k[kSortPerThread];
    uint32_t rank[kSortPerThread];
    uint32_t dig[kSortPerThread];
#pragma unroll
    for (int it = 0; it < kSortPerThread; ++it) {
        const int64_t i = sort_item(it);
        const bool valid = i < N;
        k[it] = valid ? keys_in[i] : 0ull;
        const uint32_t d = valid ? ((uint32_t)(k[it] >> shift) & mask) : 256u;
        dig[it] = d;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        const uint32_t before = valid ? s_cnt[warp][d] : 0u;
        __syncwarp();
        if (valid && (peers & lt_mask) == 0) s_cnt[warp][d] = before + (uint32_t)__popc(peers);
        __syncwarp();
        rank[it] = before + (uint32_t)__popc(peers & lt_mask);
    }
    __syncthreads();
    {   // exclusive scan over warps per digit
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t c = s_cnt[w][threadIdx.x];
            s_cnt[w][threadIdx.x] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int it = 0; it < kSortPerThread; ++it) {
        const int64_t i = sort_item(it);
        if (i < N) {
            const uint32_t d = dig[it];
            const uint32_t pos = s_goff[d] + s_cnt[warp][d] + rank[it];
            keys_out[pos] = k[it];
            vals_out[pos] = vals_in[i];
        }
    }
}

__global__ void tile_ranges_kernel(const uint64_t* __restrict__ keys, int64_t N, uint2* __restrict__ ranges)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N) return;
    const uint32_t t = (uint32_t)(keys[i] >> 32);
    if (i == 0 || (uint32_t)(keys[i - 1] >> 32) != t) ranges[t].x = (uint32_t)i;
    if (i == N - 1 || (uint32_t)(keys[i + 1] >> 32) != t) ranges[t].y = (uint32_t)(i + 1);
}

constexpr int kSmallCap = 2048;    // bucket sizes sorted by the 256-thread kernel (16 KB)
constexpr int kBigCap = 16384;     // bucket sizes sorted by the 1024-thread kernel (128 KB)

__global__ void count_tiles_kernel(const uint32_t* __restrict__ touched_cnt, const ushort4* __restrict__ rect,
                                   int64_t n, int64_t total_vn, int tiles_x, int tiles, uint32_t* __restrict__ cnt)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total_vn || touched_cnt[i] == 0) return;
    const int64_t v = i / n;
    const ushort4 r = rect[i];
    uint32_t* c = cnt + v * tiles;
    for (int ty = r.y; ty < r.w; ++ty)
        for (int tx = r.x; tx < r.z; ++tx) atomicAdd(c + ty * tiles_x + tx, 1u);
}

// stats[0] = largest bucket, stats[1] = number of buckets over kSmallCap
__global__ void bucket_stats_kernel(const uint32_t* __restrict__ cnt, const uint32_t* __restrict__ off, int64_t nb,
                                    uint32_t* __restrict__ cursor, unsigned int* __restrict__ stats,
                                    uint32_t* __restrict__ big_list)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nb) return;
    const uint32_t c = cnt[t];
    cursor[t] = off[t];
    if (c == 0) return;
    atomicMax(stats, c);
    if (c > (uint32_t)kSmallCap) big_list[atomicAdd(stats + 1, 1u)] = (uint32_t)t;
}

__global__ void scatter_tiles_kernel(const uint32_t* __restrict__ touched_cnt, const ushort4* __restrict__ rect,
                                     const float* __restrict__ depth, int64_t n, int64_t total_vn, int tiles_x,
                                     int tiles, uint32_t* __restrict__ cursor, uint64_t* __restrict__ tmp)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total_vn || touched_cnt[i] == 0) return;
    const int64_t v = i / n;
    const uint32_t g = (uint32_t)(i - v * n);
    const ushort4 r = rect[i];
    const uint64_t key = ((uint64_t)__float_as_uint(depth[i]) << 32) | g;
    uint32_t* cur = cursor + v * tiles;
    for (int ty = r.y; ty < r.w; ++ty)
        for (int tx = r.x; tx < r.z; ++tx) tmp[atomicAdd(cur + ty * tiles_x + tx, 1u)] = key;
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

__device__ __forceinline__ void sort_bucket(uint64_t* s, uint32_t t, const uint32_t* __restrict__ cnt,
                                            const uint32_t* __restrict__ off, const uint64_t* __restrict__ tmp,
                                            uint64_t* __restrict__ keys, uint32_t* __restrict__ ids)
{
    const int c = (int)cnt[t];
    const uint32_t o = off[t];
    int P = 1;
    while (P < c) P <<= 1;
    for (int i = threadIdx.x; i < P; i += blockDim.x) s[i] = i < c ? tmp[o + i] : ~0ull;
    __syncthreads();
    block_bitonic(s, P);
    const uint64_t hi = (uint64_t)t << 32;
    for (int i = threadIdx.x; i < c; i += blockDim.x) {
        const uint64_t k = s[i];
        keys[o + i] = hi | (k >> 32);
        ids[o + i] = (uint32_t)k;
    }
}

// One 256-thread CTA per bucket: writes every bucket's range, sorts buckets of
// at most kSmallCap instances.
__global__ void __launch_bounds__(256) sort_small_kernel(const uint32_t* __restrict__ cnt,
                                                         const uint32_t* __restrict__ off,
                                                         const uint64_t* __restrict__ tmp, uint64_t* __restrict__ keys,
                                                         uint32_t* __restrict__ ids, uint2* __restrict__ ranges)
{
    __shared__ uint64_t s[kSmallCap];
    const uint32_t t = blockIdx.x;
    const uint32_t c = cnt[t];
    if (threadIdx.x == 0) ranges[t] = make_uint2(off[t], off[t] + c);
    if (c == 0 || c > (uint32_t)kSmallCap) return;
    sort_bucket(s, t, cnt, off, tmp, keys, ids);
}

// One 1024-thread CTA per listed bucket of kSmallCap < size <= kBigCap.
__global__ void __launch_bounds__(1024) sort_big_kernel(const uint32_t* __restrict__ big_list,
                                                        const uint32_t* __restrict__ cnt,
                                                        const uint32_t* __restrict__ off,
                                                        const uint64_t* __restrict__ tmp, uint64_t* __restrict__ keys,
                                                        uint32_t* __restrict__ ids)
{
    extern __shared__ uint64_t s_big[];
    sort_bucket(s_big, big_list[blockIdx.x], cnt, off, tmp, keys, ids);
}

// Aligned bump layout of the workspace.
struct WsLayout {
    size_t scan_sums, offsets, totals, alt_keys, alt_ids, hist, hist_sums;
    size_t tile_cnt, tile_off, cursor, tile_sums, stats, big_list, bytes;
};

inline size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

inline WsLayout ws_layout(int64_t vn, int64_t capacity, int64_t ntile_ids)
{
    WsLayout L;
    size_t o = 0;
    L.scan_sums = o; o = align_up(o + scan_ws_bytes(vn));
    L.offsets = o;   o = align_up(o + sizeof(uint32_t) * (size_t)vn);
    L.totals = o;    o = align_up(o + 2 * sizeof(unsigned long long));
    L.alt_keys = o;  o = align_up(o + sizeof(uint64_t) * (size_t)capacity);
    L.alt_ids = o;   o = align_up(o + sizeof(uint32_t) * (size_t)capacity);
    const int64_t nb = (capacity + kSortItems - 1) / kSortItems;
    L.hist = o;      o = align_up(o + sizeof(uint32_t) * 256 * (size_t)nb);
    L.hist_sums = o; o = align_up(o + scan_ws_bytes(256 * nb));
    L.tile_cnt = o;  o = align_up(o + sizeof(uint32_t) * (size_t)ntile_ids);
    L.tile_off = o;  o = align_up(o + sizeof(uint32_t) * (size_t)ntile_ids);
    L.cursor = o;    o = align_up(o + sizeof(uint32_t) * (size_t)ntile_ids);
    L.tile_sums = o; o = align_up(o + scan_ws_bytes(ntile_ids));
    L.stats = o;     o = align_up(o + 4 * sizeof(unsigned int));
    L.big_list = o;  o = align_up(o + sizeof(uint32_t) * (size_t)ntile_ids);
    L.bytes = o;
    return L;
}

inline int bit_length(uint64_t x)
{
    int b = 0;
    while (x) { ++b; x >>= 1; }
    return b;
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_bin_sort(const gs_proj* proj, int64_t n, int32_t n_views, int32_t width, int32_t height,
                                 int64_t capacity, uint64_t* keys, uint32_t* ids, uint32_t* tile_ranges,
                                 int64_t* n_instances, void* ws, size_t* ws_bytes, void* stream)
{
    if (!ws_bytes || n < 0 || n > INT32_MAX || n_views < 1 || n_views > GS_MAX_VIEWS) return GS_ERR_INVALID_ARG;
    if (width <= 0 || height <= 0 || width > 65535 * kTile || height > 65535 * kTile) return GS_ERR_INVALID_ARG;
    if (capacity < 0 || capacity > (int64_t)UINT32_MAX) return GS_ERR_INVALID_ARG;
    const int64_t vn = n * (int64_t)n_views;
    const int tiles_x = tiles_x_of(width);
    const int64_t tiles = (int64_t)tiles_x * tiles_y_of(height);
    const int64_t ntile_ids = tiles * n_views;
    if (ntile_ids > (int64_t)INT32_MAX) return GS_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(vn, capacity, ntile_ids);
    if (!ws) {
        *ws_bytes = L.bytes;
        return GS_OK;
    }
    if (*ws_bytes < L.bytes) return GS_ERR_INVALID_ARG;
    if (!proj || !tile_ranges || !n_instances) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!proj->depth || !proj->rect || !proj->tiles_touched)) return GS_ERR_INVALID_ARG;
    if (capacity > 0 && (!keys || !ids)) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = (char*)ws;
    unsigned long long* scan_sums = (unsigned long long*)(w + L.scan_sums);
    uint32_t* offsets = (uint32_t*)(w + L.offsets);
    unsigned long long* totals = (unsigned long long*)(w + L.totals);
    uint64_t* alt_keys = (uint64_t*)(w + L.alt_keys);
    uint32_t* alt_ids = (uint32_t*)(w + L.alt_ids);
    uint32_t* hist = (uint32_t*)(w + L.hist);
    unsigned long long* hist_sums = (unsigned long long*)(w + L.hist_sums);
    uint32_t* tile_cnt = (uint32_t*)(w + L.tile_cnt);
    uint32_t* tile_off = (uint32_t*)(w + L.tile_off);
    uint32_t* cursor = (uint32_t*)(w + L.cursor);
    unsigned long long* tile_sums = (unsigned long long*)(w + L.tile_sums);
    unsigned int* stats = (unsigned int*)(w + L.stats);
    uint32_t* big_list = (uint32_t*)(w + L.big_list);
    const ushort4* rect4 = reinterpret_cast<const ushort4*>(proj->rect);
    const int threads = 256;
    const unsigned gblocks = (unsigned)((vn + threads - 1) / threads);

    // per-tile path: counts, bucket starts, totals
    GS_CUDA_TRY(cudaMemsetAsync(tile_cnt, 0, sizeof(uint32_t) * (size_t)ntile_ids, s));
    GS_CUDA_TRY(cudaMemsetAsync(stats, 0, 4 * sizeof(unsigned int), s));
    if (vn > 0) {
        count_tiles_kernel<<<gblocks, threads, 0, s>>>(proj->tiles_touched, rect4, n, vn, tiles_x, (int)tiles,
                                                        tile_cnt);
        GS_LAUNCH_CHECK();
    }
    GS_CUDA_TRY((scan_launch<uint32_t, false>(tile_cnt, ntile_ids, tile_off, tile_sums, totals, s)));
    bucket_stats_kernel<<<(unsigned)((ntile_ids + threads - 1) / threads), threads, 0, s>>>(tile_cnt, tile_off,
                                                                                           ntile_ids, cursor, stats,
                                                                                           big_list);
    GS_LAUNCH_CHECK();
    struct {
        unsigned long long total;
        unsigned int st[4];
    } host;
    GS_CUDA_TRY(cudaMemcpyAsync(&host.total, totals, sizeof(host.total), cudaMemcpyDeviceToHost, s));
    GS_CUDA_TRY(cudaMemcpyAsync(host.st, stats, sizeof(host.st), cudaMemcpyDeviceToHost, s));
    GS_CUDA_TRY(cudaStreamSynchronize(s));
    *n_instances = (int64_t)host.total;
    if ((int64_t)host.total > capacity) return GS_ERR_CAPACITY;
    if (host.total > 0 && host.st[0] <= (unsigned)kBigCap) {
        scatter_tiles_kernel<<<gblocks, threads, 0, s>>>(proj->tiles_touched, rect4, proj->depth, n, vn, tiles_x,
                                                          (int)tiles, cursor, alt_keys);
        GS_LAUNCH_CHECK();
        sort_small_kernel<<<(unsigned)ntile_ids, 256, 0, s>>>(tile_cnt, tile_off, alt_keys, keys, ids,
                                                              reinterpret_cast<uint2*>(tile_ranges));
        GS_LAUNCH_CHECK();
        if (host.st[1] > 0) {
            int P = 1;
            while (P < (int)host.st[0]) P <<= 1;
            const size_t smem = sizeof(uint64_t) * (size_t)P;
            GS_CUDA_TRY(cudaFuncSetAttribute(sort_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            sort_big_kernel<<<host.st[1], 1024, smem, s>>>(big_list, tile_cnt, tile_off, alt_keys, keys, ids);
            GS_LAUNCH_CHECK();
        }
        return GS_OK;
    }

    // LSD radix path (no instances, or a bucket too large for a block sort)
    GS_CUDA_TRY(cudaMemsetAsync(tile_ranges, 0, sizeof(uint32_t) * 2 * (size_t)ntile_ids, s));
    const int64_t N = (int64_t)host.total;
    if (N == 0) return GS_OK;
    GS_CUDA_TRY((scan_launch<uint32_t, false>(proj->tiles_touched, vn, offsets, scan_sums, totals + 1, s)));

    // passes: 32 depth bits + the tile-id bits, 8-bit digits
    const int bits = 32 + (ntile_ids > 1 ? bit_length((uint64_t)(ntile_ids - 1)) : 1);
    const int npass = (bits + 7) / 8;
    uint64_t* kbuf[2] = {keys, alt_keys};
    uint32_t* vbuf[2] = {ids, alt_ids};
    int cur = (npass & 1) ? 1 : 0;   // the last pass writes buffer 0 (the caller's)

    // emit
    emit_kernel<<<gblocks, threads, 0, s>>>(proj->tiles_touched, offsets, rect4, proj->depth, n, vn, tiles_x,
                                            (int)tiles, kbuf[cur], vbuf[cur]);
    GS_LAUNCH_CHECK();
    // radix passes
    const int64_t nb = (N + kSortItems - 1) / kSortItems;
    for (int p = 0; p < npass; ++p) {
        const int shift = 8 * p;
        const int width_bits = min(8, bits - shift);
        const uint32_t mask = (1u << width_bits) - 1u;
        radix_hist_kernel<<<(unsigned)nb, kSortThreads, 0, s>>>(kbuf[cur], N, shift, mask, hist, nb);
        GS_LAUNCH_CHECK();
        GS_CUDA_TRY((scan_launch<uint32_t, false>(hist, 256 * nb, hist, hist_sums, totals + 1, s)));
        radix_scatter_kernel<<<(unsigned)nb, kSortThreads, 0, s>>>(kbuf[cur], vbuf[cur], N, shift, mask, hist, nb,
                                                                    kbuf[cur ^ 1], vbuf[cur ^ 1]);
        GS_LAUNCH_CHECK();
        cur ^= 1;
    }
    // ranges
    tile_ranges_kernel<<<(unsigned)((N + threads - 1) / threads), threads, 0, s>>>(keys, N,
                                                                                 reinterpret_cast<uint2*>(tile_ranges));
    GS_LAUNCH_CHECK();
    return GS_OK;
}
