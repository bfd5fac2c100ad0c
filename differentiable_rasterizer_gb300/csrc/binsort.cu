// binsort.cu -- gs_bin_sort: 16x16 tile binning with (tile, depth) keys and an
// LSD radix sort, then per-tile ranges of the sorted instance list.
//
//   1. exclusive scan of tiles_touched over [V][n] -> instance offsets, total;
//   2. total read back to the host (the step's one host synchronisation);
//   3. emit: (view, Gaussian) writes key = ((v*tiles + tile) << 32) | bits(depth),
//      value = Gaussian index, for the tiles of its rect in row-major order;
//   4. LSD radix sort over the 32 depth bits and the bits of v*tiles + tile,
//      8-bit digits, each pass = block digit histograms -> scan -> stable scatter
//      (ranks within a warp from __match_any_sync, warps in order), so equal keys
//      keep emission order (ascending Gaussian index within a view);
//   5. tile ranges [start, end) from the sorted keys.
// The pass count decides which buffer the emit writes, so the last pass always
// lands in the caller's arrays.
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

// Aligned bump layout of the workspace.
struct WsLayout {
    size_t scan_sums, offsets, totals, alt_keys, alt_ids, hist, hist_sums, bytes;
};

inline size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

inline WsLayout ws_layout(int64_t vn, int64_t capacity)
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
    const WsLayout L = ws_layout(vn, capacity);
    if (!ws) {
        *ws_bytes = L.bytes;
        return GS_OK;
    }
    if (*ws_bytes < L.bytes) return GS_ERR_INVALID_ARG;
    if (!proj || !tile_ranges || !n_instances) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!proj->depth || !proj->rect || !proj->tiles_touched)) return GS_ERR_INVALID_ARG;
    if (capacity > 0 && (!keys || !ids)) return GS_ERR_INVALID_ARG;
    const int tiles_x = tiles_x_of(width);
    const int64_t tiles = (int64_t)tiles_x * tiles_y_of(height);
    const int64_t ntile_ids = tiles * n_views;
    if (ntile_ids > (int64_t)UINT32_MAX) return GS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = (char*)ws;
    unsigned long long* scan_sums = (unsigned long long*)(w + L.scan_sums);
    uint32_t* offsets = (uint32_t*)(w + L.offsets);
    unsigned long long* totals = (unsigned long long*)(w + L.totals);
    uint64_t* alt_keys = (uint64_t*)(w + L.alt_keys);
    uint32_t* alt_ids = (uint32_t*)(w + L.alt_ids);
    uint32_t* hist = (uint32_t*)(w + L.hist);
    unsigned long long* hist_sums = (unsigned long long*)(w + L.hist_sums);

    // 1-2: offsets and the instance count
    GS_CUDA_TRY((scan_launch<uint32_t, false>(proj->tiles_touched, vn, offsets, scan_sums, totals, s)));
    unsigned long long total = 0;
    GS_CUDA_TRY(cudaMemcpyAsync(&total, totals, sizeof(total), cudaMemcpyDeviceToHost, s));
    GS_CUDA_TRY(cudaStreamSynchronize(s));
    *n_instances = (int64_t)total;
    if ((int64_t)total > capacity) return GS_ERR_CAPACITY;
    const int64_t N = (int64_t)total;
    GS_CUDA_TRY(cudaMemsetAsync(tile_ranges, 0, sizeof(uint32_t) * 2 * (size_t)ntile_ids, s));
    if (N == 0) return GS_OK;

    // passes: 32 depth bits + the tile-id bits, 8-bit digits
    const int bits = 32 + (ntile_ids > 1 ? bit_length((uint64_t)(ntile_ids - 1)) : 1);
    const int npass = (bits + 7) / 8;
    uint64_t* kbuf[2] = {keys, alt_keys};
    uint32_t* vbuf[2] = {ids, alt_ids};
    int cur = (npass & 1) ? 1 : 0;   // the last pass writes buffer 0 (the caller's)

    // 3: emit
    {
        const int threads = 256;
        emit_kernel<<<(unsigned)((vn + threads - 1) / threads), threads, 0, s>>>(
            proj->tiles_touched, offsets, reinterpret_cast<const ushort4*>(proj->rect), proj->depth, n, vn, tiles_x,
            (int)tiles, kbuf[cur], vbuf[cur]);
        GS_LAUNCH_CHECK();
    }
    // 4: radix passes
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
    // 5: ranges
    {
        const int threads = 256;
        tile_ranges_kernel<<<(unsigned)((N + threads - 1) / threads), threads, 0, s>>>(
            keys, N, reinterpret_cast<uint2*>(tile_ranges));
        GS_LAUNCH_CHECK();
    }
    return GS_OK;
}
