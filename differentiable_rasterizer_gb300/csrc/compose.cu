// compose.cu -- partial render + compose (Splaxel, English abstract: each part
// renders its local subset of Gaussians and only partial pixel values (colour,
// transmittance) are exchanged and composed).
//
// Subsets are per-view depth slabs: slab s holds the Gaussians with
// z_s <= depth < z_{s+1}.  Tile lists are sorted by (depth, index), so a slab's
// entries in a tile are one contiguous part of the tile's list:
//   gs_split_ranges  per (view, tile): the S sub-ranges, by binary search of the
//                    split depths in the sorted keys (low 32 bits: depth bits)
//   gs_raster_forward_state, once per slab with its sub-ranges and a zero
//                    background: (C_s, T_s) per pixel
//   gs_compose       per pixel, front to back: C = sum_s (prod_{j<s} T_j) C_s +
//                    (prod_s T_s) bg, T = prod_s T_s
#include <algorithm>
#include <cfloat>
#include <cstring>

#include "gs_common.cuh"

namespace gs {

constexpr int kMaxSubsets = 8;

struct SplitArgs {
    const uint64_t* __restrict__ keys;
    const uint2* __restrict__ ranges;   // [V * tiles]
    uint2* sub;                         // [S][V * tiles]
    int64_t n_ranges;                   // V * tiles
    int tiles, S;
    uint32_t zbits[GS_MAX_VIEWS][kMaxSubsets - 1];   // split depths as bit patterns (positive floats)
};

__global__ void split_ranges_kernel(SplitArgs a)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.n_ranges) return;
    const int v = (int)(i / a.tiles);
    uint2 r = a.ranges[i];
    if (!GS_IN_RANGE((int64_t)r.y - (int64_t)r.x, 1ll << 32, GS_CHECK_RANGE)) r.y = r.x;
    uint32_t start = r.x;
    for (int s = 0; s < a.S; ++s) {
        uint32_t end = r.y;
        if (s < a.S - 1) {
            // first position in [start, r.y) whose depth bits are >= the split
            const uint32_t z = a.zbits[v][s];
            uint32_t lo = start, hi = r.y;
            while (lo < hi) {
                const uint32_t mid = lo + (hi - lo) / 2;
                if ((uint32_t)__ldg(a.keys + mid) < z) lo = mid + 1;
                else hi = mid;
            }
            end = lo;
        }
        a.sub[(int64_t)s * a.n_ranges + i] = make_uint2(start, end);
        start = end;
    }
}

__global__ void compose_kernel(const float* __restrict__ c_parts, const float* __restrict__ t_parts, int S,
                               int64_t n_pix /* V*H*W */, int64_t hw, float bg0, float bg1, float bg2, float* image,
                               float* t_out)
{
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n_pix; p += (int64_t)gridDim.x * blockDim.x) {
        const int64_t v = p / hw, q = p - v * hw;
        float C0 = 0.0f, C1 = 0.0f, C2 = 0.0f, T = 1.0f;
        for (int s = 0; s < S; ++s) {
            const float* cs = c_parts + ((int64_t)s * n_pix + v * hw) * 3 + q;
            C0 = __fmaf_rn(T, __ldg(cs), C0);
            C1 = __fmaf_rn(T, __ldg(cs + hw), C1);
            C2 = __fmaf_rn(T, __ldg(cs + 2 * hw), C2);
            T = T * __ldg(t_parts + (int64_t)s * n_pix + p);
        }
        float* img = image + v * 3 * hw + q;
        img[0] = __fmaf_rn(T, bg0, C0);
        img[hw] = __fmaf_rn(T, bg1, C1);
        img[2 * hw] = __fmaf_rn(T, bg2, C2);
        if (t_out) t_out[p] = T;
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_split_ranges(const uint64_t* keys, const uint32_t* tile_ranges, int32_t n_views,
                                     int32_t width, int32_t height, int32_t n_subsets, const float* depth_splits,
                                     uint32_t* sub_ranges, void* stream)
{
    GS_NVTX_RANGE("gs_split_ranges");
    if (!tile_ranges || !sub_ranges || n_subsets < 1 || n_subsets > kMaxSubsets) return GS_ERR_INVALID_ARG;
    if (n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 || height < 1) return GS_ERR_INVALID_ARG;
    if (n_subsets > 1 && (!depth_splits || !keys)) return GS_ERR_INVALID_ARG;
    SplitArgs a;
    a.keys = keys;
    a.ranges = reinterpret_cast<const uint2*>(tile_ranges);
    a.sub = reinterpret_cast<uint2*>(sub_ranges);
    a.tiles = tiles_x_of(width) * tiles_y_of(height);
    a.n_ranges = (int64_t)a.tiles * n_views;
    a.S = n_subsets;
    for (int v = 0; v < n_views; ++v)
        for (int s = 0; s + 1 < n_subsets; ++s) {
            const float z = depth_splits[v * (n_subsets - 1) + s];
            // splits must be positive, finite and ascending (depths are > near_z > 0)
            if (!(z > 0.0f && z <= FLT_MAX)) return GS_ERR_INVALID_ARG;
            if (s > 0 && !(z > depth_splits[v * (n_subsets - 1) + s - 1])) return GS_ERR_INVALID_ARG;
            uint32_t b;
            memcpy(&b, &z, 4);
            a.zbits[v][s] = b;
        }
    const int64_t blocks = (a.n_ranges + 255) / 256;
    split_ranges_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    GS_LAUNCH_CHECK();
    return GS_OK;
}

extern "C" gs_status gs_compose(const float* c_parts, const float* t_parts, int32_t n_subsets, int32_t n_views,
                                int32_t width, int32_t height, const float* bg, float* image, float* t_final,
                                void* stream)
{
    GS_NVTX_RANGE("gs_compose");
    if (!c_parts || !t_parts || !bg || !image || n_subsets < 1 || n_subsets > kMaxSubsets) return GS_ERR_INVALID_ARG;
    if (n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 || height < 1) return GS_ERR_INVALID_ARG;
    const int64_t hw = (int64_t)width * height, n_pix = hw * n_views;
    int dev = 0, sms = 0;
    GS_CUDA_TRY(cudaGetDevice(&dev));
    GS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int64_t want = (n_pix + 255) / 256;
    const int blocks = (int)std::min<int64_t>(want, (int64_t)sms * 8);
    compose_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(c_parts, t_parts, n_subsets, n_pix, hw, bg[0], bg[1],
                                                            bg[2], image, t_final);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
