// raster.cu -- gs_raster_fused_fwd_bwd: forward compositing, L1 loss and
// backward rasterization in ONE kernel (ByteSplat, English abstract: "fuses
// forward rasterization and backward rasterization into a single GPU kernel,
// retaining intermediate results on-chip").
//
// One CTA per 16x16 tile, one thread per pixel.  The tile's sorted list is
// staged through shared memory in chunks of kChunk records (gathered through
// the instance ids).  Per pixel the transmittance T, the colour, the index of
// the last composited entry and dL/dC never leave registers; the target pixel
// is read once.  Backward walks the list back to front, recovering T_i by
// division, and reduces each Gaussian's 9 gradient components over the warp
// before one atomic per warp and component.  If the part of the list that any
// pixel composited fits in the last staged chunk, backward reads no records
// from memory at all.
#include "gs_common.cuh"

namespace gs {

constexpr int kChunk = 256;   // records per shared-memory stage

struct RasterArgs {
    const float4* __restrict__ rec;     // [V][n][3]
    const uint2* __restrict__ ranges;   // [V * tiles]
    const uint32_t* __restrict__ ids;
    const float* __restrict__ target;   // [V][3][H][W] or null
    float* image;                       // [V][3][H][W]
    double* loss;                       // [V]
    float* grad2d;                      // [V][n][12]
    uint8_t* touched;                   // [V][n]
    unsigned long long* counts;         // [3] or null
    int64_t n;
    int32_t W, H, tiles_x, tiles, n_views;
    float alpha_min, alpha_max, t_min, bg0, bg1, bg2, inv3hw;
    double inv3hw_d;   // 1 / (3 H W) for the loss mean
    int32_t exclude_crossing;
};

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sums eight values over the warp with a butterfly that halves the live values
// at each of the first three stages (each lane sends the half its partner
// keeps): 4 + 2 + 1 + 1 + 1 shuffles instead of 8 x 5.  Afterwards every lane L
// holds the full sum of value (L >> 2) & 7.
__device__ __forceinline__ float warp_reduce8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                              float v7, int lane)
{
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
    float a0 = (h16 ? v4 : v0) + __shfl_xor_sync(0xffffffffu, h16 ? v0 : v4, 16);
    float a1 = (h16 ? v5 : v1) + __shfl_xor_sync(0xffffffffu, h16 ? v1 : v5, 16);
    float a2 = (h16 ? v6 : v2) + __shfl_xor_sync(0xffffffffu, h16 ? v2 : v6, 16);
    float a3 = (h16 ? v7 : v3) + __shfl_xor_sync(0xffffffffu, h16 ? v3 : v7, 16);
    float b0 = (h8 ? a2 : a0) + __shfl_xor_sync(0xffffffffu, h8 ? a0 : a2, 8);
    float b1 = (h8 ? a3 : a1) + __shfl_xor_sync(0xffffffffu, h8 ? a1 : a3, 8);
    float c0 = (h4 ? b1 : b0) + __shfl_xor_sync(0xffffffffu, h4 ? b0 : b1, 4);
    c0 += __shfl_xor_sync(0xffffffffu, c0, 2);
    c0 += __shfl_xor_sync(0xffffffffu, c0, 1);
    return c0;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

template <bool kBackward>
__global__ void __launch_bounds__(kTileThreads) raster_fused_kernel(RasterArgs a)
{
    __shared__ float4 s_r0[kChunk], s_r1[kChunk];
    __shared__ float2 s_r2[kChunk];   // (blue, tau)
    __shared__ uint32_t s_id[kChunk];
    __shared__ double s_red_d[kTileThreads / 32];
    __shared__ unsigned long long s_red_u[3][kTileThreads / 32];
    __shared__ int s_max_last[kTileThreads / 32];

    const int tile_lin = blockIdx.x;                 // v * tiles + tile
    const int v = tile_lin / a.tiles;
    const int tile = tile_lin - v * a.tiles;
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int px = tx * kTile + (threadIdx.x & (kTile - 1));
    const int py = ty * kTile + (threadIdx.x / kTile);
    const bool inside = px < a.W && py < a.H;
    const float pxf = (float)px + 0.5f, pyf = (float)py + 0.5f;
    const uint2 range = a.ranges[tile_lin];
    const int lo = (int)range.x;
    const int len = (int)(range.y - range.x);
    const float4* __restrict__ recv = a.rec + (size_t)v * (size_t)a.n * 3;

    auto stage = [&](int base) {
        const int k = base + threadIdx.x;
        if (k < len) {
            const uint32_t g = __ldg(a.ids + lo + k);
            const float4* r = recv + (size_t)g * 3;
            s_r0[threadIdx.x] = __ldg(r);
            s_r1[threadIdx.x] = __ldg(r + 1);
            const float4 r2 = __ldg(r + 2);
            s_r2[threadIdx.x] = make_float2(r2.x, r2.z);
            s_id[threadIdx.x] = g;
        }
    };

    // ------------------------------------------------------------- forward
    float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
    int last = -1, ncomp = 0;
    int stop = -1;                      // list index where this pixel stopped, -1 if it never did
    bool done = !inside;
    int resident = -1;                  // chunk currently in shared memory
    const int nchunks = (len + kChunk - 1) / kChunk;
    for (int c = 0; c < nchunks; ++c) {
        if (__syncthreads_and(done)) break;
        const int base = c * kChunk;
        stage(base);
        resident = c;
        __syncthreads();
        const int cnt = min(kChunk, len - base);
        if (!done) {
            for (int j = 0; j < cnt; ++j) {
                const float4 r0 = s_r0[j];
                const float dx = pxf - r0.x, dy = pyf - r0.y;
                const float4 r1 = s_r1[j];
                // power = -1/2 (A dx^2 + C dy^2) - B dx dy, with r0.z = -A/2, r1.x = -C/2
                const float power = ((r0.z * dx) * dx + (r1.x * dy) * dy) - (r0.w * dx) * dy;
                const float2 r2 = s_r2[j];
                // power > 0 is skipped by definition; power < tau has alpha < alpha_min
                if (power > 0.0f || power < r2.y) continue;
                const float araw = r1.y * pexp_neg(power);
                const float alpha = fminf(a.alpha_max, araw);
                if (alpha < a.alpha_min) continue;
                const float Tn = T * (1.0f - alpha);
                if (a.exclude_crossing && Tn < a.t_min) { done = true; stop = base + j; break; }
                const float wgt = alpha * T;
                C0 = C0 + r1.z * wgt;
                C1 = C1 + r1.w * wgt;
                C2 = C2 + r2.x * wgt;
                T = Tn;
                last = base + j;
                ++ncomp;
                if (!a.exclude_crossing && T < a.t_min) { done = true; stop = base + j; break; }
            }
        }
    }
    const int nev = inside ? (stop >= 0 ? stop + 1 : len) : 0;
    C0 = C0 + T * a.bg0;
    C1 = C1 + T * a.bg1;
    C2 = C2 + T * a.bg2;
    const size_t HW = (size_t)a.W * (size_t)a.H;
    const size_t pix = (size_t)v * 3 * HW + (size_t)py * a.W + px;
    float g0 = 0.0f, g1 = 0.0f, g2c = 0.0f;
    double lsum = 0.0;
    if (inside) {
        a.image[pix] = C0;
        a.image[pix + HW] = C1;
        a.image[pix + 2 * HW] = C2;
        if (kBackward) {
            const float d0 = C0 - __ldg(a.target + pix);
            const float d1 = C1 - __ldg(a.target + pix + HW);
            const float d2 = C2 - __ldg(a.target + pix + 2 * HW);
            lsum = (double)fabsf(d0) + (double)fabsf(d1) + (double)fabsf(d2);
            g0 = d0 > 0.0f ? a.inv3hw : (d0 < 0.0f ? -a.inv3hw : 0.0f);
            g1 = d1 > 0.0f ? a.inv3hw : (d1 < 0.0f ? -a.inv3hw : 0.0f);
            g2c = d2 > 0.0f ? a.inv3hw : (d2 < 0.0f ? -a.inv3hw : 0.0f);
        }
    }
    // block reductions: loss, evaluation counts, last composited index
    int warp_last;
    {
        unsigned long long ef = (unsigned long long)nev, eb = (unsigned long long)(last + 1);
        unsigned long long ec = (unsigned long long)ncomp;
        int ml = last;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
            ef += __shfl_xor_sync(0xffffffffu, ef, o);
            eb += __shfl_xor_sync(0xffffffffu, eb, o);
            ec += __shfl_xor_sync(0xffffffffu, ec, o);
            ml = max(ml, __shfl_xor_sync(0xffffffffu, ml, o));
        }
        warp_last = ml;
        if (lane == 0) {
            s_red_d[warp] = lsum;
            s_red_u[0][warp] = ef;
            s_red_u[1][warp] = eb;
            s_red_u[2][warp] = ec;
            s_max_last[warp] = ml;
        }
    }
    __syncthreads();
    int max_last = -1;
    if (threadIdx.x == 0) {
        double ls = 0.0;
        unsigned long long ef = 0, eb = 0, ec = 0;
        for (int w = 0; w < kTileThreads / 32; ++w) {
            ls += s_red_d[w];
            ef += s_red_u[0][w];
            eb += s_red_u[1][w];
            ec += s_red_u[2][w];
            max_last = max(max_last, s_max_last[w]);
        }
        if (kBackward && ls != 0.0) atomicAdd(a.loss + v, ls * a.inv3hw_d);
        if (a.counts) {
            atomicAdd(a.counts, ef);
            atomicAdd(a.counts + 1, eb);
            atomicAdd(a.counts + 2, ec);
        }
        s_max_last[0] = max_last;
    }
    if (!kBackward) return;
    __syncthreads();
    max_last = s_max_last[0];
    if (max_last < 0) return;

    // ------------------------------------------------------------- backward
    float S0 = T * a.bg0, S1 = T * a.bg1, S2 = T * a.bg2;
    float Tcur = T;
    float* __restrict__ g2v = a.grad2d + (size_t)v * (size_t)a.n * GS_GRAD2D_STRIDE;
    uint8_t* __restrict__ touchv = a.touched + (size_t)v * (size_t)a.n;
    const int red_slot = (lane >> 2) & 7;   // component this lane holds after warp_reduce8
    for (int c = max_last / kChunk; c >= 0; --c) {
        const int base = c * kChunk;
        if (c != resident) {
            __syncthreads();   // every thread is done reading the resident chunk
            stage(base);
            resident = c;
            __syncthreads();
        }
        // this warp has nothing composited beyond warp_last
        const int jtop = min(kChunk - 1, warp_last - base);
        for (int j = jtop; j >= 0; --j) {
            const int i = base + j;
            float gm0 = 0.0f, gm1 = 0.0f, gA = 0.0f, gB = 0.0f, gC = 0.0f, go = 0.0f;
            float gr = 0.0f, gg = 0.0f, gb = 0.0f;
            bool contrib = false;
            const float4 r0 = s_r0[j];
            const float dx = pxf - r0.x, dy = pyf - r0.y;
            const float4 r1 = s_r1[j];
            const float power = ((r0.z * dx) * dx + (r1.x * dy) * dy) - (r0.w * dx) * dy;
            const float2 r2 = s_r2[j];
            if (i <= last && power <= 0.0f && power >= r2.y) {
                const float G = pexp_neg(power);
                const float araw = r1.y * G;
                const float alpha = fminf(a.alpha_max, araw);
                if (alpha >= a.alpha_min) {
                    contrib = true;
                    const float oma = 1.0f - alpha;
                    const float inv_oma = rcp_approx(oma);
                    const float Ti = Tcur * inv_oma;
                    const float wgt = alpha * Ti;
                    gr = g0 * wgt;
                    gg = g1 * wgt;
                    gb = g2c * wgt;
                    const float dotc = __fmaf_rn(g0, r1.z, __fmaf_rn(g1, r1.w, g2c * r2.x));
                    const float dots = __fmaf_rn(g0, S0, __fmaf_rn(g1, S1, g2c * S2));
                    const float dalpha = __fmaf_rn(Ti, dotc, -dots * inv_oma);
                    S0 = __fmaf_rn(r1.z, wgt, S0);
                    S1 = __fmaf_rn(r1.w, wgt, S1);
                    S2 = __fmaf_rn(r2.x, wgt, S2);
                    Tcur = Ti;
                    if (araw <= a.alpha_max) {
                        go = dalpha * G;
                        const float dp = dalpha * alpha;
                        // d power / d(A, B, C) = (-dx^2/2, -dx dy, -dy^2/2);
                        // d power / d mean2d = (A dx + B dy, B dx + C dy), A = -2 r0.z, C = -2 r1.x
                        const float hdp = -0.5f * dp;
                        gA = hdp * dx * dx;
                        gB = -dp * (dx * dy);
                        gC = hdp * dy * dy;
                        gm0 = dp * __fmaf_rn(-2.0f * r0.z, dx, r0.w * dy);
                        gm1 = dp * __fmaf_rn(r0.w, dx, -2.0f * r1.x * dy);
                    }
                }
            }
            if (__any_sync(0xffffffffu, contrib)) {
                const float s8 = warp_reduce8(gm0, gm1, gA, gB, gC, go, gr, gg, lane);
                const float sb = warp_sum(gb);
                const uint32_t gid = s_id[j];
                float* dst = g2v + (size_t)gid * GS_GRAD2D_STRIDE;
                if ((lane & 3) == 0) atomicAdd(dst + red_slot, s8);
                if (lane == 1) atomicAdd(dst + 8, sb);
                if (lane == 2) touchv[gid] = 1;
            }
        }
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_raster_fused_fwd_bwd(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                             const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                             const gs_render_opts* opts, const float* target, float* image,
                                             double* loss, float* grad2d, uint8_t* touched, uint64_t* eval_counts,
                                             void* stream)
{
    if (!proj || !tile_ranges || !opts_ok(opts) || !image || n < 0 || n > INT32_MAX) return GS_ERR_INVALID_ARG;
    gs_status st = check_views(cams, n_views);
    if (st != GS_OK) return st;
    if (target && (!loss || (n > 0 && (!grad2d || !touched)))) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!proj->rec || !ids)) return GS_ERR_INVALID_ARG;
    if (!aligned16(proj->rec) || (grad2d && !aligned16(grad2d))) return GS_ERR_INVALID_ARG;
    const int W = cams[0].width, H = cams[0].height;
    RasterArgs a;
    a.rec = reinterpret_cast<const float4*>(proj->rec);
    a.ranges = reinterpret_cast<const uint2*>(tile_ranges);
    a.ids = ids;
    a.target = target;
    a.image = image;
    a.loss = loss;
    a.grad2d = grad2d;
    a.touched = touched;
    a.counts = reinterpret_cast<unsigned long long*>(eval_counts);
    a.n = n;
    a.W = W;
    a.H = H;
    a.tiles_x = tiles_x_of(W);
    a.tiles = tiles_x_of(W) * tiles_y_of(H);
    a.n_views = n_views;
    a.alpha_min = opts->alpha_min;
    a.alpha_max = opts->alpha_max;
    a.t_min = opts->t_min;
    a.bg0 = opts->bg[0];
    a.bg1 = opts->bg[1];
    a.bg2 = opts->bg[2];
    a.inv3hw_d = 1.0 / (3.0 * (double)W * (double)H);
    a.inv3hw = (float)a.inv3hw_d;
    a.exclude_crossing = opts->exclude_crossing ? 1 : 0;
    cudaStream_t s = (cudaStream_t)stream;
    const long long grid = (long long)a.tiles * n_views;
    if (grid > INT32_MAX) return GS_ERR_INVALID_ARG;
    if (target) {
        GS_CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(double) * (size_t)n_views, s));
        raster_fused_kernel<true><<<(unsigned)grid, kTileThreads, 0, s>>>(a);
    } else {
        raster_fused_kernel<false><<<(unsigned)grid, kTileThreads, 0, s>>>(a);
    }
    GS_LAUNCH_CHECK();
    return GS_OK;
}
