// project.cu -- gs_project: EWA projection of every Gaussian into every view.
//
// One thread per Gaussian reads its parameter block once (float4 loads) and
// loops over the views, so a batch of V views costs one pass over the
// parameters instead of V (Grendel, abstract: batched multi-view training).
// Culling follows GS-Scale's frustum-culling step (abstract), done on the GPU.
// The arithmetic order is fixed (see gs.h) so the cull / rect decisions are
// reproducible bit for bit on a CPU.
#include "gs_common.cuh"
#include "project_math.cuh"

namespace gs {

struct ProjectArgs {
    const float* params;
    int64_t n;
    int32_t sh_degree;
    float near_z, lowpass, alpha_min;
    int32_t tiles_x, tiles_y;
    float4* rec;
    float* depth;
    ushort4* rect;
    uint32_t* tiles_touched;
};

// Where a pixel can pass the alpha test, for the rasterizer's culling.
//  tau: a pixel whose power is below tau has alpha < alpha_min for certain
//       (o * exp(tau) <= 0.99 alpha_min; the 0.01 covers logf and exp rounding).
//  hx, hy: half-extents of a box around the mean outside which the rasterizer's
//       fp32 power is below tau.  With M = [[A, B], [B, C]] and
//       P(e) = -1/2 e^T M e, the kernel's rounded power is at most
//       P + 16u Q(e) (u = 2^-24, Q = the sum of the absolute terms), and
//       Q <= -P (1 + 2|B| / lambda_min(M)) = -P kappa; so power >= tau needs
//       e^T M e <= K = -2 tau / (1 - 16u kappa), whose bounding box is
//       |e_x| <= sqrt(K C / det M), |e_y| <= sqrt(K A / det M).  det M is
//       formed with Kahan's two-product correction; the box is widened by a
//       relative 1e-4 and by an absolute slack that covers the rounding of the
//       comparisons at the mean's magnitude.  hx = hy = -1: no pixel passes;
//       +inf: no useful bound (badly conditioned conic).
__device__ __forceinline__ void alpha_support(const ProjOut& po, float alpha_min, float& tau, float& hx, float& hy)
{
    if (!(po.opacity >= alpha_min)) {
        tau = INFINITY;
        hx = hy = -1.0f;
        return;
    }
    tau = logf(alpha_min / po.opacity) - 0.01f;
    const float A = po.cA, B = po.cB, C = po.cC;
    const float bb = B * B;
    const float bb_err = __fmaf_rn(B, B, -bb);             // exact error of B*B
    const float det = __fmaf_rn(A, C, -bb) - bb_err;       // Kahan: A C - B^2 to ~1 ulp
    const float mid = 0.5f * (A + C);
    const float lmax = mid + sqrtf(fmaxf(mid * mid - det, 0.0f));
    const float lmin = det / lmax;
    const float kappa = 1.01f * (1.0f + 2.0f * fabsf(B) / lmin) + 0.01f;
    const float eps = 16.0f * 0x1.0p-24f * kappa;
    if (!(det > 0.0f) || !(lmin > 0.0f) || !(eps < 0.5f)) {
        hx = hy = INFINITY;
        return;
    }
    const float K = -2.0f * tau / (1.0f - eps);
    hx = sqrtf(K * C / det) * 1.0001f + 1e-3f + fabsf(po.mx) * 0x1.0p-18f;
    hy = sqrtf(K * A / det) * 1.0001f + 1e-3f + fabsf(po.my) * 0x1.0p-18f;
    if (!(hx >= 0.0f) || !(hy >= 0.0f)) hx = hy = INFINITY;
}

template <int DEG>
__global__ void __launch_bounds__(128) project_kernel(ProjectArgs a, CamSet cs)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= a.n) return;
    GaussParams<DEG> gp;
    gp.load(a.params, g);
    GaussAct ac;
    activate<DEG>(gp, ac);   // view-independent: once for all views
    for (int v = 0; v < cs.n_views; ++v) {
        const size_t o = (size_t)v * (size_t)a.n + (size_t)g;
        ProjOut po;
        const bool vis = project_view<DEG>(gp, ac, cs.cam[v], a.near_z, a.lowpass, a.tiles_x, a.tiles_y, po, nullptr);
        if (!vis) {
            a.tiles_touched[o] = 0u;
            continue;
        }
        float4* r = a.rec + o * 3;
        r[0] = make_float4(po.mx, po.my, -0.5f * po.cA, po.cB);
        r[1] = make_float4(-0.5f * po.cC, po.opacity, po.col[0], po.col[1]);
        float tau, hx, hy;
        alpha_support(po, a.alpha_min, tau, hx, hy);
        r[2] = make_float4(po.col[2], tau, hx, hy);
        a.depth[o] = po.depth;
        a.rect[o] = make_ushort4((unsigned short)po.x0, (unsigned short)po.y0, (unsigned short)po.x1,
                                 (unsigned short)po.y1);
        a.tiles_touched[o] = (uint32_t)((po.x1 - po.x0) * (po.y1 - po.y0));
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_project(const float* params, int64_t n, int32_t sh_degree, const gs_camera* cams,
                                int32_t n_views, const gs_render_opts* opts, const gs_proj* out, void* stream)
{
    GS_NVTX_RANGE("gs_project");
    if (!opts_ok(opts) || !out || n < 0 || n > INT32_MAX) return GS_ERR_INVALID_ARG;
    if (param_rows(sh_degree) < 0) return GS_ERR_INVALID_ARG;
    gs_status st = check_views(cams, n_views);
    if (st != GS_OK) return st;
    if (n == 0) return GS_OK;
    if (!params || !aligned16(params) || !out->rec || !out->depth || !out->rect || !out->tiles_touched ||
        !aligned16(out->rec))
        return GS_ERR_INVALID_ARG;
    ProjectArgs a;
    a.params = params;
    a.n = n;
    a.sh_degree = sh_degree;
    a.near_z = opts->near_z;
    a.lowpass = opts->lowpass;
    a.alpha_min = opts->alpha_min;
    a.tiles_x = tiles_x_of(cams[0].width);
    a.tiles_y = tiles_y_of(cams[0].height);
    a.rec = reinterpret_cast<float4*>(out->rec);
    a.depth = out->depth;
    a.rect = reinterpret_cast<ushort4*>(out->rect);
    a.tiles_touched = out->tiles_touched;
    const CamSet cs = make_camset(cams, n_views);
    const int threads = 128;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    cudaStream_t s = (cudaStream_t)stream;
    if (sh_degree == 0)
        project_kernel<0><<<blocks, threads, 0, s>>>(a, cs);
    else
        project_kernel<3><<<blocks, threads, 0, s>>>(a, cs);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
