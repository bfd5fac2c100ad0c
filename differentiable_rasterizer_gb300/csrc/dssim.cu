// dssim.cu -- gs_dssim_loss_grad: the L1 + D-SSIM training loss of the standard
// 3DGS recipe (On Scaling Up 3D Gaussian Splatting Training, summary of the
// loss) and its gradient with respect to the rendered colour.
//
// SSIM per channel with an 11 x 11 Gaussian window (sigma 1.5), the image
// zero-padded outside its borders, C1 = 0.01^2, C2 = 0.03^2:
//   S = (2 mu_x mu_y + C1)(2 s_xy + C2) / ((mu_x^2 + mu_y^2 + C1)(s_xx + s_yy + C2))
// loss = (1 - lambda) mean|x - y| + lambda (1 - mean S).
// The gradient goes through the three windowed moments that depend on x:
//   dSSIM/dx_q = (1/N) [w * dS/dmu_x + 2 x_q (w * dS/dE[x^2]) + y_q (w * dS/dE[xy])](q)
// (w symmetric, so the adjoint of a window sum is a window sum; the maps are
// zero outside the image).  With A, B, C, D the four factors of S:
//   dS/dmu_x = (2 mu_y (B - A) - 2 mu_x S (D - C)) / (C D),
//   dS/dE[x^2] = -S / D,  dS/dE[xy] = 2 A / (C D).
//
// One CTA per (32 x 32 output tile, channel, view).  The output needs the
// derivative maps on the tile plus a 5-pixel ring (42 x 42), which need the
// moments there, which need the two images on the tile plus a 10-pixel ring
// (52 x 52).  Four separable window passes in shared memory, each thread
// sliding the 11 taps over a short run of outputs held in registers:
//   P1 rows of the 52 x 52 images  -> 5 horizontally summed products (52 x 42)
//   P2 columns                     -> moments, S and its 3 derivatives (42 x 42)
//   P3 rows of the derivative maps -> 3 x (42 x 32)
//   P4 columns                     -> dL/dC on the 32 x 32 tile
// The second moments are taken of the images minus a per-CTA constant (the mean
// of the in-image pixels of the loaded 52 x 52 region): variances and the covariance
// are invariant to the shift, so s_xx = E[x'^2] - mu_x'^2 with x' = x - c_x and
// mu_x' = mu_x - c_x sum(w), and in smooth or flat regions the cancellation that
// fp32 E[x^2] - mu_x^2 suffers is gone.  The means themselves are plain window
// sums of the (non-negative) images, accurate even where they are tiny next to a
// dark region, and the derivative maps and their combination are the unshifted
// formulas above, as in the definition.
// fp32 throughout; the loss partial sums are fp64 (one atomic per CTA).
#include "gs_common.cuh"

namespace gs {

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

namespace ssim {
constexpr int kR = 5;                 // window radius
constexpr int kWin = 2 * kR + 1;
constexpr int kTO = 32;               // output tile
constexpr int kTM = kTO + 2 * kR;     // derivative-map region (42)
constexpr int kTI = kTO + 4 * kR;     // input region (52)
constexpr int kThreads = 256;
constexpr int kK1 = 3;                // outputs per thread in P1 (kTM / kK1 runs per row)
constexpr int kK2 = 7;                // P2: 42 columns x 6 runs = 252 items, one round
constexpr int kK3 = 4;                // P3
constexpr int kK4 = 4;                // P4
static_assert(kTM % kK1 == 0 && kTM % kK2 == 0 && kTO % kK3 == 0 && kTO % kK4 == 0, "runs must tile the regions");
constexpr int kLoadIters = (kTI * kTI + kThreads - 1) / kThreads;
static_assert(kTO * (kTO / kK4) == kThreads, "P4: one run per thread");
constexpr int kSmemA = 2 * kTI * kTI;     // images (x, y interleaved), later the 3 derivative maps
constexpr int kSmemB = 5 * kTI * kTM;     // P1 sums, later the P3 sums
static_assert(3 * kTM * kTM <= kSmemA && 3 * kTM * kTO <= kSmemB, "aliased buffers must fit");
constexpr size_t kSmemBytes = sizeof(float) * (kSmemA + kSmemB);
}  // namespace ssim

struct SsimArgs {
    const float* __restrict__ image;    // [V][3][H][W]
    const float* __restrict__ target;
    float* dldc;
    double* loss;                       // [V]
    int W, H, tiles_x;
    float w[ssim::kWin];                // normalised 1-D window
    float c1, c2;
    float wsum;                         // sum of the 2-D window's fp32 weights (1 up to rounding)
    float l1_coef;                      // (1 - lambda) / N
    float ssim_coef;                    // -lambda / N (gradient of the SSIM term)
    double l1_coef_d, ssim_loss_coef_d; // (1 - lambda) / N, lambda / N
};

// Two fp32 lanes in one 64-bit register, for Blackwell's packed fp32
// instructions: each lane is an ordinary IEEE-rounded fp32 operation, so the
// results are those of the scalar operations, at one issue slot per pair.
typedef unsigned long long f2x;

__device__ __forceinline__ f2x pack2(float a, float b)
{
    f2x r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 unpack2(f2x v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ f2x fma2(f2x a, f2x b, f2x c)
{
    f2x d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2x mul2(f2x a, f2x b)
{
    f2x d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2x sub2(f2x a, f2x b)
{
    f2x d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__global__ void __launch_bounds__(ssim::kThreads, 3) dssim_kernel(SsimArgs a)
{
    using namespace ssim;
    // Shared-memory layout: pairs of quantities sit in one 8-byte slot so a
    // pass loads them with one 64-bit access and updates them with one packed
    // multiply-add.
    extern __shared__ float smem[];
    f2x* const sxy = reinterpret_cast<f2x*>(smem);                 // [kTI][kTI] (x, y)
    f2x* const dmp = reinterpret_cast<f2x*>(smem);                 // [kTM][kTM] (dS/dmu, dS/dE[x^2]) (after P1)
    float* const dms = smem + 2 * kTM * kTM;                       // [kTM][kTM] dS/dE[xy]
    f2x* const h1p = reinterpret_cast<f2x*>(smem + kSmemA);        // [2][kTI][kTM] (x, y), (x'^2, y'^2) sums
    float* const h1s = smem + kSmemA + 4 * kTI * kTM;              // [kTI][kTM] x'y' sums
    f2x* const h3p = reinterpret_cast<f2x*>(smem + kSmemA);        // [kTM][kTO] (after P2)
    float* const h3s = smem + kSmemA + 2 * kTM * kTO;              // [kTM][kTO]
    __shared__ double s_red[kThreads / 32];
    __shared__ float s_c[2][kThreads / 32];

    const int tx = blockIdx.x % a.tiles_x, ty = blockIdx.x / a.tiles_x;
    const int ch = blockIdx.y, v = blockIdx.z;
    const int ox = tx * kTO, oy = ty * kTO;       // output tile origin
    const size_t HW = (size_t)a.W * (size_t)a.H;
    const size_t plane = ((size_t)v * 3 + ch) * HW;
    const float* __restrict__ X = a.image + plane;
    const float* __restrict__ Y = a.target + plane;
    f2x w2[kWin];                                 // the window weights, one per lane
#pragma unroll
    for (int k = 0; k < kWin; ++k) w2[k] = pack2(a.w[k], a.w[k]);

    // images on the tile + 10-pixel ring, zero outside (all loads issued before
    // the first store); their means over the region's in-image pixels
    float sumx = 0.0f, sumy = 0.0f;
    {
        float lx[kLoadIters], ly[kLoadIters];
#pragma unroll
        for (int k = 0; k < kLoadIters; ++k) {
            const int i = k * kThreads + threadIdx.x;
            const int r = i / kTI, c = i - r * kTI;
            const int gy = oy - 2 * kR + r, gx = ox - 2 * kR + c;
            lx[k] = 0.0f;
            ly[k] = 0.0f;
            if (i < kTI * kTI && gy >= 0 && gy < a.H && gx >= 0 && gx < a.W) {
                const size_t o = (size_t)gy * a.W + gx;
                lx[k] = __ldg(X + o);
                ly[k] = __ldg(Y + o);
            }
        }
#pragma unroll
        for (int k = 0; k < kLoadIters; ++k) {
            const int i = k * kThreads + threadIdx.x;
            if (i < kTI * kTI) sxy[i] = pack2(lx[k], ly[k]);
            sumx += lx[k];
            sumy += ly[k];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sumx += __shfl_xor_sync(0xffffffffu, sumx, o);
        sumy += __shfl_xor_sync(0xffffffffu, sumy, o);
    }
    if ((threadIdx.x & 31) == 0) {
        s_c[0][threadIdx.x >> 5] = sumx;
        s_c[1][threadIdx.x >> 5] = sumy;
    }
    __syncthreads();
    float cx = 0.0f, cy = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        cx += s_c[0][w];
        cy += s_c[1][w];
    }
    {
        // in-image pixels of the region (at least the tile's first pixel)
        const int rows = min(oy + kTO + 2 * kR, a.H) - max(oy - 2 * kR, 0);
        const int cols = min(ox + kTO + 2 * kR, a.W) - max(ox - 2 * kR, 0);
        const float inv = 1.0f / (float)(rows * cols);
        cx = cx * inv;
        cy = cy * inv;
    }
    const f2x cxy = pack2(cx, cy);
    // this thread's P4 outputs: column tid % 32, rows 4 (tid / 32) .. + 3
    const int c4 = threadIdx.x % kTO, r4 = (threadIdx.x / kTO) * kK4;
    float ox4[kK4], oy4[kK4];
#pragma unroll
    for (int j = 0; j < kK4; ++j) {
        const float2 v2 = unpack2(sxy[(r4 + j + 2 * kR) * kTI + c4 + 2 * kR]);
        ox4[j] = v2.x;
        oy4[j] = v2.y;
    }

    // P1: horizontal window sums of (x, y), (x'^2, y'^2) and x'y'
    constexpr int kRuns1 = kTM / kK1;
    for (int it = threadIdx.x; it < kTI * kRuns1; it += kThreads) {
        const int r = it / kRuns1, c0 = (it - r * kRuns1) * kK1;
        f2x am[kK1], aq[kK1];
        float ac[kK1];
#pragma unroll
        for (int j = 0; j < kK1; ++j) {
            am[j] = 0ull;
            aq[j] = 0ull;
            ac[j] = 0.0f;
        }
#pragma unroll
        for (int t = 0; t < kK1 + 2 * kR; ++t) {
            const f2x xy = sxy[r * kTI + c0 + t];
            const f2x d = sub2(xy, cxy);
            const f2x sq = mul2(d, d);
            const float2 dd = unpack2(d);
            const float cr = dd.x * dd.y;
#pragma unroll
            for (int j = 0; j < kK1; ++j) {
                const int k = t - j;
                if (k >= 0 && k < kWin) {
                    am[j] = fma2(w2[k], xy, am[j]);
                    aq[j] = fma2(w2[k], sq, aq[j]);
                    ac[j] = __fmaf_rn(a.w[k], cr, ac[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kK1; ++j) {
            const int o = r * kTM + c0 + j;
            h1p[o] = am[j];
            h1p[kTI * kTM + o] = aq[j];
            h1s[o] = ac[j];
        }
    }
    __syncthreads();

    // P2: vertical sums -> moments; S and its derivatives on the 42 x 42 region
    // (zero outside the image); S summed over the output tile for the loss
    double ssum = 0.0;
    constexpr int kRuns2 = kTM / kK2;
    for (int it = threadIdx.x; it < kTM * kRuns2; it += kThreads) {
        const int c = it % kTM, r0 = (it / kTM) * kK2;
        f2x mm[kK2], mq[kK2];
        float mc[kK2];
#pragma unroll
        for (int j = 0; j < kK2; ++j) {
            mm[j] = 0ull;
            mq[j] = 0ull;
            mc[j] = 0.0f;
        }
#pragma unroll
        for (int t = 0; t < kK2 + 2 * kR; ++t) {
            const int o = (r0 + t) * kTM + c;
            const f2x hm = h1p[o], hq = h1p[kTI * kTM + o];
            const float hc = h1s[o];
#pragma unroll
            for (int j = 0; j < kK2; ++j) {
                const int k = t - j;
                if (k >= 0 && k < kWin) {
                    mm[j] = fma2(w2[k], hm, mm[j]);
                    mq[j] = fma2(w2[k], hq, mq[j]);
                    mc[j] = __fmaf_rn(a.w[k], hc, mc[j]);
                }
            }
        }
        const int gx = ox - kR + c;
#pragma unroll
        for (int j = 0; j < kK2; ++j) {
            const int r = r0 + j;
            const int gy = oy - kR + r;
            float dmu = 0.0f, dxx = 0.0f, dxy = 0.0f;
            if (gy >= 0 && gy < a.H && gx >= 0 && gx < a.W) {
                const float2 m01 = unpack2(mm[j]), m23 = unpack2(mq[j]);
                const float mx = m01.x, my = m01.y;
                const float mxs = mx - cx * a.wsum, mys = my - cy * a.wsum;   // means of x', y'
                const float A = 2.0f * (mx * my) + a.c1;
                const float B = 2.0f * (mc[j] - mxs * mys) + a.c2;
                const float C = (mx * mx + my * my) + a.c1;
                const float D = ((m23.x - mxs * mxs) + (m23.y - mys * mys)) + a.c2;
                // C >= C1 and D >= C2: far from the approximate reciprocal's limits
                const float rC = rcp_approx(C), rD = rcp_approx(D);
                const float inv = rC * rD;
                const float S = (A * B) * inv;
                dmu = (2.0f * my * (B - A) - 2.0f * mx * S * (D - C)) * inv;
                dxx = -S * rD;
                dxy = 2.0f * A * inv;
                if (r >= kR && r < kR + kTO && c >= kR && c < kR + kTO) ssum += (double)(1.0f - S);
            }
            dmp[r * kTM + c] = pack2(dmu, dxx);
            dms[r * kTM + c] = dxy;
        }
    }
    __syncthreads();

    // P3: horizontal sums of the derivative maps (42 rows x 32 columns)
    constexpr int kRuns3 = kTO / kK3;
    for (int it = threadIdx.x; it < kTM * kRuns3; it += kThreads) {
        const int r = it / kRuns3, c0 = (it - r * kRuns3) * kK3;
        f2x ap[kK3];
        float as[kK3];
#pragma unroll
        for (int j = 0; j < kK3; ++j) {
            ap[j] = 0ull;
            as[j] = 0.0f;
        }
#pragma unroll
        for (int t = 0; t < kK3 + 2 * kR; ++t) {
            const f2x dp = dmp[r * kTM + c0 + t];
            const float ds = dms[r * kTM + c0 + t];
#pragma unroll
            for (int j = 0; j < kK3; ++j) {
                const int k = t - j;
                if (k >= 0 && k < kWin) {
                    ap[j] = fma2(w2[k], dp, ap[j]);
                    as[j] = __fmaf_rn(a.w[k], ds, as[j]);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kK3; ++j) {
            h3p[r * kTO + c0 + j] = ap[j];
            h3s[r * kTO + c0 + j] = as[j];
        }
    }
    __syncthreads();

    // P4: vertical sums -> dL/dC on the output tile (one 4-row run per thread)
    double l1sum = 0.0;
    {
        f2x bp[kK4];
        float bs[kK4];
#pragma unroll
        for (int j = 0; j < kK4; ++j) {
            bp[j] = 0ull;
            bs[j] = 0.0f;
        }
#pragma unroll
        for (int t = 0; t < kK4 + 2 * kR; ++t) {
            const f2x hp = h3p[(r4 + t) * kTO + c4];
            const float hs = h3s[(r4 + t) * kTO + c4];
#pragma unroll
            for (int j = 0; j < kK4; ++j) {
                const int k = t - j;
                if (k >= 0 && k < kWin) {
                    bp[j] = fma2(w2[k], hp, bp[j]);
                    bs[j] = __fmaf_rn(a.w[k], hs, bs[j]);
                }
            }
        }
        const int gx = ox + c4;
#pragma unroll
        for (int j = 0; j < kK4; ++j) {
            const int gy = oy + r4 + j;
            if (gy < a.H && gx < a.W) {
                const float x = ox4[j], y = oy4[j];
                const float d = x - y;
                const float sgn = d > 0.0f ? 1.0f : (d < 0.0f ? -1.0f : 0.0f);
                const float2 b01 = unpack2(bp[j]);
                const float gs = b01.x + 2.0f * x * b01.y + y * bs[j];
                a.dldc[plane + (size_t)gy * a.W + gx] = __fmaf_rn(a.ssim_coef, gs, sgn * a.l1_coef);
                l1sum += (double)fabsf(d);
            }
        }
    }

    // loss partial: (1 - lambda)/N sum|x - y| + lambda/N sum(1 - S)
    double part = l1sum * a.l1_coef_d + ssum * a.ssim_loss_coef_d;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) t += s_red[w];
        if (t != 0.0) atomicAdd(a.loss + v, t);
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_dssim_loss_grad(const float* image, const float* target, int32_t n_views, int32_t width,
                                        int32_t height, float lambda, double* loss, float* dldc, void* stream)
{
    GS_NVTX_RANGE("gs_dssim_loss_grad");
    using namespace ssim;
    if (!image || !target || !loss || !dldc) return GS_ERR_INVALID_ARG;
    if (n_views < 1 || n_views > GS_MAX_VIEWS || width < 1 || height < 1) return GS_ERR_INVALID_ARG;
    if (!(lambda >= 0.0f && lambda <= 1.0f)) return GS_ERR_INVALID_ARG;
    SsimArgs a;
    a.image = image;
    a.target = target;
    a.dldc = dldc;
    a.loss = loss;
    a.W = width;
    a.H = height;
    a.tiles_x = (width + kTO - 1) / kTO;
    const long long tiles_y = (height + kTO - 1) / kTO;
    const long long tiles = (long long)a.tiles_x * tiles_y;
    if (tiles > INT32_MAX) return GS_ERR_INVALID_ARG;
    double g[kWin], gsum = 0.0;
    for (int i = 0; i < kWin; ++i) {
        const double t = (double)(i - kR);
        g[i] = exp(-t * t / (2.0 * 1.5 * 1.5));
        gsum += g[i];
    }
    double ws = 0.0;
    for (int i = 0; i < kWin; ++i) {
        a.w[i] = (float)(g[i] / gsum);
        ws += (double)a.w[i];
    }
    a.wsum = (float)(ws * ws);
    a.c1 = (float)(0.01 * 0.01);
    a.c2 = (float)(0.03 * 0.03);
    const double N = 3.0 * (double)width * (double)height;
    a.l1_coef_d = (1.0 - (double)lambda) / N;
    a.ssim_loss_coef_d = (double)lambda / N;
    a.l1_coef = (float)a.l1_coef_d;
    a.ssim_coef = (float)(-(double)lambda / N);
    cudaStream_t s = (cudaStream_t)stream;
    // more than the 48 KB default of dynamic shared memory (set on the current device)
    GS_CUDA_TRY(cudaFuncSetAttribute(dssim_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes));
    GS_CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(double) * (size_t)n_views, s));
    dssim_kernel<<<dim3((unsigned)tiles, 3, (unsigned)n_views), kThreads, kSmemBytes, s>>>(a);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
