// gs_common.cuh -- shared device code of the GB300 3DGS library (sm_103a).
//
// Every translation unit is compiled with -fmad=false and IEEE division and
// square root, so expressions written here round exactly as written: the
// forward decisions (cull, tile rect, alpha skip, transmittance stop) are then
// reproducible bit for bit on a CPU.  Fused multiply-adds appear only where the
// code spells them (__fmaf_rn).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/gs.h"

namespace gs {

constexpr int kTile = GS_TILE;
constexpr int kTileThreads = kTile * kTile;   // one thread per pixel of a tile

// ---------------------------------------------------------------------------
// Portable exponential (fp32).
//   x = k ln2 + r with k = rint(x log2 e) (Cody & Waite 1980 reduction with
//   ln 2 split into a 16-bit head and its remainder, both applied with fma),
//   e^r by the Taylor series to degree 7 in Horner form with fma,
//   2^k applied as two exact power-of-two multiplies 2^(k>>1) * 2^(k-(k>>1)).
// Input clamped to [-104, 89]; NaN passes through.  The constants are the fp32
// roundings of log2(e), ln 2 (head 0.693145751953125 and remainder) and 1/j!.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ float pexp(float x)
{
    if (x != x) return x;
    x = x < -104.0f ? -104.0f : x;
    x = x > 89.0f ? 89.0f : x;
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = 0x1.7f7d1cp-20f;
    const float k = rintf(x * log2e);
    float r = __fmaf_rn(-k, ln2_hi, x);
    r = __fmaf_rn(-k, ln2_lo, r);
    float p = 0x1.a01a02p-13f;               // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);    // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);     // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);     // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);     // 1/3!
    p = __fmaf_rn(p, r, 0.5f);               // 1/2!
    p = __fmaf_rn(p, r, 1.0f);               // 1/1!
    p = __fmaf_rn(p, r, 1.0f);               // 1/0!
    const int ki = (int)k;
    const int k1 = ki >> 1;
    const int k2 = ki - k1;
    return (p * pow2i(k1)) * pow2i(k2);
}

// The same function on x in [-86, 0], in fewer instructions and bit-identical
// there: rint(y) for |y| < 2^22 is (y + 1.5*2^23) - 1.5*2^23 under round-to-
// nearest-even, the reduction and polynomial are unchanged, and because
// k >= -124 the result p * 2^k is a normal number, so both the two-step scaling
// above and adding k to the exponent field (the low bits of y + 1.5*2^23 are
// k, shifted into place) are exact.
__device__ __forceinline__ float pexp_neg(float x)
{
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = 0x1.7f7d1cp-20f;
    const float magic = 12582912.0f;          // 1.5 * 2^23
    const float t = x * log2e + magic;        // -fmad=false: multiply, then add
    const float k = t - magic;
    float r = __fmaf_rn(-k, ln2_hi, x);
    r = __fmaf_rn(-k, ln2_lo, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// ---------------------------------------------------------------------------
// Real spherical harmonics up to degree 3: orthonormal on the sphere, no
// Condon-Shortley phase, coefficient k = l^2 + l + m.  Normalisations
// sqrt((2l+1)/(4pi) (l-|m|)!/(l+|m|)!) (x sqrt 2 for m != 0) folded with the
// Cartesian factors, rounded to fp32:
//   K0 = 1/(2 sqrt pi)         K1 = sqrt(3/(4 pi))      K2 = sqrt(15/pi)/2
//   K3 = sqrt(5/pi)/4          K4 = sqrt(15/pi)/4       K5 = sqrt(35/(2 pi))/4
//   K6 = sqrt(105/pi)/2        K7 = sqrt(21/(2 pi))/4   K8 = sqrt(7/pi)/4
//   K9 = sqrt(105/pi)/4
// ---------------------------------------------------------------------------
struct SH {
    static constexpr float K0 = 0x1.20dd76p-2f;
    static constexpr float K1 = 0x1.f45438p-2f;
    static constexpr float K2 = 0x1.17b142p+0f;
    static constexpr float K3 = 0x1.42f602p-2f;
    static constexpr float K4 = 0x1.17b142p-1f;
    static constexpr float K5 = 0x1.2e1a32p-1f;
    static constexpr float K6 = 0x1.71ff8ep+1f;
    static constexpr float K7 = 0x1.d403d0p-2f;
    static constexpr float K8 = 0x1.7e21f0p-2f;
    static constexpr float K9 = 0x1.71ff8ep+0f;
};

__device__ __forceinline__ void sh_basis(float x, float y, float z, float Y[16])
{
    const float xx = x * x, yy = y * y, zz = z * z, xy = x * y, yz = y * z, xz = x * z;
    Y[0] = SH::K0;
    Y[1] = SH::K1 * y;
    Y[2] = SH::K1 * z;
    Y[3] = SH::K1 * x;
    Y[4] = SH::K2 * xy;
    Y[5] = SH::K2 * yz;
    Y[6] = SH::K3 * ((2.0f * zz - xx) - yy);
    Y[7] = SH::K2 * xz;
    Y[8] = SH::K4 * (xx - yy);
    Y[9] = SH::K5 * (y * (3.0f * xx - yy));
    Y[10] = SH::K6 * (xy * z);
    Y[11] = SH::K7 * (y * ((4.0f * zz - xx) - yy));
    Y[12] = SH::K8 * (z * ((2.0f * zz - 3.0f * xx) - 3.0f * yy));
    Y[13] = SH::K7 * (x * ((4.0f * zz - xx) - yy));
    Y[14] = SH::K9 * (z * (xx - yy));
    Y[15] = SH::K5 * (x * (xx - 3.0f * yy));
}

// Cameras and options by value (kernel parameters).
struct CamSet {
    gs_camera cam[GS_MAX_VIEWS];
    int32_t n_views;
};

// One NVTX range per C-ABI call, named after the call (it groups the call's
// kernels in Nsight Systems and in ncu's --nvtx range filters).  NVTX 3 is
// header-only: with no tool attached, a push and a pop cost a pointer check.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define GS_NVTX_RANGE(name) ::gs::NvtxRange gs_nvtx_range_(name)

// ---------------------------------------------------------------------------
// Bounds checks (-DGS_CHECKED).  GS_IN_RANGE(i, n, site) is true when
// 0 <= i < n.  In the checked build a false result is counted in this
// translation unit's check record -- failures, then the site, index and bound of
// the first -- and the caller skips the access; in the plain build the macro is
// the constant true and its arguments are not evaluated.  Each unit registers a
// host reader of its record with the library (abi.cu), which gs_check_report
// calls; the registration only stores a function pointer.
// ---------------------------------------------------------------------------
#ifdef GS_CHECKED
using CheckReader = cudaError_t (*)(unsigned long long out[4]);   // copies the record out, then clears it
void register_check_reader(CheckReader reader);

namespace {
__device__ unsigned long long g_check[4];

__device__ __noinline__ void check_record(long long i, long long n, int site)
{
    if (atomicAdd(&g_check[0], 1ull) == 0ull) {
        g_check[1] = (unsigned long long)site;
        g_check[2] = (unsigned long long)i;
        g_check[3] = (unsigned long long)n;
    }
}

__device__ __forceinline__ bool in_range(long long i, long long n, int site)
{
    if (i >= 0 && i < n) return true;
    check_record(i, n, site);
    return false;
}

cudaError_t read_check_record(unsigned long long out[4])
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_check, sizeof(unsigned long long) * 4);
    if (e != cudaSuccess) return e;
    const unsigned long long zero[4] = {0ull, 0ull, 0ull, 0ull};
    return cudaMemcpyToSymbol(g_check, zero, sizeof zero);
}

struct CheckRegistrar {
    CheckRegistrar() { register_check_reader(&read_check_record); }
};
const CheckRegistrar g_check_registrar;
}  // namespace
#define GS_IN_RANGE(i, n, site) (::gs::in_range((long long)(i), (long long)(n), (site)))
#else
#define GS_IN_RANGE(i, n, site) true
#endif

// Status plumbing for host code.
#define GS_CUDA_TRY(expr)                                      \
    do {                                                       \
        cudaError_t _e = (expr);                               \
        if (_e != cudaSuccess) return GS_ERR_CUDA;             \
    } while (0)

#define GS_LAUNCH_CHECK() GS_CUDA_TRY(cudaPeekAtLastError())

inline int param_rows(int sh_degree) { return sh_degree == 0 ? 14 : (sh_degree == 3 ? 59 : -1); }
// Floats per Gaussian in the parameter, gradient and moment buffers.
inline int param_stride(int sh_degree) { return sh_degree == 0 ? 16 : (sh_degree == 3 ? 64 : -1); }

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Checks shared by the entry points: sizes and a common view resolution.
inline gs_status check_views(const gs_camera* cams, int32_t n_views)
{
    if (!cams || n_views < 1 || n_views > GS_MAX_VIEWS) return GS_ERR_INVALID_ARG;
    for (int v = 0; v < n_views; ++v) {
        if (cams[v].width <= 0 || cams[v].height <= 0) return GS_ERR_INVALID_ARG;
        if (cams[v].width != cams[0].width || cams[v].height != cams[0].height) return GS_ERR_INVALID_ARG;
        if (cams[v].width > 65535 * kTile || cams[v].height > 65535 * kTile) return GS_ERR_INVALID_ARG;
    }
    return GS_OK;
}

// alpha_min must lie in [1e-30, alpha_max], alpha_max in (0, 1), t_min >= 0: the
// rasterizer's per-Gaussian cut ln(alpha_min / o) then stays above -86, where
// pexp_neg is exact, and 1 - alpha never reaches 0.
inline bool opts_ok(const gs_render_opts* o)
{
    return o && o->alpha_min >= 1e-30f && o->alpha_min <= o->alpha_max && o->alpha_max > 0.0f &&
           o->alpha_max < 1.0f && o->t_min >= 0.0f && o->near_z > 0.0f && o->lowpass >= 0.0f;
}

inline CamSet make_camset(const gs_camera* cams, int32_t n_views)
{
    CamSet s;
    for (int v = 0; v < n_views; ++v) s.cam[v] = cams[v];
    for (int v = n_views; v < GS_MAX_VIEWS; ++v) s.cam[v] = cams[0];
    s.n_views = n_views;
    return s;
}

inline int tiles_x_of(int w) { return (w + kTile - 1) / kTile; }
inline int tiles_y_of(int h) { return (h + kTile - 1) / kTile; }

}  // namespace gs
