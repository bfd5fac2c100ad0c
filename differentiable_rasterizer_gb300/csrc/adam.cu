// adam.cu -- gs_adam_deferred: Adam applied only to the Gaussians with a
// gradient this step (GS-Scale, abstract: the optimizer update of Gaussians
// whose gradient is zero is deferred, saving their memory traffic), made exactly
// equal to dense Adam by replaying the skipped zero-gradient steps first.
//
// Work unit: a (listed Gaussian, float4 chunk of its [stride] parameter block)
// pair, 16 contiguous bytes of params, m, v and grads (grads only read: the
// decoder overwrites a Gaussian's block in the step it lists it); a grid of resident
// blocks strides over the units.  Elements with a zero gradient on a zero state
// are exact no-ops and skip the arithmetic.  The bias
// corrections of the current step come from the host (the same fp64 binary
// exponentiation as the device code, so the same values); replayed steps
// compute their own.  A row whose moments are both +0 skips the replay: a
// zero-gradient step from a zero state changes nothing, bit for bit.
// last_step is only read by the update kernel; stamp_kernel writes it after.
#include "gs_common.cuh"

#include <cfloat>

namespace gs {

__host__ __device__ __forceinline__ double powi_binary(double b, int e)
{
    double r = 1.0;
    while (e > 0) {
        if (e & 1) r *= b;
        b *= b;
        e >>= 1;
    }
    return r;
}

struct AdamArgs {
    float* __restrict__ params;
    float* __restrict__ grads;
    float* __restrict__ m;
    float* __restrict__ v;
    int32_t* __restrict__ last_step;
    int64_t n;
    const uint32_t* idx;
    const int64_t* n_idx;
    int32_t t;
    float lr[5];
    float b1, b2, eps;
    float bc1t, bc2t;   // bias corrections of step t
};

__device__ __forceinline__ void adam_one(float& p, float& m, float& v, float g, float lr, float b1, float b2, float eps,
                                         float bc1, float bc2)
{
    const float mn = b1 * m + (1.0f - b1) * g;
    const float vn = b2 * v + (1.0f - b2) * (g * g);
    const float den = sqrtf(vn / bc2) + eps;
    p = p - lr * ((mn / bc1) / den);
    m = mn;
    v = vn;
}

// A zero gradient on a zero state (m = v = +0) leaves p, m and v exactly as they
// are: m' = v' = +0 and the step is lr * (+0 / (eps + 0)) = +0 (lr >= 0 and
// finite, eps > 0, beta < 1, checked on entry).  Such elements -- the padding of
// each parameter block, colour channels that never received a gradient -- skip
// the IEEE divisions and square root, whose zero-operand paths are slow.
__device__ __forceinline__ void adam_step(float& p, float& m, float& v, float g, float lr, float b1, float b2,
                                          float eps, float bc1, float bc2)
{
    if (g == 0.0f && __float_as_uint(m) == 0u && __float_as_uint(v) == 0u) return;
    adam_one(p, m, v, g, lr, b1, b2, eps, bc1, bc2);
}

// One replayed zero-gradient step of one parameter (a zero state is skipped).
__device__ __forceinline__ void adam_zero_step(float& p, float& m, float& v, float lr, float b1, float b2, float eps,
                                               float bc1, float bc2)
{
    if (__float_as_uint(m) == 0u && __float_as_uint(v) == 0u) return;
    adam_one(p, m, v, 0.0f, lr, b1, b2, eps, bc1, bc2);
}

// Learning-rate group of parameter k: mean, log-scale, quaternion, opacity, colour.
__device__ __forceinline__ float lr_of(const AdamArgs& a, int k)
{
    return k < 3 ? a.lr[0] : (k < 6 ? a.lr[1] : (k < 10 ? a.lr[2] : (k == 10 ? a.lr[3] : a.lr[4])));
}

// Work unit: one (listed Gaussian, float4 chunk of its parameter block) pair --
// 16 contiguous bytes of params, m, v and grads -- over the chunks that hold
// parameters (4 of 4 for RGB, 15 of 16 for SH 3: the 16th is all padding).  A
// grid of resident blocks strides over the units (the list length lives on the
// device); per unit the loads come in two dependent rounds: the Gaussian index,
// then its parameter block with last_step.
template <int DEG, bool kFlush>
__global__ void __launch_bounds__(256, 5) adam_deferred_kernel(AdamArgs a)
{
    constexpr int kStride = DEG == 0 ? 16 : 64;
    constexpr int kChunks = DEG == 0 ? 4 : 15;
    const int64_t count = kFlush ? a.n : *a.n_idx;
    const int64_t total = count * kChunks;
    const float4 zero = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t e = i / kChunks;
        const int c = (int)(i - e * kChunks);
        const int64_t g = kFlush ? e : (int64_t)__ldg(a.idx + e);
        if (!kFlush && !GS_IN_RANGE(g, a.n, GS_CHECK_ADAM_ID)) continue;
        const size_t off = (size_t)g * kStride + 4 * c;
        float4 p = *reinterpret_cast<const float4*>(a.params + off);
        float4 m = *reinterpret_cast<const float4*>(a.m + off);
        float4 v = *reinterpret_cast<const float4*>(a.v + off);
        const float4 gr = kFlush ? zero : *reinterpret_cast<const float4*>(a.grads + off);
        const int s = a.last_step[g];
        if (s >= a.t) continue;
        const int k = 4 * c;
        const float l0 = lr_of(a, k), l1 = lr_of(a, k + 1), l2 = lr_of(a, k + 2), l3 = lr_of(a, k + 3);
        // catch up the zero-gradient steps s+1 .. t-1 (rare: the Gaussian was not
        // touched in the previous step)
        for (int j = s + 1; j < a.t; ++j) {
            const float bc1 = (float)(1.0 - powi_binary((double)a.b1, j));
            const float bc2 = (float)(1.0 - powi_binary((double)a.b2, j));
            adam_zero_step(p.x, m.x, v.x, l0, a.b1, a.b2, a.eps, bc1, bc2);
            adam_zero_step(p.y, m.y, v.y, l1, a.b1, a.b2, a.eps, bc1, bc2);
            adam_zero_step(p.z, m.z, v.z, l2, a.b1, a.b2, a.eps, bc1, bc2);
            adam_zero_step(p.w, m.w, v.w, l3, a.b1, a.b2, a.eps, bc1, bc2);
        }
        adam_step(p.x, m.x, v.x, gr.x, l0, a.b1, a.b2, a.eps, a.bc1t, a.bc2t);
        adam_step(p.y, m.y, v.y, gr.y, l1, a.b1, a.b2, a.eps, a.bc1t, a.bc2t);
        adam_step(p.z, m.z, v.z, gr.z, l2, a.b1, a.b2, a.eps, a.bc1t, a.bc2t);
        adam_step(p.w, m.w, v.w, gr.w, l3, a.b1, a.b2, a.eps, a.bc1t, a.bc2t);
        *reinterpret_cast<float4*>(a.params + off) = p;
        *reinterpret_cast<float4*>(a.m + off) = m;
        *reinterpret_cast<float4*>(a.v + off) = v;
    }
}

template <bool kFlush>
__global__ void __launch_bounds__(256) stamp_kernel(AdamArgs a)
{
    const int64_t count = kFlush ? a.n : *a.n_idx;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = kFlush ? i : (int64_t)a.idx[i];
        if (!kFlush && !GS_IN_RANGE(g, a.n, GS_CHECK_ADAM_ID)) continue;
        if (a.last_step[g] < a.t) a.last_step[g] = a.t;
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_adam_deferred(float* params, float* grads, float* m, float* v, int32_t* last_step, int64_t n,
                                      int32_t sh_degree, const uint32_t* idx, const int64_t* n_idx, int32_t t,
                                      const float* lr, float beta1, float beta2, float eps, int32_t flush, void* stream)
{
    GS_NVTX_RANGE("gs_adam_deferred");
    const int rows = param_rows(sh_degree);
    if (rows < 0 || !lr || n < 0 || n > INT32_MAX || t < 1) return GS_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        if (!(lr[i] >= 0.0f && lr[i] <= FLT_MAX)) return GS_ERR_INVALID_ARG;
    if (!(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f && eps > 0.0f && eps <= FLT_MAX))
        return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    if (!params || !m || !v || !last_step) return GS_ERR_INVALID_ARG;
    if (!flush && (!grads || !idx || !n_idx)) return GS_ERR_INVALID_ARG;
    if (!aligned16(params) || !aligned16(m) || !aligned16(v) || (!flush && !aligned16(grads))) return GS_ERR_INVALID_ARG;
    AdamArgs a;
    a.params = params;
    a.grads = grads;
    a.m = m;
    a.v = v;
    a.last_step = last_step;
    a.n = n;
    a.idx = idx;
    a.n_idx = n_idx;
    a.t = t;
    for (int i = 0; i < 5; ++i) a.lr[i] = lr[i];
    a.b1 = beta1;
    a.b2 = beta2;
    a.eps = eps;
    a.bc1t = (float)(1.0 - powi_binary((double)beta1, t));
    a.bc2t = (float)(1.0 - powi_binary((double)beta2, t));
    int dev = 0, sms = 0;
    GS_CUDA_TRY(cudaGetDevice(&dev));
    GS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // The list length lives on the device: a grid of resident blocks strides
    // over it (at most n entries).
    const int threads = 256;
    const int chunks = sh_degree == 0 ? 4 : 15;
    int64_t bx = (n * chunks + threads - 1) / threads;
    if (bx > (int64_t)sms * 5) bx = (int64_t)sms * 5;   // 5 resident blocks per SM
    int64_t bs = (n + threads - 1) / threads;
    if (bs > (int64_t)sms * 8) bs = (int64_t)sms * 8;
    cudaStream_t s = (cudaStream_t)stream;
    if (flush) {
        if (sh_degree == 0) adam_deferred_kernel<0, true><<<(unsigned)bx, threads, 0, s>>>(a);
        else adam_deferred_kernel<3, true><<<(unsigned)bx, threads, 0, s>>>(a);
        GS_LAUNCH_CHECK();
        stamp_kernel<true><<<(unsigned)bs, threads, 0, s>>>(a);
    } else {
        if (sh_degree == 0) adam_deferred_kernel<0, false><<<(unsigned)bx, threads, 0, s>>>(a);
        else adam_deferred_kernel<3, false><<<(unsigned)bx, threads, 0, s>>>(a);
        GS_LAUNCH_CHECK();
        stamp_kernel<false><<<(unsigned)bs, threads, 0, s>>>(a);
    }
    GS_LAUNCH_CHECK();
    return GS_OK;
}
