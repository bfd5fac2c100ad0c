// adam.cu -- gs_adam_deferred: Adam applied only to the Gaussians with a
// gradient this step (GS-Scale, abstract: "deferred optimizer update to minimize
// unnecessary memory accesses for Gaussians with zero gradients"), made exactly
// equal to dense Adam by replaying the skipped zero-gradient steps first.
//
// One thread per (listed Gaussian, group of 4 parameter rows): the loads of all
// its rows are issued before any arithmetic, and consecutive threads touch
// consecutive Gaussians of a row (coalesced when the list is dense).  The bias
// corrections of the current step come from the host (the same fp64 binary
// exponentiation as the device code, so the same values); replayed steps
// compute their own.  A row whose moments are both +0 skips the replay: a
// zero-gradient step from a zero state changes nothing, bit for bit.
// last_step is only read by the update kernel; stamp_kernel writes it after.
#include "gs_common.cuh"

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
    int32_t rows;
    const uint32_t* idx;
    const int64_t* n_idx;
    int32_t t;
    float lr[5];
    float b1, b2, eps;
    float bc1t, bc2t;   // bias corrections of step t
    int32_t flush;
};

constexpr int kRowsPerThread = 4;

__device__ __forceinline__ int row_group(int r) { return r < 3 ? 0 : (r < 6 ? 1 : (r < 10 ? 2 : (r == 10 ? 3 : 4))); }

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

__global__ void __launch_bounds__(256) adam_deferred_kernel(AdamArgs a)
{
    const int64_t count = a.flush ? a.n : *a.n_idx;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count) return;
    const int64_t g = a.flush ? i : (int64_t)a.idx[i];
    const int s = a.last_step[g];
    if (s >= a.t) return;
    const int r0 = blockIdx.y * kRowsPerThread;
    float p[kRowsPerThread], m[kRowsPerThread], v[kRowsPerThread], gr[kRowsPerThread];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const int r = r0 + k;
        if (r < a.rows) {
            const size_t e = (size_t)r * a.n + g;
            p[k] = a.params[e];
            m[k] = a.m[e];
            v[k] = a.v[e];
            gr[k] = a.flush ? 0.0f : a.grads[e];
        }
    }
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
        const int r = r0 + k;
        if (r >= a.rows) break;
        const float lr = a.lr[row_group(r)];
        for (int j = s + 1; j < a.t; ++j) {
            if (__float_as_uint(m[k]) == 0u && __float_as_uint(v[k]) == 0u) break;   // zero state: replay is a no-op
            const float bc1 = (float)(1.0 - powi_binary((double)a.b1, j));
            const float bc2 = (float)(1.0 - powi_binary((double)a.b2, j));
            adam_one(p[k], m[k], v[k], 0.0f, lr, a.b1, a.b2, a.eps, bc1, bc2);
        }
        adam_one(p[k], m[k], v[k], gr[k], lr, a.b1, a.b2, a.eps, a.bc1t, a.bc2t);
        const size_t e = (size_t)r * a.n + g;
        a.params[e] = p[k];
        a.m[e] = m[k];
        a.v[e] = v[k];
        if (!a.flush) a.grads[e] = 0.0f;
    }
}

__global__ void __launch_bounds__(256) stamp_kernel(AdamArgs a)
{
    const int64_t count = a.flush ? a.n : *a.n_idx;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = a.flush ? i : (int64_t)a.idx[i];
        if (a.last_step[g] < a.t) a.last_step[g] = a.t;
    }
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_adam_deferred(float* params, float* grads, float* m, float* v, int32_t* last_step, int64_t n,
                                      int32_t sh_degree, const uint32_t* idx, const int64_t* n_idx, int32_t t,
                                      const float* lr, float beta1, float beta2, float eps, int32_t flush, void* stream)
{
    const int rows = param_rows(sh_degree);
    if (rows < 0 || !lr || n < 0 || n > INT32_MAX || t < 1) return GS_ERR_INVALID_ARG;
    if (n == 0) return GS_OK;
    if (!params || !m || !v || !last_step) return GS_ERR_INVALID_ARG;
    if (!flush && (!grads || !idx || !n_idx)) return GS_ERR_INVALID_ARG;
    AdamArgs a;
    a.params = params;
    a.grads = grads;
    a.m = m;
    a.v = v;
    a.last_step = last_step;
    a.n = n;
    a.rows = rows;
    a.idx = idx;
    a.n_idx = n_idx;
    a.t = t;
    for (int i = 0; i < 5; ++i) a.lr[i] = lr[i];
    a.b1 = beta1;
    a.b2 = beta2;
    a.eps = eps;
    a.bc1t = (float)(1.0 - powi_binary((double)beta1, t));
    a.bc2t = (float)(1.0 - powi_binary((double)beta2, t));
    a.flush = flush ? 1 : 0;
    int dev = 0, sms = 0;
    GS_CUDA_TRY(cudaGetDevice(&dev));
    GS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // The list length lives on the device: the grid covers n entries and threads
    // beyond the list return at once.
    const int threads = 256;
    const int64_t bx = (n + threads - 1) / threads;
    const unsigned by = (unsigned)((rows + kRowsPerThread - 1) / kRowsPerThread);
    cudaStream_t s = (cudaStream_t)stream;
    adam_deferred_kernel<<<dim3((unsigned)bx, by), threads, 0, s>>>(a);
    GS_LAUNCH_CHECK();
    int64_t bs = (n + threads - 1) / threads;
    if (bs > (int64_t)sms * 8) bs = (int64_t)sms * 8;
    stamp_kernel<<<(unsigned)bs, threads, 0, s>>>(a);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
