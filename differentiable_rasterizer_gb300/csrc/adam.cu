// adam.cu -- gs_adam_deferred: Adam applied only to the Gaussians with a
// gradient this step (GS-Scale, abstract: "deferred optimizer update to minimize
// unnecessary memory accesses for Gaussians with zero gradients"), made exactly
// equal to dense Adam by replaying the skipped zero-gradient steps first.
//
// One thread per (parameter row, listed Gaussian), coalesced across the warp when
// the list is dense.  The bias corrections of the current step are computed once
// per block; replayed steps compute their own.  A row whose
// moments are both +0 is left as is during replay: a zero-gradient step from a
// zero state changes nothing, bit for bit.
#include "gs_common.cuh"

namespace gs {

__device__ __forceinline__ double powi_binary(double b, int e)
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
    int32_t flush;
};

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

// One thread per (parameter row, listed Gaussian): every thread does its own
// 4 loads and 4 stores, so the whole list streams through HBM at full width.
// last_step is only read here; stamp_kernel writes it afterwards.
__global__ void __launch_bounds__(256) adam_deferred_kernel(AdamArgs a)
{
    __shared__ float s_bc[2];
    if (threadIdx.x == 0) {
        s_bc[0] = (float)(1.0 - powi_binary((double)a.b1, a.t));
        s_bc[1] = (float)(1.0 - powi_binary((double)a.b2, a.t));
    }
    __syncthreads();
    const float bc1t = s_bc[0], bc2t = s_bc[1];
    const int64_t count = a.flush ? a.n : *a.n_idx;
    const int r = blockIdx.y;
    const float lr = a.lr[row_group(r)];
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = a.flush ? i : (int64_t)a.idx[i];
        const int s = a.last_step[g];
        if (s >= a.t) continue;
        const size_t e = (size_t)r * a.n + g;
        float p = a.params[e], m = a.m[e], v = a.v[e];
        const float gr = a.flush ? 0.0f : a.grads[e];
        for (int j = s + 1; j < a.t; ++j) {
            if (__float_as_uint(m) == 0u && __float_as_uint(v) == 0u) break;   // zero state: replay is a no-op
            const float bc1 = (float)(1.0 - powi_binary((double)a.b1, j));
            const float bc2 = (float)(1.0 - powi_binary((double)a.b2, j));
            adam_one(p, m, v, 0.0f, lr, a.b1, a.b2, a.eps, bc1, bc2);
        }
        adam_one(p, m, v, gr, lr, a.b1, a.b2, a.eps, bc1t, bc2t);
        a.params[e] = p;
        a.m[e] = m;
        a.v[e] = v;
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
    a.flush = flush ? 1 : 0;
    int dev = 0, sms = 0;
    GS_CUDA_TRY(cudaGetDevice(&dev));
    GS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // The list length lives on the device: size the grid for n and let threads
    // beyond the list exit (grid-stride beyond 8 resident blocks per SM).
    const int threads = 256;
    int64_t bx = (n + threads - 1) / threads;
    const int64_t cap = ((int64_t)sms * 8 + rows - 1) / rows;
    if (bx > cap) bx = cap;
    cudaStream_t s = (cudaStream_t)stream;
    adam_deferred_kernel<<<dim3((unsigned)bx, (unsigned)rows), threads, 0, s>>>(a);
    GS_LAUNCH_CHECK();
    int64_t bs = (n + threads - 1) / threads;
    if (bs > (int64_t)sms * 8) bs = (int64_t)sms * 8;
    stamp_kernel<<<(unsigned)bs, threads, 0, s>>>(a);
    GS_LAUNCH_CHECK();
    return GS_OK;
}
