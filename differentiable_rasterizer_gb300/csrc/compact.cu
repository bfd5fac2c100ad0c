// compact.cu -- gs_grad_compact: sparse-gradient compaction ("encoder") and
// aggregation ("decoder") for one GPU (ByteSplat, English abstract: zero partial
// gradients eliminated; encoder/decoder kernels compact the remaining records
// and aggregate them directly at their owner).
//
//   per view v: idx[v] = ascending list of Gaussians with touched[v][g] != 0
//   union:      idx[V] = ascending list of Gaussians touched in any view
//   decode:     for each Gaussian of the union, the projection VJP of every
//               touching view is summed in view order in registers and written
//               as the Gaussian's dense gradient block ([n][stride] layout,
//               float4 stores; other blocks are not touched); the consumed
//               grad2d / touched entries are cleared.
// With one owner (this GPU) no record leaves the device, so the "send" of the
// encoded list is the list itself.
#include "gs_common.cuh"
#include "project_math.cuh"
#include "scan.cuh"

namespace gs {

__global__ void union_kernel(const uint8_t* __restrict__ touched, int64_t n, int n_views, uint8_t* __restrict__ u)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= n) return;
    uint8_t any = 0;
    for (int v = 0; v < n_views; ++v) any |= touched[(size_t)v * n + g];
    u[g] = any ? 1 : 0;
}

struct VjpArgs {
    float* __restrict__ grad2d;
    uint8_t* __restrict__ touched;
    const float* __restrict__ params;
    int64_t n;
    float near_z, lowpass;
    int32_t tiles_x, tiles_y;
    const uint32_t* __restrict__ idx_union;
    const int64_t* __restrict__ n_union;
    float* __restrict__ grads;
};

// Projection VJP of Gaussian g summed over its touching views, written as its
// dense gradient block (write only: the block's previous contents are not
// read); the consumed grad2d / touched entries are cleared.
template <int DEG>
__device__ __forceinline__ void vjp_gaussian(const VjpArgs& a, const CamSet& cs, int64_t g)
{
    GaussParams<DEG> gp;
    gp.load(a.params, g);
    constexpr int kVec = GaussParams<DEG>::kVec;
    float4* gdst = reinterpret_cast<float4*>(a.grads + (size_t)g * GaussParams<DEG>::kStride);
    float grad[kVec * 4];
#pragma unroll
    for (int i = 0; i < kVec * 4; ++i) grad[i] = 0.0f;
    GaussAct ac;
    activate<DEG>(gp, ac);   // view-independent: once for all views
    for (int v = 0; v < cs.n_views; ++v) {
        const size_t o = (size_t)v * (size_t)a.n + (size_t)g;
        if (!a.touched[o]) continue;
        ProjOut po;
        ProjInter it;
        if (project_view<DEG>(gp, ac, cs.cam[v], a.near_z, a.lowpass, a.tiles_x, a.tiles_y, po, &it)) {
            float4* src = reinterpret_cast<float4*>(a.grad2d + o * GS_GRAD2D_STRIDE);
            const float4 x0 = src[0], x1 = src[1], x2 = src[2];
            const float g2[9] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w, x2.x};
            vjp_one<DEG>(gp, cs.cam[v], ac, it, po.clamp, g2, grad, grad + 11);
            const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            src[0] = z; src[1] = z; src[2] = z;
        }
        a.touched[o] = 0;
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) gdst[i] = make_float4(grad[4 * i], grad[4 * i + 1], grad[4 * i + 2], grad[4 * i + 3]);
}

// One thread per Gaussian of the union list; the list length lives on the
// device, so a grid of resident blocks strides over it.
template <int DEG>
__global__ void __launch_bounds__(128) vjp_kernel(VjpArgs a, CamSet cs)
{
    const int64_t count = *a.n_union;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t g = (int64_t)a.idx_union[i];
        if (GS_IN_RANGE(g, a.n, GS_CHECK_COMPACT_ID)) vjp_gaussian<DEG>(a, cs, g);
    }
}

struct CompactWs {
    size_t sums, flags, bytes;
};

inline CompactWs compact_ws(int64_t n)
{
    CompactWs L;
    size_t o = 0;
    L.sums = o;  o = (o + scan_ws_bytes(n) + 255) & ~(size_t)255;
    L.flags = o; o = (o + (size_t)n + 255) & ~(size_t)255;
    L.bytes = o;
    return L;
}

}  // namespace gs

using namespace gs;

extern "C" gs_status gs_grad_compact(float* grad2d, uint8_t* touched, const float* params, int64_t n,
                                     int32_t sh_degree, const gs_camera* cams, int32_t n_views,
                                     const gs_render_opts* opts, uint32_t* idx, int64_t* n_idx, float* grads,
                                     void* ws, size_t* ws_bytes, void* stream)
{
    GS_NVTX_RANGE("gs_grad_compact");
    if (!ws_bytes || n < 0 || n > INT32_MAX) return GS_ERR_INVALID_ARG;
    const CompactWs L = compact_ws(n);
    if (!ws) {
        *ws_bytes = L.bytes;
        return GS_OK;
    }
    if (*ws_bytes < L.bytes) return GS_ERR_INVALID_ARG;
    if (!opts || !n_idx) return GS_ERR_INVALID_ARG;
    if (n > 0 && (!grad2d || !touched || !params || !idx || !grads)) return GS_ERR_INVALID_ARG;
    if (param_rows(sh_degree) < 0 || !aligned16(grad2d) || !aligned16(params) || !aligned16(grads))
        return GS_ERR_INVALID_ARG;
    gs_status st = check_views(cams, n_views);
    if (st != GS_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    char* w = (char*)ws;
    unsigned long long* sums = (unsigned long long*)(w + L.sums);
    uint8_t* flags = (uint8_t*)(w + L.flags);
    unsigned long long* counts = reinterpret_cast<unsigned long long*>(n_idx);
    for (int v = 0; v < n_views; ++v)
        GS_CUDA_TRY((scan_launch<uint8_t, true>(touched + (size_t)v * n, n, idx + (size_t)v * n, sums, counts + v, s)));
    if (n_views == 1) {
        // one view: the union is that view's list
        if (n > 0)
            GS_CUDA_TRY(cudaMemcpyAsync(idx + n, idx, sizeof(uint32_t) * (size_t)n, cudaMemcpyDeviceToDevice, s));
        GS_CUDA_TRY(cudaMemcpyAsync(counts + 1, counts, sizeof(unsigned long long), cudaMemcpyDeviceToDevice, s));
    } else {
        if (n > 0) {
            union_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(touched, n, n_views, flags);
            GS_LAUNCH_CHECK();
        }
        GS_CUDA_TRY((scan_launch<uint8_t, true>(flags, n, idx + (size_t)n_views * n, sums, counts + n_views, s)));
    }
    if (n == 0) return GS_OK;
    VjpArgs a;
    a.grad2d = grad2d;
    a.touched = touched;
    a.params = params;
    a.n = n;
    a.near_z = opts->near_z;
    a.lowpass = opts->lowpass;
    a.tiles_x = tiles_x_of(cams[0].width);
    a.tiles_y = tiles_y_of(cams[0].height);
    a.idx_union = idx + (size_t)n_views * n;
    a.n_union = n_idx + n_views;
    a.grads = grads;
    const CamSet cs = make_camset(cams, n_views);
    const int threads = 128;
    int dev = 0, sms = 0, per_sm = 0;
    GS_CUDA_TRY(cudaGetDevice(&dev));
    GS_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (sh_degree == 0)
        GS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vjp_kernel<0>, threads, 0));
    else
        GS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vjp_kernel<3>, threads, 0));
    int64_t blocks = (n + threads - 1) / threads;
    const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    if (blocks > resident) blocks = resident;
    if (sh_degree == 0)
        vjp_kernel<0><<<(unsigned)blocks, threads, 0, s>>>(a, cs);
    else
        vjp_kernel<3><<<(unsigned)blocks, threads, 0, s>>>(a, cs);
    GS_LAUNCH_CHECK();
    return GS_OK;
}

// ---------------------------------------------------------------------------
// gs_grad_compact_static: the same compaction + VJP + scatter-add for callers
// that cannot allocate device memory at step time -- for example code embedded
// in a host application that owns all device memory and offers no allocator,
// or a deployment that fixes its memory budget at start-up and forbids any
// cudaMalloc afterwards.  Its scratch is a file-scope device array sized for
// GS_COMPACT_STATIC_MAX_N Gaussians, held by every GPU that loads this library
// until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kAlign256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr int64_t kStaticMaxN = GS_COMPACT_STATIC_MAX_N;
// block sums of the scans (one u64 per 4096 items, plus the total) and the union flags
constexpr size_t kStaticScratchBytes =
    kAlign256((size_t)((kStaticMaxN + 4095) / 4096 + 1) * sizeof(unsigned long long)) + kAlign256((size_t)kStaticMaxN);

__device__ __align__(256) unsigned char g_compact_scratch[kStaticScratchBytes];

// Device address of g_compact_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached together with the id of the
// context it belongs to: a device reset (cudaDeviceReset) destroys that context
// and the array with it, and the next call, seeing another context, looks the
// address up again instead of handing a stale pointer to the kernels.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Id of the current context (cuCtxGetId, through the runtime's driver entry
// point: no link dependency on the driver library); false if there is none yet.
bool current_context_id(unsigned long long* id)
{
    using CtxGetId = int (*)(void*, unsigned long long*);
    static CtxGetId fn = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetId>(p);
        looked_up = true;
    }
    return fn && fn(nullptr, id) == 0;
}

gs_status static_scratch(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long ctx = 0;
    const bool known = current_context_id(&ctx);
    if (!g_scratch_addr[dev] || !known || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_compact_scratch) != cudaSuccess || !p) return GS_ERR_CUDA;
        g_scratch_addr[dev] = p;
        // the lookup makes the device's context current if it was not yet
        g_scratch_ctx[dev] = current_context_id(&ctx) ? ctx : 0;
    }
    *out = g_scratch_addr[dev];
    return GS_OK;
}

}  // namespace

extern "C" gs_status gs_grad_compact_static(float* grad2d, uint8_t* touched, const float* params, int64_t n,
                                            int32_t sh_degree, const gs_camera* cams, int32_t n_views,
                                            const gs_render_opts* opts, uint32_t* idx, int64_t* n_idx, float* grads,
                                            void* stream)
{
    GS_NVTX_RANGE("gs_grad_compact_static");
    if (n < 0 || n > kStaticMaxN) return GS_ERR_INVALID_ARG;
    if (gs::compact_ws(n).bytes > kStaticScratchBytes) return GS_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const gs_status st = static_scratch(&scratch);
    if (st != GS_OK) return st;
    size_t bytes = kStaticScratchBytes;
    return gs_grad_compact(grad2d, touched, params, n, sh_degree, cams, n_views, opts, idx, n_idx, grads, scratch,
                           &bytes, stream);
}
