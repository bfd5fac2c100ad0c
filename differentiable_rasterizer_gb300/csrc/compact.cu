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
//               grad2d / touched entries are cleared.  (SH degree 3 with
//               several views: the geometry and colour halves run in
//               different warps, each summed in view order, and the two
//               mean terms are added at the end.)
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
// device, so a grid of resident blocks strides over it.  Used for SH degree 0
// (a 64-byte block per Gaussian; degree 3 has the two kernels below).
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

// SH degree 3 with several views: the decode with its two halves in different
// warps.  A block of 128 threads takes 64 Gaussians of the union list at a
// time: warps 0-1 run their geometry VJP (mean through the projection, scale,
// rotation, opacity) and warps 2-3 their colour VJP (48 coefficients, and the
// mean through the viewing direction), so each (Gaussian, view)'s dependent
// chain is about half as long.  Warp w + 2 serves the same 32 Gaussians as
// warp w, and the pair meets at a 64-thread named barrier: the colour warp
// passes its direction term and the gradient of the first coefficient row
// through shared memory; the geometry warp writes the first three float4 of
// the gradient block and clears the consumed grad2d / touched entries, the
// colour warp writes the rest.  (With one view the one-thread-per-Gaussian
// vjp_kernel keeps more Gaussians in flight per SM and is the faster of the
// two.)
constexpr int kSplitThreads = 128;
constexpr int kSplitGaussians = kSplitThreads / 2;

// Barrier of the warp pair (w, w + 2): ids 1 and 2, 64 threads each.
__device__ __forceinline__ void pair_sync(int warp)
{
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 1)) : "memory");
}

struct GaussGeom {
    float mu[3], ls[3], q[4], logit;
};

__global__ void __launch_bounds__(kSplitThreads) vjp_split_kernel(VjpArgs a, CamSet cs)
{
    __shared__ float4 s_x[kSplitGaussians];   // per Gaussian: (d/d coefficient row 0, d/d mean via the direction)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool geom = warp < 2;
    const int slot = ((warp & 1) << 5) | lane;
    const int64_t count = *a.n_union;
    // block-uniform loop: every thread reaches both pair barriers of every iteration
    for (int64_t base = (int64_t)blockIdx.x * kSplitGaussians; base < count;
         base += (int64_t)gridDim.x * kSplitGaussians) {
        const int64_t i = base + slot;
        int64_t g = -1;
        if (i < count) {
            const int64_t gi = (int64_t)a.idx_union[i];
            if (GS_IN_RANGE(gi, a.n, GS_CHECK_COMPACT_ID)) g = gi;
        }
        uint32_t vm = 0u;   // the views that composited g
        if (g >= 0)
            for (int v = 0; v < cs.n_views; ++v)
                if (a.touched[(size_t)v * (size_t)a.n + (size_t)g]) vm |= 1u << v;
        const float4* src = reinterpret_cast<const float4*>(a.params + (size_t)(g >= 0 ? g : 0) * 64);
        if (geom) {
            float grad[11];
#pragma unroll
            for (int k = 0; k < 11; ++k) grad[k] = 0.0f;
            if (g >= 0) {
                const float4 p0 = __ldg(src), p1 = __ldg(src + 1), p2 = __ldg(src + 2);
                const GaussGeom gp = {{p0.x, p0.y, p0.z}, {p0.w, p1.x, p1.y}, {p1.z, p1.w, p2.x, p2.y}, p2.z};
                GaussAct ac;
                activate<3>(gp, ac);
                for (uint32_t m = vm; m; m &= m - 1u) {
                    const int v = __ffs(m) - 1;
                    ProjInter it;
                    project_geom(gp, ac, cs.cam[v], a.lowpass, it);
                    const float4* g2s = reinterpret_cast<const float4*>(
                        a.grad2d + ((size_t)v * (size_t)a.n + (size_t)g) * GS_GRAD2D_STRIDE);
                    const float4 x0 = g2s[0], x1 = g2s[1];
                    const float g2[6] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y};
                    vjp_geom(gp, cs.cam[v], ac, it, g2, grad);
                }
            }
            pair_sync(warp);   // the colour warp's hand-over is in s_x, and it has read its grad2d rows
            if (g >= 0) {
                const float4 x = s_x[slot];
                float4* dst = reinterpret_cast<float4*>(a.grads + (size_t)g * 64);
                dst[0] = make_float4(grad[0] + x.y, grad[1] + x.z, grad[2] + x.w, grad[3]);
                dst[1] = make_float4(grad[4], grad[5], grad[6], grad[7]);
                dst[2] = make_float4(grad[8], grad[9], grad[10], x.x);
                const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                for (uint32_t m = vm; m; m &= m - 1u) {
                    const size_t o = (size_t)(__ffs(m) - 1) * (size_t)a.n + (size_t)g;
                    float4* g2s = reinterpret_cast<float4*>(a.grad2d + o * GS_GRAD2D_STRIDE);
                    g2s[0] = z; g2s[1] = z; g2s[2] = z;
                    a.touched[o] = 0;
                }
            }
        } else {
            if (g >= 0) {
                float mu[3], col[48];
                {
                    const float4 p0 = __ldg(src), p2 = __ldg(src + 2);
                    mu[0] = p0.x; mu[1] = p0.y; mu[2] = p0.z;
                    col[0] = p2.w;
#pragma unroll
                    for (int k = 0; k < 12; ++k) {   // floats 12 .. 59 of the block (59: padding)
                        const float4 p = __ldg(src + 3 + k);
                        col[1 + 4 * k] = p.x;
                        col[2 + 4 * k] = p.y;
                        col[3 + 4 * k] = p.z;
                        if (k < 11) col[4 + 4 * k] = p.w;
                    }
                }
                float gcol[48], gmu[3] = {0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int k = 0; k < 48; ++k) gcol[k] = 0.0f;
                for (uint32_t m = vm; m; m &= m - 1u) {
                    const int v = __ffs(m) - 1;
                    const float4* g2s = reinterpret_cast<const float4*>(
                        a.grad2d + ((size_t)v * (size_t)a.n + (size_t)g) * GS_GRAD2D_STRIDE);
                    const float4 x1 = g2s[1], x2 = g2s[2];
                    const float gc[3] = {x1.z, x1.w, x2.x};
                    vjp_colour3(mu, col, cs.cam[v], gc, gcol, gmu);
                }
                float4* dst = reinterpret_cast<float4*>(a.grads + (size_t)g * 64);
#pragma unroll
                for (int k = 0; k < 12; ++k)
                    dst[3 + k] = make_float4(gcol[1 + 4 * k], gcol[2 + 4 * k], gcol[3 + 4 * k],
                                             k < 11 ? gcol[4 + 4 * k] : 0.0f);
                s_x[slot] = make_float4(gcol[0], gmu[0], gmu[1], gmu[2]);
            }
            pair_sync(warp);   // meets the geometry warp's first barrier
        }
        pair_sync(warp);   // s_x is rewritten in the next iteration
    }
}

// SH degree 3 with one view.  A thread still differentiates one Gaussian, but
// the warp moves its 32 Gaussians' parameter and gradient blocks through shared
// memory: per load (store) instruction the warp reads (writes) two whole 240-byte
// blocks, 16 bytes a lane, where a thread reading its own block would touch 32
// blocks per instruction -- the L1 and the load-store queues, not DRAM, held
// that form back (long-scoreboard and LSU-throttle stalls at 42 % of the HBM
// peak).  The 48 colour coefficients are streamed from the staged row
// (vjp_colour3_stream) instead of held in registers, and the view's forward is
// recomputed only as far as the VJP needs it (a composited Gaussian is visible:
// no culling tests, radius or tile rectangle).
constexpr int kRowF = 68;          // floats per staged row: 16-byte accesses of 8 lanes hit distinct banks
constexpr int kStageWarps = 4;     // warps per block

// Moves the 15 used float4 of the blocks of the warp's 32 Gaussians (g: this
// lane's, -1 for none) between global blocks (stride 64 floats) and the warp's
// staged rows: instruction t covers Gaussians 2t and 2t + 1, 16 lanes each.
template <bool kToShared>
__device__ __forceinline__ void stage_rows(float* rows, int g, float* glob, int lane)
{
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        const int owner = 2 * t + (lane >> 4), piece = lane & 15;
        const int go = __shfl_sync(0xffffffffu, g, owner);
        if (go >= 0 && piece < 15) {
            float4* gp = reinterpret_cast<float4*>(glob + (size_t)go * 64) + piece;
            float4* sp = reinterpret_cast<float4*>(rows + owner * kRowF) + piece;
            if (kToShared) *sp = __ldg(gp);
            else *gp = *sp;
        }
    }
}

__global__ void __launch_bounds__(kStageWarps * 32) vjp_staged3_kernel(VjpArgs a, CamSet cs)
{
    __shared__ __align__(16) float s_rows[kStageWarps][32 * kRowF];
    const gs_camera& cam = cs.cam[0];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float* rows = s_rows[warp];
    float4* r4 = reinterpret_cast<float4*>(rows + lane * kRowF);
    const int64_t count = *a.n_union;
    const int64_t nwarps = (int64_t)gridDim.x * kStageWarps;
    // warp-uniform loop: all lanes take part in every staging step
    for (int64_t base = ((int64_t)blockIdx.x * kStageWarps + warp) * 32; base < count; base += nwarps * 32) {
        const int64_t i = base + lane;
        int g = -1;
        if (i < count) {
            const int64_t gi = (int64_t)a.idx_union[i];
            if (GS_IN_RANGE(gi, a.n, GS_CHECK_COMPACT_ID)) g = (int)gi;
        }
        stage_rows<true>(rows, g, const_cast<float*>(a.params), lane);
        __syncwarp();
        if (g >= 0) {
            float grad[11];
#pragma unroll
            for (int k = 0; k < 11; ++k) grad[k] = 0.0f;
            float gmu[3] = {0.0f, 0.0f, 0.0f};
            float gcol0 = 0.0f;
            if (a.touched[g]) {   // the one view's union is its touched set
                const float4 p0 = r4[0], p1 = r4[1], p2 = r4[2];
                const GaussGeom gp = {{p0.x, p0.y, p0.z}, {p0.w, p1.x, p1.y}, {p1.z, p1.w, p2.x, p2.y}, p2.z};
                float4* g2s = reinterpret_cast<float4*>(a.grad2d + (size_t)g * GS_GRAD2D_STRIDE);
                const float4 x0 = g2s[0], x1 = g2s[1], x2 = g2s[2];
                GaussAct ac;
                activate<3>(gp, ac);
                ProjInter it;
                project_geom(gp, ac, cam, a.lowpass, it);
                const float g2[6] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y};
                vjp_geom(gp, cam, ac, it, g2, grad);
                const float gc[3] = {x1.z, x1.w, x2.x};
                gcol0 = vjp_colour3_stream(r4, gp.mu, cam, gc, r4, gmu);
                const float4 z = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                g2s[0] = z; g2s[1] = z; g2s[2] = z;
                a.touched[g] = 0;
            } else {
#pragma unroll
                for (int k = 3; k < 15; ++k) r4[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            r4[0] = make_float4(grad[0] + gmu[0], grad[1] + gmu[1], grad[2] + gmu[2], grad[3]);
            r4[1] = make_float4(grad[4], grad[5], grad[6], grad[7]);
            r4[2] = make_float4(grad[8], grad[9], grad[10], gcol0);
        }
        __syncwarp();
        stage_rows<false>(rows, g, a.grads, lane);
        __syncwarp();   // the rows are refilled in the next iteration
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
    if (sh_degree == 0 || n_views == 1) {
        auto kernel = sh_degree == 0 ? vjp_kernel<0> : vjp_staged3_kernel;
        GS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0));
        int64_t blocks = (n + threads - 1) / threads;
        const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > resident) blocks = resident;
        kernel<<<(unsigned)blocks, threads, 0, s>>>(a, cs);
    } else {
        GS_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vjp_split_kernel, kSplitThreads, 0));
        int64_t blocks = (n + kSplitGaussians - 1) / kSplitGaussians;
        const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
        if (blocks > resident) blocks = resident;
        vjp_split_kernel<<<(unsigned)blocks, kSplitThreads, 0, s>>>(a, cs);
    }
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
