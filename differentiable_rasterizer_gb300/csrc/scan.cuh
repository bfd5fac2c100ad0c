// scan.cuh -- device-wide exclusive scan and stream compaction (three launches:
// per-block sums, one-block scan of the sums, per-block rescan with the block
// prefix).  Blocks of 256 threads own 16 consecutive items per thread, so each
// block covers kScanItems consecutive items and no inter-block waiting is needed;
// a thread reads its items with 16-byte loads where the input is aligned.
#pragma once

#include "gs_common.cuh"

namespace gs {
namespace {   // internal linkage: each translation unit gets its own copy

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 16;
constexpr int kScanItems = kScanThreads * kScanPerThread;

template <typename T>
__device__ __forceinline__ unsigned long long load_item(const T* in, int64_t i, int64_t n)
{
    return i < n ? (unsigned long long)in[i] : 0ull;
}

// Counts of "nonzero" (flag mode) or values (value mode).
template <typename T, bool kFlag>
__device__ __forceinline__ unsigned long long item_value(const T* in, int64_t i, int64_t n)
{
    if (i >= n) return 0ull;
    const T x = in[i];
    return kFlag ? (x != 0 ? 1ull : 0ull) : (unsigned long long)x;
}

// The kScanPerThread items of one thread, from base: 16-byte vector loads when
// the input is 16-byte aligned and all the items are in range (one load for
// bytes, four for 32-bit words), else one item at a time.
template <typename T, bool kFlag>
__device__ __forceinline__ void load_items(const T* in, int64_t base, int64_t n, bool vec, uint32_t (&v)[kScanPerThread])
{
    static_assert(sizeof(T) == 1 || sizeof(T) == 4, "bytes or 32-bit words");
    if (vec && base + kScanPerThread <= n) {
        constexpr int kQ = kScanPerThread * (int)sizeof(T) / 16;   // uint4 loads
        const uint4* q = reinterpret_cast<const uint4*>(in + base);
#pragma unroll
        for (int l = 0; l < kQ; ++l) {
            const uint4 u = q[l];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (sizeof(T) == 1) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const uint32_t x = (w[e] >> (8 * b)) & 0xffu;
                        v[16 * l + 4 * e + b] = kFlag ? (x != 0u ? 1u : 0u) : x;
                    }
                } else {
                    v[4 * l + e] = kFlag ? (w[e] != 0u ? 1u : 0u) : w[e];
                }
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < kScanPerThread; ++k) v[k] = (uint32_t)item_value<T, kFlag>(in, base + k, n);
    }
}

// Block-wide exclusive scan of one u64 per thread; returns the exclusive prefix,
// *total receives the block total.
__device__ __forceinline__ unsigned long long block_exclusive_scan(unsigned long long x, unsigned long long* total)
{
    __shared__ unsigned long long s_warp[kScanThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    unsigned long long woff = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
        const unsigned long long s = s_warp[w];
        if (w < warp) woff += s;
        tot += s;
    }
    __syncthreads();
    *total = tot;
    return woff + inc - x;
}

template <typename T, bool kFlag>
__global__ void __launch_bounds__(kScanThreads) scan_block_sums(const T* in, int64_t n, unsigned long long* sums,
                                                                bool vec)
{
    const int64_t base = (int64_t)blockIdx.x * kScanItems + (int64_t)threadIdx.x * kScanPerThread;
    uint32_t v[kScanPerThread];
    load_items<T, kFlag>(in, base, n, vec, v);
    unsigned long long s = 0;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) s += v[k];
    unsigned long long tot;
    block_exclusive_scan(s, &tot);
    if (threadIdx.x == 0) sums[blockIdx.x] = tot;
}

// One block scans the block sums in place (exclusive) and writes the grand total.
__global__ void __launch_bounds__(kScanThreads) scan_sums_kernel(unsigned long long* sums, int64_t nb,
                                                                 unsigned long long* total)
{
    unsigned long long carry = 0;
    for (int64_t base = 0; base < nb; base += kScanThreads) {
        const int64_t i = base + threadIdx.x;
        const unsigned long long x = i < nb ? sums[i] : 0ull;
        unsigned long long tot;
        const unsigned long long ex = block_exclusive_scan(x, &tot);
        if (i < nb) sums[i] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) *total = carry;
}

// Value mode: out[i] = exclusive prefix (u32).  Flag mode: out[prefix] = i for nonzero in[i].
template <typename T, bool kFlag>
__global__ void __launch_bounds__(kScanThreads) scan_block_apply(const T* in, int64_t n,
                                                                 const unsigned long long* sums, uint32_t* out,
                                                                 bool vec)
{
    const int64_t base = (int64_t)blockIdx.x * kScanItems + (int64_t)threadIdx.x * kScanPerThread;
    uint32_t vals[kScanPerThread];
    load_items<T, kFlag>(in, base, n, vec, vals);
    unsigned long long s = 0;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) s += vals[k];
    unsigned long long tot;
    unsigned long long run = sums[blockIdx.x] + block_exclusive_scan(s, &tot);
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        const int64_t i = base + k;
        if (i < n) {
            if (kFlag) {
                if (vals[k]) out[run] = (uint32_t)i;
            } else {
                out[i] = (uint32_t)run;
            }
        }
        run += vals[k];
    }
}

inline int64_t scan_blocks(int64_t n) { return (n + kScanItems - 1) / kScanItems; }

// Bytes of scratch for a scan of n items: block sums + total.
inline size_t scan_ws_bytes(int64_t n) { return (size_t)(scan_blocks(n) + 1) * sizeof(unsigned long long); }

// Exclusive scan (kFlag = false) or compaction (kFlag = true) of n items.
// ws must hold scan_ws_bytes(n); *d_total (device) receives the total.
template <typename T, bool kFlag>
inline cudaError_t scan_launch(const T* in, int64_t n, uint32_t* out, unsigned long long* ws,
                               unsigned long long* d_total, cudaStream_t s)
{
    const int64_t nb = scan_blocks(n);
    if (nb == 0) return cudaMemsetAsync(d_total, 0, sizeof(unsigned long long), s);
    const bool vec = ((uintptr_t)in & 15u) == 0;   // 16-byte loads need an aligned start
    scan_block_sums<T, kFlag><<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, ws, vec);
    scan_sums_kernel<<<1, kScanThreads, 0, s>>>(ws, nb, d_total);
    scan_block_apply<T, kFlag><<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, ws, out, vec);
    return cudaPeekAtLastError();
}

}  // namespace
}  // namespace gs
