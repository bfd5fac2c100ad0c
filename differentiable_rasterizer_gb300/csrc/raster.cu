// raster.cu -- gs_raster_fused_fwd_bwd: forward compositing, L1 loss and
// backward rasterization in ONE kernel (ByteSplat, English abstract: the two
// rasterization passes are one kernel whose intermediate results stay on chip
// instead of going through off-chip memory).
//
// One CTA per 16x16 tile, one pixel per thread; warp w owns the 8x4 pixel block
// (w % 2, w / 2) of the tile (compact blocks: their pixels' walks are of more
// similar length than those of two tile rows).  The tile's
// sorted list is staged through shared memory in chunks of kChunk records
// (gathered through the instance ids).  Per chunk, thread t turns entry t's
// alpha-support box (from gs_project; it provably contains every pixel whose
// fp32 power can reach the entry's cut tau) into row and column spans, and the
// warps transpose them by ballots into one 256-bit candidate mask per tile row
// and per tile column.  Each pixel then ANDs its row and column masks and walks
// its candidates in list order: the pass test (power, tau, exp, alpha) and, for
// the entries that pass, compositing, with T, the colour, the stop index and
// dL/dC in registers; the entries that passed set bits in the pixel's own
// 256-bit row.
//
// Entries that do not pass are skipped by definition, so the image, stop index
// and evaluation counts are those of walking every list entry.  The entries a
// pixel composited are exactly its passing bits up to its last index, so
// backward needs no per-pixel list.  Backward walks the chunks last to first;
// per chunk each pixel walks its own composited entries newest first, with T
// before an entry = T after it / (1 - alpha) and dL/dC . (colour behind it)
// carried in registers; each (entry, pixel) pair's 9 gradient terms go to the
// Gaussian's grad2d row with vector atomics.  The pass bits of
// the last kRing chunks stay in shared memory (a ring), so backward re-gathers
// only their records; the bits of older chunks, written to a scratch buffer by
// the forward as the ring evicts them, are read back from it (recomputed when
// no scratch is given or it is too small).  A chunk in
// which the warp's pixels mostly composite the same entries (large Gaussians) is
// walked one entry at a time for all 32 pixels instead, its gradient terms summed
// over the warp by shuffles before one atomic per component.
//
// All decisions use the same fp32 operations in the same order as the CPU
// definition (see gs_common.cuh); boxes, tau and bits only avoid work whose
// outcome is already known.
//
// Modes (template argument): kFused -- forward, L1 loss and backward in one
// pass; kFwd -- forward only, optionally storing per pixel the final T and last
// index, and the pass bits of every chunk in the scratch; kBwdState -- the
// backward alone, started from that stored state with dL/dC given per pixel
// (for losses whose gradient needs other tiles' colours).
// Views are interleaved over the grid (CTA i: view i mod V, tile i / V) so the
// heavy central tiles of all views spread over the launch.
#include "gs_common.cuh"

namespace gs {

constexpr int kChunk = 256;      // records per shared-memory stage
constexpr int kWords = kChunk / 32;
constexpr int kWarps = kTileThreads / 32;
constexpr int kRing = 3;         // chunks whose pass bits stay in shared memory
constexpr int kDense = 12;       // backward: entries per distinct Gaussian from which a warp reduces per Gaussian

// Kernel modes.
constexpr int kFwd = 0;          // forward only (image; optionally final T and last index per pixel)
constexpr int kFused = 1;        // forward, L1 loss and backward in one pass
constexpr int kBwdState = 2;     // backward only, from a stored final T / last index and a given dL/dC

struct RasterArgs {
    const float4* __restrict__ rec;     // [V][n][3]
    const uint2* __restrict__ ranges;   // [V * tiles]
    const uint32_t* __restrict__ ids;
    const float* __restrict__ target;   // [V][3][H][W] or null
    const float* __restrict__ dldc;     // [V][3][H][W]: dL/dC (backward from stored state)
    float* t_final;                     // [V][H][W]: final transmittance per pixel, or null
    int32_t* last_idx;                  // [V][H][W]: last composited list index per pixel (-1: none)
    uint32_t* bits_ws;                  // saved pass bits by list position (kWords words per entry), or null
    int64_t bits_ws_words;              // its size in 32-bit words
    float* image;                       // [V][3][H][W]
    double* loss;                       // [V]
    float* grad2d;                      // [V][n][12]
    uint8_t* touched;                   // [V][n]
    unsigned long long* counts;         // [3] or null
    unsigned long long* work;           // [kWCount] executed-work counters (counting variant) or null
    int64_t n;
    int32_t W, H, tiles_x, tiles, n_views;
    float alpha_min, alpha_max, t_min, bg0, bg1, bg2, inv3hw;
    double inv3hw_d;                    // 1 / (3 H W) for the loss mean
    int32_t exclude_crossing;
};

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Pixels of the tile at (ox, oy) whose centres lie in the box |x - mx| <= hx,
// |y - my| <= hy, as half-open column/row ranges packed x0 | x1<<8 | y0<<16 | y1<<24
// (0: none).
__device__ __forceinline__ uint32_t tile_box(float mx, float my, float hx, float hy, int ox, int oy)
{
    if (!(hx >= 0.0f && hy >= 0.0f)) return 0u;
    const float fx0 = fmaxf(ceilf(mx - hx - (float)ox - 0.5f), 0.0f);
    const float fx1 = fminf(floorf(mx + hx - (float)ox - 0.5f) + 1.0f, (float)kTile);
    const float fy0 = fmaxf(ceilf(my - hy - (float)oy - 0.5f), 0.0f);
    const float fy1 = fminf(floorf(my + hy - (float)oy - 0.5f) + 1.0f, (float)kTile);
    if (!(fx0 < fx1 && fy0 < fy1)) return 0u;
    return (uint32_t)fx0 | ((uint32_t)fx1 << 8) | ((uint32_t)fy0 << 16) | ((uint32_t)fy1 << 24);
}

// Gradient terms of one composited entry (9: mean2d x y, conic A B C, opacity,
// colour r g b).
struct EntryGrad {
    float gm0, gm1, gA, gB, gC, go, gr, gg, gb;
};

// One step of the halving sum below: of the 2H partial sums v (the lower half
// kept by lanes with `upper` clear), a lane keeps its half and adds the
// partner's (lane ^ o) copy of that half.
template <int H>
__device__ __forceinline__ void halve(const float (&v)[2 * H], float (&k)[H], bool upper, int o)
{
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float send = upper ? v[i] : v[H + i];
        const float keep = upper ? v[H + i] : v[i];
        k[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
}

// Warp sum of the nine gradient terms by recursive halving: at xor distances
// 16, 8, 4, 2, 1 each lane keeps the half of its partial sums that its lane bit
// selects (12 shuffles instead of a full butterfly's 45).  Every partial sum is
// own + partner at the same distances as the butterfly, so the totals are the
// butterfly's bit for bit.  Returns the total of term reduce_term(lane).
__device__ __forceinline__ float warp_sum_terms(const EntryGrad& e, int lane)
{
    const float v10[10] = {e.gm0, e.gm1, e.gA, e.gB, e.gC, e.go, e.gr, e.gg, e.gb, 0.0f};
    float k5[5];
    halve<5>(v10, k5, (lane & 16) != 0, 16);            // terms 0..4 | 5..9
    const float v6[6] = {k5[0], k5[1], k5[2], k5[3], k5[4], 0.0f};
    float k3[3];
    halve<3>(v6, k3, (lane & 8) != 0, 8);               // 0..2 | 3, 4, pad
    const float v4[4] = {k3[0], k3[1], k3[2], 0.0f};
    float k2[2];
    halve<2>(v4, k2, (lane & 4) != 0, 4);               // 0, 1 | 2, pad
    float k1[1];
    halve<1>(k2, k1, (lane & 2) != 0, 2);
    return k1[0] + __shfl_xor_sync(0xffffffffu, k1[0], 1);
}

// The term whose warp total warp_sum_terms leaves in this lane (even lanes
// only; -1: a padding slot or an odd lane).
__device__ __forceinline__ int reduce_term(int lane)
{
    const int m = ((lane & 4) ? 2 : 0) + ((lane & 2) ? 1 : 0);   // of the 3 kept after distance 8
    const int i = ((lane & 8) ? 3 : 0) + m;                        // of the 5 kept after distance 16
    const int t = ((lane & 16) ? 5 : 0) + i;
    return ((lane & 1) || m > 2 || i > 4 || t > 8) ? -1 : t;
}

// Gradient terms of one composited entry from its transmittance before it (Ti),
// dotc = dL/dC . its colour, dots = dL/dC . the colour composited behind it, and
// rc = 1 / (1 - alpha).
__device__ __forceinline__ EntryGrad entry_grad_at(const float4 r0, const float4 r1, float dx, float dy, float G,
                                                   float araw, float alpha, float alpha_max, float g0, float g1,
                                                   float g2c, float Ti, float dotc, float dots, float rc)
{
    EntryGrad e;
    const float wgt = alpha * Ti;
    e.gr = g0 * wgt;
    e.gg = g1 * wgt;
    e.gb = g2c * wgt;
    const float dalpha = __fmaf_rn(Ti, dotc, -dots * rc);
    if (araw <= alpha_max) {
        e.go = dalpha * G;
        const float dp = dalpha * alpha;
        const float hdp = -0.5f * dp;
        e.gA = hdp * dx * dx;
        e.gB = -dp * (dx * dy);
        e.gC = hdp * dy * dy;
        e.gm0 = dp * __fmaf_rn(-2.0f * r0.z, dx, r0.w * dy);
        e.gm1 = dp * __fmaf_rn(r0.w, dx, -2.0f * r1.x * dy);
    } else {
        e.go = e.gA = e.gB = e.gC = e.gm0 = e.gm1 = 0.0f;
    }
    return e;
}

// 16-byte asynchronous global -> shared copy (cp.async, L2 only) and its group
// commit / wait.  The wait is the hardware's: it ends when the copies land.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Executed-work counters of the counting variant (kCount): what the kernel
// actually does, as opposed to the E_fwd / E_bwd evaluations the method defines.
enum WorkCounter {
    kWPairs = 0,        // (entry, pixel) candidates tested: power evaluated
    kWPairExp,          // ... of which reached the exponential (tau <= power <= 0)
    kWCompWalk,         // ... of which passed and were composited (T, colour)
    kWSparseEntries,    // backward, per-pixel walk: (entry, pixel) evaluations
    kWSparseSteps,      // ... warp steps (the most entries any lane of the warp walked, per chunk)
    kWDenseEntries,     // backward, per-Gaussian path: (entry, pixel) evaluations
    kWDenseSteps,       // ... warp steps (one union entry for 32 lanes, one warp sum)
    kWChunks,           // chunks staged in the forward
    kWRestaged,         // chunks staged again in the backward
    kWRecomputed,       // ... of which had their pass bits recomputed
    kWCount
};

// Shared memory of one block (dynamic: about 54 KB, four blocks per SM).
struct RasterSmem {
    float4 r0[2][kChunk], r1[2][kChunk], r2[2][kChunk];   // records of two chunks; r2: (blue, tau, hx, hy)
    uint32_t id[2][kChunk];                                // their instance ids
    uint32_t bits[kRing][kWords][kTileThreads];            // per ring slot: bit j of pixel p = entry j passes at p
    uint32_t rowm[2][kTile][kWords];                       // per mask buffer: entries whose box covers tile row y
    uint32_t colm[2][kTile][kWords + 1];                   // ... column x (padded: conflict-free reads)
    double red_loss[kWarps];                               // per warp: loss sum ...
    unsigned long long red_counts[3][kWarps];              // ... and evaluation counts
};

template <int kMode, bool kCount>
__global__ void __launch_bounds__(kTileThreads, kCount ? 1 : 4) raster_fused_kernel(RasterArgs a)
{
    constexpr bool kBackward = kMode != kFwd;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RasterSmem& sm = *reinterpret_cast<RasterSmem*>(smem_raw);
    auto& s_r0 = sm.r0;
    auto& s_r1 = sm.r1;
    auto& s_r2 = sm.r2;
    auto& s_id = sm.id;
    auto& s_bits = sm.bits;
    auto& s_rowm = sm.rowm;
    auto& s_colm = sm.colm;

    // Views interleaved (CTA i: view i mod V, tile i / V) so the heavy central
    // tiles of all views are spread over the launch instead of queued view by
    // view (batched: 45.5 -> 43.2 ms).
    const int v = (int)(blockIdx.x % (unsigned)a.n_views);
    const int tile = (int)(blockIdx.x / (unsigned)a.n_views);
    const int tile_lin = v * a.tiles + tile;
    const int tx = tile % a.tiles_x, ty = tile / a.tiles_x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int red_term = reduce_term(lane);   // dense backward: the gradient term this lane adds
    const int ox = tx * kTile, oy = ty * kTile;
    const int px = ox + ((warp & 1) << 3) + (lane & 7);   // warp w: the 8 x 4 block (w % 2, w / 2)
    const int py = oy + ((warp >> 1) << 2) + (lane >> 3);
    const bool inside = px < a.W && py < a.H;
    const float pxf = (float)px + 0.5f, pyf = (float)py + 0.5f;
    const uint2 range = a.ranges[tile_lin];
    const size_t lo = range.x;                      // list start: instance counts up to 2^32 - 1
    const int len = GS_IN_RANGE((int64_t)range.y - (int64_t)range.x, 1ll << 32, GS_CHECK_RANGE)
                        ? (int)(range.y - range.x) : 0;
    const float4* __restrict__ recv = a.rec + (size_t)v * (size_t)a.n * 3;
    const float alpha_min = a.alpha_min, alpha_max = a.alpha_max;
    unsigned long long work[kCount ? kWCount : 1];
    if (kCount)
#pragma unroll
        for (int k = 0; k < kWCount; ++k) work[k] = 0ull;

    // Staging of a chunk, asynchronous: the instance ids are loaded into a
    // register one chunk before they are used, then the three record float4s
    // are copied into buffer b with cp.async while the block works on the chunk
    // before (forward: issued as that chunk starts, so the copy overlaps its
    // candidate walk).  Waiting for them (cp_async_wait_all) and a block
    // barrier make them visible.
    constexpr uint32_t kNone = 0xffffffffu;        // no entry (ids are < 2^31)
    auto stage_id = [&](int base) -> uint32_t {
        const int k = base + (int)threadIdx.x;
        return k < len ? __ldg(a.ids + lo + k) : kNone;
    };
    auto stage_copy = [&](uint32_t g, int b) {
        if (g != kNone && !GS_IN_RANGE(g, a.n, GS_CHECK_RASTER_ID)) {
            // dropped: an empty extent gives the entry an empty box, so it never
            // passes a pixel and no later phase reads its record or index
            s_r2[b][threadIdx.x] = make_float4(0.0f, 0.0f, -1.0f, -1.0f);
            g = kNone;
        }
        if (g != kNone) {
            const float4* r = recv + (size_t)g * 3;
            cp_async16(&s_r0[b][threadIdx.x], r);
            cp_async16(&s_r1[b][threadIdx.x], r + 1);
            cp_async16(&s_r2[b][threadIdx.x], r + 2);
        }
        s_id[b][threadIdx.x] = g;
        cp_async_commit();
    };
    // Chunk c's slot in the saved-bits scratch: its rows (word w of every pixel
    // = 256 words, 32 list entries' bits) for the words that hold entries, from
    // word (lo + 32 l + c kChunk) kWords on, l = the list's index.  32 bytes
    // per list entry plus 32 entries' worth per list keep a list's partial last
    // chunk clear of the next list.  A chunk past the scratch's end has no slot
    // and is recomputed instead.
    auto saved_words = [&](int c) -> int { return (min(kChunk, len - c * kChunk) + 31) >> 5; };
    auto saved_base = [&](int c) -> size_t { return lo + (size_t)tile_lin * 32 + (size_t)c * kChunk; };
    auto saved = [&](int c) -> bool {
        return a.bits_ws != nullptr &&
               (int64_t)((saved_base(c) + (size_t)saved_words(c) * 32) * kWords) <= a.bits_ws_words;
    };
    auto saved_row = [&](int c) -> uint32_t* { return a.bits_ws + saved_base(c) * kWords + threadIdx.x; };

    // Candidate masks of the chunk in buffer b, into mask buffer mb: bit j of
    // row mask y (column mask x) is set when entry j's alpha-support box (from
    // gs_project, clipped to the tile; it provably holds every pixel whose fp32
    // power can reach the entry's cut tau) covers tile row y (column x), so
    // pixel (x, y)'s candidates are the AND of its two masks -- exactly the
    // (entry, box pixel) pairs.  Thread t reads entry t's record (copied by
    // itself); each warp transposes its 32 entries' spans with ballots.
    auto build_masks = [&](int cnt, int b, int mb) {
        uint32_t box = 0u;
        if ((int)threadIdx.x < cnt) {
            const float4 q0 = s_r0[b][threadIdx.x], q2 = s_r2[b][threadIdx.x];
            box = tile_box(q0.x, q0.y, q2.z, q2.w, ox, oy);
        }
        const int x0 = box & 0xff, x1 = (box >> 8) & 0xff;   // an empty box is all zero
        const int y0 = (box >> 16) & 0xff, y1 = box >> 24;
        uint32_t mine = 0u;
#pragma unroll
        for (int r = 0; r < kTile; ++r) {
            const uint32_t br = __ballot_sync(0xffffffffu, r >= y0 && r < y1);
            const uint32_t bc = __ballot_sync(0xffffffffu, r >= x0 && r < x1);
            if (lane == r) mine = br;
            if (lane == kTile + r) mine = bc;
        }
        if (lane < kTile) s_rowm[mb][lane][warp] = mine;
        else s_colm[mb][lane - kTile][warp] = mine;
    };
    // This pixel's candidates in word w of the chunk (masks in buffer mb).
    const int tx_l = px - ox, ty_l = py - oy;
    auto candidates = [&](int mb, int w) -> uint32_t { return s_rowm[mb][ty_l][w] & s_colm[mb][tx_l][w]; };
    // Pass test of entry j at this pixel: alpha from the same fp32 operations as
    // the CPU definition; power > 0 is skipped by definition, power < tau has
    // alpha < alpha_min.  Returns alpha, or -1 if the entry does not pass.
    auto pass_alpha = [&](int b, int j, float4& r0, float4& r1) -> float {
        r0 = s_r0[b][j];
        r1 = s_r1[b][j];
        const float dx = pxf - r0.x, dy = pyf - r0.y;
        // power = -1/2 (A dx^2 + C dy^2) - B dx dy, with r0.z = -A/2, r1.x = -C/2
        const float power = ((r0.z * dx) * dx + (r1.x * dy) * dy) - (r0.w * dx) * dy;
        if (kCount) ++work[kWPairs];
        if (power > 0.0f || power < s_r2[b][j].y) return -1.0f;
        if (kCount) ++work[kWPairExp];
        const float alpha = fminf(alpha_max, r1.y * pexp_neg(power));
        return alpha < alpha_min ? -1.0f : alpha;
    };
    // Pass bits of this pixel for the chunk in buffer b (masks in mb), entries
    // up to lim only, into its row of ring slot sl (zero when lim < 0).
    auto eval_bits = [&](int b, int mb, int sl, int lim) {
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            const int top = lim - (w << 5);
            uint32_t cand = top >= 0 ? candidates(mb, w) : 0u;
            if (top >= 0 && top < 31) cand &= (2u << top) - 1u;
            uint32_t pass = 0u;
            while (cand) {
                const int bt = __ffs(cand) - 1;
                cand &= cand - 1u;
                float4 r0, r1;
                if (pass_alpha(b, (w << 5) | bt, r0, r1) >= 0.0f) pass |= 1u << bt;
            }
            s_bits[sl][w][threadIdx.x] = pass;
        }
    };

    // This lane's entry bits (passing, up to lim) and their count; returns the
    // warp total.
    auto gather = [&](uint32_t (&words)[kWords], int lim, int sl, int& nmine) {
        nmine = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            const int top = lim - (w << 5);
            uint32_t word = top >= 0 ? s_bits[sl][w][threadIdx.x] : 0u;
            if (top >= 0 && top < 31) word &= (2u << top) - 1u;
            words[w] = word;
            nmine += __popc(word);
        }
        return (int)__reduce_add_sync(0xffffffffu, (unsigned)nmine);
    };


    // ------------------------------------------------------------- forward
    float T = 1.0f, C0 = 0.0f, C1 = 0.0f, C2 = 0.0f;
    int last = -1, ncomp = 0;
    int stop = -1;                      // list index where this pixel stopped, -1 if it never did
    bool done = !inside;
    int resident = -1;                  // chunk whose records the block last worked on (buffer resident & 1)
    const size_t HW = (size_t)a.W * (size_t)a.H;
    const size_t spix = (size_t)v * HW + (size_t)py * a.W + px;   // per-pixel state index
    if (kMode == kBwdState && inside) {
        T = a.t_final[spix];
        last = a.last_idx[spix];
    }
    const int nchunks = kMode == kBwdState ? 0 : (len + kChunk - 1) / kChunk;
    uint32_t g_ahead = nchunks > 1 ? stage_id(kChunk) : kNone;   // ids of the chunk after the next
    // the target, loaded before the forward so that its latency is hidden
    float t0v = 0.0f, t1v = 0.0f, t2v = 0.0f;
    if (kBackward && kMode != kBwdState && inside) {
        const size_t tp = (size_t)v * 3 * HW + (size_t)py * a.W + px;
        t0v = __ldg(a.target + tp);
        t1v = __ldg(a.target + tp + HW);
        t2v = __ldg(a.target + tp + 2 * HW);
    }
    if (nchunks > 0) stage_copy(stage_id(0), 0);
    for (int c = 0; c < nchunks; ++c) {
        const int base = c * kChunk, b = c & 1, sl = c % kRing;
        cp_async_wait_all();
        build_masks(min(kChunk, len - base), b, b);
        // one barrier: chunk c's records and masks visible, chunk c - 1 finished
        if (__syncthreads_and(done)) break;
        resident = c;
        if (kCount && threadIdx.x == 0) ++work[kWChunks];
        if (c + 1 < nchunks) stage_copy(g_ahead, b ^ 1);
        g_ahead = c + 2 < nchunks ? stage_id(base + 2 * kChunk) : kNone;
        if (kMode != kBwdState && c >= kRing && saved(c - kRing)) {
            // slot sl still holds chunk c - kRing, which the ring now evicts: its
            // rows go to the scratch, where the backward reads them back
            uint32_t* dst = saved_row(c - kRing);
#pragma unroll
            for (int w = 0; w < kWords; ++w) dst[w * kTileThreads] = s_bits[sl][w][threadIdx.x];   // a full chunk
        }
        // Each pixel tests its candidates in list order and composites the ones
        // that pass, with T, the colour, the stop index and dL/dC in registers;
        // its pass bits go to its own row of ring slot sl for the backward.
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            uint32_t cand = done ? 0u : candidates(b, w);
            uint32_t pass = 0u;
            while (cand) {
                const int bt = __ffs(cand) - 1;
                cand &= cand - 1u;
                const int j = (w << 5) | bt;
                float4 r0, r1;
                const float alpha = pass_alpha(b, j, r0, r1);
                if (alpha < 0.0f) continue;
                pass |= 1u << bt;
                const float Tn = T * (1.0f - alpha);
                if (kCount) ++work[kWCompWalk];
                if (a.exclude_crossing && Tn < a.t_min) { done = true; stop = base + j; break; }
                const float wgt = alpha * T;
                C0 = C0 + r1.z * wgt;
                C1 = C1 + r1.w * wgt;
                C2 = C2 + s_r2[b][j].x * wgt;
                T = Tn;
                last = base + j;
                ++ncomp;
                if (!a.exclude_crossing && T < a.t_min) { done = true; stop = base + j; break; }
            }
            s_bits[sl][w][threadIdx.x] = pass;
        }
    }
    cp_async_wait_all();   // a break above can leave the next chunk's copies in flight
    const int nev = inside ? (stop >= 0 ? stop + 1 : len) : 0;
    C0 = C0 + T * a.bg0;
    C1 = C1 + T * a.bg1;
    C2 = C2 + T * a.bg2;
    const size_t pix = (size_t)v * 3 * HW + (size_t)py * a.W + px;
    float g0 = 0.0f, g1 = 0.0f, g2c = 0.0f;
    double lsum = 0.0;
    if (kMode == kBwdState) {
        if (inside) {
            g0 = __ldg(a.dldc + pix);
            g1 = __ldg(a.dldc + pix + HW);
            g2c = __ldg(a.dldc + pix + 2 * HW);
        }
    } else if (inside) {
        a.image[pix] = C0;
        a.image[pix + HW] = C1;
        a.image[pix + 2 * HW] = C2;
        if (kMode == kFwd && a.t_final) {
            a.t_final[spix] = T;
            a.last_idx[spix] = last;
        }
        if (kBackward) {
            const float d0 = C0 - t0v;
            const float d1 = C1 - t1v;
            const float d2 = C2 - t2v;
            lsum = (double)fabsf(d0) + (double)fabsf(d1) + (double)fabsf(d2);
            g0 = d0 > 0.0f ? a.inv3hw : (d0 < 0.0f ? -a.inv3hw : 0.0f);
            g1 = d1 > 0.0f ? a.inv3hw : (d1 < 0.0f ? -a.inv3hw : 0.0f);
            g2c = d2 > 0.0f ? a.inv3hw : (d2 < 0.0f ? -a.inv3hw : 0.0f);
        }
    }
    // Warp sums of the loss and the evaluation counts go to shared memory; the
    // block's are added to global memory once, after the barrier that ends the
    // forward.  (Deferring that barrier to the end of the kernel, so that the
    // warps start their backward without waiting for one another, measured
    // slower on every workload.)
    if (kMode != kBwdState) {
        unsigned long long ef = (unsigned long long)nev, eb = (unsigned long long)(last + 1);
        unsigned long long ec = (unsigned long long)ncomp;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
            ef += __shfl_xor_sync(0xffffffffu, ef, o);
            eb += __shfl_xor_sync(0xffffffffu, eb, o);
            ec += __shfl_xor_sync(0xffffffffu, ec, o);
        }
        if (lane == 0) {
            sm.red_loss[warp] = lsum;
            sm.red_counts[0][warp] = ef;
            sm.red_counts[1][warp] = eb;
            sm.red_counts[2][warp] = ec;
        }
    }
    // Adds the block's loss and counts (after a barrier that every thread reaches).
    auto flush_sums = [&]() {
        if (threadIdx.x == 0) {
            double ls = 0.0;
            unsigned long long x0 = 0ull, x1 = 0ull, x2 = 0ull;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                ls += sm.red_loss[w];
                x0 += sm.red_counts[0][w];
                x1 += sm.red_counts[1][w];
                x2 += sm.red_counts[2][w];
            }
            if (kMode == kFused && ls != 0.0) atomicAdd(a.loss + v, ls * a.inv3hw_d);
            if (a.counts) {
                atomicAdd(a.counts, x0);
                atomicAdd(a.counts + 1, x1);
                atomicAdd(a.counts + 2, x2);
            }
        }
    };
    if (kMode == kFwd) {
        __syncthreads();
        flush_sums();
        // the chunks still in the ring go to the scratch as well (the evicted ones
        // went there during the forward), for a backward from this state
        for (int cc = max(0, resident - kRing + 1); cc <= resident; ++cc) {
            if (!saved(cc)) continue;
            uint32_t* dst = saved_row(cc);
            const int nw = saved_words(cc);
#pragma unroll
            for (int w = 0; w < kWords; ++w)
                if (w < nw) dst[w * kTileThreads] = s_bits[cc % kRing][w][threadIdx.x];
        }
        return;
    }

    // ------------------------------------------------------------- backward
    // The chunks are visited from the forward's last (still in shared memory) down
    // to 0; the ring holds the pass bits of chunks last_fwd - kRing + 1 .. last_fwd
    // (none when the forward ran in an earlier launch: then every chunk's bits
    // come from the scratch, or are recomputed).  A chunk other than the
    // resident one is staged again only if some pixel of the tile composited an
    // entry at or after its start (one vote at the barrier that precedes it); the
    // chunk below it is copied in while the warps work on it.
    if (kMode == kFused) {
        __syncthreads();
        flush_sums();
    }
    const int last_fwd = kMode == kBwdState ? INT32_MAX / 2 : resident;
    const int c_top = kMode == kBwdState ? (len > 0 ? (len - 1) / kChunk : -1) : resident;
    int fetched = -1;    // chunk whose records were last copied into buffer fetched & 1
    uint32_t g_pre = kNone;   // ids of chunk pre_chunk, loaded a step before their copy
    int pre_chunk = -1;
    if (resident >= 1) {
        // the chunk below the resident one, copied in speculatively; its buffer
        // held chunk resident + 1 (never read) or resident - 1 (finished)
        stage_copy(stage_id((resident - 1) * kChunk), (resident - 1) & 1);
        fetched = resident - 1;
        if (resident >= 2) {
            g_pre = stage_id((resident - 2) * kChunk);
            pre_chunk = resident - 2;
        }
    }
    // dL/dC . (colour composited behind the next entry to visit), per pixel
    float Sg = T * __fmaf_rn(g0, a.bg0, __fmaf_rn(g1, a.bg1, g2c * a.bg2));
    float Tcur = T;
    float* __restrict__ g2v = a.grad2d + (size_t)v * (size_t)a.n * GS_GRAD2D_STRIDE;
    uint8_t* __restrict__ touchv = a.touched + (size_t)v * (size_t)a.n;
    for (int c = c_top; c >= 0; --c) {
        const int base = c * kChunk;
        const int sl = c % kRing;
        const int b = c & 1;
        if (c != resident) {
            if (fetched != c) {
                // not copied in ahead (the chunk above was skipped): copy it now;
                // its buffer's previous chunk was finished before the last barrier
                stage_copy(stage_id(base), b);
                fetched = c;
            }
            cp_async_wait_all();
            // barrier: the chunk above is finished by every warp, this one's records visible
            if (!__syncthreads_or(last >= base)) continue;   // no pixel composited anything here or after
            if (c >= 1) {
                stage_copy(pre_chunk == c - 1 ? g_pre : stage_id(base - kChunk), b ^ 1);
                fetched = c - 1;
                if (c >= 2) {
                    g_pre = stage_id(base - 2 * kChunk);
                    pre_chunk = c - 2;
                }
            }
            if (kCount && threadIdx.x == 0) ++work[kWRestaged];
            if (c <= last_fwd - kRing) {
                if (saved(c)) {
                    // pass bits saved by the forward (evicted from the ring, or all
                    // of them for a backward from a stored state)
                    const uint32_t* src = saved_row(c);
                    const int nw = saved_words(c);
#pragma unroll
                    for (int w = 0; w < kWords; ++w) s_bits[sl][w][threadIdx.x] = w < nw ? src[w * kTileThreads] : 0u;
                } else {
                    // pass bits no longer in the ring: recompute them, each pixel up
                    // to its last composited entry (mask buffer 0: the forward is over)
                    build_masks(min(kChunk, len - base), b, 0);
                    __syncthreads();
                    eval_bits(b, 0, sl, last - base);
                    if (kCount && threadIdx.x == 0) ++work[kWRecomputed];
                }
            }
            // (no barrier: a pixel reads back only its own row of pass bits)
            resident = c;
        }
        // This pixel's composited entries in the chunk are its passing bits up to
        // last.
        uint32_t words[kWords];
        int nmine;
        const int nq = gather(words, last - base, sl, nmine);
        if (nq == 0) continue;
        // Distinct entries composited by any of the warp's pixels in this chunk.
        uint32_t uni[kWords];
        int nu = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) {
            uni[w] = __reduce_or_sync(0xffffffffu, words[w]);
            nu += __popc(uni[w]);
        }
        if (nq >= kDense * nu) {
            // Dense chunk (large Gaussians: most of the warp's pixels composite
            // the same entries): walk the union newest first, every lane updating
            // its own pixel's T and dL/dC . (colour behind); the 9 gradient
            // terms are summed over the warp (warp_sum_terms) and added with one
            // atomic per component.
#pragma unroll
            for (int w = kWords - 1; w >= 0; --w) {
                uint32_t u = uni[w];
                while (u) {
                    const int bt = 31 - __clz(u);
                    u &= ~(1u << bt);
                    const int j = (w << 5) | bt;
                    EntryGrad e;
                    e.gm0 = e.gm1 = e.gA = e.gB = e.gC = e.go = e.gr = e.gg = e.gb = 0.0f;
                    if ((words[w] >> bt) & 1u) {
                        const float4 r0 = s_r0[b][j];
                        const float4 r1 = s_r1[b][j];
                        const float cb = s_r2[b][j].x;
                        const float dx = pxf - r0.x, dy = pyf - r0.y;
                        const float power = ((r0.z * dx) * dx + (r1.x * dy) * dy) - (r0.w * dx) * dy;
                        const float G = pexp_neg(power);
                        const float araw = r1.y * G;
                        const float alpha = fminf(alpha_max, araw);
                        const float rc = rcp_approx(1.0f - alpha);
                        const float Tb = Tcur * rc;   // transmittance before this entry
                        const float dotc = __fmaf_rn(g0, r1.z, __fmaf_rn(g1, r1.w, g2c * cb));
                        e = entry_grad_at(r0, r1, dx, dy, G, araw, alpha, alpha_max, g0, g1, g2c, Tb, dotc, Sg, rc);
                        Sg += dotc * alpha * Tb;
                        Tcur = Tb;
                        if (kCount) ++work[kWDenseEntries];
                    }
                    if (kCount && lane == 0) ++work[kWDenseSteps];
                    const float sum = warp_sum_terms(e, lane);
                    const uint32_t gid = s_id[b][j];
                    if (GS_IN_RANGE(gid, a.n, GS_CHECK_RASTER_ID)) {   // a dropped entry never has pass bits
                        if (red_term >= 0) atomicAdd(g2v + (size_t)gid * GS_GRAD2D_STRIDE + red_term, sum);
                        if (lane == 1) touchv[gid] = 1;
                    }
                }
            }
            continue;
        }
        // Sparse chunk: each lane walks its own pixel's entries newest first,
        // T and dL/dC . (colour behind) in registers (no exchange between lanes);
        // each (entry, pixel) pair adds its terms with vector atomics.
        if (kCount) {
            const unsigned steps = __reduce_max_sync(0xffffffffu, (unsigned)nmine);
            if (lane == 0) work[kWSparseSteps] += steps;
        }
#pragma unroll
        for (int w = kWords - 1; w >= 0; --w) {
            uint32_t word = words[w];
            while (word) {
                const int bt = 31 - __clz(word);
                word &= ~(1u << bt);
                const int j = (w << 5) | bt;
                const float4 r0 = s_r0[b][j];
                const float4 r1 = s_r1[b][j];
                const float cb = s_r2[b][j].x;
                const float dx = pxf - r0.x, dy = pyf - r0.y;
                const float power = ((r0.z * dx) * dx + (r1.x * dy) * dy) - (r0.w * dx) * dy;
                const float G = pexp_neg(power);
                const float araw = r1.y * G;
                const float alpha = fminf(alpha_max, araw);
                const float rc = rcp_approx(1.0f - alpha);
                const float Tb = Tcur * rc;
                const float dotc = __fmaf_rn(g0, r1.z, __fmaf_rn(g1, r1.w, g2c * cb));
                const EntryGrad e = entry_grad_at(r0, r1, dx, dy, G, araw, alpha, alpha_max, g0, g1, g2c, Tb, dotc, Sg, rc);
                Sg += dotc * alpha * Tb;
                Tcur = Tb;
                if (kCount) ++work[kWSparseEntries];
                const uint32_t gid = s_id[b][j];
                if (GS_IN_RANGE(gid, a.n, GS_CHECK_RASTER_ID)) {
                    float* dst = g2v + (size_t)gid * GS_GRAD2D_STRIDE;
                    atomicAdd(reinterpret_cast<float4*>(dst), make_float4(e.gm0, e.gm1, e.gA, e.gB));
                    atomicAdd(reinterpret_cast<float4*>(dst + 4), make_float4(e.gC, e.go, e.gr, e.gg));
                    atomicAdd(dst + 8, e.gb);
                    touchv[gid] = 1;
                }
            }
        }
    }
    cp_async_wait_all();   // no copy outlives the block
    if (kCount) {
#pragma unroll
        for (int k = 0; k < kWCount; ++k) {
            unsigned long long x = work[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (lane == 0 && x) atomicAdd(a.work + k, x);
        }
    }
}

}  // namespace gs

using namespace gs;

// Launch with the block's dynamic shared memory (opted in once per variant; the
// maximum shared-memory carveout lets four blocks share an SM).
template <int kMode, bool kCount>
static gs_status launch_raster(const RasterArgs& a, long long grid, cudaStream_t s)
{
    static bool configured = false;
    if (!configured) {
        GS_CUDA_TRY(cudaFuncSetAttribute(raster_fused_kernel<kMode, kCount>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(RasterSmem)));
        GS_CUDA_TRY(cudaFuncSetAttribute(raster_fused_kernel<kMode, kCount>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout, 100));
        configured = true;
    }
    raster_fused_kernel<kMode, kCount><<<(unsigned)grid, kTileThreads, sizeof(RasterSmem), s>>>(a);
    GS_LAUNCH_CHECK();
    return GS_OK;
}

// Arguments shared by the three launches.
static gs_status raster_args(RasterArgs& a, const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                             const uint32_t* ids, const gs_camera* cams, int32_t n_views, const gs_render_opts* opts,
                             long long& grid)
{
    if (!proj || !tile_ranges || !opts_ok(opts) || n < 0 || n > INT32_MAX) return GS_ERR_INVALID_ARG;
    gs_status st = check_views(cams, n_views);
    if (st != GS_OK) return st;
    if (n > 0 && (!proj->rec || !ids)) return GS_ERR_INVALID_ARG;
    if (!aligned16(proj->rec)) return GS_ERR_INVALID_ARG;
    const int W = cams[0].width, H = cams[0].height;
    a = RasterArgs{};
    a.rec = reinterpret_cast<const float4*>(proj->rec);
    a.ranges = reinterpret_cast<const uint2*>(tile_ranges);
    a.ids = ids;
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
    grid = (long long)a.tiles * n_views;
    if (grid > INT32_MAX) return GS_ERR_INVALID_ARG;
    return GS_OK;
}

extern "C" gs_status gs_raster_fused_fwd_bwd(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                             const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                             const gs_render_opts* opts, const float* target, float* image,
                                             double* loss, float* grad2d, uint8_t* touched, uint64_t* eval_counts,
                                             uint32_t* bits_ws, int64_t bits_ws_words, void* stream)
{
    GS_NVTX_RANGE("gs_raster_fused_fwd_bwd");
    RasterArgs a;
    long long grid = 0;
    gs_status st = raster_args(a, proj, n, tile_ranges, ids, cams, n_views, opts, grid);
    if (st != GS_OK) return st;
    if (!image) return GS_ERR_INVALID_ARG;
    if (target && (!loss || (n > 0 && (!grad2d || !touched)))) return GS_ERR_INVALID_ARG;
    if (grad2d && !aligned16(grad2d)) return GS_ERR_INVALID_ARG;
    if (bits_ws_words < 0 || (bits_ws && bits_ws_words == 0)) return GS_ERR_INVALID_ARG;
    a.target = target;
    a.image = image;
    a.loss = loss;
    a.grad2d = grad2d;
    a.touched = touched;
    a.counts = reinterpret_cast<unsigned long long*>(eval_counts);
    a.bits_ws = bits_ws;
    a.bits_ws_words = bits_ws ? bits_ws_words : 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (target) {
        GS_CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(double) * (size_t)n_views, s));
        return launch_raster<kFused, false>(a, grid, s);
    }
    return launch_raster<kFwd, false>(a, grid, s);
}

extern "C" gs_status gs_raster_work_counts(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                           const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                           const gs_render_opts* opts, const float* target, float* image,
                                           double* loss, float* grad2d, uint8_t* touched, uint64_t* work,
                                           uint32_t* bits_ws, int64_t bits_ws_words, void* stream)
{
    GS_NVTX_RANGE("gs_raster_work_counts");
    RasterArgs a;
    long long grid = 0;
    gs_status st = raster_args(a, proj, n, tile_ranges, ids, cams, n_views, opts, grid);
    if (st != GS_OK) return st;
    if (!image || !target || !loss || !work || (n > 0 && (!grad2d || !touched))) return GS_ERR_INVALID_ARG;
    if (grad2d && !aligned16(grad2d)) return GS_ERR_INVALID_ARG;
    if (bits_ws_words < 0 || (bits_ws && bits_ws_words == 0)) return GS_ERR_INVALID_ARG;
    static_assert(kWCount == GS_RASTER_WORK_COUNTERS, "counter layout");
    a.bits_ws = bits_ws;
    a.bits_ws_words = bits_ws ? bits_ws_words : 0;
    a.target = target;
    a.image = image;
    a.loss = loss;
    a.grad2d = grad2d;
    a.touched = touched;
    a.work = reinterpret_cast<unsigned long long*>(work);
    cudaStream_t s = (cudaStream_t)stream;
    GS_CUDA_TRY(cudaMemsetAsync(loss, 0, sizeof(double) * (size_t)n_views, s));
    return launch_raster<kFused, true>(a, grid, s);
}

extern "C" gs_status gs_raster_forward_state(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                             const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                             const gs_render_opts* opts, float* image, float* t_final,
                                             int32_t* last_idx, uint32_t* bits_ws, int64_t bits_ws_words,
                                             uint64_t* eval_counts, void* stream)
{
    GS_NVTX_RANGE("gs_raster_forward_state");
    RasterArgs a;
    long long grid = 0;
    gs_status st = raster_args(a, proj, n, tile_ranges, ids, cams, n_views, opts, grid);
    if (st != GS_OK) return st;
    if (!image || !t_final || !last_idx) return GS_ERR_INVALID_ARG;
    if (bits_ws_words < 0 || (bits_ws && bits_ws_words == 0)) return GS_ERR_INVALID_ARG;
    a.image = image;
    a.t_final = t_final;
    a.last_idx = last_idx;
    a.bits_ws = bits_ws;
    a.bits_ws_words = bits_ws ? bits_ws_words : 0;
    a.counts = reinterpret_cast<unsigned long long*>(eval_counts);
    return launch_raster<kFwd, false>(a, grid, (cudaStream_t)stream);
}

extern "C" gs_status gs_raster_backward_state(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                              const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                              const gs_render_opts* opts, const float* t_final,
                                              const int32_t* last_idx, const uint32_t* bits_ws,
                                              int64_t bits_ws_words, const float* dldc, float* grad2d,
                                              uint8_t* touched, void* stream)
{
    GS_NVTX_RANGE("gs_raster_backward_state");
    RasterArgs a;
    long long grid = 0;
    gs_status st = raster_args(a, proj, n, tile_ranges, ids, cams, n_views, opts, grid);
    if (st != GS_OK) return st;
    if (!t_final || !last_idx || !dldc || (n > 0 && (!grad2d || !touched))) return GS_ERR_INVALID_ARG;
    if (bits_ws_words < 0 || (bits_ws && bits_ws_words == 0)) return GS_ERR_INVALID_ARG;
    a.bits_ws = const_cast<uint32_t*>(bits_ws);   // only read in this mode
    a.bits_ws_words = bits_ws ? bits_ws_words : 0;
    if (grad2d && !aligned16(grad2d)) return GS_ERR_INVALID_ARG;
    a.t_final = const_cast<float*>(t_final);
    a.last_idx = const_cast<int32_t*>(last_idx);
    a.dldc = dldc;
    a.grad2d = grad2d;
    a.touched = touched;
    return launch_raster<kBwdState, false>(a, grid, (cudaStream_t)stream);
}
