/*
 * gs.h -- C ABI of the GB300 (sm_103a) 3D Gaussian Splatting training step.
 *
 * One training step is five calls on one CUDA stream:
 *
 *   gs_project               EWA projection, culling, colour (per Gaussian x view)
 *   gs_bin_sort              16x16 tile binning with (tile, depth) keys + sort
 *   gs_raster_fused_fwd_bwd  forward compositing, L1 loss and backward in ONE kernel
 *   gs_grad_compact          touched-set compaction, projection VJP, scatter-add
 *   gs_adam_deferred         Adam on the touched Gaussians only, with catch-up
 *
 * Method sources (pages, by title and section):
 *   ByteSplat: Efficient Distributed 3DGS Training via Intra- and Inter-GPU
 *     Communication Reduction -- English abstract: forward and backward
 *     rasterization fused into a single kernel that keeps intermediate results
 *     on chip; zero partial gradients eliminated, the remaining records compacted
 *     by an encoder and aggregated by a decoder.
 *   On Scaling Up 3D Gaussian Splatting Training (Grendel) -- abstract: batched
 *     training over multiple views, sqrt(batch size) hyper-parameter scaling;
 *     method-details section: L1 loss.
 *   GS-Scale: Unlocking Large-Scale 3DGS Training via Host Offloading --
 *     abstract: frustum culling; deferred optimizer update that avoids memory
 *     traffic for Gaussians with zero gradients.
 * The rasterizer arithmetic is the standard tile-based 3DGS one: EWA projection
 * to a 2D conic and radius, alpha = min(0.99, o * exp(-1/2 d^T Sigma2D^-1 d)),
 * alpha < 1/255 skipped, compositing stops once T < 1e-4.
 *
 * Conventions for every call
 *   - Returns gs_status; nothing is thrown across the ABI.
 *   - All array pointers are DEVICE pointers owned by the caller unless the
 *     argument says "host".  The library allocates no device memory and keeps no
 *     state between calls (two exceptions, both stated with their calls:
 *     gs_bin_sort's 24-byte pinned host buffer per calling thread and
 *     gs_grad_compact_static's device scratch); calls that need scratch take
 *     (ws, ws_bytes): pass ws == NULL to query the size into *ws_bytes.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  gs_bin_sort is the only call that synchronises the host
 *     (it reads the instance count back to size the sort).
 *   - Arithmetic is fp32 (fp64 for the loss sum).  The forward decisions (cull,
 *     tile rect, alpha skip, transmittance stop) are computed with IEEE-rounded
 *     + - * / sqrt, no contraction, and one portable exp (Cody-Waite reduction,
 *     degree-7 Taylor polynomial in Horner form with fma, exact 2^k scaling),
 *     so they are reproducible bit for bit by a CPU implementation.
 *   - Sizes: n <= 2^31 - 1 Gaussians, n_views <= GS_MAX_VIEWS, all views share
 *     one resolution, instance count < 2^32.
 *   - Thread-compatible: no hidden globals; concurrent calls on different
 *     buffers are safe.
 *
 * Parameter buffer ([n][stride] fp32, Gaussian-major: Gaussian g's parameters
 * are params[g * stride + k], stride = gs_param_stride(sh_degree) = 16 or 64 so
 * each Gaussian is one aligned 64- or 256-byte block; entries k >= P are padding,
 * never read by the projection and left as given by the optimizer when zero):
 *   k 0-2 mean (world), 3-5 log-scale, 6-9 quaternion (w, x, y, z; any norm),
 *   10 opacity logit, colour: degree 0 -> k 11-13 RGB (P = 14);
 *   degree 3 -> SH coefficient j (0..15, j = l^2 + l + m, real orthonormal basis
 *   without Condon-Shortley phase), channel c at k = 11 + 3j + c (P = 59);
 *   colour = max(0, sum_j coef_j Y_j(dir) + 0.5), dir = unit(mean - camera centre).
 * Gradients and the Adam moments use the same layout.
 */
#ifndef GS_H
#define GS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GS_API __attribute__((visibility("default")))
#else
#define GS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gs_status {
    GS_OK = 0,
    GS_ERR_INVALID_ARG = 1, /* a pointer, size or option is out of range          */
    GS_ERR_CAPACITY = 2,    /* instance buffers too small; needed count reported  */
    GS_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed        */
    GS_ERR_TIMEOUT = 4,     /* reserved: no call waits on the device              */
    GS_ERR_DEVICE = 5       /* a kernel reported an error through the device word */
} gs_status;

#define GS_TILE 16          /* tile edge in pixels                                */
#define GS_MAX_VIEWS 32     /* views per call (cameras are passed by value)       */
#define GS_REC_FLOAT4 3     /* float4 per projected record                        */
#define GS_GRAD2D_STRIDE 12 /* floats per (view, Gaussian) in grad2d              */

/* Pinhole camera.  World -> camera: x_c = R x_w + t (R row-major).  Camera looks
 * along +z, image x right, y down; pixel (i, j) has its centre at (i + .5, j + .5);
 * u = fx * x_c / z_c + cx,  v = fy * y_c / z_c + cy. */
typedef struct gs_camera {
    float R[9];
    float t[3];
    float fx, fy, cx, cy;
    int32_t width, height;
} gs_camera;

/* Render options.  Defaults: near_z 0.2, lowpass 0.3 (px^2 added to the 2D
 * covariance diagonal), alpha_min 1/255 (skip below), alpha_max 0.99 (clamp),
 * t_min 1e-4 (stop once T falls below it; the Gaussian that crosses is
 * composited unless exclude_crossing = 1), bg = background colour.
 * Valid ranges (else GS_ERR_INVALID_ARG): 1e-30 <= alpha_min <= alpha_max < 1,
 * alpha_max > 0, t_min >= 0, near_z > 0, lowpass >= 0. */
typedef struct gs_render_opts {
    float near_z, lowpass, alpha_min, alpha_max, t_min;
    float bg[3];
    int32_t exclude_crossing;
    int32_t reserved;
} gs_render_opts;

/* Per-view projected records, caller-allocated, each [n_views][n]:
 *   rec            3 float4 per (view, Gaussian), 16-byte aligned:
 *                  {mx, my, -A/2, B}, {-C/2, opacity, r, g}, {b, tau, hx, hy}
 *                  (mean in pixels, conic (A, B, C) = Sigma2D^-1;
 *                  tau = ln(alpha_min / opacity) - 0.01: any pixel with power
 *                  below tau has alpha < alpha_min, +inf if opacity < alpha_min;
 *                  hx, hy: half-extents of a box around the mean outside which
 *                  the rasterizer's fp32 power is below tau, -1 if no pixel can
 *                  pass, +inf if no bound is available);
 *                  written only for visible Gaussians
 *   depth          float z_c (written only for visible Gaussians)
 *   rect           4 x uint16 tile bounds x0, y0, x1, y1, half-open, clipped
 *                  to the grid (written only for visible Gaussians)
 *   tiles_touched  (x1 - x0) * (y1 - y0), 0 = culled (always written)
 */
typedef struct gs_proj {
    float* rec;
    float* depth;
    uint16_t* rect;
    uint32_t* tiles_touched;
} gs_proj;

/* EWA projection of every Gaussian into every view (one pass over params).
 * Cull: z_c <= near_z, non-finite values, zero quaternion, det(Sigma2D) <= 0,
 * or an empty tile rect.  Radius = ceil(3 sqrt(lambda_max(Sigma2D))); rect =
 * tiles floor((m -/+ r)/16).  Opacity = sigmoid(logit).
 * params: [n][stride]; cams/opts: HOST; out: device arrays described above.
 * Errors: INVALID_ARG for NULL pointers, n < 0, n_views outside 1..GS_MAX_VIEWS,
 * sh_degree not 0 or 3, differing view sizes; CUDA on launch failure. */
GS_API gs_status gs_project(const float* params, int64_t n, int32_t sh_degree, const gs_camera* cams, int32_t n_views,
                     const gs_render_opts* opts, const gs_proj* out, void* stream);

/* Tile binning and sort.  Every visible (view v, Gaussian g) emits one instance
 * per tile of its rect with key = ((v * tiles + tile) << 32) | bits(depth) and
 * value g; instances are sorted by key, stably, so equal keys keep ascending g
 * (a counting sort on v * tiles + tile, then every (view, tile) bucket sorted on
 * (bits(depth), g): the same order as an LSD radix sort of the keys).
 * keys, ids: [capacity] outputs (sorted); tile_ranges: [n_views * tiles][2]
 * uint32 [start, end) into the sorted arrays (start == end: empty tile).
 * n_instances: HOST out, set even when the capacity is too small.
 * ws / ws_bytes: scratch (ws == NULL: query).  Synchronises the host once, on
 * the read-back of the instance count (an event after the copy, so the scatter
 * and the sorts of buckets up to 2048 instances, already queued, run
 * meanwhile), and a second time only when some tile holds more than 16384
 * instances: the key-range splitter of such buckets reports a range it could
 * not sort through a device error word, read back before returning.  The
 * count is read into a 24-byte pinned host buffer that each calling thread
 * allocates on its first call and keeps for its lifetime.
 * Errors: CAPACITY if n_instances > capacity (outputs untouched: the queued
 * kernels check the count on the device and write nothing);
 * INVALID_ARG for bad sizes (width above 655360, i.e. more than 40960 tiles in a
 * row) or a too small workspace; DEVICE if the splitter's pending-range stack
 * overflowed (impossible for unique keys: each split level narrows the key
 * interval by at least 512, so at most seven levels are pending). */
GS_API gs_status gs_bin_sort(const gs_proj* proj, int64_t n, int32_t n_views, int32_t width, int32_t height,
                      int64_t capacity, uint64_t* keys, uint32_t* ids, uint32_t* tile_ranges,
                      int64_t* n_instances, void* ws, size_t* ws_bytes, void* stream);

/* Hardware-aware pruning of the sorted tile lists (ByteSplat, English abstract:
 * pruning that weighs rendering quality against the per-tile shared-memory
 * budget).  A tile list longer than `budget` keeps its `budget` most opaque
 * entries (equal opacities: the earlier, nearer entry) in depth order; its
 * ids are compacted in place at the start of its range and the range end
 * becomes start + budget.  Other lists are untouched.  The fused raster kernel
 * keeps the pass bits of 3 x 256 entries per tile on chip, so budget = 768
 * bounds every list to what its backward can take without recomputing them.
 * proj: as given to gs_bin_sort (opacity = record float 5).  ids, tile_ranges:
 * gs_bin_sort's outputs, updated in place (keys are left as sorted).
 * budget >= 1.
 * Errors: INVALID_ARG for bad pointers, sizes or budget; CUDA on launch failure. */
GS_API gs_status gs_prune_tiles(const gs_proj* proj, int64_t n, int32_t n_views, int32_t width, int32_t height,
                                int32_t budget, uint32_t* ids, uint32_t* tile_ranges, void* stream);

/* Fused forward + backward rasterization: one CTA per 16x16 tile (256 threads,
 * one pixel each).  Forward: front-to-back over the tile's sorted list, skip
 * power > 0 or alpha < alpha_min, C += c * alpha * T, T *= 1 - alpha, stop at
 * T < t_min; C += T * bg.  The list's records pass through shared memory in
 * chunks of 256, the next chunk copied in (cp.async) while the block works on
 * the current one; each pixel walks the entries whose support box covers it
 * (per-chunk row and column candidate masks) in list order.  The per-pixel T,
 * colour and last index stay in registers, and the entries that pass set bits
 * in the pixel's row of an on-chip ring that keeps the last three chunks.  With
 * a target: L1 loss per view, mean over 3*H*W values, summed in fp64, and its
 * gradient sign(C - target) / (3HW) on chip; backward walks each pixel's
 * composited entries back to front, T recovered by division and
 * dL/dC . (colour behind) carried in registers, and adds each entry's 9
 * gradient terms to the Gaussian's grad2d row with vector atomics (their order
 * varies from run to run); where most of a warp's pixels share the entries it
 * sums the terms over the warp first.
 * target: [V][3][H][W] or NULL (forward only: no loss, gradients or touched).
 * image: [V][3][H][W] out.  loss: [V] fp64 out (overwritten).
 * grad2d: [V][n][GS_GRAD2D_STRIDE] accumulated (+=): d/d mean2d (x, y),
 *   d/d conic (A, B, C), d/d opacity, d/d colour (r, g, b), 3 pad floats.
 * touched: [V][n] u8 set to 1 for every Gaussian composited at least once.
 *   grad2d and touched must be zero on entry; gs_grad_compact returns them to
 *   zero, so a step loop needs to clear them only once.
 * eval_counts: NULL or [3] u64 accumulated (+=): E_fwd = list entries evaluated
 *   up to the stop (skipped ones included), E_bwd = sum of (last index + 1),
 *   E_comp = entries composited (alpha >= alpha_min and not stopped).
 * bits_ws, bits_ws_words: NULL and 0, or a DEVICE u32 scratch and its size in
 *   words.  The pass bits of the chunks the on-chip ring evicts are saved there
 *   in the forward and read back by the backward instead of being recomputed.
 *   Layout: list l's chunk c (256 entries) from word (start of l + 32 l +
 *   256 c) * 8 on, word w of pixel p at 256 w + p (bit j: entry 32 w + j of the
 *   chunk passes at p), only the words that hold entries; a chunk whose slot
 *   lies past the scratch's end is recomputed.  GS_RASTER_BITS_WS_WORDS(I, L)
 *   words cover I instances in L = n_views * tiles lists laid out in tile order
 *   (as gs_bin_sort and gs_prune_tiles leave them).  Contents on entry are
 *   ignored and left undefined; results do not depend on the scratch.
 * Errors: INVALID_ARG for bad pointers or sizes; CUDA on launch failure. */
#define GS_RASTER_BITS_WS_WORDS(n_instances, n_lists) (((int64_t)(n_instances) + 32 * (int64_t)(n_lists)) * 8)
GS_API gs_status gs_raster_fused_fwd_bwd(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges, const uint32_t* ids,
                                  const gs_camera* cams, int32_t n_views, const gs_render_opts* opts,
                                  const float* target, float* image, double* loss, float* grad2d, uint8_t* touched,
                                  uint64_t* eval_counts, uint32_t* bits_ws, int64_t bits_ws_words, void* stream);

/* Executed-work counters of the fused kernel -- a measurement aid with no
 * counterpart on the pages: the kernel skips, with results unchanged, the
 * (entry, pixel) pairs its per-Gaussian support box and alpha cut prove
 * cannot pass, so the work it executes is far below E_fwd + E_bwd.  Runs the
 * same step as gs_raster_fused_fwd_bwd (target required; same outputs, eval
 * counts not taken; bits_ws as there) in a variant that also counts, into
 * work[] (DEVICE u64,
 * accumulated +=), in this order:
 *   0 candidates tested (power)          1 of which reached the exponential
 *   2 of which were composited            3 backward per-pixel walk entries
 *   4 ... walk steps (per warp)           5 backward per-Gaussian evaluations
 *   6 backward per-Gaussian steps (warp)  7 chunks staged in the forward
 *   8 chunks staged again in the backward 9 of which had pass bits recomputed
 * The counting makes it slower; time gs_raster_fused_fwd_bwd, count here.
 * Errors: INVALID_ARG for bad pointers or sizes; CUDA on launch failure. */
#define GS_RASTER_WORK_COUNTERS 10
GS_API gs_status gs_raster_work_counts(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                       const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                       const gs_render_opts* opts, const float* target, float* image, double* loss,
                                       float* grad2d, uint8_t* touched, uint64_t* work, uint32_t* bits_ws,
                                       int64_t bits_ws_words, void* stream);

/* ---- L1 + D-SSIM loss (the standard 3DGS loss: On Scaling Up 3D Gaussian
 * Splatting Training, summary of the loss) ----
 * The SSIM window reaches 10 pixels beyond a tile, into tiles other CTAs
 * render, so this loss cannot live inside the fused kernel.  A step with it is
 * three launches instead of one:
 *   gs_raster_forward_state   image + per-pixel final T and last index
 *   gs_dssim_loss_grad        loss and dL/dC from image and target
 *   gs_raster_backward_state  backward from the stored state and dL/dC
 * The forward saves every chunk's pass bits to a scratch (as the fused kernel
 * saves the chunks its on-chip ring evicts) and the backward reads them back
 * instead of recomputing them; otherwise it is the fused kernel's backward. */

/* Forward rasterization as in gs_raster_fused_fwd_bwd without a target, that
 * also stores per pixel the final transmittance and the last composited list
 * index (-1 if none), and optionally the pass bits of every chunk of 256 list
 * entries it works on (the backward reads them instead of recomputing them).
 * image: [V][3][H][W] out.  t_final: [V][H][W] fp32 out.  last_idx: [V][H][W]
 * int32 out.  bits_ws, bits_ws_words: NULL and 0, or a DEVICE u32 scratch and
 * its size in words, laid out as for gs_raster_fused_fwd_bwd (8 words per list
 * entry at its list position: word w of pixel p of a chunk at 256 w + p, bit j
 * set when entry 32 w + j of the chunk passes at p); chunks whose slot lies past
 * the scratch's end are not stored.  eval_counts: NULL or [3] u64 accumulated
 * (+=), as for the fused call.
 * Errors: INVALID_ARG for bad pointers or sizes; CUDA on launch failure. */
GS_API gs_status gs_raster_forward_state(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                         const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                         const gs_render_opts* opts, float* image, float* t_final, int32_t* last_idx,
                                         uint32_t* bits_ws, int64_t bits_ws_words, uint64_t* eval_counts,
                                         void* stream);

/* Loss (1 - lambda) L1 + lambda (1 - SSIM) per view and its gradient
 * dL/dC.  L1 = mean |image - target| over 3*H*W values; SSIM = mean over
 * channels and pixels of the SSIM map, per channel with an 11 x 11 Gaussian
 * window (sigma 1.5, weights normalised to sum 1), the images zero outside
 * their borders, C1 = 0.01^2, C2 = 0.03^2.  dL/dC = (1 - lambda) sign(image -
 * target) / (3HW) - lambda dSSIM/dimage.  fp32 arithmetic, loss summed in fp64.
 * image, target: [V][3][H][W].  loss: [V] fp64 out (overwritten).
 * dldc: [V][3][H][W] fp32 out.  0 <= lambda <= 1 (3DGS uses 0.2).
 * Errors: INVALID_ARG for bad pointers, sizes or lambda; CUDA on launch failure. */
GS_API gs_status gs_dssim_loss_grad(const float* image, const float* target, int32_t n_views, int32_t width,
                                    int32_t height, float lambda, double* loss, float* dldc, void* stream);

/* Backward rasterization from a stored forward state: the pixels' composited
 * entries are walked back to front exactly as in gs_raster_fused_fwd_bwd, with
 * dL/dC taken from dldc instead of the L1 sign.  proj, tile lists, cams and
 * opts must be those of the gs_raster_forward_state call that wrote t_final,
 * last_idx and (if given) the scratch bits_ws / bits_ws_words, read here; a
 * chunk without a slot in it (or all, without a scratch) has its pass bits
 * recomputed.  dldc: [V][3][H][W].  grad2d, touched: as for the fused call
 * (accumulated; zero on entry).
 * Errors: INVALID_ARG for bad pointers or sizes; CUDA on launch failure. */
GS_API gs_status gs_raster_backward_state(const gs_proj* proj, int64_t n, const uint32_t* tile_ranges,
                                          const uint32_t* ids, const gs_camera* cams, int32_t n_views,
                                          const gs_render_opts* opts, const float* t_final, const int32_t* last_idx,
                                          const uint32_t* bits_ws, int64_t bits_ws_words, const float* dldc,
                                          float* grad2d, uint8_t* touched, void* stream);

/* ---- Partial render + compose (Splaxel, English abstract: each part renders
 * its local subset of Gaussians; only partial pixel values -- colour and
 * transmittance -- are exchanged and composed) ----
 * Subsets are per-view depth slabs: slab s = the Gaussians with
 * z_s <= depth < z_{s+1} (z_0 = 0, z_S = +inf).  A slab's entries in a tile are a
 * contiguous part of the tile's sorted list, so a partial render is
 * gs_raster_forward_state over the slab's sub-ranges with a zero background.
 * Composing the slabs front to back regroups the one-pass compositing; it
 * differs from the one-pass render only where a pixel stops before its last
 * slab, by at most the transmittance at the stop (below t_min, or below
 * t_min / (1 - alpha_max) with the crossing entry excluded) times the largest
 * colour value. */

/* Sub-ranges of every tile list per slab.
 * keys, tile_ranges: gs_bin_sort's outputs (unpruned lists).  depth_splits: HOST
 * [V][S-1] fp32, positive, finite and ascending per view.  sub_ranges:
 * [S][V * tiles][2] u32 out (slab s of view v, tile t at (s * V + v) * tiles + t).
 * 1 <= n_subsets <= 8.
 * Errors: INVALID_ARG for bad pointers, sizes or splits; CUDA on launch failure. */
GS_API gs_status gs_split_ranges(const uint64_t* keys, const uint32_t* tile_ranges, int32_t n_views, int32_t width,
                                 int32_t height, int32_t n_subsets, const float* depth_splits, uint32_t* sub_ranges,
                                 void* stream);

/* Front-to-back composition of partial renders, per pixel in fp32 with fused
 * multiply-adds: C = sum_s (prod_{j<s} T_j) C_s + (prod_s T_s) bg,
 * T = prod_s T_s.
 * c_parts: [S][V][3][H][W]; t_parts: [S][V][H][W]; bg: HOST [3].
 * image: [V][3][H][W] out; t_final: [V][H][W] out or NULL.  1 <= n_subsets <= 8.
 * Errors: INVALID_ARG for bad pointers or sizes; CUDA on launch failure. */
GS_API gs_status gs_compose(const float* c_parts, const float* t_parts, int32_t n_subsets, int32_t n_views,
                            int32_t width, int32_t height, const float* bg, float* image, float* t_final,
                            void* stream);

/* Sparse-gradient compaction ("encoder") and aggregation ("decoder"):
 * per view, idx[v] = ascending list of touched Gaussians, n_idx[v] its length;
 * idx[n_views] / n_idx[n_views] = the union over views.  For every Gaussian of
 * the union the projection VJP of each touching view is summed in view order
 * and written as its gradient block (write only; the blocks of Gaussians
 * outside the union are not touched, so they keep whatever an earlier step
 * left there).  grad2d and touched are cleared for the entries consumed.
 * touched and grad2d are those a gs_raster_* call left for the same params,
 * cams and opts: a touched (Gaussian, view) was composited, hence visible, and
 * for SH degree 3 the VJP recomputes the projection without repeating the
 * culling tests (it differentiates the projection a composited record came
 * from).  With SH degree 3 and several views the geometry and colour terms are
 * each summed in view order and then added.
 * idx: [(n_views + 1) * n] u32 out; n_idx: [n_views + 1] int64 DEVICE out.
 * grads: [n][stride] fp32 out (union blocks only).  cams/opts: HOST, as given to gs_project.
 * Errors: INVALID_ARG for bad pointers, sizes or a too small workspace. */
GS_API gs_status gs_grad_compact(float* grad2d, uint8_t* touched, const float* params, int64_t n, int32_t sh_degree,
                          const gs_camera* cams, int32_t n_views, const gs_render_opts* opts,
                          uint32_t* idx, int64_t* n_idx, float* grads, void* ws, size_t* ws_bytes, void* stream);

/* Maximum Gaussian count of gs_grad_compact_static (its scratch: ~4.2 MB per GPU). */
#define GS_COMPACT_STATIC_MAX_N (1 << 22)

/* gs_grad_compact without a workspace argument, for callers that cannot
 * allocate device memory while they run -- e.g. code embedded in a host
 * application that owns all GPU memory and exposes no allocator, or a
 * deployment that fixes its memory budget at start-up.  The pages have no
 * counterpart; this is an interface convenience of this library.
 * Scratch lives in one file-scope device array of this library (about 4.2 MB,
 * sized for GS_COMPACT_STATIC_MAX_N Gaussians), which every GPU that loads the
 * library keeps until the process exits.  The call allocates nothing (no
 * cudaMalloc/cudaFree, no allocating library routine).
 * Same arguments, outputs and errors as gs_grad_compact, minus (ws, ws_bytes);
 * n > GS_COMPACT_STATIC_MAX_N returns GS_ERR_INVALID_ARG.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  A device reset (cudaDeviceReset)
 * destroys the array's context: the next call on that device sees a new
 * context, looks the address up again (make it, too, before any capture) and
 * finds the array's contents undefined, which the call does not rely on.  All calls share the one array: calls
 * whose work overlaps on the GPU (other streams, other threads) race on it and
 * must be serialised by the caller.  Nothing in it needs to start at zero; it
 * keeps whatever the last call left there. */
GS_API gs_status gs_grad_compact_static(float* grad2d, uint8_t* touched, const float* params, int64_t n,
                                        int32_t sh_degree, const gs_camera* cams, int32_t n_views,
                                        const gs_render_opts* opts, uint32_t* idx, int64_t* n_idx, float* grads,
                                        void* stream);

/* Deferred Adam (dense-equivalent).  For every listed Gaussian g with
 * s = last_step[g] < t: the skipped zero-gradient steps j = s+1 .. t-1 are
 * replayed, then step t uses grads; last_step[g] = t.  grads is only read (the
 * listed Gaussians' blocks, as gs_grad_compact wrote them this step).
 * One step: m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2;
 *           p -= lr * ((m / bc1) / (sqrt(v / bc2) + eps)),
 * bc = 1 - beta^j with beta^j by binary exponentiation in fp64, rounded to fp32.
 * flush = 1: every Gaussian with last_step < t is brought to step t with zero
 *   gradients (idx, n_idx, grads unused) -- call before reading or saving params.
 * params, grads, m, v: [n][stride]; last_step: [n] int32 (0 = never stepped).
 * idx: [>= *n_idx] u32, n_idx: DEVICE int64.  lr: HOST [5] per group (mean,
 * log-scale, quaternion, opacity, colour), each finite and >= 0; 0 <= beta1,
 * beta2 < 1; eps > 0 and finite; t >= 1.  Padding entries k >= P of a block are
 * never touched.
 * Errors: INVALID_ARG for bad pointers, t < 1, or lr / beta / eps out of range. */
GS_API gs_status gs_adam_deferred(float* params, float* grads, float* m, float* v, int32_t* last_step, int64_t n,
                           int32_t sh_degree, const uint32_t* idx, const int64_t* n_idx, int32_t t, const float* lr,
                           float beta1, float beta2, float eps, int32_t flush, void* stream);

/* ---------------------------------------------------------------------------
 * Bounds-checked build.  The same sources compiled with -DGS_CHECKED give
 * libgs_gb300_checked.so, in which every kernel tests the indexes it reads from
 * memory before it uses them: the Gaussian index of a sorted, listed or
 * compacted entry against n, a projected tile rect against the tile grid, a
 * scatter slot against the instance capacity, a tile range's end against its
 * start.  A failing index is counted and the access it would make is skipped
 * (the entry is dropped, the write not made), so a bad index never reaches
 * memory; no kernel traps.  The plain library compiles the tests away.
 * Sites, reported as the `site` word below: */
typedef enum gs_check_site {
    GS_CHECK_NONE = 0,
    GS_CHECK_BIN_RECT = 1,    /* gs_bin_sort: a touched Gaussian's rect outside the grid (index: its end)  */
    GS_CHECK_BIN_SLOT = 2,    /* gs_bin_sort: a scatter slot >= capacity                                     */
    GS_CHECK_SORT_SLOT = 3,   /* gs_bin_sort: a sorted entry's position >= capacity                          */
    GS_CHECK_SORT_ID = 4,     /* gs_bin_sort: a sorted entry's Gaussian index >= n                           */
    GS_CHECK_RANGE = 5,       /* raster / prune / split: a tile range whose end precedes its start           */
    GS_CHECK_RASTER_ID = 6,   /* raster kernels: a listed Gaussian index >= n (entry dropped)                */
    GS_CHECK_PRUNE_ID = 7,    /* gs_prune_tiles: a listed Gaussian index >= n (read as opacity 0)            */
    GS_CHECK_COMPACT_ID = 8,  /* gs_grad_compact: a union-list index >= n (entry skipped)                    */
    GS_CHECK_ADAM_ID = 9      /* gs_adam_deferred: a listed index >= n (entry skipped)                       */
} gs_check_site;

/* Report of the bounds checks since the previous report, then reset.
 * report: HOST [4] u64 out: number of failed checks; the site (gs_check_site),
 *   index and bound of one of the first to fail (zeros when none failed).
 *   An index read as a negative number is reported in two's complement.
 * checked: HOST int32 out: 1 from the bounds-checked build, 0 from the plain
 *   one (whose report is always zeros and which does no device work here).
 * The checked build synchronizes the device first (all streams), so the report
 * covers every kernel launched before the call.
 * Errors: INVALID_ARG for NULL pointers; DEVICE when a check failed; CUDA when a
 * copy of the records fails. */
GS_API gs_status gs_check_report(uint64_t* report, int32_t* checked);

/* Static helpers (no device work). */
GS_API const char* gs_error_string(gs_status s);
GS_API int32_t gs_param_rows(int32_t sh_degree);                     /* P: 14, 59, or -1 */
GS_API int32_t gs_param_stride(int32_t sh_degree);                   /* 16, 64, or -1 */
GS_API int64_t gs_num_tiles(int32_t width, int32_t height);          /* ceil(W/16) * ceil(H/16) */
GS_API const char* gs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GS_H */
