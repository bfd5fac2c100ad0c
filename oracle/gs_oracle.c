/*
 * gs_oracle.c -- CPU oracle for the tile-based 3D Gaussian Splatting training step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  The product path never calls it;
 * it shares no code, header or constant with the CUDA library.
 *
 * Plain, slow, single-threaded and untiled: every step is the definition written
 * out in the order the method states it.  The file is compiled twice:
 *   REAL=float  (symbols *_f32): the precision the workloads fix (fp32); its
 *                forward decisions (cull, rect, skip, stop) are the reference for
 *                bit-exact indexing.
 *   REAL=double (symbols *_f64): the same definition in fp64 with libm exp, used
 *                by the finite-difference checks of the gradients.
 * Gradients (per-pixel contributions and their sums) are always accumulated in
 * fp64, from the forward values of the chosen precision.
 *
 * Sources of the method (pages, by title and section):
 *   - ByteSplat (distributed 3DGS training with less intra-/inter-GPU data
 *     movement), English abstract: one fused forward+backward rasterization,
 *     gradient sparsity, encoder (compaction) / decoder (aggregation).
 *   - On Scaling Up 3D Gaussian Splatting Training (Grendel), abstract: batched
 *     multi-view training, sqrt(batch) learning-rate scaling; method details
 *     section: L1 loss.
 *   - GS-Scale, abstract: frustum culling, deferred optimizer update that skips
 *     Gaussians with zero gradient.
 *   The rasterizer's arithmetic (EWA projection, 16x16 tiles, (tile, depth) keys,
 *   alpha = min(0.99, o*exp(-1/2 d^T Sigma2D^-1 d)), skip alpha < 1/255, stop at
 *   T < 1e-4) is the standard tile-based 3DGS formulation the pages build on;
 *   where a step is left open, the reading taken is marked [reading].
 *
 * Build (both precisions into one library):
 *   gcc -O2 -std=c11 -fPIC -ffp-contract=off -fno-fast-math -DREAL=float  -c ...
 *   gcc -O2 -std=c11 -fPIC -ffp-contract=off -fno-fast-math -DREAL=double -c ...
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL float
#endif

#define CAT2(a, b) a##b
#define CAT(a, b) CAT2(a, b)

#if defined(REAL_IS_DOUBLE)
#define SFX _f64
#define SQRT(x) sqrt(x)
#define FLOOR(x) floor(x)
#define CEIL(x) ceil(x)
#define FABS(x) fabs(x)
#define ISFIN(x) isfinite(x)
#else
#define SFX _f32
#define SQRT(x) sqrtf(x)
#define FLOOR(x) floorf(x)
#define CEIL(x) ceilf(x)
#define FABS(x) fabsf(x)
#define ISFIN(x) isfinite(x)
#endif
#define FN(name) CAT(name, SFX)

#define TILE 16

/* ------------------------------------------------------------------------- */
/* Portable exponential.                                                      */
/*                                                                           */
/* The cull/rect/skip/stop decisions depend on exp(); platform expf() results  */
/* differ in the last ulp between libraries, so the fp32 method uses one exp   */
/* specified from first principles and implemented independently on each side: */
/*   Cody & Waite (1980) argument reduction  x = k*ln2 + r,  k = rint(x*log2 e),*/
/*   r = fma(-k, ln2_hi, x);  r = fma(-k, ln2_lo, r)  (ln2 split hi + lo),      */
/*   e^r by its Taylor series to degree 7 in Horner form with fma,             */
/*   scaling by 2^k as two exact power-of-two multiplies 2^(k>>1) * 2^(k-(k>>1)).*/
/* Input is clamped to [-104, 89] (beyond: 0 / +inf after scaling); NaN passes.*/
/* fp64 mode uses libm exp (its decisions are not compared with the GPU).     */
/* ------------------------------------------------------------------------- */
#if !defined(REAL_IS_DOUBLE)
static float pow2i_f(int e) /* 2^e for e in [-126, 127], built from the exponent field */
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)(e + 127) << 23;
    return v.f;
}

static float pexp32(float x)
{
    if (x != x) return x;
    if (x < -104.0f) x = -104.0f;
    if (x > 89.0f) x = 89.0f;
    /* constants from the mathematics: log2(e), ln 2 split into a 16-bit head and its remainder */
    const float log2e = (float)1.4426950408889634;
    const float ln2_hi = 0.693145751953125f;             /* ln 2 truncated to 16 significant bits */
    const float ln2_lo = (float)(0.6931471805599453 - 0.693145751953125);
    float k = rintf(x * log2e);
    float r = fmaf(-k, ln2_hi, x);
    r = fmaf(-k, ln2_lo, r);
    /* Taylor coefficients 1/j!, j = 0..7, rounded to fp32 once */
    static float c[8];
    static int ready = 0;
    if (!ready) {
        double f = 1.0;
        for (int j = 0; j < 8; ++j) { if (j > 0) f *= (double)j; c[j] = (float)(1.0 / f); }
        ready = 1;
    }
    float p = c[7];
    for (int j = 6; j >= 0; --j) p = fmaf(p, r, c[j]);
    int ki = (int)k;
    int k1 = ki >> 1;            /* floor(k/2) */
    int k2 = ki - k1;
    return (p * pow2i_f(k1)) * pow2i_f(k2);
}

float oracle_pexp_f32(float x) { return pexp32(x); }
#define PEXP(x) pexp32(x)
#else
#define PEXP(x) exp(x)
#endif

/* ------------------------------------------------------------------------- */
/* Inputs                                                                     */
/* ------------------------------------------------------------------------- */
typedef struct {
    REAL R[9], t[3], fx, fy, cx, cy;
    int W, H;
} cam_t;

typedef struct {
    REAL near_z, lowpass, alpha_min, alpha_max, t_min, bg[3];
    int exclude_crossing;
    int64_t tile_budget;   /* 0: no pruning */
} opts_t;

/* cam16 = R(9, row-major world->camera), t(3), fx, fy, cx, cy */
static void load_cam(const double* c16, int W, int H, cam_t* c)
{
    for (int i = 0; i < 9; ++i) c->R[i] = (REAL)c16[i];
    for (int i = 0; i < 3; ++i) c->t[i] = (REAL)c16[9 + i];
    c->fx = (REAL)c16[12]; c->fy = (REAL)c16[13]; c->cx = (REAL)c16[14]; c->cy = (REAL)c16[15];
    c->W = W; c->H = H;
}

/* optsv = near_z, lowpass, alpha_min, alpha_max, t_min, bg r, g, b, exclude_crossing, tile_budget */
static void load_opts(const double* ov, opts_t* o)
{
    o->near_z = (REAL)ov[0]; o->lowpass = (REAL)ov[1]; o->alpha_min = (REAL)ov[2];
    o->alpha_max = (REAL)ov[3]; o->t_min = (REAL)ov[4];
    o->bg[0] = (REAL)ov[5]; o->bg[1] = (REAL)ov[6]; o->bg[2] = (REAL)ov[7];
    o->exclude_crossing = (int)ov[8];
    o->tile_budget = (int64_t)ov[9];
}

/* ------------------------------------------------------------------------- */
/* Real spherical harmonics, degree <= 3, orthonormal on the unit sphere.      */
/* Y_lm = N_lm * (homogeneous harmonic polynomial in x, y, z), with             */
/* N_lm = sqrt((2l+1)/(4 pi) * (l-|m|)!/(l+|m|)!) * (sqrt 2 if m != 0) times the */
/* Cartesian factor of the associated Legendre polynomial; sin(|m| phi) for     */
/* m < 0, cos(m phi) for m > 0; no Condon-Shortley phase.                      */
/* Coefficient k = l^2 + l + m.                                                */
/* ------------------------------------------------------------------------- */
static double sh_const_d[10];
static int sh_const_ready = 0;

static void sh_constants(void)
{
    if (sh_const_ready) return;
    const double pi = 3.14159265358979323846;
    sh_const_d[0] = 0.5 * sqrt(1.0 / pi);          /* Y00                        */
    sh_const_d[1] = sqrt(3.0 / (4.0 * pi));        /* Y1,-1 Y10 Y11  (y, z, x)     */
    sh_const_d[2] = 0.5 * sqrt(15.0 / pi);         /* Y2,-2 Y2,-1 Y21 (xy, yz, xz) */
    sh_const_d[3] = 0.25 * sqrt(5.0 / pi);         /* Y20  (2zz - xx - yy)         */
    sh_const_d[4] = 0.25 * sqrt(15.0 / pi);        /* Y22  (xx - yy)               */
    sh_const_d[5] = 0.25 * sqrt(35.0 / (2.0 * pi));/* Y3,-3 Y33                    */
    sh_const_d[6] = 0.5 * sqrt(105.0 / pi);        /* Y3,-2 (xyz)                  */
    sh_const_d[7] = 0.25 * sqrt(21.0 / (2.0 * pi));/* Y3,-1 Y31                    */
    sh_const_d[8] = 0.25 * sqrt(7.0 / pi);         /* Y30                          */
    sh_const_d[9] = 0.25 * sqrt(105.0 / pi);       /* Y32  z(xx - yy)              */
    sh_const_ready = 1;
}

/* Basis values at unit direction (x, y, z), in REAL, fixed evaluation order. */
static void sh_basis(REAL x, REAL y, REAL z, REAL Y[16])
{
    sh_constants();
    const REAL K00 = (REAL)sh_const_d[0], K1 = (REAL)sh_const_d[1], K2a = (REAL)sh_const_d[2];
    const REAL K20 = (REAL)sh_const_d[3], K22 = (REAL)sh_const_d[4], K33 = (REAL)sh_const_d[5];
    const REAL K32 = (REAL)sh_const_d[6], K31 = (REAL)sh_const_d[7], K30 = (REAL)sh_const_d[8];
    const REAL K32h = (REAL)sh_const_d[9];
    const REAL xx = x * x, yy = y * y, zz = z * z, xy = x * y, yz = y * z, xz = x * z;
    const REAL two = (REAL)2, three = (REAL)3, four = (REAL)4;
    Y[0] = K00;
    Y[1] = K1 * y;
    Y[2] = K1 * z;
    Y[3] = K1 * x;
    Y[4] = K2a * xy;
    Y[5] = K2a * yz;
    Y[6] = K20 * ((two * zz - xx) - yy);
    Y[7] = K2a * xz;
    Y[8] = K22 * (xx - yy);
    Y[9] = K33 * (y * (three * xx - yy));
    Y[10] = K32 * (xy * z);
    Y[11] = K31 * (y * ((four * zz - xx) - yy));
    Y[12] = K30 * (z * ((two * zz - three * xx) - three * yy));
    Y[13] = K31 * (x * ((four * zz - xx) - yy));
    Y[14] = K32h * (z * (xx - yy));
    Y[15] = K33 * (x * (xx - three * yy));
}

/* d Y_k / d(x, y, z) of the homogeneous polynomials (fp64). */
static void sh_basis_grad(double x, double y, double z, double dY[16][3])
{
    sh_constants();
    const double K1 = sh_const_d[1], K2a = sh_const_d[2], K20 = sh_const_d[3], K22 = sh_const_d[4];
    const double K33 = sh_const_d[5], K32 = sh_const_d[6], K31 = sh_const_d[7], K30 = sh_const_d[8];
    const double K32h = sh_const_d[9];
    memset(dY, 0, sizeof(double) * 48);
    dY[1][1] = K1;
    dY[2][2] = K1;
    dY[3][0] = K1;
    dY[4][0] = K2a * y; dY[4][1] = K2a * x;
    dY[5][1] = K2a * z; dY[5][2] = K2a * y;
    dY[6][0] = -2 * K20 * x; dY[6][1] = -2 * K20 * y; dY[6][2] = 4 * K20 * z;
    dY[7][0] = K2a * z; dY[7][2] = K2a * x;
    dY[8][0] = 2 * K22 * x; dY[8][1] = -2 * K22 * y;
    dY[9][0] = 6 * K33 * x * y; dY[9][1] = K33 * (3 * x * x - 3 * y * y);
    dY[10][0] = K32 * y * z; dY[10][1] = K32 * x * z; dY[10][2] = K32 * x * y;
    dY[11][0] = -2 * K31 * x * y; dY[11][1] = K31 * (4 * z * z - x * x - 3 * y * y); dY[11][2] = 8 * K31 * y * z;
    dY[12][0] = -6 * K30 * x * z; dY[12][1] = -6 * K30 * y * z; dY[12][2] = K30 * (6 * z * z - 3 * x * x - 3 * y * y);
    dY[13][0] = K31 * (4 * z * z - 3 * x * x - y * y); dY[13][1] = -2 * K31 * x * y; dY[13][2] = 8 * K31 * x * z;
    dY[14][0] = 2 * K32h * x * z; dY[14][1] = -2 * K32h * y * z; dY[14][2] = K32h * (x * x - y * y);
    dY[15][0] = K33 * (3 * x * x - 3 * y * y); dY[15][1] = -6 * K33 * x * y;
}

void FN(oracle_sh_basis)(const REAL* dirs, int64_t n, REAL* out)
{
    for (int64_t i = 0; i < n; ++i) sh_basis(dirs[3 * i], dirs[3 * i + 1], dirs[3 * i + 2], out + 16 * i);
}

/* ------------------------------------------------------------------------- */
/* O1..O6: projection of one Gaussian into one view.                          */
/* rec: mx, my, conicA, conicB, conicC, opacity, r, g, b, depth               */
/* rect: x0, y0, x1, y1 in tiles, half-open; visible = 0 means culled.        */
/* clampmask bit c: colour channel c clamped at 0 (degree 3 only).            */
/* ------------------------------------------------------------------------- */
static int project_one(const REAL* P, int64_t n, int64_t g, int deg, const cam_t* cam,
                       const opts_t* op, REAL* rec, int32_t* rect, uint8_t* clampmask)
{
    const REAL one = (REAL)1, two = (REAL)2, half = (REAL)0.5, three = (REAL)3;
    REAL mu[3] = {P[0 * n + g], P[1 * n + g], P[2 * n + g]};
    /* O2: view transform, near-plane cull */
    REAL t[3];
    for (int i = 0; i < 3; ++i)
        t[i] = ((cam->R[3 * i + 0] * mu[0] + cam->R[3 * i + 1] * mu[1]) + cam->R[3 * i + 2] * mu[2]) + cam->t[i];
    if (!(t[2] > op->near_z)) return 0;
    /* O1: activations */
    REAL s[3];
    for (int j = 0; j < 3; ++j) s[j] = PEXP(P[(3 + j) * n + g]);
    REAL q0 = P[6 * n + g], q1 = P[7 * n + g], q2 = P[8 * n + g], q3 = P[9 * n + g];
    REAL qn = SQRT(((q0 * q0 + q1 * q1) + q2 * q2) + q3 * q3);
    if (!(qn > 0)) return 0;
    REAL w = q0 / qn, x = q1 / qn, y = q2 / qn, z = q3 / qn;
    REAL xx = x * x, yy = y * y, zz = z * z, xy = x * y, xz = x * z, yz = y * z;
    REAL wx = w * x, wy = w * y, wz = w * z;
    REAL R[9];
    R[0] = one - two * (yy + zz); R[1] = two * (xy - wz);        R[2] = two * (xz + wy);
    R[3] = two * (xy + wz);       R[4] = one - two * (xx + zz);  R[5] = two * (yz - wx);
    R[6] = two * (xz - wy);       R[7] = two * (yz + wx);        R[8] = one - two * (xx + yy);
    REAL M[9];
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j) M[3 * i + j] = R[3 * i + j] * s[j];
    REAL S[9];  /* Sigma = M M^T */
    for (int i = 0; i < 3; ++i)
        for (int j = 0; j < 3; ++j)
            S[3 * i + j] = (M[3 * i + 0] * M[3 * j + 0] + M[3 * i + 1] * M[3 * j + 1]) + M[3 * i + 2] * M[3 * j + 2];
    /* O3: EWA projection, Sigma2D = (J W) Sigma (J W)^T + lowpass * I */
    const REAL fx = cam->fx, fy = cam->fy;
    const REAL tz2 = t[2] * t[2];
    const REAL j00 = fx / t[2], j11 = fy / t[2];
    const REAL j02 = -(fx * t[0]) / tz2, j12 = -(fy * t[1]) / tz2;
    const REAL* W = cam->R;
    REAL T0[3], T1[3];
    for (int k = 0; k < 3; ++k) {
        T0[k] = j00 * W[0 + k] + j02 * W[6 + k];
        T1[k] = j11 * W[3 + k] + j12 * W[6 + k];
    }
    REAL u[3], v[3];
    for (int k = 0; k < 3; ++k) {
        u[k] = (T0[0] * S[0 + k] + T0[1] * S[3 + k]) + T0[2] * S[6 + k];
        v[k] = (T1[0] * S[0 + k] + T1[1] * S[3 + k]) + T1[2] * S[6 + k];
    }
    REAL a = ((u[0] * T0[0] + u[1] * T0[1]) + u[2] * T0[2]) + op->lowpass;
    REAL b = (u[0] * T1[0] + u[1] * T1[1]) + u[2] * T1[2];
    REAL c = ((v[0] * T1[0] + v[1] * T1[1]) + v[2] * T1[2]) + op->lowpass;
    REAL mx = (fx * t[0]) / t[2] + cam->cx;
    REAL my = (cam->fy * t[1]) / t[2] + cam->cy;
    /* O4: conic and radius */
    REAL det = a * c - b * b;
    if (!(det > 0)) return 0;
    REAL cA = c / det, cB = (-b) / det, cC = a / det;
    REAL mid = half * (a + c);
    REAL disc = mid * mid - det;
    if (disc < 0) disc = 0;
    REAL lmax = mid + SQRT(disc);
    REAL r = CEIL(three * SQRT(lmax));
    if (!(ISFIN(mx) && ISFIN(my) && ISFIN(r) && ISFIN(cA) && ISFIN(cB) && ISFIN(cC))) return 0;
    /* O5: tile rect [x0, x1) x [y0, y1), clipped to the grid */
    const int tiles_x = (cam->W + TILE - 1) / TILE, tiles_y = (cam->H + TILE - 1) / TILE;
    const REAL inv_tile = (REAL)(1.0 / TILE);
    REAL fx0 = FLOOR((mx - r) * inv_tile), fx1 = FLOOR((mx + r) * inv_tile) + one;
    REAL fy0 = FLOOR((my - r) * inv_tile), fy1 = FLOOR((my + r) * inv_tile) + one;
    if (fx0 < 0) fx0 = 0;
    if (fy0 < 0) fy0 = 0;
    if (fx1 > (REAL)tiles_x) fx1 = (REAL)tiles_x;
    if (fy1 > (REAL)tiles_y) fy1 = (REAL)tiles_y;
    if (!(fx0 < fx1 && fy0 < fy1)) return 0;
    /* O1 (opacity): o = sigmoid(logit) */
    REAL o = one / (one + PEXP(-P[10 * n + g]));
    /* O6: colour */
    REAL col[3];
    uint8_t cm = 0;
    if (deg == 0) {
        for (int ch = 0; ch < 3; ++ch) col[ch] = P[(11 + ch) * n + g];
    } else {
        REAL cc[3];
        for (int j = 0; j < 3; ++j)  /* camera centre = -R^T t */
            cc[j] = -((W[0 + j] * cam->t[0] + W[3 + j] * cam->t[1]) + W[6 + j] * cam->t[2]);
        REAL dv[3] = {mu[0] - cc[0], mu[1] - cc[1], mu[2] - cc[2]};
        REAL nv = SQRT((dv[0] * dv[0] + dv[1] * dv[1]) + dv[2] * dv[2]);
        REAL Y[16];
        sh_basis(dv[0] / nv, dv[1] / nv, dv[2] / nv, Y);
        for (int ch = 0; ch < 3; ++ch) {
            REAL acc = P[(11 + ch) * n + g] * Y[0];
            for (int k = 1; k < 16; ++k) acc = acc + P[(11 + 3 * k + ch) * n + g] * Y[k];
            acc = acc + half;
            if (acc < 0) { acc = 0; cm |= (uint8_t)(1u << ch); }
            col[ch] = acc;
        }
    }
    if (!(ISFIN(o) && ISFIN(col[0]) && ISFIN(col[1]) && ISFIN(col[2]))) return 0;
    rec[0] = mx; rec[1] = my; rec[2] = cA; rec[3] = cB; rec[4] = cC; rec[5] = o;
    rec[6] = col[0]; rec[7] = col[1]; rec[8] = col[2]; rec[9] = t[2];
    rect[0] = (int32_t)fx0; rect[1] = (int32_t)fy0; rect[2] = (int32_t)fx1; rect[3] = (int32_t)fy1;
    *clampmask = cm;
    return 1;
}

int FN(oracle_project)(const REAL* params, int64_t n, int sh_degree, const double* cam16, int width, int height,
                       const double* optsv, REAL* rec, int32_t* rect, uint8_t* visible, uint8_t* clampmask)
{
    cam_t cam; opts_t op;
    load_cam(cam16, width, height, &cam);
    load_opts(optsv, &op);
    for (int64_t g = 0; g < n; ++g) {
        memset(rec + 10 * g, 0, sizeof(REAL) * 10);
        rect[4 * g + 0] = rect[4 * g + 1] = rect[4 * g + 2] = rect[4 * g + 3] = 0;
        clampmask[g] = 0;
        visible[g] = (uint8_t)project_one(params, n, g, sh_degree, &cam, &op, rec + 10 * g, rect + 4 * g, clampmask + g);
        if (!visible[g]) {
            memset(rec + 10 * g, 0, sizeof(REAL) * 10);
            rect[4 * g + 0] = rect[4 * g + 1] = rect[4 * g + 2] = rect[4 * g + 3] = 0;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* O7: per-pixel candidate list = every visible g whose rect holds the pixel's */
/* tile, ordered by (depth, index).  Depth > near_z > 0, so ordering the float */
/* values equals ordering their bit patterns.                                  */
/* ------------------------------------------------------------------------- */
typedef struct { REAL depth; int64_t g; } cand_t;

static int cand_cmp(const void* pa, const void* pb)
{
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->depth < b->depth) return -1;
    if (a->depth > b->depth) return 1;
    return (a->g < b->g) ? -1 : (a->g > b->g) ? 1 : 0;
}

static int in_rect(const int32_t* rc, int tx, int ty)
{
    return tx >= rc[0] && tx < rc[2] && ty >= rc[1] && ty < rc[3];
}

/* ------------------------------------------------------------------------- */
/* Hardware-aware pruning (ByteSplat, English abstract: pruning that weighs   */
/* rendering quality against the per-tile shared-memory budget).  [reading]   */
/* A tile list longer than the budget K keeps its K most opaque entries        */
/* (opacity = the projected o; equal opacities: the nearer entry, i.e. the     */
/* earlier list position, is kept) and stays in depth order.                   */
/* ------------------------------------------------------------------------- */
typedef struct { REAL o; int64_t pos; } prune_t;

static int prune_cmp(const void* pa, const void* pb)
{
    const prune_t* a = (const prune_t*)pa;
    const prune_t* b = (const prune_t*)pb;
    if (a->o > b->o) return -1;
    if (a->o < b->o) return 1;
    return (a->pos < b->pos) ? -1 : (a->pos > b->pos) ? 1 : 0;
}

static int pos_cmp(const void* pa, const void* pb)
{
    const prune_t* a = (const prune_t*)pa;
    const prune_t* b = (const prune_t*)pb;
    return (a->pos < b->pos) ? -1 : (a->pos > b->pos) ? 1 : 0;
}

/* Prunes list[0..len) in place; returns the new length (-1 on allocation failure). */
static int64_t prune_list(const REAL* rec, cand_t* list, int64_t len, int64_t budget)
{
    if (budget <= 0 || len <= budget) return len;
    prune_t* p = (prune_t*)malloc(sizeof(prune_t) * (size_t)len);
    if (!p) return -1;
    for (int64_t i = 0; i < len; ++i) { p[i].o = rec[10 * list[i].g + 5]; p[i].pos = i; }
    qsort(p, (size_t)len, sizeof(prune_t), prune_cmp);     /* most opaque first */
    qsort(p, (size_t)budget, sizeof(prune_t), pos_cmp);    /* the kept ones back in list order */
    for (int64_t i = 0; i < budget; ++i) list[i] = list[p[i].pos];   /* p[i].pos >= i: forward copy is safe */
    free(p);
    return budget;
}

/* Literal mode: scan all n Gaussians for this pixel's tile. */
static int64_t list_literal(const REAL* rec, const int32_t* rect, const uint8_t* visible, int64_t n,
                            int tx, int ty, int64_t budget, cand_t* buf)
{
    int64_t m = 0;
    for (int64_t g = 0; g < n; ++g)
        if (visible[g] && in_rect(rect + 4 * g, tx, ty)) { buf[m].depth = rec[10 * g + 9]; buf[m].g = g; ++m; }
    qsort(buf, (size_t)m, sizeof(cand_t), cand_cmp);
    return prune_list(rec, buf, m, budget);
}

/* Tile-list mode: the same list, computed once per tile (every pixel of a tile */
/* has the same candidate list under the support rule), by bucketing then qsort. */
typedef struct { int64_t* off; int64_t* len; cand_t* items; } tile_lists_t;   /* tile t: items[off[t] .. + len[t]) */

static int build_tile_lists(const REAL* rec, const int32_t* rect, const uint8_t* visible, int64_t n,
                            int tiles_x, int tiles_y, const uint8_t* tile_mask, int64_t budget, tile_lists_t* tl)
{
    int64_t nt = (int64_t)tiles_x * tiles_y;
    int64_t* cnt = (int64_t*)calloc((size_t)nt + 1, sizeof(int64_t));
    if (!cnt) return -1;
    for (int64_t g = 0; g < n; ++g) {
        if (!visible[g]) continue;
        const int32_t* rc = rect + 4 * g;
        for (int ty = rc[1]; ty < rc[3]; ++ty)
            for (int tx = rc[0]; tx < rc[2]; ++tx)
                if (!tile_mask || tile_mask[(int64_t)ty * tiles_x + tx]) cnt[(int64_t)ty * tiles_x + tx + 1]++;
    }
    for (int64_t i = 0; i < nt; ++i) cnt[i + 1] += cnt[i];
    cand_t* items = (cand_t*)malloc(sizeof(cand_t) * (size_t)(cnt[nt] > 0 ? cnt[nt] : 1));
    int64_t* fill = (int64_t*)malloc(sizeof(int64_t) * (size_t)nt);
    if (!items || !fill) { free(cnt); free(items); free(fill); return -1; }
    memcpy(fill, cnt, sizeof(int64_t) * (size_t)nt);
    for (int64_t g = 0; g < n; ++g) {
        if (!visible[g]) continue;
        const int32_t* rc = rect + 4 * g;
        for (int ty = rc[1]; ty < rc[3]; ++ty)
            for (int tx = rc[0]; tx < rc[2]; ++tx) {
                if (tile_mask && !tile_mask[(int64_t)ty * tiles_x + tx]) continue;
                int64_t k = fill[(int64_t)ty * tiles_x + tx]++;
                items[k].depth = rec[10 * g + 9];
                items[k].g = g;
            }
    }
    /* fill is reused for the (pruned) lengths */
    for (int64_t i = 0; i < nt; ++i) {
        qsort(items + cnt[i], (size_t)(cnt[i + 1] - cnt[i]), sizeof(cand_t), cand_cmp);
        fill[i] = prune_list(rec, items + cnt[i], cnt[i + 1] - cnt[i], budget);
        if (fill[i] < 0) { free(cnt); free(items); free(fill); return -1; }
    }
    tl->off = cnt;
    tl->len = fill;
    tl->items = items;
    return 0;
}

/* Sorted per-tile lists as flat arrays (for the bit-exact sort-order check). */
/* With budget > 0 the lists are the pruned ones, concatenated. */
int64_t FN(oracle_tile_lists)(const REAL* rec, const int32_t* rect, const uint8_t* visible, int64_t n,
                              int width, int height, int64_t budget, int64_t* offsets /* [tiles+1] */,
                              int64_t* ids /* [I] or NULL */)
{
    int tiles_x = (width + TILE - 1) / TILE, tiles_y = (height + TILE - 1) / TILE;
    int64_t nt = (int64_t)tiles_x * tiles_y;
    tile_lists_t tl;
    if (build_tile_lists(rec, rect, visible, n, tiles_x, tiles_y, 0, budget, &tl)) return -1;
    offsets[0] = 0;
    for (int64_t t = 0; t < nt; ++t) {
        if (ids)
            for (int64_t i = 0; i < tl.len[t]; ++i) ids[offsets[t] + i] = tl.items[tl.off[t] + i].g;
        offsets[t + 1] = offsets[t] + tl.len[t];
    }
    int64_t total = offsets[nt];
    free(tl.off);
    free(tl.len);
    free(tl.items);
    return total;
}

/* ------------------------------------------------------------------------- */
/* O8..O10: compositing, L1 loss and reverse-mode gradients, pixel by pixel.   */
/* ------------------------------------------------------------------------- */
typedef struct { int64_t g; REAL alpha, T, G, dx, dy; int clamped; } comp_t;

static uint64_t fnv(uint64_t h, uint64_t v)
{
    for (int i = 0; i < 8; ++i) { h ^= (v >> (8 * i)) & 0xffu; h *= 1099511628211ull; }
    return h;
}

/*
 * mode 0: literal per-pixel candidate scan; mode 1: per-tile lists.
 * target == NULL: forward only (no loss, no gradients).
 * grad2d: [n][9] fp64 accumulated (+=): d mean2d x, y; d conic A, B, C; d opacity; d colour r, g, b.
 * touched: [n] set to 1 for every Gaussian composited at least once.
 * counts: E_fwd (entries evaluated up to the stop, skipped ones included), E_bwd (sum of last+1),
 *         E_comp (entries composited).
 * last_idx: [H*W] list position of the last composited entry (-1 if none), or NULL.
 * t_final: [H*W] transmittance after the last composited entry, or NULL.
 * dldc_extra: [3][H][W] another loss term's dL/dC, added to the L1 one, or NULL.
 * l1_weight: weight of the L1 term in the loss and in dL/dC (1 for plain L1).
 * sig: decision signature (hash of every discrete decision), or NULL.
 * tile_mask: NULL, or [tiles] u8: only pixels of tiles with a nonzero entry are
 *   rendered (the rest of image is left untouched and is excluded from the loss,
 *   the gradients and the counts); used to check large images tile by tile.
 * grad2d_mag: NULL, or [n][9] fp64 accumulated (+=) beside grad2d: for every term
 *   added to a grad2d entry, the same term with every factor and every sum inside
 *   it taken by absolute value (dL/dalpha as T |dL/dC|.c + |dL/dC|.S / (1 - alpha),
 *   d power / d mean2d as |A dx| + |B dy|, ...).  It bounds |grad2d| and is the
 *   scale at which a sum of these terms in another order, or each term formed
 *   in fp32, may differ from grad2d: the tolerance of a GPU comparison.  It
 *   changes nothing else.
 */
int FN(oracle_render)(const REAL* rec, const int32_t* rect, const uint8_t* visible, int64_t n,
                      int width, int height, const double* optsv, int mode, const REAL* target,
                      REAL* image, double* loss, double* grad2d, uint8_t* touched, int64_t* counts,
                      int32_t* last_idx, uint64_t* sig, const uint8_t* tile_mask, const REAL* dldc_extra,
                      double l1_weight, REAL* t_final, double* grad2d_mag)
{
    opts_t op;
    load_opts(optsv, &op);
    const int tiles_x = (width + TILE - 1) / TILE, tiles_y = (height + TILE - 1) / TILE;
    const int64_t HW = (int64_t)width * height;
    tile_lists_t tl = {0, 0, 0};
    cand_t* buf = 0;
    if (mode == 1) {
        if (build_tile_lists(rec, rect, visible, n, tiles_x, tiles_y, tile_mask, op.tile_budget, &tl)) return -1;
    } else {
        buf = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
        if (!buf) return -1;
    }
    comp_t* comp = (comp_t*)malloc(sizeof(comp_t) * (size_t)(n > 0 ? n : 1));
    if (!comp) { free(buf); free(tl.off); free(tl.items); return -1; }
    /* dL/dC = w sign(C - target) / (3HW) [reading: L1 = mean absolute error over pixels and channels,
       weighted by w = l1_weight], plus dldc_extra (another loss term's dL/dC, e.g. D-SSIM) if given */
    const REAL inv3hw = (REAL)(l1_weight * (1.0 / (3.0 * (double)HW)));
    double lsum = 0.0;
    int64_t efwd = 0, ebwd = 0, ecomp = 0;
    uint64_t h = 1469598103934665603ull;
    if (sig)
        for (int64_t g = 0; g < n; ++g) {
            h = fnv(h, (uint64_t)visible[g]);
            for (int k = 0; k < 4; ++k) h = fnv(h, (uint64_t)(uint32_t)rect[4 * g + k]);
        }
    for (int py = 0; py < height; ++py) {
        for (int px = 0; px < width; ++px) {
            const int tx = px / TILE, ty = py / TILE;
            if (tile_mask && !tile_mask[(int64_t)ty * tiles_x + tx]) continue;
            const cand_t* list;
            int64_t len;
            if (mode == 1) {
                int64_t t = (int64_t)ty * tiles_x + tx;
                list = tl.items + tl.off[t];
                len = tl.len[t];
            } else {
                len = list_literal(rec, rect, visible, n, tx, ty, op.tile_budget, buf);
                if (len < 0) { free(comp); free(buf); return -1; }
                list = buf;
            }
            const REAL pxc = (REAL)px + (REAL)0.5, pyc = (REAL)py + (REAL)0.5;
            REAL T = (REAL)1, C[3] = {0, 0, 0};
            int64_t last = -1, nev = 0, ncomp = 0;
            for (int64_t k = 0; k < len; ++k) {
                ++nev;
                const REAL* r = rec + 10 * list[k].g;
                const REAL dx = pxc - r[0], dy = pyc - r[1];
                /* power = -1/2 d^T Sigma2D^-1 d with conic (A, B, C) */
                const REAL power = (REAL)(-0.5) * ((r[2] * dx) * dx + (r[4] * dy) * dy) - (r[3] * dx) * dy;
                if (power > 0) continue;
                const REAL G = PEXP(power);
                const REAL araw = r[5] * G;
                const REAL alpha = araw < op.alpha_max ? araw : op.alpha_max;
                if (alpha < op.alpha_min) continue;
                const REAL Tn = T * ((REAL)1 - alpha);
                if (op.exclude_crossing && Tn < op.t_min) break;
                const REAL wgt = alpha * T;
                for (int ch = 0; ch < 3; ++ch) C[ch] = C[ch] + r[6 + ch] * wgt;
                comp[ncomp].g = list[k].g; comp[ncomp].alpha = alpha; comp[ncomp].T = T;
                comp[ncomp].G = G; comp[ncomp].dx = dx; comp[ncomp].dy = dy;
                comp[ncomp].clamped = araw > op.alpha_max;
                ++ncomp;
                T = Tn;
                last = k;
                if (!op.exclude_crossing && T < op.t_min) break;  /* [reading] crossing entry included */
            }
            for (int ch = 0; ch < 3; ++ch) C[ch] = C[ch] + T * op.bg[ch];
            efwd += nev;
            ebwd += last + 1;
            ecomp += ncomp;
            if (last_idx) last_idx[(int64_t)py * width + px] = (int32_t)last;
            if (t_final) t_final[(int64_t)py * width + px] = T;
            for (int ch = 0; ch < 3; ++ch) image[ch * HW + (int64_t)py * width + px] = C[ch];
            if (sig) {
                h = fnv(h, (uint64_t)ncomp);
                h = fnv(h, (uint64_t)nev);
                for (int64_t i = 0; i < ncomp; ++i) { h = fnv(h, (uint64_t)comp[i].g); h = fnv(h, (uint64_t)comp[i].clamped); }
            }
            for (int64_t i = 0; i < ncomp; ++i) touched[comp[i].g] = 1;
            if (!target) continue;
            /* O9: L1 loss and its gradient */
            REAL gC[3];
            for (int ch = 0; ch < 3; ++ch) {
                const REAL diff = C[ch] - target[ch * HW + (int64_t)py * width + px];
                lsum += (double)FABS(diff);
                gC[ch] = diff > 0 ? inv3hw : (diff < 0 ? -inv3hw : (REAL)0);
                if (dldc_extra) gC[ch] = gC[ch] + dldc_extra[ch * HW + (int64_t)py * width + px];
                if (sig) h = fnv(h, (uint64_t)(diff > 0 ? 2 : (diff < 0 ? 1 : 0)));
            }
            if (!grad2d) continue;
            /* O10: back to front over the composited entries, in fp64 */
            double S[3];
            for (int ch = 0; ch < 3; ++ch) S[ch] = (double)T * (double)op.bg[ch];
            for (int64_t i = ncomp - 1; i >= 0; --i) {
                const comp_t* e = comp + i;
                const REAL* r = rec + 10 * e->g;
                double* gg = grad2d + 9 * e->g;
                const double al = e->alpha, Ti = e->T, wgt = al * Ti;
                double dotc = 0, dots = 0, dotc_m = 0, dots_m = 0;
                for (int ch = 0; ch < 3; ++ch) {
                    gg[6 + ch] += (double)gC[ch] * wgt;
                    dotc += (double)gC[ch] * (double)r[6 + ch];
                    dots += (double)gC[ch] * S[ch];
                    dotc_m += fabs((double)gC[ch] * (double)r[6 + ch]);
                    dots_m += fabs((double)gC[ch] * S[ch]);
                }
                const double dalpha = Ti * dotc - dots / (1.0 - al);
                const double dalpha_m = Ti * dotc_m + dots_m / (1.0 - al);
                for (int ch = 0; ch < 3; ++ch) S[ch] += (double)r[6 + ch] * wgt;
                double* mm = grad2d_mag ? grad2d_mag + 9 * e->g : 0;
                if (mm)
                    for (int ch = 0; ch < 3; ++ch) mm[6 + ch] += fabs((double)gC[ch]) * wgt;
                if (e->clamped) continue;  /* alpha = 0.99 constant: no gradient to o or power */
                const double dx = e->dx, dy = e->dy;
                const double dpow = dalpha * al;
                gg[5] += dalpha * (double)e->G;
                gg[2] += dpow * (-0.5 * dx * dx);
                gg[3] += dpow * (-dx * dy);
                gg[4] += dpow * (-0.5 * dy * dy);
                gg[0] += dpow * ((double)r[2] * dx + (double)r[3] * dy);
                gg[1] += dpow * ((double)r[3] * dx + (double)r[4] * dy);
                if (mm) {
                    const double dpow_m = dalpha_m * al;
                    mm[5] += dalpha_m * (double)e->G;
                    mm[2] += dpow_m * (0.5 * dx * dx);
                    mm[3] += dpow_m * fabs(dx * dy);
                    mm[4] += dpow_m * (0.5 * dy * dy);
                    mm[0] += dpow_m * (fabs((double)r[2] * dx) + fabs((double)r[3] * dy));
                    mm[1] += dpow_m * (fabs((double)r[3] * dx) + fabs((double)r[4] * dy));
                }
            }
        }
    }
    if (loss) *loss = l1_weight * (lsum / (3.0 * (double)HW));
    if (counts) { counts[0] = efwd; counts[1] = ebwd; counts[2] = ecomp; }
    if (sig) *sig = h;
    free(comp);
    free(buf);
    free(tl.off);
    free(tl.len);
    free(tl.items);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* O10 (continued): the projection's vector-Jacobian product, in fp64.        */
/* grads [P][n] += d loss / d params for every touched g.                     */
/* ------------------------------------------------------------------------- */
int FN(oracle_vjp)(const REAL* params, int64_t n, int sh_degree, const double* cam16, int width, int height,
                   const double* optsv, const double* grad2d, const uint8_t* touched, const uint8_t* clampmask,
                   double* grads)
{
    (void)width; (void)height;
    opts_t op;
    load_opts(optsv, &op);
    const double* W = cam16;  /* row-major world->camera rotation */
    const double* tc = cam16 + 9;
    const double fx = cam16[12], fy = cam16[13];
    const double lowpass = (double)op.lowpass;
    for (int64_t g = 0; g < n; ++g) {
        if (!touched[g]) continue;
        const double* G2 = grad2d + 9 * g;
        double mu[3], ls[3], q[4];
        for (int i = 0; i < 3; ++i) mu[i] = (double)params[i * n + g];
        for (int i = 0; i < 3; ++i) ls[i] = (double)params[(3 + i) * n + g];
        for (int i = 0; i < 4; ++i) q[i] = (double)params[(6 + i) * n + g];
        const double logit = (double)params[10 * n + g];
        /* forward intermediates */
        double t[3];
        for (int i = 0; i < 3; ++i) t[i] = W[3 * i] * mu[0] + W[3 * i + 1] * mu[1] + W[3 * i + 2] * mu[2] + tc[i];
        double s[3] = {exp(ls[0]), exp(ls[1]), exp(ls[2])};
        double qn = sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
        double w = q[0] / qn, x = q[1] / qn, y = q[2] / qn, z = q[3] / qn;
        double R[9] = {1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y),
                       2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x),
                       2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)};
        double M[9], S[9];
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j) M[3 * i + j] = R[3 * i + j] * s[j];
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j) S[3 * i + j] = M[3 * i] * M[3 * j] + M[3 * i + 1] * M[3 * j + 1] + M[3 * i + 2] * M[3 * j + 2];
        const double tz = t[2], tz2 = tz * tz, tz3 = tz2 * tz;
        const double j00 = fx / tz, j11 = fy / tz, j02 = -fx * t[0] / tz2, j12 = -fy * t[1] / tz2;
        double T0[3], T1[3];
        for (int k = 0; k < 3; ++k) { T0[k] = j00 * W[k] + j02 * W[6 + k]; T1[k] = j11 * W[3 + k] + j12 * W[6 + k]; }
        double ST0[3], ST1[3];  /* Sigma T0^T, Sigma T1^T */
        for (int k = 0; k < 3; ++k) {
            ST0[k] = S[3 * k] * T0[0] + S[3 * k + 1] * T0[1] + S[3 * k + 2] * T0[2];
            ST1[k] = S[3 * k] * T1[0] + S[3 * k + 1] * T1[1] + S[3 * k + 2] * T1[2];
        }
        const double a = T0[0] * ST0[0] + T0[1] * ST0[1] + T0[2] * ST0[2] + lowpass;
        const double b = T0[0] * ST1[0] + T0[1] * ST1[1] + T0[2] * ST1[2];
        const double c = T1[0] * ST1[0] + T1[1] * ST1[1] + T1[2] * ST1[2] + lowpass;
        const double det = a * c - b * b, id = 1.0 / det;
        /* conic (A, B, C) = (c, -b, a) / det */
        const double gA = G2[2], gB = G2[3], gCc = G2[4];
        const double g_id = gA * c - gB * b + gCc * a;
        const double g_det = -g_id * id * id;
        const double ga = gCc * id + g_det * c;
        const double gc = gA * id + g_det * a;
        const double gb = -gB * id + g_det * (-2.0 * b);
        /* a = T0 S T0^T + l, b = T0 S T1^T, c = T1 S T1^T + l */
        double gT0[3], gT1[3], Gs[9];
        for (int k = 0; k < 3; ++k) {
            gT0[k] = 2.0 * ga * ST0[k] + gb * ST1[k];
            gT1[k] = gb * ST0[k] + 2.0 * gc * ST1[k];
        }
        for (int k = 0; k < 3; ++k)
            for (int l = 0; l < 3; ++l)
                Gs[3 * k + l] = ga * T0[k] * T0[l] + 0.5 * gb * (T0[k] * T1[l] + T1[k] * T0[l]) + gc * T1[k] * T1[l];
        /* Sigma = M M^T, Gs symmetric: dM = 2 Gs M */
        double gM[9];
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j)
                gM[3 * i + j] = 2.0 * (Gs[3 * i] * M[j] + Gs[3 * i + 1] * M[3 + j] + Gs[3 * i + 2] * M[6 + j]);
        double gR[9], gs[3] = {0, 0, 0};
        for (int i = 0; i < 3; ++i)
            for (int j = 0; j < 3; ++j) { gR[3 * i + j] = gM[3 * i + j] * s[j]; gs[j] += gM[3 * i + j] * R[3 * i + j]; }
        /* R(w, x, y, z) */
        double gw = 2 * (-z * gR[1] + y * gR[2] + z * gR[3] - x * gR[5] - y * gR[6] + x * gR[7]);
        double gx = 2 * (y * gR[1] + z * gR[2] + y * gR[3] - 2 * x * gR[4] - w * gR[5] + z * gR[6] + w * gR[7] - 2 * x * gR[8]);
        double gy = 2 * (-2 * y * gR[0] + x * gR[1] + w * gR[2] + x * gR[3] + z * gR[5] - w * gR[6] + z * gR[7] - 2 * y * gR[8]);
        double gz = 2 * (-2 * z * gR[0] - w * gR[1] + x * gR[2] + w * gR[3] - 2 * z * gR[4] + y * gR[5] + x * gR[6] + y * gR[7]);
        double qh[4] = {w, x, y, z}, gqh[4] = {gw, gx, gy, gz};
        double dotq = qh[0] * gqh[0] + qh[1] * gqh[1] + qh[2] * gqh[2] + qh[3] * gqh[3];
        double gq[4];
        for (int i = 0; i < 4; ++i) gq[i] = (gqh[i] - qh[i] * dotq) / qn;
        /* T = J W */
        double gj00 = 0, gj02 = 0, gj11 = 0, gj12 = 0;
        for (int k = 0; k < 3; ++k) {
            gj00 += gT0[k] * W[k]; gj02 += gT0[k] * W[6 + k];
            gj11 += gT1[k] * W[3 + k]; gj12 += gT1[k] * W[6 + k];
        }
        const double gmx = G2[0], gmy = G2[1];
        double gt[3];
        gt[0] = gj02 * (-fx / tz2) + gmx * (fx / tz);
        gt[1] = gj12 * (-fy / tz2) + gmy * (fy / tz);
        gt[2] = gj00 * (-fx / tz2) + gj02 * (2.0 * fx * t[0] / tz3) + gj11 * (-fy / tz2) + gj12 * (2.0 * fy * t[1] / tz3)
              + gmx * (-fx * t[0] / tz2) + gmy * (-fy * t[1] / tz2);
        double gmu[3];
        for (int j = 0; j < 3; ++j) gmu[j] = W[j] * gt[0] + W[3 + j] * gt[1] + W[6 + j] * gt[2];
        /* colour */
        if (sh_degree == 0) {
            for (int ch = 0; ch < 3; ++ch) grads[(11 + ch) * n + g] += G2[6 + ch];
        } else {
            double cc[3];
            for (int j = 0; j < 3; ++j) cc[j] = -(W[j] * tc[0] + W[3 + j] * tc[1] + W[6 + j] * tc[2]);
            double v[3] = {mu[0] - cc[0], mu[1] - cc[1], mu[2] - cc[2]};
            double nv = sqrt(v[0] * v[0] + v[1] * v[1] + v[2] * v[2]);
            double d[3] = {v[0] / nv, v[1] / nv, v[2] / nv};
            double Yd[16];
            {   /* fp64 basis values from the same polynomials */
                sh_constants();
                const double* K = sh_const_d;
                const double X = d[0], Yv = d[1], Z = d[2];
                Yd[0] = K[0]; Yd[1] = K[1] * Yv; Yd[2] = K[1] * Z; Yd[3] = K[1] * X;
                Yd[4] = K[2] * X * Yv; Yd[5] = K[2] * Yv * Z; Yd[6] = K[3] * (2 * Z * Z - X * X - Yv * Yv);
                Yd[7] = K[2] * X * Z; Yd[8] = K[4] * (X * X - Yv * Yv);
                Yd[9] = K[5] * Yv * (3 * X * X - Yv * Yv); Yd[10] = K[6] * X * Yv * Z;
                Yd[11] = K[7] * Yv * (4 * Z * Z - X * X - Yv * Yv); Yd[12] = K[8] * Z * (2 * Z * Z - 3 * X * X - 3 * Yv * Yv);
                Yd[13] = K[7] * X * (4 * Z * Z - X * X - Yv * Yv); Yd[14] = K[9] * Z * (X * X - Yv * Yv);
                Yd[15] = K[5] * X * (X * X - 3 * Yv * Yv);
            }
            double dY[16][3];
            sh_basis_grad(d[0], d[1], d[2], dY);
            double gd[3] = {0, 0, 0};
            for (int ch = 0; ch < 3; ++ch) {
                if (clampmask[g] & (1u << ch)) continue;
                const double gcol = G2[6 + ch];
                for (int k = 0; k < 16; ++k) {
                    grads[(11 + 3 * k + ch) * n + g] += gcol * Yd[k];
                    const double kc = (double)params[(11 + 3 * k + ch) * n + g];
                    gd[0] += gcol * kc * dY[k][0];
                    gd[1] += gcol * kc * dY[k][1];
                    gd[2] += gcol * kc * dY[k][2];
                }
            }
            double dd = d[0] * gd[0] + d[1] * gd[1] + d[2] * gd[2];
            for (int j = 0; j < 3; ++j) gmu[j] += (gd[j] - d[j] * dd) / nv;
        }
        /* opacity: o = sigmoid(logit) */
        const double o = 1.0 / (1.0 + exp(-logit));
        grads[10 * n + g] += G2[5] * o * (1.0 - o);
        for (int j = 0; j < 3; ++j) grads[j * n + g] += gmu[j];
        for (int j = 0; j < 3; ++j) grads[(3 + j) * n + g] += gs[j] * s[j];
        for (int i = 0; i < 4; ++i) grads[(6 + i) * n + g] += gq[i];
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* O11: compaction ("encoder"): ascending list of touched Gaussians.          */
/* ------------------------------------------------------------------------- */
int64_t FN(oracle_compact)(const uint8_t* touched, int64_t n, uint32_t* idx)
{
    int64_t m = 0;
    for (int64_t g = 0; g < n; ++g)
        if (touched[g]) idx[m++] = (uint32_t)g;
    return m;
}

/* ------------------------------------------------------------------------- */
/* O12: Adam (Kingma & Ba) and its deferred form (GS-Scale, abstract: the     */
/* update of Gaussians with zero gradients is deferred).                      */
/* beta^j is computed in fp64 by right-to-left binary exponentiation; the bias */
/* corrections are rounded to REAL once.  One step j on one scalar:            */
/*   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g);                           */
/*   p = p - lr * ((m / bc1) / (sqrt(v / bc2) + eps))                         */
/* ------------------------------------------------------------------------- */
static double powi_binary(double b, int e)
{
    double r = 1.0;
    while (e > 0) {
        if (e & 1) r *= b;
        b *= b;
        e >>= 1;
    }
    return r;
}

static void adam_one(REAL* p, REAL* m, REAL* v, REAL g, int j, REAL lr, REAL b1, REAL b2, REAL eps)
{
    const REAL one = (REAL)1;
    const REAL bc1 = (REAL)(1.0 - powi_binary((double)b1, j));
    const REAL bc2 = (REAL)(1.0 - powi_binary((double)b2, j));
    const REAL mn = b1 * (*m) + (one - b1) * g;
    const REAL vn = b2 * (*v) + (one - b2) * (g * g);
    const REAL den = SQRT(vn / bc2) + eps;
    *p = *p - lr * ((mn / bc1) / den);
    *m = mn;
    *v = vn;
}

void FN(oracle_adam_dense_step)(REAL* p, REAL* m, REAL* v, const REAL* g, int64_t rows, int64_t n,
                                const REAL* lr_rows, int t, REAL b1, REAL b2, REAL eps)
{
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t i = 0; i < n; ++i)
            adam_one(p + r * n + i, m + r * n + i, v + r * n + i, g[r * n + i], t, lr_rows[r], b1, b2, eps);
}

/* Deferred: for each listed g, run the skipped zero-gradient steps
 * last_step+1 .. t-1, then step t with the stored gradient, set last_step = t and
 * clear the gradient.  flush: every g with last_step < t is brought to step t
 * with zero gradients (the gradient buffer is neither read nor cleared). */
void FN(oracle_adam_deferred)(REAL* p, REAL* m, REAL* v, REAL* g, int32_t* last_step, int64_t rows, int64_t n,
                              const REAL* lr_rows, const uint32_t* idx, int64_t nidx, int t,
                              REAL b1, REAL b2, REAL eps, int flush)
{
    int64_t cnt = flush ? n : nidx;
    for (int64_t k = 0; k < cnt; ++k) {
        int64_t i = flush ? k : (int64_t)idx[k];
        int s = last_step[i];
        if (s >= t) continue;
        for (int64_t r = 0; r < rows; ++r) {
            int64_t e = r * n + i;
            for (int j = s + 1; j < t; ++j) adam_one(p + e, m + e, v + e, (REAL)0, j, lr_rows[r], b1, b2, eps);
            if (flush) {
                adam_one(p + e, m + e, v + e, (REAL)0, t, lr_rows[r], b1, b2, eps);
            } else {
                adam_one(p + e, m + e, v + e, g[e], t, lr_rows[r], b1, b2, eps);
                g[e] = 0;
            }
        }
        last_step[i] = t;
    }
}
