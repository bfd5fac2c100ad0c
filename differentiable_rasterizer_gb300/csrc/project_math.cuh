// project_math.cuh -- per-Gaussian projection and its vector-Jacobian product.
//
// project_one() (= activate() once per Gaussian + project_view() per view)
// evaluates, in a fixed IEEE operation order:
//   activation   s = exp(log_scale), q^ = q / |q|, R(q^), M = R diag(s), Sigma = M M^T,
//                o = 1 / (1 + exp(-logit))
//   view         t = R_cam mu + t_cam, culled unless t_z > near_z
//   EWA          J = [[fx/tz, 0, -fx tx/tz^2], [0, fy/tz, -fy ty/tz^2]],
//                T = J R_cam, Sigma2D = T Sigma T^T + lowpass I, mean2d = (fx tx/tz + cx, fy ty/tz + cy)
//   conic        det = a c - b^2 (> 0), conic = (c, -b, a) / det
//   radius       mid = (a + c)/2, lambda_max = mid + sqrt(max(0, mid^2 - det)), r = ceil(3 sqrt(lambda_max))
//   tile rect    floor((m - r)/16) .. floor((m + r)/16) per axis, clipped; empty -> culled
//   colour       degree 0: rgb; degree 3: max(0, sum_k coef_k Y_k(unit(mu - C_cam)) + 1/2)
// and vjp_one() is its reverse-mode derivative (fp32, fma allowed).
#pragma once

#include "gs_common.cuh"

namespace gs {

template <int DEG>
struct GaussParams {
    static constexpr int kCol = DEG == 0 ? 3 : 48;
    static constexpr int kRows = 11 + kCol;                 // parameters used (P)
    static constexpr int kStride = DEG == 0 ? 16 : 64;      // floats per Gaussian in memory
    static constexpr int kVec = (kRows + 3) / 4;            // float4 loads covering P
    float mu[3], ls[3], q[4], logit;
    float col[kCol];   // degree 3: col[3j + c] = coefficient j, channel c
    // Gaussian g's block of the [n][kStride] parameter buffer, as float4 loads.
    __device__ __forceinline__ void load(const float* __restrict__ P, int64_t g)
    {
        const float4* src = reinterpret_cast<const float4*>(P + (size_t)g * kStride);
        float v[kVec * 4];
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            const float4 t = __ldg(src + i);
            v[4 * i] = t.x;
            v[4 * i + 1] = t.y;
            v[4 * i + 2] = t.z;
            v[4 * i + 3] = t.w;
        }
#pragma unroll
        for (int i = 0; i < 3; ++i) mu[i] = v[i];
#pragma unroll
        for (int i = 0; i < 3; ++i) ls[i] = v[3 + i];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = v[6 + i];
        logit = v[10];
#pragma unroll
        for (int i = 0; i < kCol; ++i) col[i] = v[11 + i];
    }
};

// The same parameters with the colour coefficients left in a shared-memory row
// (col[3 k + c]) instead of registers.
template <int DEG>
struct GaussParamsShared {
    static constexpr int kCol = GaussParams<DEG>::kCol;
    float mu[3], ls[3], q[4], logit;
    const float* col;
};

struct ProjOut {
    float mx, my, cA, cB, cC, opacity, col[3], depth;
    int x0, y0, x1, y1;
    uint32_t clamp;   // bit c: colour channel c clamped at 0
};

// Per-view forward intermediates kept for the VJP (the view-independent ones
// are the Gaussian's GaussAct).
struct ProjInter {
    float t[3], T0[3], T1[3];
    float a, b, c, det;
    float dir[3], nv;
};

// The view-independent part of the projection of one Gaussian: scale, rotation,
// 3D covariance and opacity (computed once for all views).
struct GaussAct {
    float s[3], qn, qh[4], R[9], M[9], S[9], o;
};

template <int DEG, class GP>
__device__ __forceinline__ void activate(const GP& gp, GaussAct& ac)
{
#pragma unroll
    for (int j = 0; j < 3; ++j) ac.s[j] = pexp(gp.ls[j]);
    const float q0 = gp.q[0], q1 = gp.q[1], q2 = gp.q[2], q3 = gp.q[3];
    const float qn = sqrtf(((q0 * q0 + q1 * q1) + q2 * q2) + q3 * q3);
    ac.qn = qn;
    const float w = q0 / qn, x = q1 / qn, y = q2 / qn, z = q3 / qn;
    ac.qh[0] = w; ac.qh[1] = x; ac.qh[2] = y; ac.qh[3] = z;
    const float xx = x * x, yy = y * y, zz = z * z, xy = x * y, xz = x * z, yz = y * z;
    const float wx = w * x, wy = w * y, wz = w * z;
    float* R = ac.R;
    R[0] = 1.0f - 2.0f * (yy + zz); R[1] = 2.0f * (xy - wz);        R[2] = 2.0f * (xz + wy);
    R[3] = 2.0f * (xy + wz);        R[4] = 1.0f - 2.0f * (xx + zz); R[5] = 2.0f * (yz - wx);
    R[6] = 2.0f * (xz - wy);        R[7] = 2.0f * (yz + wx);        R[8] = 1.0f - 2.0f * (xx + yy);
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) ac.M[3 * i + j] = R[3 * i + j] * ac.s[j];
    const float* M = ac.M;
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j)
            ac.S[3 * i + j] = (M[3 * i + 0] * M[3 * j + 0] + M[3 * i + 1] * M[3 * j + 1]) + M[3 * i + 2] * M[3 * j + 2];
    ac.o = 1.0f / (1.0f + pexp(-gp.logit));
}

// The per-view part, given the Gaussian's activation (same operations and
// order as evaluating everything per view).
template <int DEG, class GP>
__device__ __forceinline__ bool project_view(const GP& gp, const GaussAct& ac, const gs_camera& cam,
                                             float near_z, float lowpass, int tiles_x, int tiles_y, ProjOut& out,
                                             ProjInter* it)
{
    const float* W = cam.R;
    float t[3];
#pragma unroll
    for (int i = 0; i < 3; ++i)
        t[i] = ((W[3 * i + 0] * gp.mu[0] + W[3 * i + 1] * gp.mu[1]) + W[3 * i + 2] * gp.mu[2]) + cam.t[i];
    if (!(t[2] > near_z)) return false;
    if (!(ac.qn > 0.0f)) return false;
    const float* S = ac.S;
    const float fx = cam.fx, fy = cam.fy;
    const float tz2 = t[2] * t[2];
    const float j00 = fx / t[2], j11 = fy / t[2];
    const float j02 = -(fx * t[0]) / tz2, j12 = -(fy * t[1]) / tz2;
    float T0[3], T1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        T0[k] = j00 * W[0 + k] + j02 * W[6 + k];
        T1[k] = j11 * W[3 + k] + j12 * W[6 + k];
    }
    float u[3], v[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        u[k] = (T0[0] * S[0 + k] + T0[1] * S[3 + k]) + T0[2] * S[6 + k];
        v[k] = (T1[0] * S[0 + k] + T1[1] * S[3 + k]) + T1[2] * S[6 + k];
    }
    const float a = ((u[0] * T0[0] + u[1] * T0[1]) + u[2] * T0[2]) + lowpass;
    const float b = (u[0] * T1[0] + u[1] * T1[1]) + u[2] * T1[2];
    const float c = ((v[0] * T1[0] + v[1] * T1[1]) + v[2] * T1[2]) + lowpass;
    const float mx = (fx * t[0]) / t[2] + cam.cx;
    const float my = (fy * t[1]) / t[2] + cam.cy;
    const float det = a * c - b * b;
    if (!(det > 0.0f)) return false;
    const float cA = c / det, cB = (-b) / det, cC = a / det;
    const float mid = 0.5f * (a + c);
    float disc = mid * mid - det;
    if (disc < 0.0f) disc = 0.0f;
    const float lmax = mid + sqrtf(disc);
    const float r = ceilf(3.0f * sqrtf(lmax));
    if (!(isfinite(mx) && isfinite(my) && isfinite(r) && isfinite(cA) && isfinite(cB) && isfinite(cC))) return false;
    float fx0 = floorf((mx - r) * 0.0625f), fx1 = floorf((mx + r) * 0.0625f) + 1.0f;
    float fy0 = floorf((my - r) * 0.0625f), fy1 = floorf((my + r) * 0.0625f) + 1.0f;
    if (fx0 < 0.0f) fx0 = 0.0f;
    if (fy0 < 0.0f) fy0 = 0.0f;
    if (fx1 > (float)tiles_x) fx1 = (float)tiles_x;
    if (fy1 > (float)tiles_y) fy1 = (float)tiles_y;
    if (!(fx0 < fx1 && fy0 < fy1)) return false;
    const float o = ac.o;
    float col[3];
    uint32_t cm = 0;
    float dir[3] = {0.0f, 0.0f, 0.0f}, nv = 0.0f;
    if (DEG == 0) {
        col[0] = gp.col[0]; col[1] = gp.col[1]; col[2] = gp.col[2];
    } else {
        float cc[3];
#pragma unroll
        for (int j = 0; j < 3; ++j) cc[j] = -((W[0 + j] * cam.t[0] + W[3 + j] * cam.t[1]) + W[6 + j] * cam.t[2]);
        const float dv0 = gp.mu[0] - cc[0], dv1 = gp.mu[1] - cc[1], dv2 = gp.mu[2] - cc[2];
        nv = sqrtf((dv0 * dv0 + dv1 * dv1) + dv2 * dv2);
        dir[0] = dv0 / nv; dir[1] = dv1 / nv; dir[2] = dv2 / nv;
        float Y[16];
        sh_basis(dir[0], dir[1], dir[2], Y);
#pragma unroll
        for (int ch = 0; ch < 3; ++ch) {
            float acc = gp.col[ch] * Y[0];
#pragma unroll
            for (int k = 1; k < 16; ++k) acc = acc + gp.col[(3 * k + ch) % GaussParams<DEG>::kCol] * Y[k];
            acc = acc + 0.5f;
            if (acc < 0.0f) { acc = 0.0f; cm |= 1u << ch; }
            col[ch] = acc;
        }
    }
    if (!(isfinite(o) && isfinite(col[0]) && isfinite(col[1]) && isfinite(col[2]))) return false;
    out.mx = mx; out.my = my; out.cA = cA; out.cB = cB; out.cC = cC; out.opacity = o;
    out.col[0] = col[0]; out.col[1] = col[1]; out.col[2] = col[2];
    out.depth = t[2];
    out.x0 = (int)fx0; out.y0 = (int)fy0; out.x1 = (int)fx1; out.y1 = (int)fy1;
    out.clamp = cm;
    if (it) {
#pragma unroll
        for (int i = 0; i < 3; ++i) { it->t[i] = t[i]; it->dir[i] = dir[i]; it->T0[i] = T0[i]; it->T1[i] = T1[i]; }
        it->a = a; it->b = b; it->c = c; it->det = det; it->nv = nv;
    }
    return true;
}

template <int DEG>
__device__ __forceinline__ bool project_one(const GaussParams<DEG>& gp, const gs_camera& cam, float near_z,
                                            float lowpass, int tiles_x, int tiles_y, ProjOut& out, ProjInter* it)
{
    GaussAct ac;
    activate<DEG>(gp, ac);
    return project_view<DEG>(gp, ac, cam, near_z, lowpass, tiles_x, tiles_y, out, it);
}

// d loss / d params of one (Gaussian, view) given d loss / d (mean2d, conic, opacity, colour).
// g2: mx, my, A, B, C, o, r, g, b.  Accumulated (+=): grad[0..10] the geometry rows,
// gcol[0..kCol) the colour rows (row 11 + i), as in the parameter buffer; the
// derivative of each SH basis polynomial is formed where it is used.
template <int DEG, class GP>
__device__ __forceinline__ void vjp_one(const GP& gp, const gs_camera& cam, const GaussAct& ac, const ProjInter& it,
                                        uint32_t clamp, const float g2[9], float* grad, float* gcol_out)
{
    const float* W = cam.R;
    const float fx = cam.fx, fy = cam.fy;
    const float a = it.a, b = it.b, c = it.c;
    const float id = 1.0f / it.det;
    // conic (A, B, C) = (c, -b, a) / det
    const float gA = g2[2], gB = g2[3], gC = g2[4];
    const float g_id = __fmaf_rn(gA, c, __fmaf_rn(-gB, b, gC * a));
    const float g_det = -g_id * id * id;
    const float ga = __fmaf_rn(gC, id, g_det * c);
    const float gc = __fmaf_rn(gA, id, g_det * a);
    const float gb = __fmaf_rn(-gB, id, g_det * (-2.0f * b));
    // a = T0 S T0^T + l, b = T0 S T1^T, c = T1 S T1^T + l
    float ST0[3], ST1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        ST0[k] = __fmaf_rn(ac.S[3 * k], it.T0[0], __fmaf_rn(ac.S[3 * k + 1], it.T0[1], ac.S[3 * k + 2] * it.T0[2]));
        ST1[k] = __fmaf_rn(ac.S[3 * k], it.T1[0], __fmaf_rn(ac.S[3 * k + 1], it.T1[1], ac.S[3 * k + 2] * it.T1[2]));
    }
    float gT0[3], gT1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        gT0[k] = __fmaf_rn(2.0f * ga, ST0[k], gb * ST1[k]);
        gT1[k] = __fmaf_rn(gb, ST0[k], 2.0f * gc * ST1[k]);
    }
    float Gs[9];
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int l = 0; l < 3; ++l)
            Gs[3 * k + l] = __fmaf_rn(ga * it.T0[k], it.T0[l],
                                      __fmaf_rn(0.5f * gb, __fmaf_rn(it.T0[k], it.T1[l], it.T1[k] * it.T0[l]),
                                                gc * it.T1[k] * it.T1[l]));
    // Sigma = M M^T: dM = 2 Gs M
    float gR[9], gs[3] = {0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const float gM = 2.0f * __fmaf_rn(Gs[3 * i], ac.M[j], __fmaf_rn(Gs[3 * i + 1], ac.M[3 + j], Gs[3 * i + 2] * ac.M[6 + j]));
            gR[3 * i + j] = gM * ac.s[j];
            gs[j] = __fmaf_rn(gM, ac.R[3 * i + j], gs[j]);
        }
    const float w = ac.qh[0], x = ac.qh[1], y = ac.qh[2], z = ac.qh[3];
    const float gw = 2.0f * (-z * gR[1] + y * gR[2] + z * gR[3] - x * gR[5] - y * gR[6] + x * gR[7]);
    const float gx = 2.0f * (y * gR[1] + z * gR[2] + y * gR[3] - 2.0f * x * gR[4] - w * gR[5] + z * gR[6] + w * gR[7] - 2.0f * x * gR[8]);
    const float gy = 2.0f * (-2.0f * y * gR[0] + x * gR[1] + w * gR[2] + x * gR[3] + z * gR[5] - w * gR[6] + z * gR[7] - 2.0f * y * gR[8]);
    const float gz = 2.0f * (-2.0f * z * gR[0] - w * gR[1] + x * gR[2] + w * gR[3] - 2.0f * z * gR[4] + y * gR[5] + x * gR[6] + y * gR[7]);
    const float dotq = w * gw + x * gx + y * gy + z * gz;
    const float iqn = 1.0f / ac.qn;
    // T = J W
    float gj00 = 0.0f, gj02 = 0.0f, gj11 = 0.0f, gj12 = 0.0f;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        gj00 = __fmaf_rn(gT0[k], W[k], gj00);
        gj02 = __fmaf_rn(gT0[k], W[6 + k], gj02);
        gj11 = __fmaf_rn(gT1[k], W[3 + k], gj11);
        gj12 = __fmaf_rn(gT1[k], W[6 + k], gj12);
    }
    const float tx = it.t[0], ty = it.t[1], tz = it.t[2];
    const float itz = 1.0f / tz, itz2 = itz * itz, itz3 = itz2 * itz;
    const float gmx = g2[0], gmy = g2[1];
    float gt[3];
    gt[0] = gj02 * (-fx * itz2) + gmx * (fx * itz);
    gt[1] = gj12 * (-fy * itz2) + gmy * (fy * itz);
    gt[2] = gj00 * (-fx * itz2) + gj02 * (2.0f * fx * tx * itz3) + gj11 * (-fy * itz2) + gj12 * (2.0f * fy * ty * itz3)
          + gmx * (-fx * tx * itz2) + gmy * (-fy * ty * itz2);
    float gmu[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) gmu[j] = __fmaf_rn(W[j], gt[0], __fmaf_rn(W[3 + j], gt[1], W[6 + j] * gt[2]));
    if (DEG == 0) {
        gcol_out[0] += g2[6];
        gcol_out[1] += g2[7];
        gcol_out[2] += g2[8];
    } else {
        const float X = it.dir[0], Yv = it.dir[1], Z = it.dir[2];
        float Y[16];
        sh_basis(X, Yv, Z, Y);
        // gradient of each basis polynomial w.r.t. (x, y, z)
        const float XX = X * X, YY = Yv * Yv, ZZ = Z * Z;
        float gd0 = 0.0f, gd1 = 0.0f, gd2 = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            // gradient of basis polynomial k w.r.t. (x, y, z)
            float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f;
            switch (k) {
                case 1: d1 = SH::K1; break;
                case 2: d2 = SH::K1; break;
                case 3: d0 = SH::K1; break;
                case 4: d0 = SH::K2 * Yv; d1 = SH::K2 * X; break;
                case 5: d1 = SH::K2 * Z; d2 = SH::K2 * Yv; break;
                case 6: d0 = -2.0f * SH::K3 * X; d1 = -2.0f * SH::K3 * Yv; d2 = 4.0f * SH::K3 * Z; break;
                case 7: d0 = SH::K2 * Z; d2 = SH::K2 * X; break;
                case 8: d0 = 2.0f * SH::K4 * X; d1 = -2.0f * SH::K4 * Yv; break;
                case 9: d0 = 6.0f * SH::K5 * X * Yv; d1 = SH::K5 * (3.0f * XX - 3.0f * YY); break;
                case 10: d0 = SH::K6 * Yv * Z; d1 = SH::K6 * X * Z; d2 = SH::K6 * X * Yv; break;
                case 11: d0 = -2.0f * SH::K7 * X * Yv; d1 = SH::K7 * (4.0f * ZZ - XX - 3.0f * YY); d2 = 8.0f * SH::K7 * Yv * Z; break;
                case 12: d0 = -6.0f * SH::K8 * X * Z; d1 = -6.0f * SH::K8 * Yv * Z; d2 = SH::K8 * (6.0f * ZZ - 3.0f * XX - 3.0f * YY); break;
                case 13: d0 = SH::K7 * (4.0f * ZZ - 3.0f * XX - YY); d1 = -2.0f * SH::K7 * X * Yv; d2 = 8.0f * SH::K7 * X * Z; break;
                case 14: d0 = 2.0f * SH::K9 * X * Z; d1 = -2.0f * SH::K9 * Yv * Z; d2 = SH::K9 * (XX - YY); break;
                case 15: d0 = SH::K5 * (3.0f * XX - 3.0f * YY); d1 = -6.0f * SH::K5 * X * Yv; break;
                default: break;
            }
#pragma unroll
            for (int ch = 0; ch < 3; ++ch) {
                if (clamp & (1u << ch)) continue;
                const float gcol = g2[6 + ch];
                const int row = 3 * k + ch;
                gcol_out[row] = __fmaf_rn(gcol, Y[k], gcol_out[row]);
                const float kc = gcol * gp.col[row % GP::kCol];
                gd0 = __fmaf_rn(kc, d0, gd0);
                gd1 = __fmaf_rn(kc, d1, gd1);
                gd2 = __fmaf_rn(kc, d2, gd2);
            }
        }
        const float dd = X * gd0 + Yv * gd1 + Z * gd2;
        const float inv = 1.0f / it.nv;
        gmu[0] += (gd0 - X * dd) * inv;
        gmu[1] += (gd1 - Yv * dd) * inv;
        gmu[2] += (gd2 - Z * dd) * inv;
    }
    grad[10] += g2[5] * ac.o * (1.0f - ac.o);
    grad[0] += gmu[0];
    grad[1] += gmu[1];
    grad[2] += gmu[2];
    grad[3] += gs[0] * ac.s[0];
    grad[4] += gs[1] * ac.s[1];
    grad[5] += gs[2] * ac.s[2];
    grad[6] += (gw - w * dotq) * iqn;
    grad[7] += (gx - x * dotq) * iqn;
    grad[8] += (gy - y * dotq) * iqn;
    grad[9] += (gz - z * dotq) * iqn;
}

// ---------------------------------------------------------------------------
// The VJP of one (Gaussian, view) split in two independent halves, for a
// decoder that runs them in different warps: the geometry (mean through the
// projection, scale, rotation, opacity) and the SH-3 colour (coefficients, and
// the mean through the viewing direction).  Both recompute their forward
// intermediates with the operations of project_view, so the colour's clamp
// decisions are the forward's; a composited (Gaussian, view) is always visible,
// so no culling test is repeated.
// ---------------------------------------------------------------------------

// Geometry intermediates of project_view (t, T0, T1, the 2D covariance).
template <class GP>
__device__ __forceinline__ void project_geom(const GP& gp, const GaussAct& ac, const gs_camera& cam, float lowpass,
                                             ProjInter& it)
{
    const float* W = cam.R;
    float t[3];
#pragma unroll
    for (int i = 0; i < 3; ++i)
        t[i] = ((W[3 * i + 0] * gp.mu[0] + W[3 * i + 1] * gp.mu[1]) + W[3 * i + 2] * gp.mu[2]) + cam.t[i];
    const float* S = ac.S;
    const float fx = cam.fx, fy = cam.fy;
    const float tz2 = t[2] * t[2];
    const float j00 = fx / t[2], j11 = fy / t[2];
    const float j02 = -(fx * t[0]) / tz2, j12 = -(fy * t[1]) / tz2;
    float T0[3], T1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        T0[k] = j00 * W[0 + k] + j02 * W[6 + k];
        T1[k] = j11 * W[3 + k] + j12 * W[6 + k];
    }
    float u[3], v[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        u[k] = (T0[0] * S[0 + k] + T0[1] * S[3 + k]) + T0[2] * S[6 + k];
        v[k] = (T1[0] * S[0 + k] + T1[1] * S[3 + k]) + T1[2] * S[6 + k];
    }
    it.a = ((u[0] * T0[0] + u[1] * T0[1]) + u[2] * T0[2]) + lowpass;
    it.b = (u[0] * T1[0] + u[1] * T1[1]) + u[2] * T1[2];
    it.c = ((v[0] * T1[0] + v[1] * T1[1]) + v[2] * T1[2]) + lowpass;
    it.det = it.a * it.c - it.b * it.b;
#pragma unroll
    for (int i = 0; i < 3; ++i) { it.t[i] = t[i]; it.T0[i] = T0[i]; it.T1[i] = T1[i]; }
}

// Geometry half of vjp_one: grad[0..10] += d loss / d (mean through the
// projection, log-scale, quaternion, opacity logit).
template <class GP>
__device__ __forceinline__ void vjp_geom(const GP& gp, const gs_camera& cam, const GaussAct& ac, const ProjInter& it,
                                         const float g2[6], float* grad)
{
    const float* W = cam.R;
    const float fx = cam.fx, fy = cam.fy;
    const float a = it.a, b = it.b, c = it.c;
    const float id = 1.0f / it.det;
    const float gA = g2[2], gB = g2[3], gC = g2[4];
    const float g_id = __fmaf_rn(gA, c, __fmaf_rn(-gB, b, gC * a));
    const float g_det = -g_id * id * id;
    const float ga = __fmaf_rn(gC, id, g_det * c);
    const float gc = __fmaf_rn(gA, id, g_det * a);
    const float gb = __fmaf_rn(-gB, id, g_det * (-2.0f * b));
    float ST0[3], ST1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        ST0[k] = __fmaf_rn(ac.S[3 * k], it.T0[0], __fmaf_rn(ac.S[3 * k + 1], it.T0[1], ac.S[3 * k + 2] * it.T0[2]));
        ST1[k] = __fmaf_rn(ac.S[3 * k], it.T1[0], __fmaf_rn(ac.S[3 * k + 1], it.T1[1], ac.S[3 * k + 2] * it.T1[2]));
    }
    float gT0[3], gT1[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        gT0[k] = __fmaf_rn(2.0f * ga, ST0[k], gb * ST1[k]);
        gT1[k] = __fmaf_rn(gb, ST0[k], 2.0f * gc * ST1[k]);
    }
    float Gs[9];
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
        for (int l = 0; l < 3; ++l)
            Gs[3 * k + l] = __fmaf_rn(ga * it.T0[k], it.T0[l],
                                      __fmaf_rn(0.5f * gb, __fmaf_rn(it.T0[k], it.T1[l], it.T1[k] * it.T0[l]),
                                                gc * it.T1[k] * it.T1[l]));
    float gR[9], gs[3] = {0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const float gM = 2.0f * __fmaf_rn(Gs[3 * i], ac.M[j], __fmaf_rn(Gs[3 * i + 1], ac.M[3 + j], Gs[3 * i + 2] * ac.M[6 + j]));
            gR[3 * i + j] = gM * ac.s[j];
            gs[j] = __fmaf_rn(gM, ac.R[3 * i + j], gs[j]);
        }
    const float w = ac.qh[0], x = ac.qh[1], y = ac.qh[2], z = ac.qh[3];
    const float gw = 2.0f * (-z * gR[1] + y * gR[2] + z * gR[3] - x * gR[5] - y * gR[6] + x * gR[7]);
    const float gx = 2.0f * (y * gR[1] + z * gR[2] + y * gR[3] - 2.0f * x * gR[4] - w * gR[5] + z * gR[6] + w * gR[7] - 2.0f * x * gR[8]);
    const float gy = 2.0f * (-2.0f * y * gR[0] + x * gR[1] + w * gR[2] + x * gR[3] + z * gR[5] - w * gR[6] + z * gR[7] - 2.0f * y * gR[8]);
    const float gz = 2.0f * (-2.0f * z * gR[0] - w * gR[1] + x * gR[2] + w * gR[3] - 2.0f * z * gR[4] + y * gR[5] + x * gR[6] + y * gR[7]);
    const float dotq = w * gw + x * gx + y * gy + z * gz;
    const float iqn = 1.0f / ac.qn;
    float gj00 = 0.0f, gj02 = 0.0f, gj11 = 0.0f, gj12 = 0.0f;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        gj00 = __fmaf_rn(gT0[k], W[k], gj00);
        gj02 = __fmaf_rn(gT0[k], W[6 + k], gj02);
        gj11 = __fmaf_rn(gT1[k], W[3 + k], gj11);
        gj12 = __fmaf_rn(gT1[k], W[6 + k], gj12);
    }
    const float tx = it.t[0], ty = it.t[1], tz = it.t[2];
    const float itz = 1.0f / tz, itz2 = itz * itz, itz3 = itz2 * itz;
    const float gmx = g2[0], gmy = g2[1];
    float gt[3];
    gt[0] = gj02 * (-fx * itz2) + gmx * (fx * itz);
    gt[1] = gj12 * (-fy * itz2) + gmy * (fy * itz);
    gt[2] = gj00 * (-fx * itz2) + gj02 * (2.0f * fx * tx * itz3) + gj11 * (-fy * itz2) + gj12 * (2.0f * fy * ty * itz3)
          + gmx * (-fx * tx * itz2) + gmy * (-fy * ty * itz2);
#pragma unroll
    for (int j = 0; j < 3; ++j) grad[j] += __fmaf_rn(W[j], gt[0], __fmaf_rn(W[3 + j], gt[1], W[6 + j] * gt[2]));
    grad[10] += g2[5] * ac.o * (1.0f - ac.o);
    grad[3] += gs[0] * ac.s[0];
    grad[4] += gs[1] * ac.s[1];
    grad[5] += gs[2] * ac.s[2];
    grad[6] += (gw - w * dotq) * iqn;
    grad[7] += (gx - x * dotq) * iqn;
    grad[8] += (gy - y * dotq) * iqn;
    grad[9] += (gz - z * dotq) * iqn;
}

// Colour half of vjp_one for SH degree 3: the view's colour forward (the
// operations of project_view, so the same clamp decisions), then gcol[48] +=
// d loss / d coefficients and gmu[3] += d loss / d mean through the viewing
// direction.  gc: d loss / d (r, g, b) of the view.
__device__ __forceinline__ void vjp_colour3(const float mu[3], const float col[48], const gs_camera& cam,
                                            const float gc[3], float gcol[48], float gmu[3])
{
    const float* W = cam.R;
    float cc[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) cc[j] = -((W[0 + j] * cam.t[0] + W[3 + j] * cam.t[1]) + W[6 + j] * cam.t[2]);
    const float dv0 = mu[0] - cc[0], dv1 = mu[1] - cc[1], dv2 = mu[2] - cc[2];
    const float nv = sqrtf((dv0 * dv0 + dv1 * dv1) + dv2 * dv2);
    const float X = dv0 / nv, Yv = dv1 / nv, Z = dv2 / nv;
    float Y[16];
    sh_basis(X, Yv, Z, Y);
    uint32_t clamp = 0;
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) {
        float acc = col[ch] * Y[0];
#pragma unroll
        for (int k = 1; k < 16; ++k) acc = acc + col[3 * k + ch] * Y[k];
        acc = acc + 0.5f;
        if (acc < 0.0f) clamp |= 1u << ch;
    }
    const float XX = X * X, YY = Yv * Yv, ZZ = Z * Z;
    float gd0 = 0.0f, gd1 = 0.0f, gd2 = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f;
        switch (k) {
            case 1: d1 = SH::K1; break;
            case 2: d2 = SH::K1; break;
            case 3: d0 = SH::K1; break;
            case 4: d0 = SH::K2 * Yv; d1 = SH::K2 * X; break;
            case 5: d1 = SH::K2 * Z; d2 = SH::K2 * Yv; break;
            case 6: d0 = -2.0f * SH::K3 * X; d1 = -2.0f * SH::K3 * Yv; d2 = 4.0f * SH::K3 * Z; break;
            case 7: d0 = SH::K2 * Z; d2 = SH::K2 * X; break;
            case 8: d0 = 2.0f * SH::K4 * X; d1 = -2.0f * SH::K4 * Yv; break;
            case 9: d0 = 6.0f * SH::K5 * X * Yv; d1 = SH::K5 * (3.0f * XX - 3.0f * YY); break;
            case 10: d0 = SH::K6 * Yv * Z; d1 = SH::K6 * X * Z; d2 = SH::K6 * X * Yv; break;
            case 11: d0 = -2.0f * SH::K7 * X * Yv; d1 = SH::K7 * (4.0f * ZZ - XX - 3.0f * YY); d2 = 8.0f * SH::K7 * Yv * Z; break;
            case 12: d0 = -6.0f * SH::K8 * X * Z; d1 = -6.0f * SH::K8 * Yv * Z; d2 = SH::K8 * (6.0f * ZZ - 3.0f * XX - 3.0f * YY); break;
            case 13: d0 = SH::K7 * (4.0f * ZZ - 3.0f * XX - YY); d1 = -2.0f * SH::K7 * X * Yv; d2 = 8.0f * SH::K7 * X * Z; break;
            case 14: d0 = 2.0f * SH::K9 * X * Z; d1 = -2.0f * SH::K9 * Yv * Z; d2 = SH::K9 * (XX - YY); break;
            case 15: d0 = SH::K5 * (3.0f * XX - 3.0f * YY); d1 = -6.0f * SH::K5 * X * Yv; break;
            default: break;
        }
#pragma unroll
        for (int ch = 0; ch < 3; ++ch) {
            if (clamp & (1u << ch)) continue;
            const int row = 3 * k + ch;
            gcol[row] = __fmaf_rn(gc[ch], Y[k], gcol[row]);
            const float kc = gc[ch] * col[row];
            gd0 = __fmaf_rn(kc, d0, gd0);
            gd1 = __fmaf_rn(kc, d1, gd1);
            gd2 = __fmaf_rn(kc, d2, gd2);
        }
    }
    const float dd = X * gd0 + Yv * gd1 + Z * gd2;
    const float inv = 1.0f / nv;
    gmu[0] += (gd0 - X * dd) * inv;
    gmu[1] += (gd1 - Yv * dd) * inv;
    gmu[2] += (gd2 - Z * dd) * inv;
}

// Colour half for SH degree 3 and ONE view, streaming the 48 coefficients from
// the Gaussian's parameter block (global or shared memory; src may be dst: every
// read comes before the first write) instead of holding them: coefficient i = 3 k + c
// (float 11 + i of the block) adds to channel c's forward colour sum (in the
// order of project_view, so the clamp decisions are the forward's) and to its
// three sums col * dY_k / d(direction); once the clamps are known, the mean's
// direction term is gmu += (gd - dir (dir . gd)) / |mu - C| with
// gd = sum over unclamped c of gc[c] (channel c's sums).  With one view a
// coefficient's gradient is gc[c] Y_k (0 if c clamped): written straight to
// floats 12 .. 59 of dst (float4 3 .. 14; 59 is padding); the gradient of
// coefficient 0 (float 11) is returned for the caller's float4 2.
__device__ __forceinline__ float vjp_colour3_stream(const float4* src, const float mu[3], const gs_camera& cam,
                                                    const float gc[3], float4* dst, float gmu[3])
{
    const float* W = cam.R;
    float cc[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) cc[j] = -((W[0 + j] * cam.t[0] + W[3 + j] * cam.t[1]) + W[6 + j] * cam.t[2]);
    const float dv0 = mu[0] - cc[0], dv1 = mu[1] - cc[1], dv2 = mu[2] - cc[2];
    const float nv = sqrtf((dv0 * dv0 + dv1 * dv1) + dv2 * dv2);
    const float X = dv0 / nv, Yv = dv1 / nv, Z = dv2 / nv;
    float Y[16];
    sh_basis(X, Yv, Z, Y);
    const float XX = X * X, YY = Yv * Yv, ZZ = Z * Z;
    float fwd[3] = {0.0f, 0.0f, 0.0f}, sd0[3] = {0.0f, 0.0f, 0.0f}, sd1[3] = {0.0f, 0.0f, 0.0f}, sd2[3] = {0.0f, 0.0f, 0.0f};
    // coefficient i: forward sum and direction-derivative sums of its channel
    auto take = [&](int i, float col) {
        const int k = i / 3, ch = i - 3 * (i / 3);
        fwd[ch] = k == 0 ? col * Y[0] : fwd[ch] + col * Y[k];
        float d0 = 0.0f, d1 = 0.0f, d2 = 0.0f;
        switch (k) {
            case 1: d1 = SH::K1; break;
            case 2: d2 = SH::K1; break;
            case 3: d0 = SH::K1; break;
            case 4: d0 = SH::K2 * Yv; d1 = SH::K2 * X; break;
            case 5: d1 = SH::K2 * Z; d2 = SH::K2 * Yv; break;
            case 6: d0 = -2.0f * SH::K3 * X; d1 = -2.0f * SH::K3 * Yv; d2 = 4.0f * SH::K3 * Z; break;
            case 7: d0 = SH::K2 * Z; d2 = SH::K2 * X; break;
            case 8: d0 = 2.0f * SH::K4 * X; d1 = -2.0f * SH::K4 * Yv; break;
            case 9: d0 = 6.0f * SH::K5 * X * Yv; d1 = SH::K5 * (3.0f * XX - 3.0f * YY); break;
            case 10: d0 = SH::K6 * Yv * Z; d1 = SH::K6 * X * Z; d2 = SH::K6 * X * Yv; break;
            case 11: d0 = -2.0f * SH::K7 * X * Yv; d1 = SH::K7 * (4.0f * ZZ - XX - 3.0f * YY); d2 = 8.0f * SH::K7 * Yv * Z; break;
            case 12: d0 = -6.0f * SH::K8 * X * Z; d1 = -6.0f * SH::K8 * Yv * Z; d2 = SH::K8 * (6.0f * ZZ - 3.0f * XX - 3.0f * YY); break;
            case 13: d0 = SH::K7 * (4.0f * ZZ - 3.0f * XX - YY); d1 = -2.0f * SH::K7 * X * Yv; d2 = 8.0f * SH::K7 * X * Z; break;
            case 14: d0 = 2.0f * SH::K9 * X * Z; d1 = -2.0f * SH::K9 * Yv * Z; d2 = SH::K9 * (XX - YY); break;
            case 15: d0 = SH::K5 * (3.0f * XX - 3.0f * YY); d1 = -6.0f * SH::K5 * X * Yv; break;
            default: break;
        }
        sd0[ch] = __fmaf_rn(col, d0, sd0[ch]);
        sd1[ch] = __fmaf_rn(col, d1, sd1[ch]);
        sd2[ch] = __fmaf_rn(col, d2, sd2[ch]);
    };
    take(0, src[2].w);
#pragma unroll
    for (int m = 0; m < 12; ++m) {   // floats 12 .. 59 = coefficients 1 .. 47 (+ padding)
        const float4 p = src[3 + m];
        take(1 + 4 * m, p.x);
        take(2 + 4 * m, p.y);
        take(3 + 4 * m, p.z);
        if (m < 11) take(4 + 4 * m, p.w);
    }
    // (a clamped channel's sums are never used: a visible Gaussian may hold an
    // infinite coefficient in a channel that the clamp zeroes)
    float gm[3], gd0 = 0.0f, gd1 = 0.0f, gd2 = 0.0f;
#pragma unroll
    for (int ch = 0; ch < 3; ++ch) {
        const bool clamped = fwd[ch] + 0.5f < 0.0f;
        gm[ch] = clamped ? 0.0f : gc[ch];
        if (!clamped) {
            gd0 = __fmaf_rn(gc[ch], sd0[ch], gd0);
            gd1 = __fmaf_rn(gc[ch], sd1[ch], gd1);
            gd2 = __fmaf_rn(gc[ch], sd2[ch], gd2);
        }
    }
    auto gcol = [&](int i) -> float { return gm[i - 3 * (i / 3)] * Y[i / 3]; };
#pragma unroll
    for (int m = 0; m < 12; ++m)
        dst[3 + m] = make_float4(gcol(1 + 4 * m), gcol(2 + 4 * m), gcol(3 + 4 * m), m < 11 ? gcol(4 + 4 * m) : 0.0f);
    const float dd = X * gd0 + Yv * gd1 + Z * gd2;
    const float inv = 1.0f / nv;
    gmu[0] += (gd0 - X * dd) * inv;
    gmu[1] += (gd1 - Yv * dd) * inv;
    gmu[2] += (gd2 - Z * dd) * inv;
    return gcol(0);
}

}  // namespace gs
