// Logit transform chains ("[WS2] Framework for ablation experiment", LogProb
// knobs table, row 7: temperature, soft-cap, logit scale), applied in fp32 to
// each real logit before any softmax arithmetic.  Shared by the streaming row
// kernel and the fused LM-head epilogue, which pick the same form for a chain
// (scales only, at most one soft-cap per side, or the general per-op loop), so
// a logit gets the same transformed bits on either path.
#pragma once

#include <cmath>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"

namespace lpd {

// A side's chain as the consumers read it: one {kind, p, 1/p} entry per op in
// a shared-memory table (dynamic indexing stays cheap there), walked by a real
// loop so each op body is emitted once per call site.
struct XformView {
    const float4 *ops;  // x: kind (as int bits), y: p, z: 1/p
    int n;
};

__device__ __forceinline__ void xform_table(const Xform &c, float4 *ops) {
    for (int k = 0; k < c.n_ops; ++k)
        ops[k] = make_float4(__int_as_float(c.kind[k]), c.param[k], __frcp_rn(c.param[k]), 0.f);
}

// ---- soft-cap p * tanh(x / p) ---------------------------------------------
// Near-identical logits on the two sides must get near-identical transformed
// values, so tanh has to stay at the level of fp32 rounding (the hardware
// tanh.approx, about 2^-11 relative, does not).  Own tanh, from its series
// and its exponential form, with y = x / p and z = y^2:
//   z < 0.36:   p tanh(y) = x (1 + z P(z)), P of degree 4 fitted to
//               (tanh(y)/y - 1)/z (csrc/tanh_coeffs.py: tanh within 0.63 ulp
//               in float32 Horner evaluation; degree 5 gained nothing, the
//               final rounding dominates); p y is written as x itself;
//   otherwise:  p tanh(y) = p sign(y) (1 - 2 / (1 + 2^(2|y| log2 e))), with
//               ex2.approx and rcp.approx (a few ulp where |y| >= 0.6,
//               exactly +-p once the power overflows; NaN stays NaN).
// Every path takes the same per-element decision on the same rounded z, and
// the packed path rounds each half like the scalar one, so a column's value
// does not depend on which load path or lane handled it.
constexpr float kTanhZMax = 0.36f;
constexpr int kTanhDegree = 4;
__host__ __device__ constexpr float tanh_c(int k) {
    return k == 0 ? -3.333327174e-01f : k == 1 ? 1.333131194e-01f : k == 2 ? -5.373601243e-02f
         : k == 3 ? 2.064501122e-02f : -5.728444550e-03f;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// z P(z)
__device__ __forceinline__ float tanh_q(float z) {
    float p = tanh_c(kTanhDegree);
#pragma unroll
    for (int k = kTanhDegree - 1; k >= 0; --k) p = __fmaf_rn(p, z, tanh_c(k));
    return __fmul_rn(z, p);
}

__device__ __forceinline__ float tanh_exp(float y) {
    const float e = ex2(__fmul_rn(fabsf(y), 2.8853900817779268f));  // 2^(2|y| log2 e)
    const float t = __fmaf_rn(-2.f, rcp_approx(__fadd_rn(1.f, e)), 1.f);
    return copysignf(t, y);
}

__device__ __forceinline__ float softcap1(float x, float p, float rcp) {
    const float y = __fmul_rn(x, rcp), z = __fmul_rn(y, y);
    return z < kTanhZMax ? __fmaf_rn(x, tanh_q(z), x) : __fmul_rn(p, tanh_exp(y));
}

// Sixteen values in place.  When no value of the warp needs the exponential
// form (the usual case: |x| < 0.6 p everywhere) only the packed polynomial runs.
__device__ __forceinline__ void softcap16(f2_t *v, float p, float rcp) {
    const f2_t r2 = f2(rcp, rcp);
    f2_t y[8], z[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        y[q] = mul2(v[q], r2);
        z[q] = mul2(y[q], y[q]);
    }
    const float zmax = max16(z);
    f2_t o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        f2_t pp = f2(tanh_c(kTanhDegree), tanh_c(kTanhDegree));
#pragma unroll
        for (int k = kTanhDegree - 1; k >= 0; --k) pp = fma2(pp, z[q], f2(tanh_c(k), tanh_c(k)));
        o[q] = fma2(v[q], mul2(z[q], pp), v[q]);
    }
    if (__any_sync(0xffffffffu, !(zmax < kTanhZMax))) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float lo = f2_lo(z[q]) < kTanhZMax ? f2_lo(o[q]) : __fmul_rn(p, tanh_exp(f2_lo(y[q])));
            const float hi = f2_hi(z[q]) < kTanhZMax ? f2_hi(o[q]) : __fmul_rn(p, tanh_exp(f2_hi(y[q])));
            o[q] = f2(lo, hi);
        }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = o[q];
}

// ---- the reduced single soft-cap (kRowSoftcap) --------------------------------
// Its own fit: degree 3 on |y| < 0.45 (csrc/tanh_coeffs.py 0.45 3: 0.67 ulp in
// float32, one fused multiply-add less per value than the degree-4 fit above),
// evaluated on u = x^2 with the coefficients pre-multiplied by the powers of
// 1/p^2 (SoftcapSide::q), so p tanh(x / p) = x (1 + u Q(u)).  Beyond the range,
// the exponential form above.  With logits of a few units and p around 30 the
// exponential form is almost never needed.
constexpr float kSoftcapZMax = 0.2025f;  // 0.45^2
__host__ __device__ constexpr float softcap_c(int k) {
    return k == 0 ? -3.333319426e-01f : k == 1 ? 1.332776695e-01f : k == 2 ? -5.322368443e-02f : 1.772576943e-02f;
}

__device__ __forceinline__ float softcap_series(float x, float u, const SoftcapSide &c) {
    float q = c.q[kSoftcapTerms - 1];
#pragma unroll
    for (int k = kSoftcapTerms - 2; k >= 0; --k) q = __fmaf_rn(q, u, c.q[k]);
    return __fmaf_rn(__fmul_rn(x, u), q, x);
}

// One value: the series when u / p^2 < 0.45^2, else the exponential form.
__device__ __forceinline__ float softcap_u1(float x, const SoftcapSide &c) {
    const float u = __fmul_rn(x, x);
    return __fmul_rn(u, c.r2) < kSoftcapZMax ? softcap_series(x, u, c) : __fmul_rn(c.p, tanh_exp(__fmul_rn(x, c.r)));
}

__device__ __forceinline__ float amax16(const f2_t *v) {
    const float a0 = max3_abs(f2_lo(v[0]), f2_hi(v[0]), f2_lo(v[1]));
    const float a1 = max3_abs(f2_hi(v[1]), f2_lo(v[2]), f2_hi(v[2]));
    const float a2 = max3_abs(f2_lo(v[3]), f2_hi(v[3]), f2_lo(v[4]));
    const float a3 = max3_abs(f2_hi(v[4]), f2_lo(v[5]), f2_hi(v[5]));
    const float a4 = max3_abs(f2_lo(v[6]), f2_hi(v[6]), f2_lo(v[7]));
    return fmaxf(max3(a0, a1, a2), max3_abs(a3, a4, f2_hi(v[7])));
}

// The series on one value pair: x + (x u) Q(u).
__device__ __forceinline__ f2_t softcap_series2(f2_t x, const SoftcapSide &c) {
    const f2_t u = mul2(x, x);
    const f2_t xu = mul2(x, u);
    f2_t w = f2(c.q[kSoftcapTerms - 1], c.q[kSoftcapTerms - 1]);
#pragma unroll
    for (int k = kSoftcapTerms - 2; k >= 0; --k) w = fma2(w, u, f2(c.q[k], c.q[k]));
    return fma2(xu, w, x);
}

// Sixteen values of each side in place, both sides' soft-caps at once.  When
// every |x| of the warp is below its side's c.thr (set on the host a little
// under 0.45 p, so that softcap_u1 takes its series for each of them) the
// series runs packed on both sides, one range test and one warp vote per
// tile.  Otherwise each value takes softcap_u1.  Either way a value gets
// softcap_u1's bits.  A side without a soft-cap carries zero coefficients (its
// series is x + (x u) 0 = x for every |x| below its threshold of 1e12) and is
// left alone on the slow path.
__device__ __forceinline__ void softcap32_u(f2_t *vt, f2_t *vr, const SoftcapSide &ct, const SoftcapSide &cr) {
    const float at = amax16(vt), ar = amax16(vr);
    // NaN is skipped by the maxima; the series carries it through
    if (__all_sync(0xffffffffu, at < ct.thr && ar < cr.thr)) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            vt[q] = softcap_series2(vt[q], ct);
            vr[q] = softcap_series2(vr[q], cr);
        }
    } else {
        if (ct.on) {
#pragma unroll
            for (int q = 0; q < 8; ++q) vt[q] = f2(softcap_u1(f2_lo(vt[q]), ct), softcap_u1(f2_hi(vt[q]), ct));
        }
        if (cr.on) {
#pragma unroll
            for (int q = 0; q < 8; ++q) vr[q] = f2(softcap_u1(f2_lo(vr[q]), cr), softcap_u1(f2_hi(vr[q]), cr));
        }
    }
}

// (host) A side's chain in the reduced form of the soft-cap passes: at most one
// soft-cap, every scale behind it (softcap_p(a x) = a softcap_{p/a}(x)), the
// product of all scales in *post.  False when the chain has more than one
// soft-cap, or when the pre-multiplied series coefficients would leave the
// range of normal floats (p far from 1); such chains take the general pass.
inline bool reduce_softcap(const Xform &c, SoftcapSide *out, double *post) {
    *out = SoftcapSide{};
    double pre = 1.0, after = 1.0, cap = 0.0;
    int n_cap = 0;
    for (int k = 0; k < c.n_ops; ++k) {
        if (c.kind[k] == LPD_OP_SCALE) {
            (n_cap ? after : pre) *= static_cast<double>(c.param[k]);
        } else {
            ++n_cap;
            cap = static_cast<double>(c.param[k]);
        }
    }
    *post = pre * after;
    if (n_cap == 0) {
        // no soft-cap: zero series coefficients leave every |x| below the
        // threshold as it is (x + (x u) 0; x u = x^3 stays finite below 1e12),
        // larger values take the slow path, which leaves this side alone
        out->thr = 1e12f;
        return true;
    }
    if (n_cap > 1) return false;
    const double p = cap / pre, r = pre / cap;
    const double lo = 1e-36, hi = 1e36;
    if (!(p > lo && p < hi && r * r > lo && r * r < hi)) return false;
    out->on = 1;
    out->p = static_cast<float>(p);
    out->r = static_cast<float>(r);
    out->r2 = static_cast<float>(r * r);
    // |x| < 0.449 p gives fl(fl(x^2) fl(1/p^2)) < 0.45^2 after every rounding
    out->thr = static_cast<float>(0.449 * p);
    double rk = r * r;
    for (int k = 0; k < kSoftcapTerms; ++k, rk *= r * r) {
        const double q = static_cast<double>(softcap_c(k)) * rk;
        if (!(std::fabs(q) > lo && std::fabs(q) < hi)) return false;
        out->q[k] = static_cast<float>(q);
    }
    return true;
}

__device__ __forceinline__ float xform1(float x, const XformView &c) {
#pragma unroll 1
    for (int k = 0; k < c.n; ++k) {
        const float4 op = c.ops[k];
        if (__float_as_int(op.x) == LPD_OP_SCALE)
            x = __fmul_rn(x, op.y);
        else
            x = softcap1(x, op.y, op.z);
    }
    return x;
}

// The chain over sixteen values: ops outermost, so each op's kind is decided
// once per chunk (it is the same for every thread); both ops run packed.
__device__ __forceinline__ void xform16(f2_t *v, const XformView &c) {
#pragma unroll 1
    for (int k = 0; k < c.n; ++k) {
        const float4 op = c.ops[k];
        if (__float_as_int(op.x) == LPD_OP_SCALE) {
            const f2_t p2 = f2(op.y, op.y);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = mul2(v[q], p2);
        } else {
            softcap16(v, op.y, op.z);
        }
    }
}

}  // namespace lpd
