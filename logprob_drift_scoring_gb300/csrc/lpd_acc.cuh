// Online log-sum-exp state of one row (or one vocab segment of a row) for both
// sides at once, and its merge.  Used by the row kernel (per thread, per warp)
// and by the finalise kernel (across warps and segments), so both sides of
// every merge use the same arithmetic bit for bit.
//
// State (fp32):
//   mt, st   train side: running max and sum exp(x_t - mt)
//   mr, sr   rollout side: running max and sum exp(x_r - mr)
//   dd       sum of exp(x_t - mt) - exp(x_r - mr), i.e. st - sr carried
//            separately.  Identical logits on both sides contribute exactly 0,
//            so dd's rounding is relative to the drift itself, and
//            log(sr / st) = log1p(-dd / st) stays accurate when the two rows
//            nearly agree ("WS2 Cross-Config Logprob Drift Contract",
//            "Measurement Contract": dlogp = train - rollout logp).
// When the maxima move, the sums are rescaled by f = 2^alpha (train) and
// g = 2^beta (rollout) and dd by
//   dd' = dd * f + sr * (f - g),
// which keeps dd = st - sr.  f - g is formed as g * expm1((alpha - beta) ln 2)
// with a short Taylor series when the exponents are close (exactly 0 when they
// are equal), so the correction is accurate relative to itself.
#pragma once

#include <cfloat>

#include "lpd_internal.cuh"

namespace lpd {

// 2^x on the special-function unit.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct Acc {
    float mt, st, dd, mr, sr;
};

__device__ __forceinline__ Acc acc_init() {
    Acc a;
    a.mt = -FLT_MAX;
    a.mr = -FLT_MAX;
    a.st = a.dd = a.sr = 0.f;
    return a;
}

// f - g for f = 2^alpha, g = 2^beta, accurate when alpha ~ beta.
// expm1(u) = u + u^2/2 + u^3/6 + u^4/24 + O(u^5); for |alpha - beta| < 2^-6
// (|u| < 0.011) the omitted terms are below 1e-10 relative.
__device__ __forceinline__ float scale_diff(float f, float g, float alpha, float beta) {
    const float dl = __fsub_rn(alpha, beta);
    if (dl == 0.f) return 0.f;
    if (fabsf(dl) < 0.015625f) {
        const float u = __fmul_rn(dl, 0.6931471805599453f);
        float p = __fmaf_rn(u, 1.f / 24.f, 1.f / 6.f);
        p = __fmaf_rn(u, p, 0.5f);
        p = __fmaf_rn(u, p, 1.f);
        return __fmul_rn(g, __fmul_rn(u, p));
    }
    return __fsub_rn(f, g);  // also the NaN/inf path for empty states
}

// Merge state b into a.  Symmetric in a and b bit for bit (max and IEEE
// addition commute), so a butterfly leaves every lane with the same value.
__device__ __forceinline__ void merge_acc(Acc &a, const Acc &b) {
    const float mt = fmaxf(a.mt, b.mt), mr = fmaxf(a.mr, b.mr);
    const float aa = __fmul_rn(__fsub_rn(a.mt, mt), kLog2e), ab = __fmul_rn(__fsub_rn(b.mt, mt), kLog2e);
    const float ba = __fmul_rn(__fsub_rn(a.mr, mr), kLog2e), bb = __fmul_rn(__fsub_rn(b.mr, mr), kLog2e);
    const float fa = ex2(aa), fb = ex2(ab), ga = ex2(ba), gb = ex2(bb);
    const float xa = __fadd_rn(__fmul_rn(a.dd, fa), __fmul_rn(a.sr, scale_diff(fa, ga, aa, ba)));
    const float xb = __fadd_rn(__fmul_rn(b.dd, fb), __fmul_rn(b.sr, scale_diff(fb, gb, ab, bb)));
    a.st = __fadd_rn(__fmul_rn(a.st, fa), __fmul_rn(b.st, fb));
    a.sr = __fadd_rn(__fmul_rn(a.sr, ga), __fmul_rn(b.sr, gb));
    a.dd = __fadd_rn(xa, xb);
    a.mt = mt;
    a.mr = mr;
}

}  // namespace lpd
