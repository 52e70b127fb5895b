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

// ht, hr (entropy variant only, else 0): sum of e_j * a_j per side, where
// e_j = 2^a_j is the term and a_j = (x_j - m) log2(e) its exponent, so that
// the softmax entropy is H = ln(s) - ln(2) * h / s.  When the max moves by
// delta = (m_old - m_new) log2(e) and the terms are scaled by f = 2^delta,
// h becomes f * (h + delta * s).
struct Acc {
    float mt, st, dd, mr, sr, ht, hr;
};

__device__ __forceinline__ Acc acc_init() {
    Acc a;
    a.mt = -FLT_MAX;
    a.mr = -FLT_MAX;
    a.st = a.dd = a.sr = a.ht = a.hr = 0.f;
    return a;
}

// f * (h + delta * s), with an empty state (s == 0, delta possibly -inf)
// contributing exactly 0.
__device__ __forceinline__ float ent_rescale(float h, float s, float f, float delta) {
    return s == 0.f ? 0.f : __fmul_rn(f, __fmaf_rn(delta, s, h));
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
// Without kEntropy the entropy sums are left alone (they are not carried);
// the other fields are the same either way.
// lt, lr: each side's factor from a logit difference to a base-2 exponent
// (log2 e, or s log2 e when the maxima are kept in unscaled units of a side
// whose logits are scaled by s).
template <bool kEntropy = true>
__device__ __forceinline__ void merge_acc(Acc &a, const Acc &b, float lt = kLog2e, float lr = kLog2e) {
    const float mt = fmaxf(a.mt, b.mt), mr = fmaxf(a.mr, b.mr);
    const float aa = __fmul_rn(__fsub_rn(a.mt, mt), lt), ab = __fmul_rn(__fsub_rn(b.mt, mt), lt);
    const float ba = __fmul_rn(__fsub_rn(a.mr, mr), lr), bb = __fmul_rn(__fsub_rn(b.mr, mr), lr);
    const float fa = ex2(aa), fb = ex2(ab), ga = ex2(ba), gb = ex2(bb);
    const float xa = __fadd_rn(__fmul_rn(a.dd, fa), __fmul_rn(a.sr, scale_diff(fa, ga, aa, ba)));
    const float xb = __fadd_rn(__fmul_rn(b.dd, fb), __fmul_rn(b.sr, scale_diff(fb, gb, ab, bb)));
    if (kEntropy) {
        a.ht = __fadd_rn(ent_rescale(a.ht, a.st, fa, aa), ent_rescale(b.ht, b.st, fb, ab));
        a.hr = __fadd_rn(ent_rescale(a.hr, a.sr, ga, ba), ent_rescale(b.hr, b.sr, gb, bb));
    }
    a.st = __fadd_rn(__fmul_rn(a.st, fa), __fmul_rn(b.st, fb));
    a.sr = __fadd_rn(__fmul_rn(a.sr, ga), __fmul_rn(b.sr, gb));
    a.dd = __fadd_rn(xa, xb);
    a.mt = mt;
    a.mr = mr;
}

// Every lane's state reduced over the warp, the result held by all lanes: the
// two maxima first (exact), then each lane's sums rescaled once to them (dd
// with the same exact-difference correction as merge_acc) and added in a
// fixed xor butterfly.  IEEE addition commutes, so partner lanes form the same
// sums and every lane ends with the same bits.
template <bool kEntropy>
__device__ __forceinline__ Acc warp_reduce_acc(Acc a, float lt = kLog2e, float lr = kLog2e) {
    float mt = a.mt, mr = a.mr;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
    }
    const float at = __fmul_rn(__fsub_rn(a.mt, mt), lt), ar = __fmul_rn(__fsub_rn(a.mr, mr), lr);
    const float ft = ex2(at), fr = ex2(ar);
    float dd = __fadd_rn(__fmul_rn(a.dd, ft), __fmul_rn(a.sr, scale_diff(ft, fr, at, ar)));
    float st = __fmul_rn(a.st, ft), sr = __fmul_rn(a.sr, fr);
    float ht = 0.f, hr = 0.f;
    if (kEntropy) {
        ht = ent_rescale(a.ht, a.st, ft, at);
        hr = ent_rescale(a.hr, a.sr, fr, ar);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        st = __fadd_rn(st, __shfl_xor_sync(0xffffffffu, st, off));
        sr = __fadd_rn(sr, __shfl_xor_sync(0xffffffffu, sr, off));
        dd = __fadd_rn(dd, __shfl_xor_sync(0xffffffffu, dd, off));
        if (kEntropy) {
            ht = __fadd_rn(ht, __shfl_xor_sync(0xffffffffu, ht, off));
            hr = __fadd_rn(hr, __shfl_xor_sync(0xffffffffu, hr, off));
        }
    }
    Acc r;
    r.mt = mt;
    r.mr = mr;
    r.st = st;
    r.sr = sr;
    r.dd = dd;
    r.ht = ht;
    r.hr = hr;
    return r;
}

// ---- packed fp32 pairs ---------------------------------------------------------
// Two fp32 values in one 64-bit register pair, operated on with the f32x2
// instructions.  Each half is rounded exactly like the scalar .rn operation, so
// packing changes the instruction count, not the arithmetic.
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2(float a, float b) {
    f2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float f2_lo(f2_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(f2_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ f2_t add2(f2_t a, f2_t b) {
    f2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t sub2(f2_t a, f2_t b) {
    f2_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t mul2(f2_t a, f2_t b) {
    f2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c) {
    f2_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ f2_t ex2_2(f2_t a) { return f2(ex2(f2_lo(a)), ex2(f2_hi(a))); }

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// max(|a|, |b|, |c|) in one instruction (NaN inputs are skipped)
__device__ __forceinline__ float max3_abs(float a, float b, float c) {
    float r;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// ---- streaming form (row kernel and fused epilogue) -------------------------------
// Streaming form of the state of lpd_acc.cuh: the three sums are kept as
// packed (even column, odd column) pairs, folded into one Acc at the end of a
// segment.
struct Acc2 {
    float mt, mr;
    f2_t st, sr, dd, ht, hr;
};

__device__ __forceinline__ Acc2 acc2_init() {
    Acc2 a;
    a.mt = -FLT_MAX;
    a.mr = -FLT_MAX;
    a.st = a.sr = a.dd = a.ht = a.hr = f2(0.f, 0.f);
    return a;
}

__device__ __forceinline__ Acc acc2_fold(const Acc2 &a) {
    Acc r;
    r.mt = a.mt;
    r.mr = a.mr;
    r.st = __fadd_rn(f2_lo(a.st), f2_hi(a.st));
    r.sr = __fadd_rn(f2_lo(a.sr), f2_hi(a.sr));
    r.dd = __fadd_rn(f2_lo(a.dd), f2_hi(a.dd));
    r.ht = __fadd_rn(f2_lo(a.ht), f2_hi(a.ht));
    r.hr = __fadd_rn(f2_lo(a.hr), f2_hi(a.hr));
    return r;
}

// packed form of ent_rescale (both halves share f and delta, not s)
__device__ __forceinline__ f2_t ent_rescale2(f2_t h, f2_t s, float f, float delta) {
    return f2(ent_rescale(f2_lo(h), f2_lo(s), f, delta), ent_rescale(f2_hi(h), f2_hi(s), f, delta));
}

__device__ __forceinline__ float max16(const f2_t *v) {
    const float a = max3(f2_lo(v[0]), f2_hi(v[0]), f2_lo(v[1]));
    const float b = max3(f2_hi(v[1]), f2_lo(v[2]), f2_hi(v[2]));
    const float c = max3(f2_lo(v[3]), f2_hi(v[3]), f2_lo(v[4]));
    const float d = max3(f2_hi(v[4]), f2_lo(v[5]), f2_hi(v[5]));
    const float e = max3(f2_lo(v[6]), f2_hi(v[6]), f2_lo(v[7]));
    return fmaxf(max3(a, b, c), max3(d, e, f2_hi(v[7])));
}

// Fixed pairwise tree over eight packed pairs.
__device__ __forceinline__ f2_t tree8(const f2_t *e) {
    return add2(add2(add2(e[0], e[1]), add2(e[2], e[3])), add2(add2(e[4], e[5]), add2(e[6], e[7])));
}

// Online log-sum-exp of sixteen columns of both sides into the state (see
// lpd_acc.cuh).  Each side's chunk maximum is taken first and the sums are
// rescaled at most once per chunk; the sixteen terms of each sum are added in a
// fixed pairwise tree.  -inf columns (masked tails) contribute exactly 0; the
// -FLT_MAX floor keeps (x - m) defined for rows that are -inf everywhere.
// kClamp (entropy sums only): clamp each term's exponent to a finite floor
// before forming e * a, so that -inf columns add 0 instead of 0 * -inf = NaN.
// Without it a -inf column turns the sum into NaN, which the caller must then
// recompute (the row kernel does, for the warps whose sum came out NaN).
template <bool kEntropy = false, bool kClamp = true>
__device__ __forceinline__ void accumulate16(const f2_t *vt, const f2_t *vr, Acc2 &a, float lt = kLog2e,
                                             float lr = kLog2e) {
    const float cmt = max16(vt), cmr = max16(vr);
    if (cmt > a.mt || cmr > a.mr) {
        const float nmt = fmaxf(a.mt, cmt), nmr = fmaxf(a.mr, cmr);
        const float at = __fmul_rn(__fsub_rn(a.mt, nmt), lt);
        const float ar = __fmul_rn(__fsub_rn(a.mr, nmr), lr);
        const float ft = ex2(at), fr = ex2(ar);
        const float corr = scale_diff(ft, fr, at, ar);
        if (kEntropy) {
            a.ht = ent_rescale2(a.ht, a.st, ft, at);
            a.hr = ent_rescale2(a.hr, a.sr, fr, ar);
        }
        a.dd = add2(mul2(a.dd, f2(ft, ft)), mul2(a.sr, f2(corr, corr)));
        a.st = mul2(a.st, f2(ft, ft));
        a.sr = mul2(a.sr, f2(fr, fr));
        a.mt = nmt;
        a.mr = nmr;
    }
    const f2_t mt2 = f2(a.mt, a.mt), mr2 = f2(a.mr, a.mr), lt2 = f2(lt, lt), lr2 = f2(lr, lr);
    f2_t et[8], er[8], dq[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const f2_t xt = mul2(sub2(vt[p], mt2), lt2), xr = mul2(sub2(vr[p], mr2), lr2);
        et[p] = ex2_2(xt);
        er[p] = ex2_2(xr);
        dq[p] = sub2(et[p], er[p]);
        if (kEntropy && kClamp) {
            // -inf columns give e = 0 and a = -inf; clamping a to a finite
            // floor makes their product 0 instead of NaN (finite terms are
            // never below the floor: their e would be 0 anyway)
            a.ht = fma2(et[p], f2(fmaxf(f2_lo(xt), -1e30f), fmaxf(f2_hi(xt), -1e30f)), a.ht);
            a.hr = fma2(er[p], f2(fmaxf(f2_lo(xr), -1e30f), fmaxf(f2_hi(xr), -1e30f)), a.hr);
        } else if (kEntropy) {
            a.ht = fma2(et[p], xt, a.ht);
            a.hr = fma2(er[p], xr, a.hr);
        }
    }
    a.st = add2(a.st, tree8(et));
    a.sr = add2(a.sr, tree8(er));
    a.dd = add2(a.dd, tree8(dq));
}

}  // namespace lpd
