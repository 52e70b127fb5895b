// Streaming row pass: for every active row, the partial log-sum-exp of each
// vocab segment of both the training-side and the rollout-side logits, in one
// read of each row, plus the selected-logit gather.
//
// Method: "WS2 Cross-Config Logprob Drift Contract", section "Measurement
// Contract" (teacher-forced selected-token logp on both sides); "[WS2]
// Framework for ablation experiment", LogProb knobs table, rows 3-5 and 8
// (per-shard partial (max, sum exp) and single-owner gather).
//
// Layout of the work.  One persistent CTA per SM takes active rows i =
// blockIdx.x, blockIdx.x + gridDim.x, ...  A producer thread streams each row
// through a ring of shared-memory stages with 1-D bulk copies (TMA,
// cp.async.bulk, completion on an mbarrier); every stage holds the same tile of
// 16 * 32 W columns of both sides (W consumer warps: 23, so 11776 columns; 20
// for the reduced soft-cap; 16 for the general transform chain; 23, 20, 19 or
// 16 for the plain pass over several vocab segments, whichever pads the
// segments' last tiles least, see row_pass_warps).  The W warps read the
// stage, and thread t owns columns [G g + 4t, G g + 4t + 4), g = 0..3, G =
// 128 W, of every tile.  Each thread keeps an online (max, sum exp) pair per
// side in fp32 plus the sum of the two sides' term differences; at the end of
// a segment each warp reduces its 32 states (both maxima first, then the
// rescaled sums in a fixed xor butterfly) and writes one state to the
// workspace.  The finalise kernel merges the W warp states and the segments
// and does the fp64 row arithmetic.
//
// Batch invariance ("Attention Debug Matrix", section "Metrics": the
// batch-composition control must be bitwise zero): the value that reaches a
// thread, the order in which it accumulates, and the merge trees depend only
// on the logical column index, never on the row index, the grid, the load path
// or the storage dtype (bf16 and fp32 inputs are widened to fp32 first and
// then share one arithmetic path, written with explicit round-to-nearest
// intrinsics so the compiler cannot contract it differently per dtype).
#include <cfloat>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"
#include "lpd_xform.cuh"

namespace lpd {
namespace {

struct Bf16 {
    static constexpr int kBytes = 2;
};
struct F32 {
    static constexpr int kBytes = 4;
};

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s: a stage takes microseconds
constexpr uint32_t kWaitLimitIters = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier and bulk copy (inline PTX) ----------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Bounded wait for phase `parity` of an mbarrier.  Gives up (and tells every
// other thread of the CTA to give up) after kWaitLimitNs, recording
// LPD_STATUS_TIMEOUT; a pipeline stage normally completes in microseconds.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           uint32_t *status, bool honour_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t n = 1; n < kWaitLimitIters; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 0) {
            if (honour_abort && *abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
    }
    *abort_flag = 1;
    atomicOr(status, LPD_STATUS_TIMEOUT);
    return false;
}

// ---- -inf tiles ------------------------------------------------------------
// A whole tile's worth of -inf in each storage format, the source of the bulk
// copies that pad a segment's last stage (constant data of the module).
template <uint32_t kWord, int kWords>
struct __align__(16) FillWords {
    uint32_t w[kWords];
    constexpr FillWords() : w{} {
        for (int i = 0; i < kWords; ++i) w[i] = kWord;
    }
};
constexpr int kMaxTileCols = kColsPerThread * 32 * kConsumerWarps;
__device__ const FillWords<0xFF800000u, kMaxTileCols> g_neg_inf_f32;       // fp32 -inf
__device__ const FillWords<0xFF80FF80u, kMaxTileCols / 2> g_neg_inf_bf16;  // bf16 -inf pairs

template <class D>
__device__ __forceinline__ const void *neg_inf_words();
template <>
__device__ __forceinline__ const void *neg_inf_words<Bf16>() { return g_neg_inf_bf16.w; }
template <>
__device__ __forceinline__ const void *neg_inf_words<F32>() { return g_neg_inf_f32.w; }

// ---- element access ------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <class D>
__device__ __forceinline__ float ldg_elem(const char *p);
template <>
__device__ __forceinline__ float ldg_elem<Bf16>(const char *p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
}
template <>
__device__ __forceinline__ float ldg_elem<F32>(const char *p) {
    return __ldg(reinterpret_cast<const float *>(p));
}

// Four consecutive columns starting at `col` (a multiple of 4) of a stage, as
// two packed pairs.
template <class D>
__device__ __forceinline__ void lds4(const char *stage, int col, f2_t *v);
template <>
__device__ __forceinline__ void lds4<Bf16>(const char *stage, int col, f2_t *v) {
    const uint2 w = *reinterpret_cast<const uint2 *>(stage + 2 * col);
    v[0] = f2(bf16_lo(w.x), bf16_hi(w.x));
    v[1] = f2(bf16_lo(w.y), bf16_hi(w.y));
}
template <>
__device__ __forceinline__ void lds4<F32>(const char *stage, int col, f2_t *v) {
    const float4 w = *reinterpret_cast<const float4 *>(stage + 4 * col);
    v[0] = f2(w.x, w.y);
    v[1] = f2(w.z, w.w);
}

// The logit transform chain ("[WS2] Framework for ablation experiment", LogProb
// knobs table, row 7), applied in order to one logit in fp32: scale x * p
// (temperature 1/T or logit scale) or soft-cap p * tanh(x * (1/p)).  The chain
// is copied into registers once per thread (constant indices only, so it never
// lives in local memory); ops past n are skipped.  Only real columns are
// transformed; masked tail columns stay -inf.
// Column of slot q (0..15) of consumer thread t within a tile of groups of kGroup columns.
template <int kGroup>
__device__ __forceinline__ int slot_col(int t, int q) { return (q >> 2) * kGroup + 4 * t + (q & 3); }

// Tile kinds for the tile body: known full, known ragged (the segment's last,
// shorter tile), or decided at run time from the tile's width.
enum TileKind { kTileFull, kTileRagged, kTileAny };
template <int K>
struct TileTag {
    static constexpr int kind = K;
};

// ---- the arithmetic: accumulate16 and the packed state live in lpd_acc.cuh ----

__device__ __forceinline__ float select16(const f2_t *v, int q) {
    float x = f2_lo(v[0]);
#pragma unroll
    for (int k = 1; k < 16; ++k) x = (q == k) ? ((k & 1) ? f2_hi(v[k >> 1]) : f2_lo(v[k >> 1])) : x;
    return x;
}

// Sum over consumer thread t's columns of one row segment (its slots of every
// tile, read from global memory) of e * max(a, -1e30), a = (x - m) l and
// e = 2^a, then over the warp in a fixed xor butterfly: the entropy sum of a
// warp state relative to the warp's maximum m, with -inf logits adding 0.
template <class D, int kTile, int kGroupCols>
__device__ __noinline__ float entropy_terms(const char *row, int64_t len, float m, float l, int t) {
    float h = 0.f;
    for (int64_t c0 = 0; c0 < len; c0 += kTile) {
#pragma unroll
        for (int q = 0; q < kColsPerThread; ++q) {
            const int64_t col = c0 + slot_col<kGroupCols>(t, q);
            if (col < len) {
                const float x = __fmul_rn(__fsub_rn(ldg_elem<D>(row + col * D::kBytes), m), l);
                h = __fmaf_rn(ex2(x), fmaxf(x, -1e30f), h);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) h = __fadd_rn(h, __shfl_xor_sync(0xffffffffu, h, off));
    return h;
}

// kW: consumer warps.  kMulti: the plain pass over several vocab segments,
// with the -inf tail copies.
// kMode: 0 plain, 1 with a general transform chain, 2 with the entropy sums,
// 3 with a scale-only chain (each side's product of scales folded into its
// exponent factor, so no tanh code and no extra arithmetic per element), 4
// with a chain of at most one soft-cap per side in its reduced form (the
// soft-cap on each loaded value, the scales folded into the exponent factor
// as in mode 3).
template <class DT, class DR, bool kTma, int kMode, int kW, bool kMulti>
__global__ void __launch_bounds__(kW * 32 + 32, 1)
    row_kernel(const __grid_constant__ RowArgs a, int n_stages) {
    constexpr bool kXform = kMode == kRowTransform;
    constexpr bool kEntropy = kMode == kRowEntropy;
    constexpr bool kScale = kMode == kRowScale;
    constexpr bool kSoftcap = kMode == kRowSoftcap;
    constexpr int kWarps = kW;
    constexpr int kGroupCols = 4 * 32 * kWarps;
    constexpr int kTile = kColsPerThread * 32 * kWarps;
    extern __shared__ __align__(1024) char smem[];
    __shared__ int abort_flag;
    __shared__ float4 xf_ops[kXform ? 2 * LPD_MAX_TRANSFORM_OPS : 1];
    constexpr int kStageT = kTile * DT::kBytes;
    constexpr int kStageR = kTile * DR::kBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + n_stages;
    char *ring = smem + 1024;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_active = a.hdr->n_active;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (kXform) {
            xform_table(a.xt, xf_ops);
            xform_table(a.xr, xf_ops + LPD_MAX_TRANSFORM_OPS);
        }
        if (kTma) {
            for (int s = 0; s < n_stages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kWarps);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
    }
    __syncthreads();

    // The plain pass over several vocab segments (kMulti: every segment's last
    // tile is ragged): when a segment's length in bytes is a multiple of 16 on
    // both sides, the producer also copies -inf into the columns of its last
    // stage past the segment's end (from the constant arrays above), so the
    // consumers read that tile like any full one.  It gives every column the
    // value the branch-free ragged path would (-inf past the end), so the bits
    // are the same either way; passes over one segment (one ragged tile a row)
    // are instantiated without it, as they measured slower with it.
    constexpr bool kFillTail = kMulti && !kXform && !kSoftcap;
    auto tail_filled = [&](const Segment &sg) {
        return kFillTail && (sg.len * DT::kBytes) % 16 == 0 && (sg.len * DR::kBytes) % 16 == 0;
    };

    if (warp == kWarps) {
        // ------------------------------------------------------ producer
        if (!kTma || lane != 0) return;
        uint64_t policy;
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
        uint32_t it = 0;
        bool ok = true;
        for (int64_t i = blockIdx.x; ok && i < n_active; i += gridDim.x) {
            const int64_t r = a.rowid[i].x;
            for (int k = 0; ok && k < a.n_seg; ++k) {
                const Segment &sg = a.seg[k];
                const char *tb = sg.t + r * sg.t_stride;
                const char *rb = sg.r + r * sg.r_stride;
                const bool fill = tail_filled(sg);
                for (int64_t c0 = 0; c0 < sg.len; c0 += kTile) {
                    const uint32_t stage = it % n_stages, round = it / n_stages;
                    if (round > 0 && !wait_phase(&empty[stage], (round - 1) & 1, &abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const int64_t nv = min(static_cast<int64_t>(kTile), sg.len - c0);
                    const uint32_t bt = static_cast<uint32_t>(nv * DT::kBytes) & ~15u;
                    const uint32_t br = static_cast<uint32_t>(nv * DR::kBytes) & ~15u;
                    // -inf tails (multiples of 16 bytes when fill holds)
                    const uint32_t ft = (fill && nv < kTile) ? kStageT - bt : 0u;
                    const uint32_t fr = (fill && nv < kTile) ? kStageR - br : 0u;
                    char *st = ring + static_cast<size_t>(stage) * (kStageT + kStageR);
                    mbar_arrive_expect_tx(&full[stage], bt + br + ft + fr);
                    // a.stall (tests of the timeout path only): CTA 0 never
                    // issues its first copy, so its consumers run into the
                    // bounded wait; no copy is in flight for that stage
                    const bool withhold = a.stall && it == 0 && blockIdx.x == 0;
                    if (!withhold) {
                        if (bt) bulk_g2s(st, tb + c0 * DT::kBytes, bt, &full[stage], policy);
                        if (br) bulk_g2s(st + kStageT, rb + c0 * DR::kBytes, br, &full[stage], policy);
                        if (ft) bulk_g2s(st + bt, neg_inf_words<DT>(), ft, &full[stage], policy);
                        if (fr) bulk_g2s(st + kStageT + br, neg_inf_words<DR>(), fr, &full[stage], policy);
                    }
                    ++it;
                }
            }
        }
        // Before the CTA (and its shared memory) goes away, every copy this
        // thread issued must have landed: the last n_stages ones are the only
        // ones that can still be in flight.  Normally they completed long ago
        // (the consumers waited for them); after an abandoned pipeline this is
        // the bounded wait for the stragglers.
        (void)ok;
        const uint32_t first = it > static_cast<uint32_t>(n_stages) ? it - n_stages : 0;
        for (uint32_t j = first; j < it; ++j)
            wait_phase(&full[j % n_stages], (j / n_stages) & 1, &abort_flag, a.status, false);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int t = threadIdx.x;
    // Scale-only chains keep the logits unscaled: the scale s rides in the
    // factor to base-2 exponents, (x - m) s log2 e, and the finalise forms
    // s m and s x[id] in fp64.
    const float lg_t = (kScale || kSoftcap) ? a.lt : kLog2e, lg_r = (kScale || kSoftcap) ? a.lr : kLog2e;
    const XformView cxt{xf_ops, kXform ? a.xt.n_ops : 0}, cxr{xf_ops + (kXform ? LPD_MAX_TRANSFORM_OPS : 0),
                                                              kXform ? a.xr.n_ops : 0};
    // one real logit of each side through that side's chain (modes 1 and 4)
    auto tf_t = [&](float x) -> float {
        if constexpr (kXform) return xform1(x, cxt);
        else if constexpr (kSoftcap) return a.cap[0].on ? softcap_u1(x, a.cap[0]) : x;
        else return x;
    };
    auto tf_r = [&](float x) -> float {
        if constexpr (kXform) return xform1(x, cxr);
        else if constexpr (kSoftcap) return a.cap[1].on ? softcap_u1(x, a.cap[1]) : x;
        else return x;
    };
    uint32_t it = 0;
    for (int64_t i = blockIdx.x; i < n_active; i += gridDim.x) {
        const int2 rid = a.rowid[i];
        const int64_t r = rid.x, id = rid.y;
        // Which segment, tile and slot hold the selected column, and whether
        // this thread owns it (single-owner gather).
        int pick_seg = -1, pick_slot = 0;
        int64_t pick_c0 = -1;
        bool pick_mine = false;
        if (id >= 0 && id < a.vocab) {
            for (int k = 0; k < a.n_seg; ++k) {
                const int64_t c = id - a.seg[k].v_start;
                if (c >= 0 && c < a.seg[k].len) {
                    const int pos = static_cast<int>(c % kTile);
                    pick_seg = k;
                    pick_c0 = c - pos;
                    pick_slot = (pos / kGroupCols) * 4 + (pos & 3);
                    pick_mine = ((pos % kGroupCols) >> 2) == t;
                }
            }
        }
        for (int k = 0; k < a.n_seg; ++k) {
            const Segment &sg = a.seg[k];
            const char *tb = sg.t + r * sg.t_stride;
            const char *rb = sg.r + r * sg.r_stride;
            Acc2 acc2 = acc2_init();
            const bool seg_filled = tail_filled(sg);
            auto tile = [&](const int64_t c0, auto tag) -> bool {
                constexpr int kKind = decltype(tag)::kind;
                const int nv = kKind == kTileFull ? kTile : static_cast<int>(min(static_cast<int64_t>(kTile), sg.len - c0));
                f2_t vt[8], vr[8];  // slots (2p, 2p+1) in pair p
                if (kTma) {
                    const uint32_t stage = it % n_stages, round = it / n_stages;
                    // the whole warp leaves together if any lane gave up, so no
                    // lane is left behind at a warp-synchronous instruction
                    const bool ok = wait_phase(&full[stage], round & 1, &abort_flag, a.status);
                    if (__any_sync(0xffffffffu, !ok)) return false;
                    const char *stg = ring + static_cast<size_t>(stage) * (kStageT + kStageR);
                    if (kKind == kTileFull || (kKind == kTileAny && (nv == kTile || seg_filled))) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            lds4<DT>(stg, g * kGroupCols + 4 * t, vt + 2 * g);
                            lds4<DR>(stg + kStageT, g * kGroupCols + 4 * t, vr + 2 * g);
                        }
                        if (kXform) {
                            xform16(vt, cxt);
                            xform16(vr, cxr);
                        }
                        if (kSoftcap) softcap32_u(vt, vr, a.cap[0], a.cap[1]);
                    } else {
                        // ragged last tile: the same vector loads, then the
                        // columns the bulk copy did not cover (a few bytes at the
                        // end of the row) come from global, and columns past the
                        // segment are -inf
                        const int nbt = static_cast<int>((static_cast<uint32_t>(nv * DT::kBytes) & ~15u) / DT::kBytes);
                        const int nbr = static_cast<int>((static_cast<uint32_t>(nv * DR::kBytes) & ~15u) / DR::kBytes);
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            lds4<DT>(stg, g * kGroupCols + 4 * t, vt + 2 * g);
                            lds4<DR>(stg + kStageT, g * kGroupCols + 4 * t, vr + 2 * g);
                        }
                        constexpr bool kChain = kXform || kSoftcap;
                        if (nbt == nv && nbr == nv) {
                            // the copy holds every real column (the segment's
                            // length in bytes is a multiple of 16 on both sides,
                            // the same for every thread): columns past the end
                            // are selected away without branches; a chain runs
                            // packed on all sixteen values, as in a full tile,
                            // with 0 in those columns, which become -inf after it
                            const float fill = kChain ? 0.f : -INFINITY;
#pragma unroll
                            for (int p = 0; p < 8; ++p) {
                                const int col0 = slot_col<kGroupCols>(t, 2 * p);
                                const bool in0 = col0 < nv, in1 = col0 + 1 < nv;
                                vt[p] = f2(in0 ? f2_lo(vt[p]) : fill, in1 ? f2_hi(vt[p]) : fill);
                                vr[p] = f2(in0 ? f2_lo(vr[p]) : fill, in1 ? f2_hi(vr[p]) : fill);
                            }
                            if constexpr (kChain) {
                                if constexpr (kXform) {
                                    xform16(vt, cxt);
                                    xform16(vr, cxr);
                                } else {
                                    softcap32_u(vt, vr, a.cap[0], a.cap[1]);
                                }
#pragma unroll
                                for (int p = 0; p < 8; ++p) {
                                    const int col0 = slot_col<kGroupCols>(t, 2 * p);
                                    const bool in0 = col0 < nv, in1 = col0 + 1 < nv;
                                    vt[p] = f2(in0 ? f2_lo(vt[p]) : -INFINITY, in1 ? f2_hi(vt[p]) : -INFINITY);
                                    vr[p] = f2(in0 ? f2_lo(vr[p]) : -INFINITY, in1 ? f2_hi(vr[p]) : -INFINITY);
                                }
                            }
                        } else if constexpr (kSoftcap) {
                            // the soft-cap runs packed on all sixteen values, as
                            // in a full tile: columns past the segment hold 0 while
                            // it runs and become -inf afterwards
#pragma unroll
                            for (int p = 0; p < 8; ++p) {
                                const int col0 = slot_col<kGroupCols>(t, 2 * p);
                                if (col0 >= nv) {
                                    vt[p] = vr[p] = f2(0.f, 0.f);
                                } else if (col0 + 1 >= min(nbt, nbr)) {
                                    float x[2] = {f2_lo(vt[p]), f2_hi(vt[p])}, y[2] = {f2_lo(vr[p]), f2_hi(vr[p])};
#pragma unroll
                                    for (int h = 0; h < 2; ++h) {
                                        const int col = col0 + h;
                                        if (col >= nbt) x[h] = col < nv ? ldg_elem<DT>(tb + (c0 + col) * DT::kBytes) : 0.f;
                                        if (col >= nbr) y[h] = col < nv ? ldg_elem<DR>(rb + (c0 + col) * DR::kBytes) : 0.f;
                                    }
                                    vt[p] = f2(x[0], x[1]);
                                    vr[p] = f2(y[0], y[1]);
                                }
                            }
                            softcap32_u(vt, vr, a.cap[0], a.cap[1]);
#pragma unroll
                            for (int p = 0; p < 8; ++p) {
                                const int col0 = slot_col<kGroupCols>(t, 2 * p);
                                if (col0 + 1 >= nv) {
                                    const float lt = col0 < nv ? f2_lo(vt[p]) : -INFINITY;
                                    const float lr = col0 < nv ? f2_lo(vr[p]) : -INFINITY;
                                    vt[p] = f2(lt, -INFINITY);
                                    vr[p] = f2(lr, -INFINITY);
                                }
                            }
                        } else {
#pragma unroll
                        for (int p = 0; p < 8; ++p) {
                            const int col0 = slot_col<kGroupCols>(t, 2 * p);  // the pair is col0, col0 + 1
                            if (col0 >= nv) {
                                vt[p] = vr[p] = f2(-INFINITY, -INFINITY);  // wholly past the segment
                            } else if (col0 + 1 >= min(nbt, nbr)) {
                                float x[2] = {f2_lo(vt[p]), f2_hi(vt[p])}, y[2] = {f2_lo(vr[p]), f2_hi(vr[p])};
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int col = col0 + h;
                                    if (col >= nbt) x[h] = col < nv ? ldg_elem<DT>(tb + (c0 + col) * DT::kBytes) : -INFINITY;
                                    if (col >= nbr) y[h] = col < nv ? ldg_elem<DR>(rb + (c0 + col) * DR::kBytes) : -INFINITY;
                                    if (kXform && col < nv) {
                                        x[h] = tf_t(x[h]);
                                        y[h] = tf_r(y[h]);
                                    }
                                }
                                vt[p] = f2(x[0], x[1]);
                                vr[p] = f2(y[0], y[1]);
                            } else if (kXform) {
                                vt[p] = f2(tf_t(f2_lo(vt[p])), tf_t(f2_hi(vt[p])));
                                vr[p] = f2(tf_r(f2_lo(vr[p])), tf_r(f2_hi(vr[p])));
                            }
                        }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[stage]);  // values are in registers now
                    ++it;
                } else {
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        float x[2], y[2];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int col = slot_col<kGroupCols>(t, 2 * p + h);
                            x[h] = col < nv ? ldg_elem<DT>(tb + (c0 + col) * DT::kBytes) : -INFINITY;
                            y[h] = col < nv ? ldg_elem<DR>(rb + (c0 + col) * DR::kBytes) : -INFINITY;
                            if ((kXform || kSoftcap) && col < nv) {
                                x[h] = tf_t(x[h]);
                                y[h] = tf_r(y[h]);
                            }
                        }
                        vt[p] = f2(x[0], x[1]);
                        vr[p] = f2(y[0], y[1]);
                    }
                }
                if (pick_mine && k == pick_seg && c0 == pick_c0)
                    a.pick[i] = make_float2(select16(vt, pick_slot), select16(vr, pick_slot));
                // entropy sums: full tiles skip the clamp of -inf exponents
                // (a -inf logit there leaves a NaN sum, recomputed below)
                accumulate16<kEntropy, kKind != kTileFull>(vt, vr, acc2, lg_t, lg_r);
                return true;
            };
            if constexpr (kXform || kEntropy) {
                // full tiles in a tight loop, the segment's ragged last tile
                // after it (measured faster for the transform chain's larger
                // body; for the entropy sums, only the last tile clamps)
                int64_t c0 = 0;
                for (; c0 + kTile <= sg.len; c0 += kTile)
                    if (!tile(c0, TileTag<kTileFull>{})) return;
                if (c0 < sg.len && !tile(c0, TileTag<kTileRagged>{})) return;
            } else {
                for (int64_t c0 = 0; c0 < sg.len; c0 += kTile)
                    if (!tile(c0, TileTag<kTileAny>{})) return;
            }
            Acc acc = warp_reduce_acc<kEntropy>(acc2_fold(acc2), lg_t, lg_r);
            if constexpr (kEntropy) {
                // A -inf logit in a full tile made this warp's entropy sum NaN
                // (0 * -inf, see accumulate16): the warp sums its columns'
                // terms again, clamped, relative to its final maxima (the same
                // quantity; the test is warp-uniform, every lane holds the
                // reduced sums).  NaN logits stay NaN.
                if (isnan(acc.ht)) acc.ht = entropy_terms<DT, kTile, kGroupCols>(tb, sg.len, acc.mt, lg_t, t);
                if (isnan(acc.hr)) acc.hr = entropy_terms<DR, kTile, kGroupCols>(rb, sg.len, acc.mr, lg_r, t);
            }
            if (lane == 0) {
                float4 *dst = a.part + ((i * a.n_seg + k) * kConsumerWarps + warp) * 2;
                dst[0] = make_float4(acc.mt, acc.st, acc.dd, acc.mr);
                dst[1] = make_float4(acc.sr, acc.ht, acc.hr, 0.f);
            }
        }
    }
}

template <class DT, class DR, bool kTma, int kMode, int kW, bool kMulti>
cudaError_t launch_typed(const RowArgs &a, cudaStream_t stream) {
    constexpr int kThreads = kW * 32 + 32;  // + producer warp
    const int stage_bytes = kColsPerThread * 32 * kW * (DT::kBytes + DR::kBytes);
    const int n_stages = kTma ? min(16, kRingBytes / stage_bytes) : 0;
    const size_t smem = kTma ? 1024 + static_cast<size_t>(n_stages) * stage_bytes : 0;
    auto kern = row_kernel<DT, DR, kTma, kMode, kW, kMulti>;
    static std::atomic<uint64_t> configured{0};
    const cudaError_t e = set_smem_once(kern, smem, configured);
    if (e != cudaSuccess) return e;
    kern<<<device_sm_count(), kThreads, smem, stream>>>(a, n_stages);
    return cudaGetLastError();
}

template <bool kTma, int kMode, int kW = row_warps(kMode), bool kMulti = false>
cudaError_t dispatch(const RowArgs &a, int dt, int dr, cudaStream_t stream) {
    if (dt == LPD_BF16 && dr == LPD_BF16) return launch_typed<Bf16, Bf16, kTma, kMode, kW, kMulti>(a, stream);
    if (dt == LPD_BF16 && dr == LPD_F32) return launch_typed<Bf16, F32, kTma, kMode, kW, kMulti>(a, stream);
    if (dt == LPD_F32 && dr == LPD_BF16) return launch_typed<F32, Bf16, kTma, kMode, kW, kMulti>(a, stream);
    return launch_typed<F32, F32, kTma, kMode, kW, kMulti>(a, stream);
}

template <int kMode>
cudaError_t dispatch_path(const RowArgs &a, int dt, int dr, bool use_tma, cudaStream_t stream) {
    return use_tma ? dispatch<true, kMode>(a, dt, dr, stream) : dispatch<false, kMode>(a, dt, dr, stream);
}

}  // namespace

int row_pass_warps(const Segment *segs, int n_seg, int mode, bool use_tma) {
    if (mode != kRowPlain || !use_tma || n_seg < 2) return row_warps(mode);
    // the plain bulk-copy pass over several vocab segments: the consumer-warp
    // count (tile width 512 W) whose tiles cover the segments with the fewest
    // columns; each segment's last tile is padded to a whole tile, which costs
    // as much as real columns.  Ties keep the most warps.
    int best = row_warps(mode);
    int64_t best_cols = -1;
    for (int w : {23, 20, 19, 16}) {
        const int64_t tile = static_cast<int64_t>(kColsPerThread) * 32 * w;
        int64_t cols = 0;
        for (int k = 0; k < n_seg; ++k) cols += (segs[k].len + tile - 1) / tile * tile;
        if (best_cols < 0 || cols < best_cols) {
            best = w;
            best_cols = cols;
        }
    }
    return best;
}

cudaError_t launch_rows(const RowArgs &a, int dtype_t, int dtype_r, bool use_tma, int mode, int warps,
                        cudaStream_t stream) {
    if (mode == kRowPlain && use_tma && a.n_seg > 1) {
        if (warps == 23) return dispatch<true, kRowPlain, 23, true>(a, dtype_t, dtype_r, stream);
        if (warps == 19) return dispatch<true, kRowPlain, 19, true>(a, dtype_t, dtype_r, stream);
        if (warps == 16) return dispatch<true, kRowPlain, 16, true>(a, dtype_t, dtype_r, stream);
        return dispatch<true, kRowPlain, 20, true>(a, dtype_t, dtype_r, stream);
    }
    if (mode == kRowTransform) return dispatch_path<1>(a, dtype_t, dtype_r, use_tma, stream);
    if (mode == kRowSoftcap) return dispatch_path<4>(a, dtype_t, dtype_r, use_tma, stream);
    if (mode == kRowEntropy) return dispatch_path<2>(a, dtype_t, dtype_r, use_tma, stream);
    if (mode == kRowScale) return dispatch_path<3>(a, dtype_t, dtype_r, use_tma, stream);
    return dispatch_path<0>(a, dtype_t, dtype_r, use_tma, stream);
}

}  // namespace lpd
