// Active-row selection, per-row finalisation, and the drift metrics.
//
// Method: "WS2 Cross-Config Logprob Drift Contract", sections "Measurement
// Contract" (dlogp = train - rollout on active response/action tokens only)
// and "Diagnostics" (ratio0, clipfrac0, approx_kl0, mean/p95/p99/max |dlogp|),
// and roadmap item B1 (zero active tokens, worst-token metadata).
//
// Every reduction here has a fixed shape: block partials over fixed row
// ranges, merged in block order, trees with a fixed pairing.  There are no
// floating-point atomics, so results are bitwise repeatable.
#include <cfloat>
#include <climits>

#include <math_constants.h>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"

namespace lpd {
namespace {

// lse of a side whose maxima are kept in unscaled units (scale 1 otherwise):
// the product of two floats is exact in fp64.
__device__ __forceinline__ double lse_train(const Acc &a, float scale) {
    return static_cast<double>(scale) * static_cast<double>(a.mt) + log(static_cast<double>(a.st));
}
__device__ __forceinline__ double lse_rollout(const Acc &a, float scale) {
    return static_cast<double>(scale) * static_cast<double>(a.mr) + log(static_cast<double>(a.sr));
}

// ---------------------------------------------------------------- stage 1
// One CTA walks the mask in chunks of 16384 rows (16 consecutive rows per
// thread), block-scans the per-thread counts and writes the (row, token id)
// pairs of active rows in row order.
__global__ void __launch_bounds__(1024) select_active_kernel(int64_t n_rows, const uint8_t *__restrict__ mask,
                                                             const int32_t *__restrict__ ids,
                                                             float *__restrict__ out_lt, float *__restrict__ out_lr,
                                                             float *__restrict__ out_d, lpd_metrics *metrics,
                                                             WsHeader *hdr, int2 *__restrict__ rowid) {
    __shared__ int warp_excl[32];
    __shared__ int chunk_total;
    __shared__ long long base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) base = 0;
    __syncthreads();
    for (int64_t chunk = 0; chunk < n_rows; chunk += 1024 * 16) {
        const int64_t r0 = chunk + static_cast<int64_t>(tid) * 16;
        // all of this thread's loads first (independent), then the stores
        uint8_t mk[16];
        int32_t idv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) mk[q] = (r0 + q < n_rows) ? mask[r0 + q] : 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) idv[q] = (mk[q] && ids) ? ids[r0 + q] : 0;
        uint32_t bits = 0;
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int64_t r = r0 + q;
            if (mk[q]) {
                bits |= 1u << q;
                ++cnt;
            } else if (r < n_rows) {
                if (out_lt) out_lt[r] = 0.f;
                if (out_lr) out_lr[r] = 0.f;
                if (out_d) out_d[r] = 0.f;
            }
        }
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) warp_excl[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int w = warp_excl[lane];
            int wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += y;
            }
            warp_excl[lane] = wi - w;
            if (lane == 31) chunk_total = wi;
        }
        __syncthreads();
        int64_t pos = base + warp_excl[warp] + (incl - cnt);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            if (bits >> q & 1u) rowid[pos++] = make_int2(static_cast<int>(r0 + q), idv[q]);
        }
        __syncthreads();
        if (tid == 0) base += chunk_total;
        __syncthreads();
    }
    if (tid == 0) {
        hdr->n_active = base;
        metrics->status = 0u;
    }
}

// The same compaction spread over blocks of kSelBlockRows rows, for batches
// of 2 to kSelMaxBlocks such blocks: one kernel counts each block's active
// rows into the workspace header's spare slots, a second lets every block
// take its base from the counts of the blocks before it and write its pairs.
// The output is the single-CTA kernel's, pair for pair.
constexpr int kSelBlockThreads = 256;
constexpr int kSelBlockRows = kSelBlockThreads * 16;  // 4096
constexpr int kSelMaxBlocks = 31;                     // spare int64 slots in WsHeader

__device__ __forceinline__ int block_excl_scan(int v, int *warp_sum, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kSelBlockThreads / 32 ? warp_sum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += y;
        }
        if (lane < kSelBlockThreads / 32) warp_sum[lane] = wi - w;
        if (lane == 31) warp_sum[31] = wi;
    }
    __syncthreads();
    total = warp_sum[31];
    return warp_sum[warp] + incl - v;
}

__global__ void __launch_bounds__(kSelBlockThreads) count_active_kernel(int64_t n_rows,
                                                                       const uint8_t *__restrict__ mask,
                                                                       WsHeader *hdr) {
    __shared__ int warp_sum[32];
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kSelBlockRows + threadIdx.x * 16;
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) cnt += (r0 + q < n_rows && mask[r0 + q]) ? 1 : 0;
    int total;
    block_excl_scan(cnt, warp_sum, total);
    if (threadIdx.x == 0) hdr->reserved[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kSelBlockThreads) compact_active_kernel(
    int64_t n_rows, const uint8_t *__restrict__ mask, const int32_t *__restrict__ ids, float *__restrict__ out_lt,
    float *__restrict__ out_lr, float *__restrict__ out_d, lpd_metrics *metrics, WsHeader *hdr,
    int2 *__restrict__ rowid) {
    __shared__ int warp_sum[32];
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kSelBlockRows + threadIdx.x * 16;
    uint8_t mk[16];
    int32_t idv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) mk[q] = (r0 + q < n_rows) ? mask[r0 + q] : 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) idv[q] = (mk[q] && ids) ? ids[r0 + q] : 0;
    int64_t base = 0;
    for (unsigned b = 0; b < blockIdx.x; ++b) base += hdr->reserved[b];  // the blocks before this one
    uint32_t bits = 0;
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const int64_t r = r0 + q;
        if (mk[q]) {
            bits |= 1u << q;
            ++cnt;
        } else if (r < n_rows) {
            if (out_lt) out_lt[r] = 0.f;
            if (out_lr) out_lr[r] = 0.f;
            if (out_d) out_d[r] = 0.f;
        }
    }
    int total;
    int64_t pos = base + block_excl_scan(cnt, warp_sum, total);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        if (bits >> q & 1u) rowid[pos++] = make_int2(static_cast<int>(r0 + q), idv[q]);
    }
    if (threadIdx.x == 0) {
        if (blockIdx.x == gridDim.x - 1) hdr->n_active = base + total;
        if (blockIdx.x == 0) metrics->status = 0u;
    }
}

// Metrics over caller-given per-row dlogp (the union of several ranks' rows):
// active row i takes d = dlogp[row] widened to fp64 and the key |d| in fp32;
// a non-finite value on an active row sets LPD_STATUS_NONFINITE.
__global__ void __launch_bounds__(kFinThreads) dlogp_rows_kernel(const float *__restrict__ dlogp,
                                                                 const WsHeader *hdr, const int2 *rowid,
                                                                 double *dval, uint32_t *keys, uint32_t *status) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x;
    if (i >= hdr->n_active) return;
    const float d = dlogp[rowid[i].x];
    dval[i] = static_cast<double>(d);
    keys[i] = __float_as_uint(fabsf(d));
    if (!isfinite(d)) atomicOr(status, static_cast<uint32_t>(LPD_STATUS_NONFINITE));
}

// ---------------------------------------------------------------- stage 2b
struct Part {
    double sum_abs, sum_k3, sum_em1, max_abs;
    long long argmax_row, n_clip;
};

__device__ __forceinline__ void combine(Part &x, const Part &y) {
    x.sum_abs += y.sum_abs;
    x.sum_k3 += y.sum_k3;
    x.sum_em1 += y.sum_em1;
    x.n_clip += y.n_clip;
    if (y.max_abs > x.max_abs || (y.max_abs == x.max_abs && y.argmax_row < x.argmax_row)) {
        x.max_abs = y.max_abs;
        x.argmax_row = y.argmax_row;
    }
}

__device__ __forceinline__ Part neutral_part() {
    Part p;
    p.sum_abs = p.sum_k3 = p.sum_em1 = 0.0;
    p.max_abs = -1.0;
    p.argmax_row = LLONG_MAX;
    p.n_clip = 0;
    return p;
}

// Fixed-pairing tree over a block's Part values held in shared memory.
template <int kN>
__device__ __forceinline__ void block_tree(Part *sh) {
#pragma unroll 1
    for (int stride = kN / 2; stride > 0; stride >>= 1) {
        if (threadIdx.x < stride) combine(sh[threadIdx.x], sh[threadIdx.x + stride]);
        __syncthreads();
    }
}

// One thread per active row: merge the warp states of each segment, then
// the segments in vocab order (and optionally in a given permutation), then
// the per-row arithmetic in fp64:
//   lse = m + log(s),  logp = x[id] - lse,
//   dlogp = (x_t[id] - x_r[id]) - (m_t - m_r) + log(s_r / s_t),
// with log(s_r / s_t) = log1p(-dd / s_t) when |dd| < s_t / 2 (dd = s_t - s_r
// carried separately, see lpd_acc.cuh), which keeps dlogp accurate when the
// two rows nearly agree and exactly 0 when they differ by a constant shift.
// One thread per active row in small blocks, so that a batch of a few
// thousand rows still spreads over every SM (the fp64 row arithmetic is
// latency-bound).
constexpr int kFinalizeThreads = 64;

__global__ void __launch_bounds__(kFinalizeThreads) finalize_kernel(const __grid_constant__ FinArgs a) {
    const int64_t n_active = a.hdr->n_active;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kFinalizeThreads + threadIdx.x;
    if (i >= n_active) return;
    const int2 rid = a.rowid[i];
    const int64_t r = rid.x, id = rid.y;
    uint32_t bad = 0;
    double d;
    if (id < 0 || id >= a.vocab) {
        bad |= LPD_STATUS_TOKEN_OOB;
        d = CUDART_NAN;
        if (a.out_lt) a.out_lt[r] = CUDART_NAN_F;
        if (a.out_lr) a.out_lr[r] = CUDART_NAN_F;
        if (a.out_perm_lt) a.out_perm_lt[r] = CUDART_NAN_F;
        if (a.out_perm_lr) a.out_perm_lr[r] = CUDART_NAN_F;
        if (a.out_ent_t) a.out_ent_t[r] = CUDART_NAN_F;
        if (a.out_ent_r) a.out_ent_r[r] = CUDART_NAN_F;
    } else {
        const float2 xs = a.pick[i];
        Acc seg[kMaxSegments];
        for (int k = 0; k < a.n_seg; ++k) {
            Acc sk = acc_init();
            const float4 *pw = a.part + (i * a.n_seg + k) * kConsumerWarps * 2;
#pragma unroll 4
            for (int w = 0; w < a.n_warps; ++w) {
                const float4 p0 = pw[2 * w], p1 = pw[2 * w + 1];
                Acc o;
                o.mt = p0.x;
                o.st = p0.y;
                o.dd = p0.z;
                o.mr = p0.w;
                o.sr = p1.x;
                o.ht = p1.y;
                o.hr = p1.z;
                merge_acc(sk, o, a.lg_t, a.lg_r);
            }
            seg[k] = sk;
        }
        // the selected logits, scaled by a scale-only chain (exact in fp64)
        const double xt = static_cast<double>(a.scale_t) * xs.x, xr = static_cast<double>(a.scale_r) * xs.y;
        Acc row = acc_init();
        double lse_t, lse_r;
        if (a.topo == LPD_TOPO_ALLREDUCE_PARTIALS) {
            // a max reduction, then a sum reduction of s_k 2^((m_k - M) log2 e)
            // in reduction order, each side on its own
            float mt = -FLT_MAX, mr = -FLT_MAX;
            for (int k = 0; k < a.n_seg; ++k) {
                mt = fmaxf(mt, seg[k].mt);
                mr = fmaxf(mr, seg[k].mr);
            }
            float st = 0.f, sr = 0.f;
            for (int j = 0; j < a.n_seg; ++j) {
                const Acc &sk = seg[a.n_order ? a.order[j] : j];
                st = __fadd_rn(st, __fmul_rn(sk.st, ex2(__fmul_rn(__fsub_rn(sk.mt, mt), a.lg_t))));
                sr = __fadd_rn(sr, __fmul_rn(sk.sr, ex2(__fmul_rn(__fsub_rn(sk.mr, mr), a.lg_r))));
            }
            lse_t = static_cast<double>(a.scale_t) * static_cast<double>(mt) + log(static_cast<double>(st));
            lse_r = static_cast<double>(a.scale_r) * static_cast<double>(mr) + log(static_cast<double>(sr));
            d = (xt - lse_t) - (xr - lse_r);
        } else {
            // online pairwise merge in global vocab-shard order (or the given one)
            for (int j = 0; j < a.n_seg; ++j) merge_acc(row, seg[a.n_order ? a.order[j] : j], a.lg_t, a.lg_r);
            lse_t = lse_train(row, a.scale_t);
            lse_r = lse_rollout(row, a.scale_r);
            const double st = row.st, sr = row.sr, dd = row.dd;
            const double l_ratio = fabs(dd) < 0.5 * st ? log1p(-dd / st) : log(sr / st);
            d = ((xt - xr) - (static_cast<double>(a.scale_t) * static_cast<double>(row.mt) -
                              static_cast<double>(a.scale_r) * static_cast<double>(row.mr))) +
                l_ratio;
        }
        if (!(isfinite(lse_t) && isfinite(lse_r) && isfinite(xt) && isfinite(xr))) bad |= LPD_STATUS_NONFINITE;
        if (a.out_lt) a.out_lt[r] = static_cast<float>(xt - lse_t);
        if (a.out_lr) a.out_lr[r] = static_cast<float>(xr - lse_r);
        // entropy H = ln(s) - ln(2) * h / s of each side's softmax
        if (a.out_ent_t) a.out_ent_t[r] = static_cast<float>(log((double)row.st) - 0.6931471805599453 * (double)row.ht / row.st);
        if (a.out_ent_r) a.out_ent_r[r] = static_cast<float>(log((double)row.sr) - 0.6931471805599453 * (double)row.hr / row.sr);
        if (a.n_perm) {
            Acc pr = acc_init();
            for (int j = 0; j < a.n_perm; ++j) merge_acc(pr, seg[a.perm[j]], a.lg_t, a.lg_r);
            if (a.out_perm_lt) a.out_perm_lt[r] = static_cast<float>(xt - lse_train(pr, a.scale_t));
            if (a.out_perm_lr) a.out_perm_lr[r] = static_cast<float>(xr - lse_rollout(pr, a.scale_r));
        }
    }
    if (a.out_d) a.out_d[r] = static_cast<float>(d);
    a.dval[i] = d;
    a.keys[i] = __float_as_uint(fabsf(static_cast<float>(d)));
    if (bad) atomicOr(a.status, bad);
}

// ---------------------------------------------------------------- stage 3a
// Per-row metric terms of the Diagnostics table, reduced per block of 256
// active rows with a fixed tree: sum |d|, sum (exp(d) - 1 - d) evaluated as
// expm1(d) - d, sum expm1(d) (ratio0 mean = 1 + that / A), the count of
// ratio0 outside [lo, hi] (as d < ln lo or d > ln hi), and max |d| with the
// lowest row index among ties.  Also the first pass of the percentile select:
// the block's histogram of the keys' first digit (bits 30..20) in shared
// memory, added to the zeroed global one bin by bin (integer counts, so the
// order of the additions does not matter).
constexpr int kKeyShift0 = 20;

__global__ void __launch_bounds__(kFinThreads) terms_kernel(double ln_clip_lo, double ln_clip_hi,
                                                            const WsHeader *hdr, const int2 *rowid,
                                                            const double *dval, const uint32_t *keys,
                                                            BlockPartial *bp, uint32_t *hist) {
    __shared__ Part sh[kFinThreads];
    __shared__ uint32_t bh[kKeyHistBins];
    const int64_t n_active = hdr->n_active;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * kFinThreads + threadIdx.x;
    for (int b = threadIdx.x; b < kKeyHistBins; b += kFinThreads) bh[b] = 0;
    Part p = neutral_part();
    __syncthreads();
    if (i < n_active) {
        atomicAdd(&bh[(keys[i] >> kKeyShift0) & (kKeyHistBins - 1)], 1u);
        const double d = dval[i];
        const double em1 = expm1(d);
        p.sum_abs = fabs(d);
        p.sum_em1 = em1;
        p.sum_k3 = em1 - d;
        p.max_abs = fabs(d);
        p.argmax_row = rowid[i].x;
        p.n_clip = (d < ln_clip_lo || d > ln_clip_hi) ? 1 : 0;
    }
    sh[threadIdx.x] = p;
    __syncthreads();
    for (int b = threadIdx.x; b < kKeyHistBins; b += kFinThreads)
        if (bh[b]) atomicAdd(&hist[b], bh[b]);
    block_tree<kFinThreads>(sh);
    if (threadIdx.x == 0) {
        BlockPartial &o = bp[blockIdx.x];
        o.sum_abs = sh[0].sum_abs;
        o.sum_k3 = sh[0].sum_k3;
        o.sum_em1 = sh[0].sum_em1;
        o.max_abs = sh[0].max_abs;
        o.argmax_row = sh[0].argmax_row;
        o.n_clip = sh[0].n_clip;
    }
}

// ---------------------------------------------------------------- stage 3b
// One CTA: merge the finalise blocks' partials (thread tid < 256 folds blocks
// tid, tid+256, ... in order, then a fixed tree), then nearest-rank p95 and
// p99 of |dlogp| by a most-significant-digit radix select over the fp32 bit
// patterns of |dlogp| (monotone for non-negative floats; the sign bit is always
// 0), in three passes of 11, 10 and 10 bits, both ranks in the same passes.
// The first digit covers the exponent and four mantissa bits, so keys that
// share an order of magnitude still spread over several histogram bins; its
// histogram (one for both ranks) comes from the terms kernel's blocks, and
// this CTA reads the keys only for the two narrower passes.  The maximum comes
// exact from the partials.
constexpr int kSelBins = kKeyHistBins;
constexpr int kSelBatch = 8;

__global__ void __launch_bounds__(kSelThreads) metrics_kernel(int64_t n_blocks, const WsHeader *hdr,
                                                              const uint32_t *keys, const BlockPartial *bp,
                                                              const uint32_t *hist0, lpd_metrics *out) {
    constexpr int kFold = 256;  // threads that fold block partials
    __shared__ Part sh[kFold];
    __shared__ uint32_t hist[2][kSelBins];
    __shared__ uint32_t prefix[2];
    __shared__ long long rank[2];
    __shared__ uint32_t wsum[2][32];    // per-warp bin totals, then their exclusive scan
    __shared__ uint32_t sel_bin[2];     // the bin holding each rank in this pass
    __shared__ long long sel_rank[2];   // the rank within that bin
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n_active = hdr->n_active;

    Part p = neutral_part();
    for (int64_t b = tid; tid < kFold && b < n_blocks; b += kFold) {
        Part q;
        q.sum_abs = bp[b].sum_abs;
        q.sum_k3 = bp[b].sum_k3;
        q.sum_em1 = bp[b].sum_em1;
        q.max_abs = bp[b].max_abs;
        q.argmax_row = bp[b].argmax_row;
        q.n_clip = bp[b].n_clip;
        combine(p, q);
    }
    if (tid < kFold) sh[tid] = p;
    if (tid < 2) {
        prefix[tid] = 0;
        const long long pct = tid == 0 ? 95 : 99;
        rank[tid] = (pct * n_active + 99) / 100;  // ceil(p * A / 100), 1-based
    }
    __syncthreads();
    block_tree<kFold>(sh);

    if (n_active > 0) {
        const int shifts[3] = {kKeyShift0, 10, 0};
        const int widths[3] = {11, 10, 10};
        for (int pass = 0; pass < 3; ++pass) {
            const int shift = shifts[pass];
            const uint32_t dmask = (1u << widths[pass]) - 1u;
            const int nbins = 1 << widths[pass];
            const uint32_t hi_mask = pass == 0 ? 0u : (0xffffffffu << (shift + widths[pass]));
            if (pass == 0) {
                // the first digit's histogram, built by the terms kernel's
                // blocks (one histogram serves both ranks: empty prefix)
                for (int b = tid; b < kSelBins; b += kSelThreads) hist[0][b] = hist0[b];
                __syncthreads();
            } else {
                for (int b = tid; b < 2 * kSelBins; b += kSelThreads) (&hist[0][0])[b] = 0;
                __syncthreads();
            }
            const uint32_t p0 = prefix[0], p1 = prefix[1];
            // kSelBatch keys a thread in flight before their histogram updates
            const int64_t step = static_cast<int64_t>(kSelThreads) * kSelBatch;
            for (int64_t base = tid; pass > 0 && base < n_active; base += step) {
                uint32_t key[kSelBatch];
#pragma unroll
                for (int j = 0; j < kSelBatch; ++j) {
                    const int64_t i = base + static_cast<int64_t>(j) * kSelThreads;
                    key[j] = i < n_active ? keys[i] : 0u;
                }
#pragma unroll
                for (int j = 0; j < kSelBatch; ++j) {
                    if (base + static_cast<int64_t>(j) * kSelThreads >= n_active) break;
                    const uint32_t dig = (key[j] >> shift) & dmask;
                    if ((key[j] & hi_mask) == p0) atomicAdd(&hist[0][dig], 1u);
                    if ((key[j] & hi_mask) == p1) atomicAdd(&hist[1][dig], 1u);
                }
            }
            __syncthreads();
            // Both ranks' bins at once, over the whole block: thread t owns
            // bins [t per, (t + 1) per) of each histogram; counts are scanned
            // within warps by shuffles, then across the 32 warp totals.
            const int per = nbins / kSelThreads;
            uint32_t tot[2], incl[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t *h = hist[pass == 0 ? 0 : r];
                tot[r] = 0;
                for (int b = 0; b < per; ++b) tot[r] += h[tid * per + b];
                incl[r] = tot[r];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl[r], off);
                    if (lane >= off) incl[r] += y;
                }
                if (lane == 31) wsum[r][warp] = incl[r];
            }
            __syncthreads();
            if (warp < 2) {
                // exclusive scan of warp `warp`'s rank over the 32 warp totals
                const uint32_t t = wsum[warp][lane];
                uint32_t x = t;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                wsum[warp][lane] = x - t;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t *h = hist[pass == 0 ? 0 : r];
                const long long k = rank[r];
                const long long before = static_cast<long long>(wsum[r][warp]) + (incl[r] - tot[r]);
                if (before < k && k <= before + static_cast<long long>(tot[r])) {
                    long long acc = before;
                    for (int b = 0; b < per; ++b) {
                        const uint32_t c = h[tid * per + b];
                        if (acc + c >= k) {
                            sel_bin[r] = static_cast<uint32_t>(tid * per + b);
                            sel_rank[r] = k - acc;
                            break;
                        }
                        acc += c;
                    }
                }
            }
            __syncthreads();
            if (tid < 2) {
                prefix[tid] |= sel_bin[tid] << shift;
                rank[tid] = sel_rank[tid];
            }
            __syncthreads();
        }
    }

    if (tid == 0) {
        const Part &t = sh[0];
        out->n_active = n_active;
        if (n_active > 0) {
            const double A = static_cast<double>(n_active);
            out->argmax_row = t.argmax_row;
            out->flags = 0u;
            out->ratio0_mean = 1.0 + t.sum_em1 / A;
            out->clipfrac0 = static_cast<double>(t.n_clip) / A;
            out->approx_kl0 = t.sum_k3 / A;
            out->mean_abs_dlogp = t.sum_abs / A;
            out->p95_abs_dlogp = static_cast<double>(__uint_as_float(prefix[0]));
            out->p99_abs_dlogp = static_cast<double>(__uint_as_float(prefix[1]));
            out->max_abs_dlogp = t.max_abs;
        } else {
            out->argmax_row = -1;
            out->flags = LPD_FLAG_NO_ACTIVE;
            out->ratio0_mean = out->clipfrac0 = out->approx_kl0 = out->mean_abs_dlogp = 0.0;
            out->p95_abs_dlogp = out->p99_abs_dlogp = out->max_abs_dlogp = 0.0;
        }
    }
}

}  // namespace

cudaError_t launch_select_active(int64_t n_rows, const uint8_t *mask, const int32_t *ids, float *out_lt,
                                 float *out_lr, float *out_d, lpd_metrics *metrics, WsHeader *hdr,
                                 int2 *rowid, cudaStream_t stream) {
    const int64_t blocks = (n_rows + kSelBlockRows - 1) / kSelBlockRows;
    if (blocks < 2 || blocks > kSelMaxBlocks) {
        select_active_kernel<<<1, 1024, 0, stream>>>(n_rows, mask, ids, out_lt, out_lr, out_d, metrics, hdr, rowid);
        return cudaGetLastError();
    }
    count_active_kernel<<<static_cast<unsigned>(blocks), kSelBlockThreads, 0, stream>>>(n_rows, mask, hdr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    compact_active_kernel<<<static_cast<unsigned>(blocks), kSelBlockThreads, 0, stream>>>(
        n_rows, mask, ids, out_lt, out_lr, out_d, metrics, hdr, rowid);
    return cudaGetLastError();
}

cudaError_t launch_dlogp_rows(int64_t n_rows, const float *dlogp, const WsHeader *hdr, const int2 *rowid,
                              double *dval, uint32_t *keys, uint32_t *status, cudaStream_t stream) {
    const int64_t blocks = (n_rows + kFinThreads - 1) / kFinThreads;
    if (blocks == 0) return cudaSuccess;
    dlogp_rows_kernel<<<static_cast<unsigned>(blocks), kFinThreads, 0, stream>>>(dlogp, hdr, rowid, dval, keys,
                                                                                 status);
    return cudaGetLastError();
}

cudaError_t launch_finalize(const FinArgs &a, int64_t n_rows, cudaStream_t stream) {
    const int64_t blocks = (n_rows + kFinalizeThreads - 1) / kFinalizeThreads;
    if (blocks == 0) return cudaSuccess;
    finalize_kernel<<<static_cast<unsigned>(blocks), kFinalizeThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_metrics(int64_t n_rows, double ln_clip_lo, double ln_clip_hi, const WsHeader *hdr,
                           const int2 *rowid, const double *dval, const uint32_t *keys, BlockPartial *bp,
                           uint32_t *hist, lpd_metrics *metrics, cudaStream_t stream) {
    const int64_t blocks = (n_rows + kFinThreads - 1) / kFinThreads;
    if (blocks > 0) {
        cudaError_t e = cudaMemsetAsync(hist, 0, kKeyHistBins * sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
        terms_kernel<<<static_cast<unsigned>(blocks), kFinThreads, 0, stream>>>(ln_clip_lo, ln_clip_hi, hdr,
                                                                               rowid, dval, keys, bp, hist);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    metrics_kernel<<<1, kSelThreads, 0, stream>>>(blocks, hdr, keys, bp, hist, metrics);
    return cudaGetLastError();
}

}  // namespace lpd
