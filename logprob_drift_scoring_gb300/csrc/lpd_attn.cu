// Split-KV / context-parallel attention (out, lse) merge and its merge-order
// diagnostic.
//
// Method: "Attention Debug Matrix", row A7 (merge_order), and "[WS2] Framework
// for ablation experiment", Attention knobs table, rows 6-7.  Part k holds,
// for every query row r, the attention output over one key block, normalised
// within the block, and that block's log-sum-exp.  The merged row is
//   lse = log(sum_k exp(lse_k)),  out = sum_k exp(lse_k - lse) out_k,
// folded one part at a time in a caller-given order (the A7 knob).
//
// Layout: the merge streams K * n_rows * head_dim values once and writes one
// n_rows * head_dim result, so it is bound by HBM.  Each thread owns one or
// two adjacent 16-byte chunks of one row (4 or 8 f32 columns, 8 or 16 bf16),
// so the per-part scalar work of the fold is shared by them; a block of 128 threads
// copies the lse values of the rows it touches, then the chunks of every part
// whose lse is finite (a causal split leaves many (row, part) pairs without
// keys), into shared memory with cp.async (every copy of a thread in flight at
// once, no registers held); each thread then folds its chunk over the parts in
// the requested order straight from shared memory.  The order-drift diagnostic
// folds the same staged data a second time in the other order, so it reads
// HBM no more than the plain merge does.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"

namespace lpd {
namespace {

constexpr int kMergeThreads = 128;
constexpr int kMaxParts = LPD_ATTN_MAX_PARTS;
constexpr int kSmallParts = 8;  // part counts up to this run fully unrolled

// A thread's unit is kV adjacent 16-byte chunks of one row (merge_kv picks kV).
struct MergeArgs {
    const char *parts;       // [K][n][d] as 16-byte chunks
    const float *lse;        // [K][n]
    float *out;              // [n][d]
    float *out_lse;          // [n]
    unsigned *row_dout;      // [n], float bits, zeroed by the caller (drift only)
    float *row_dlse;         // [n] (drift only)
    int64_t n;               // rows
    int64_t part_bytes;      // bytes of one part
    uint32_t units;          // units per part = n * cpr / kV (below 2^32, checked by the caller)
    uint32_t upr;            // units per row
    int upr_shift;           // log2(upr) when upr is a power of two, else -1
    int n_parts;
    int nr_max;              // bound on the rows one block touches
    int base2;
    int row_in_warp;         // upr divides 32: a row's units are lanes of one warp
    uint8_t order_a[kMaxParts], order_b[kMaxParts];
    uint8_t slot_b[kSmallParts];  // staging slot (order-A visit position) of order B's k-th part
    int64_t off_a[kSmallParts];  // order_a[k] * part_bytes for the first parts
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(dst))),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<unsigned>(__cvta_generic_to_shared(dst))),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <bool kBf16>
__device__ __forceinline__ void unpack(const uint4 w, float *v) {
    if constexpr (kBf16) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(ws[q] << 16);
            v[2 * q + 1] = __uint_as_float(ws[q] & 0xffff0000u);
        }
    } else {
        v[0] = __uint_as_float(w.x);
        v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z);
        v[3] = __uint_as_float(w.w);
    }
}

// Staged shared memory of one block: chunk_s[(k * kV + v) * 128 + t] holds
// chunk v of thread t's unit in slot k (consecutive threads, consecutive 16
// bytes: no bank conflicts).  Slot k is part k, except in the plain merge of
// up to kSmallParts parts, where it is the k-th part visited.  lse_s[rr *
// kMaxK + k] is the lse of the block's row rr in part k; ord_s holds both
// orders (the looped kMaxK = 64 form only).
template <int kV, int kMaxK>
struct Staged {
    const uint4 *chunk_s;
    const float *lse_s;
    const uint8_t *ord_s;
};

// Part visited k-th in order A (kB false) or B.  The unrolled form (every k a
// constant) reads the order straight from the kernel parameters.
template <int kMaxK, bool kB>
__device__ __forceinline__ int order_at(const MergeArgs &a, const uint8_t *ord_s, int k) {
    if constexpr (kMaxK <= kSmallParts)
        return kB ? a.order_b[k] : a.order_a[k];
    else
        return ord_s[(kB ? kMaxParts : 0) + k];
}

// Running state of one unit's fold: max m, sum s of exp(lse_k - m) and the
// unnormalised accumulator acc.  A part above the running max rescales the
// state instead of being scaled itself.  cvt converts an lse difference to
// base 2 for ex2.
template <int N>
struct FoldState {
    float m, s, acc[N];
};

template <int N>
__device__ __forceinline__ void fold_init(FoldState<N> &f) {
    f.m = -CUDART_INF_F;
    f.s = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e) f.acc[e] = 0.f;
}

template <int N>
__device__ __forceinline__ void fold_step(FoldState<N> &f, float l, const float *v, float cvt) {
    if (l > f.m) {
        const float sc = ex2(__fmul_rn(__fsub_rn(f.m, l), cvt));  // 0 while m is still -inf
        f.s = __fmaf_rn(f.s, sc, 1.f);
#pragma unroll
        for (int e = 0; e < N; ++e) f.acc[e] = __fmaf_rn(f.acc[e], sc, v[e]);
        f.m = l;
    } else {
        const float w = ex2(__fmul_rn(__fsub_rn(l, f.m), cvt));
        f.s = __fadd_rn(f.s, w);
#pragma unroll
        for (int e = 0; e < N; ++e) f.acc[e] = __fmaf_rn(w, v[e], f.acc[e]);
    }
}

// out = acc / s and (only where asked: the row's first unit) lse = m + log s;
// a unit no part saw gives out 0 and lse -inf.
template <int N>
__device__ __forceinline__ void fold_finish(const FoldState<N> &f, bool want_lse, bool base2, float *o, float &lse) {
    if (f.s > 0.f) {
        const float inv = __frcp_rn(f.s);
#pragma unroll
        for (int e = 0; e < N; ++e) o[e] = __fmul_rn(f.acc[e], inv);
        if (want_lse) lse = __fadd_rn(f.m, base2 ? log2f(f.s) : logf(f.s));
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e) o[e] = 0.f;
        lse = -CUDART_INF_F;
    }
}

// One unit folded over the parts in order A or B, chunks staged by part index.
// A part with lse = -inf is skipped.
template <bool kBf16, int kV, int kMaxK, bool kB>
__device__ __forceinline__ void fold(const MergeArgs &a, const Staged<kV, kMaxK> &st, int K, int t, int rl, float cvt,
                                     bool want_lse, float *o, float &lse) {
    constexpr int E = kBf16 ? 8 : 4;
    FoldState<kV * E> f;
    fold_init(f);
#pragma unroll(kMaxK <= kSmallParts ? kMaxK : 1)
    for (int k = 0; k < kMaxK; ++k) {
        if (k >= K) break;
        const int p = order_at<kMaxK, kB>(a, st.ord_s, k);
        const float l = st.lse_s[rl * kMaxK + p];
        if (l == -CUDART_INF_F) continue;
        float v[kV * E];
#pragma unroll
        for (int u = 0; u < kV; ++u) unpack<kBf16>(st.chunk_s[(p * kV + u) * kMergeThreads + t], v + u * E);
        fold_step(f, l, v, cvt);
    }
    fold_finish(f, want_lse, a.base2, o, lse);
}

// Merges of up to kSmallParts parts with one chunk per thread: the row's lse
// values sit in registers in visiting order and chunk k of order A's visit is
// staged in slot k.  Order A folds slot k at step k; order B (the drift
// form's second fold) folds slot slot_b[k], a kernel parameter.
template <bool kBf16, bool kB>
__device__ __forceinline__ void fold_seq(const MergeArgs &a, const float (&l)[kSmallParts], const uint4 *chunk_s,
                                         int t, float cvt, bool want_lse, float *o, float &lse) {
    constexpr int E = kBf16 ? 8 : 4;
    FoldState<E> f;
    fold_init(f);
#pragma unroll
    for (int k = 0; k < kSmallParts; ++k) {
        if (l[k] == -CUDART_INF_F) continue;  // also every k >= K
        float v[E];
        unpack<kBf16>(chunk_s[(kB ? a.slot_b[k] : k) * kMergeThreads + t], v);
        fold_step(f, l[k], v, cvt);
    }
    fold_finish(f, want_lse, a.base2, o, lse);
}

// Row of a unit index: a shift for the usual power-of-two head sizes.
__device__ __forceinline__ uint32_t unit_row(const MergeArgs &a, uint32_t u) {
    return a.upr_shift >= 0 ? u >> a.upr_shift : u / a.upr;
}

// A tile is 128 consecutive units: the rows [r0, r0 + nr) it touches.
struct Tile {
    uint32_t u0, r0;
    int nr;
};

__device__ __forceinline__ Tile tile_at(const MergeArgs &a, uint32_t tile) {
    Tile g;
    g.u0 = tile * static_cast<uint32_t>(kMergeThreads);
    g.r0 = unit_row(a, g.u0);
    const uint32_t u_last = (a.units - g.u0 > static_cast<uint32_t>(kMergeThreads) ? g.u0 + kMergeThreads : a.units) - 1;
    g.nr = static_cast<int>(unit_row(a, u_last) - g.r0 + 1);
    return g;
}

// Copy the lse of every part for the tile's rows into lse_s[rr * kMaxK + k].
template <int kMaxK>
__device__ __forceinline__ void stage_lse(const MergeArgs &a, const Tile &g, float *lse_s, int t, int K) {
    for (int rr = t; rr < g.nr; rr += kMergeThreads) {
#pragma unroll(kMaxK <= kSmallParts ? kMaxK : 1)
        for (int k = 0; k < kMaxK; ++k) {
            if (k >= K) break;
            cp_async4(lse_s + rr * kMaxK + k, a.lse + static_cast<int64_t>(k) * a.n + g.r0 + rr);
        }
    }
}

// Persistent blocks walk tiles blockIdx.x, blockIdx.x + gridDim.x, ...  The
// lse of a block's next tile is copied while the current tile's chunks are in
// flight, so each tile costs one memory round trip, not two.
template <bool kBf16, bool kDrift, int kV, int kMaxK>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeArgs a) {
    constexpr int E = kBf16 ? 8 : 4;
    // few parts, one chunk per thread: visiting orders fixed per launch, lse in registers
    constexpr bool kSeq = kMaxK <= kSmallParts && kV == 1;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = a.n_parts;
    const int lse_stride = a.nr_max * kMaxK;
    uint4 *chunk_s = reinterpret_cast<uint4 *>(smem);
    float *lse_s = reinterpret_cast<float *>(smem + static_cast<size_t>(K) * kV * kMergeThreads * 16);  // [2][lse_stride]
    unsigned *rowmax_s = reinterpret_cast<unsigned *>(lse_s + 2 * lse_stride);
    uint8_t *ord_s = reinterpret_cast<uint8_t *>(rowmax_s + a.nr_max);

    const int t = threadIdx.x;
    const uint32_t n_tiles = static_cast<uint32_t>((static_cast<uint64_t>(a.units) + kMergeThreads - 1) / kMergeThreads);
    uint32_t tile = blockIdx.x;
    if (tile >= n_tiles) return;  // whole block
    if constexpr (kMaxK > kSmallParts) {
        if (t < K) {
            ord_s[t] = a.order_a[t];
            if (kDrift) ord_s[kMaxParts + t] = a.order_b[t];
        }
    }
    Tile g = tile_at(a, tile);
    stage_lse<kMaxK>(a, g, lse_s, t, K);
    cp_async_wait_all();
    __syncthreads();

    const float cvt = a.base2 ? 1.f : kLog2e;
    int buf = 0;
    for (;;) {
        const float *lcur = lse_s + buf * lse_stride;
        const uint32_t u = g.u0 + t;
        const bool live = u < a.units;
        const uint32_t row = unit_row(a, u);
        const int rl = static_cast<int>(row - g.r0);
        // a part with lse = -inf saw no keys for this row: its chunks are never copied
        const char *src = a.parts + static_cast<int64_t>(u) * (16 * kV);
        float lseq[kSmallParts], lseq_b[kSmallParts];  // kSeq: the row's lse in each visiting order
        if constexpr (kSeq) {
#pragma unroll
            for (int k = 0; k < kSmallParts; ++k) {
                lseq[k] = (live && k < K) ? lcur[rl * kMaxK + a.order_a[k]] : -CUDART_INF_F;
                if (kDrift) lseq_b[k] = (live && k < K) ? lcur[rl * kMaxK + a.order_b[k]] : -CUDART_INF_F;
                if (lseq[k] != -CUDART_INF_F) cp_async16(chunk_s + k * kMergeThreads + t, src + a.off_a[k]);
            }
        } else if (live) {
#pragma unroll(kMaxK <= kSmallParts ? kMaxK : 1)
            for (int k = 0; k < kMaxK; ++k) {
                if (k >= K) break;
                if (lcur[rl * kMaxK + k] != -CUDART_INF_F) {
#pragma unroll
                    for (int v = 0; v < kV; ++v)
                        cp_async16(chunk_s + (k * kV + v) * kMergeThreads + t, src + k * a.part_bytes + 16 * v);
                }
            }
        }
        const uint32_t next = tile + gridDim.x;
        const bool more = next < n_tiles;
        Tile gn = g;
        if (more) {
            gn = tile_at(a, next);
            stage_lse<kMaxK>(a, gn, lse_s + (buf ^ 1) * lse_stride, t, K);
        }
        if (kDrift && !a.row_in_warp)
            for (int i = t; i < g.nr; i += kMergeThreads) rowmax_s[i] = 0u;
        cp_async_wait_all();
        __syncthreads();  // the next tile's lse and the zeroed row maxima are visible

        const Staged<kV, kMaxK> st{chunk_s, lcur, ord_s};
        const bool head = live && row * a.upr == u;  // first unit of its row
        float oa[kV * E], la = 0.f;
        if (live) {
            if constexpr (kSeq)
                fold_seq<kBf16, false>(a, lseq, chunk_s, t, cvt, head, oa, la);
            else
                fold<kBf16, kV, kMaxK, false>(a, st, K, t, rl, cvt, head, oa, la);
            float4 *dst = reinterpret_cast<float4 *>(a.out + static_cast<int64_t>(u) * (kV * E));
#pragma unroll
            for (int q = 0; q < kV * E / 4; ++q)
                dst[q] = make_float4(oa[4 * q], oa[4 * q + 1], oa[4 * q + 2], oa[4 * q + 3]);
            if (head) a.out_lse[row] = la;
        }
        if constexpr (kDrift) {
            float dmax = 0.f;
            if (live) {
                float ob[kV * E], lb;
                if constexpr (kSeq)
                    fold_seq<kBf16, true>(a, lseq_b, chunk_s, t, cvt, head, ob, lb);
                else
                    fold<kBf16, kV, kMaxK, true>(a, st, K, t, rl, cvt, head, ob, lb);
#pragma unroll
                for (int e = 0; e < kV * E; ++e) {
                    const float d = oa[e] == ob[e] ? 0.f : fabsf(__fsub_rn(oa[e], ob[e]));
                    dmax = (d > dmax || d != d) ? d : dmax;  // NaN wins
                }
                if (head) a.row_dlse[row] = la == lb ? 0.f : fabsf(__fsub_rn(la, lb));
            }
            if (a.row_in_warp) {
                // the row's units are the aligned group of upr lanes: reduce
                // there (float bits of non-negative values and NaN order like
                // the numbers, NaN above all) and let the row's first lane write
                for (uint32_t off = 1; off < a.upr; off <<= 1) {
                    const float o = __shfl_xor_sync(0xffffffffu, dmax, off);
                    dmax = (o > dmax || o != o) ? o : dmax;
                }
                if (head) a.row_dout[row] = __float_as_uint(dmax);
            } else {
                if (live) atomicMax(rowmax_s + rl, __float_as_uint(dmax));
                __syncthreads();
                for (int i = t; i < g.nr; i += kMergeThreads) atomicMax(a.row_dout + g.r0 + i, rowmax_s[i]);
            }
        }
        if (!more) break;
        __syncthreads();  // every thread is done with this tile's lse buffer before it is refilled
        tile = next;
        g = gn;
        buf ^= 1;
    }
}

// Maximum and lowest arg-max row of the two per-row drift columns.  Keys pack
// the non-negative float's bits above (2^32 - 1 - row), so one unsigned
// 64-bit max gives both, whatever order the blocks finish in.
constexpr int kReduceThreads = 256;

__global__ void __launch_bounds__(kReduceThreads) drift_reduce_kernel(const float *row_dout, const float *row_dlse,
                                                                      int64_t n, unsigned long long *keys) {
    unsigned long long ko = 0, kl = 0;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x; r < n;
         r += static_cast<int64_t>(gridDim.x) * kReduceThreads) {
        const unsigned long long lo = 0xffffffffull - static_cast<unsigned long long>(r);
        const unsigned long long a = (static_cast<unsigned long long>(__float_as_uint(row_dout[r])) << 32) | lo;
        const unsigned long long b = (static_cast<unsigned long long>(__float_as_uint(row_dlse[r])) << 32) | lo;
        ko = a > ko ? a : ko;
        kl = b > kl ? b : kl;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, ko, off);
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, kl, off);
        ko = x > ko ? x : ko;
        kl = y > kl ? y : kl;
    }
    __shared__ unsigned long long wo[kReduceThreads / 32], wl[kReduceThreads / 32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) {
        wo[warp] = ko;
        wl[warp] = kl;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kReduceThreads / 32; ++w) {
            ko = wo[w] > ko ? wo[w] : ko;
            kl = wl[w] > kl ? wl[w] : kl;
        }
        atomicMax(keys, ko);
        atomicMax(keys + 1, kl);
    }
}

__global__ void drift_finalize_kernel(lpd_merge_drift *d, int64_t n) {
    if (threadIdx.x != 0) return;
    const unsigned long long ko = d->scratch[0], kl = d->scratch[1];
    if (n == 0) {
        d->max_abs_dout = 0.0;
        d->max_abs_dlse = 0.0;
        d->row_dout = -1;
        d->row_dlse = -1;
        return;
    }
    d->max_abs_dout = static_cast<double>(__uint_as_float(static_cast<unsigned>(ko >> 32)));
    d->max_abs_dlse = static_cast<double>(__uint_as_float(static_cast<unsigned>(kl >> 32)));
    d->row_dout = static_cast<int64_t>(0xffffffffull - (ko & 0xffffffffull));
    d->row_dlse = static_cast<int64_t>(0xffffffffull - (kl & 0xffffffffull));
}

// Plain merge: a persistent grid, as many blocks as fit on every SM at once,
// each walking tiles blockIdx.x, blockIdx.x + gridDim.x, ...  Order drift:
// one block per tile.
template <bool kBf16, bool kDrift, int kV, int kMaxK>
cudaError_t launch_merge(const MergeArgs &a, size_t smem, cudaStream_t stream) {
    auto *fn = merge_kernel<kBf16, kDrift, kV, kMaxK>;
    static std::atomic<uint64_t> raised{0};
    cudaError_t e;
    if (smem > 48 * 1024 && (e = set_smem_max_once(fn, raised)) != cudaSuccess) return e;
    const int64_t tiles = (static_cast<int64_t>(a.units) + kMergeThreads - 1) / kMergeThreads;
    int64_t grid = tiles;
    if (!kDrift) {
        // the drift form's second fold and extra barriers leave each block's
        // memory idle for longer: one block per tile keeps more copies in flight
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kMergeThreads, smem)) != cudaSuccess)
            return e;
        const int64_t resident = static_cast<int64_t>(device_sm_count()) * (per_sm > 0 ? per_sm : 1);
        grid = tiles < resident ? tiles : resident;
    }
    fn<<<static_cast<unsigned>(grid), kMergeThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <bool kBf16, bool kDrift>
cudaError_t launch_merge_shape(const MergeArgs &a, int kv, size_t smem, cudaStream_t stream) {
    if (a.n_parts <= kSmallParts) return launch_merge<kBf16, kDrift, 1, kSmallParts>(a, smem, stream);  // kv is 1
    return kv == 2 ? launch_merge<kBf16, kDrift, 2, kMaxParts>(a, smem, stream)
                   : launch_merge<kBf16, kDrift, 1, kMaxParts>(a, smem, stream);
}

// Chunks per thread: one up to kSmallParts parts (more resident blocks beat
// sharing the per-part scalar work between two chunks, in the plain merge and
// in the order-drift form alike: measured); beyond, two when a row has an even
// number of chunks and the staging of up to 32 parts fits.
int merge_kv(int n_parts, int cpr) {
    if (n_parts <= kSmallParts) return 1;
    return (cpr % 2 == 0 && n_parts <= 32) ? 2 : 1;
}

size_t attn_merge_smem(int n_parts, int cpr) {
    const int kv = merge_kv(n_parts, cpr);
    const int max_k = n_parts <= kSmallParts ? kSmallParts : kMaxParts;
    const int nr_max = kMergeThreads / (cpr / kv) + 2;
    return static_cast<size_t>(n_parts) * kv * kMergeThreads * 16 + 2 * static_cast<size_t>(nr_max) * max_k * 4 +
           static_cast<size_t>(nr_max) * 4 + 2 * kMaxParts;
}

}  // namespace

cudaError_t launch_attn_merge(const AttnMergeCall &c, cudaStream_t stream) {
    const int es = c.bf16 ? 2 : 4;
    const int cpr = static_cast<int>(static_cast<int64_t>(c.head_dim) * es / 16);
    const bool drift = c.diag;
    const int kv = merge_kv(c.n_parts, cpr);
    const int upr = cpr / kv;
    // a row's units fill an aligned group of lanes: its drift maximum is a
    // warp reduction written once, otherwise atomics into zeroed memory
    const bool row_in_warp = upr <= 32 && 32 % upr == 0;
    if (drift) {
        cudaError_t e = cudaMemsetAsync(c.drift, 0, sizeof(lpd_merge_drift), stream);
        if (e == cudaSuccess && c.n_rows > 0 && !row_in_warp)
            e = cudaMemsetAsync(c.row_dout, 0, c.n_rows * sizeof(float), stream);
        if (e != cudaSuccess) return e;
    }
    if (c.n_rows > 0) {
        MergeArgs a{};
        a.parts = static_cast<const char *>(c.parts);
        a.lse = c.lse;
        a.out = c.out;
        a.out_lse = c.out_lse;
        a.row_dout = reinterpret_cast<unsigned *>(c.row_dout);
        a.row_dlse = c.row_dlse;
        a.n = c.n_rows;
        a.part_bytes = c.n_rows * cpr * 16;
        a.units = static_cast<uint32_t>(c.n_rows * upr);
        a.upr = static_cast<uint32_t>(upr);
        a.upr_shift = (upr & (upr - 1)) == 0 ? __builtin_ctz(static_cast<unsigned>(upr)) : -1;
        a.n_parts = c.n_parts;
        a.nr_max = kMergeThreads / upr + 2;
        a.base2 = c.base2;
        a.row_in_warp = row_in_warp ? 1 : 0;
        int pos_a[kMaxParts] = {};
        for (int k = 0; k < c.n_parts; ++k) {
            a.order_a[k] = static_cast<uint8_t>(c.order_a[k]);
            a.order_b[k] = static_cast<uint8_t>(drift ? c.order_b[k] : c.order_a[k]);
            pos_a[c.order_a[k]] = k;
            if (k < kSmallParts) a.off_a[k] = static_cast<int64_t>(c.order_a[k]) * a.part_bytes;
        }
        for (int k = 0; k < c.n_parts && k < kSmallParts; ++k) a.slot_b[k] = static_cast<uint8_t>(pos_a[a.order_b[k]]);
        const size_t smem = attn_merge_smem(c.n_parts, cpr);
        cudaError_t e;
        if (c.bf16)
            e = drift ? launch_merge_shape<true, true>(a, kv, smem, stream)
                      : launch_merge_shape<true, false>(a, kv, smem, stream);
        else
            e = drift ? launch_merge_shape<false, true>(a, kv, smem, stream)
                      : launch_merge_shape<false, false>(a, kv, smem, stream);
        if (e != cudaSuccess) return e;
        if (drift) {
            const int64_t want = (c.n_rows + kReduceThreads - 1) / kReduceThreads;
            const int64_t cap = static_cast<int64_t>(device_sm_count()) * 2;
            drift_reduce_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kReduceThreads, 0, stream>>>(
                c.row_dout, c.row_dlse, c.n_rows, reinterpret_cast<unsigned long long *>(c.drift->scratch));
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    if (drift) {
        drift_finalize_kernel<<<1, 32, 0, stream>>>(c.drift, c.n_rows);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace lpd
