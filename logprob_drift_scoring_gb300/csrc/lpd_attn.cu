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
// n_rows * head_dim result, so it is bound by HBM.  Each thread owns one
// 16-byte chunk of one row (4 f32 or 8 bf16 columns); a block of 128 threads
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

struct MergeArgs {
    const char *parts;       // [K][n][d] chunks of 16 bytes
    const float *lse;        // [K][n]
    float *out;              // [n][d]
    float *out_lse;          // [n]
    unsigned *row_dout;      // [n], float bits, zeroed by the caller (drift only)
    float *row_dlse;         // [n] (drift only)
    int64_t n;               // rows
    int64_t total;           // chunks per part = n * cpr
    int cpr;                 // 16-byte chunks per row
    int n_parts;
    int nr_max;              // bound on the rows one block touches
    int base2;
    uint8_t order_a[kMaxParts], order_b[kMaxParts];
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
__device__ __forceinline__ void unpack(const uint4 w, float (&v)[kBf16 ? 8 : 4]) {
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

// One row chunk folded over the parts in `ord`: running max m, running sum s
// of exp(lse_k - m), unnormalised accumulator acc; a part above the running
// max rescales the state instead of being scaled itself.  A part with
// lse = -inf is skipped.  c converts an lse difference to base 2 for ex2.
template <bool kBf16>
__device__ __forceinline__ void fold(const uint4 *chunk_s, const float *lse_s, int nr_max, const uint8_t *ord, int K,
                                     int t, int rl, float c, bool base2, float (&o)[kBf16 ? 8 : 4], float &lse) {
    constexpr int E = kBf16 ? 8 : 4;
    float m = -CUDART_INF_F, s = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int k = 0; k < K; ++k) {
        const int p = ord[k];
        const float l = lse_s[p * nr_max + rl];
        if (l == -CUDART_INF_F) continue;
        float v[E];
        unpack<kBf16>(chunk_s[p * kMergeThreads + t], v);
        if (l > m) {
            const float sc = ex2(__fmul_rn(__fsub_rn(m, l), c));  // 0 while m is still -inf
            s = __fmaf_rn(s, sc, 1.f);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(acc[e], sc, v[e]);
            m = l;
        } else {
            const float w = ex2(__fmul_rn(__fsub_rn(l, m), c));
            s = __fadd_rn(s, w);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = __fmaf_rn(w, v[e], acc[e]);
        }
    }
    if (s > 0.f) {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = __fdiv_rn(acc[e], s);
        lse = __fadd_rn(m, base2 ? log2f(s) : logf(s));
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = 0.f;
        lse = -CUDART_INF_F;
    }
}

template <bool kBf16, bool kDrift>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeArgs a) {
    constexpr int E = kBf16 ? 8 : 4;
    extern __shared__ __align__(16) unsigned char smem[];
    const int K = a.n_parts;
    uint4 *chunk_s = reinterpret_cast<uint4 *>(smem);                                   // [K][128]
    float *lse_s = reinterpret_cast<float *>(smem + static_cast<size_t>(K) * kMergeThreads * 16);  // [K][nr_max]
    unsigned *rowmax_s = reinterpret_cast<unsigned *>(lse_s + K * a.nr_max);           // [nr_max]
    uint8_t *ord_s = reinterpret_cast<uint8_t *>(rowmax_s + a.nr_max);                  // [2][kMaxParts]

    const int t = threadIdx.x;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kMergeThreads;
    const int64_t c = c0 + t;
    const bool live = c < a.total;
    const int64_t r0 = c0 / a.cpr;
    const int64_t c_end = c0 + kMergeThreads < a.total ? c0 + kMergeThreads : a.total;
    const int nr = static_cast<int>((c_end - 1) / a.cpr - r0 + 1);

    // lse of the rows this block touches first: a part with lse = -inf saw no
    // keys for that row, and its chunk is never copied
    for (int i = t; i < K * nr; i += kMergeThreads) {
        const int k = i / nr, rr = i - k * nr;
        cp_async4(lse_s + k * a.nr_max + rr, a.lse + k * a.n + r0 + rr);
    }
    if (t < K) {
        ord_s[t] = a.order_a[t];
        if (kDrift) ord_s[kMaxParts + t] = a.order_b[t];
    }
    if (kDrift)
        for (int i = t; i < nr; i += kMergeThreads) rowmax_s[i] = 0u;
    cp_async_wait_all();
    __syncthreads();

    const int64_t row = c / a.cpr;
    const int rl = static_cast<int>(row - r0);
    if (live) {
        const char *src = a.parts + c * 16;
        const int64_t part_bytes = a.total * 16;
        for (int k = 0; k < K; ++k)
            if (lse_s[k * a.nr_max + rl] != -CUDART_INF_F)
                cp_async16(chunk_s + k * kMergeThreads + t, src + k * part_bytes);
        cp_async_wait_all();  // each thread reads back only its own chunks
    }

    const float cvt = a.base2 ? 1.f : kLog2e;
    const bool head = live && row * a.cpr == c;  // first chunk of its row
    float oa[E], la = 0.f;
    if (live) {
        fold<kBf16>(chunk_s, lse_s, a.nr_max, ord_s, K, t, rl, cvt, a.base2, oa, la);
        float4 *dst = reinterpret_cast<float4 *>(a.out + c * E);
        dst[0] = make_float4(oa[0], oa[1], oa[2], oa[3]);
        if constexpr (kBf16) dst[1] = make_float4(oa[4], oa[5], oa[6], oa[7]);
        if (head) a.out_lse[row] = la;
    }
    if constexpr (kDrift) {
        if (live) {
            float ob[E], lb;
            fold<kBf16>(chunk_s, lse_s, a.nr_max, ord_s + kMaxParts, K, t, rl, cvt, a.base2, ob, lb);
            float dmax = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float d = oa[e] == ob[e] ? 0.f : fabsf(__fsub_rn(oa[e], ob[e]));
                dmax = (d > dmax || d != d) ? d : dmax;  // NaN wins
            }
            atomicMax(rowmax_s + rl, __float_as_uint(dmax));
            if (head) a.row_dlse[row] = la == lb ? 0.f : fabsf(__fsub_rn(la, lb));
        }
        __syncthreads();
        for (int i = t; i < nr; i += kMergeThreads) atomicMax(a.row_dout + r0 + i, rowmax_s[i]);
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

template <bool kBf16, bool kDrift>
cudaError_t launch_merge(const MergeArgs &a, size_t smem, unsigned blocks, cudaStream_t stream) {
    auto *fn = merge_kernel<kBf16, kDrift>;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    fn<<<blocks, kMergeThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

size_t attn_merge_smem(int n_parts, int cpr) {
    const int nr_max = kMergeThreads / cpr + 2;
    return static_cast<size_t>(n_parts) * kMergeThreads * 16 + static_cast<size_t>(n_parts) * nr_max * 4 +
           static_cast<size_t>(nr_max) * 4 + 2 * kMaxParts;
}

cudaError_t launch_attn_merge(const AttnMergeCall &c, cudaStream_t stream) {
    const int es = c.bf16 ? 2 : 4;
    const int cpr = static_cast<int>(static_cast<int64_t>(c.head_dim) * es / 16);
    const bool drift = c.diag;
    if (drift) {
        cudaError_t e = cudaMemsetAsync(c.drift, 0, sizeof(lpd_merge_drift), stream);
        if (e == cudaSuccess && c.n_rows > 0) e = cudaMemsetAsync(c.row_dout, 0, c.n_rows * sizeof(float), stream);
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
        a.total = c.n_rows * cpr;
        a.cpr = cpr;
        a.n_parts = c.n_parts;
        a.nr_max = kMergeThreads / cpr + 2;
        a.base2 = c.base2;
        for (int k = 0; k < c.n_parts; ++k) {
            a.order_a[k] = static_cast<uint8_t>(c.order_a[k]);
            a.order_b[k] = static_cast<uint8_t>(drift ? c.order_b[k] : c.order_a[k]);
        }
        const size_t smem = attn_merge_smem(c.n_parts, cpr);
        const unsigned blocks = static_cast<unsigned>((a.total + kMergeThreads - 1) / kMergeThreads);
        cudaError_t e;
        if (c.bf16)
            e = drift ? launch_merge<true, true>(a, smem, blocks, stream) : launch_merge<true, false>(a, smem, blocks, stream);
        else
            e = drift ? launch_merge<false, true>(a, smem, blocks, stream) : launch_merge<false, false>(a, smem, blocks, stream);
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
