// Gradient of the selected-token logprob with respect to the logits.
//
// Method: "[WS2] Framework for ablation experiment", LogProb knobs table, row
// 11 (training-only state: the logprob's gradient must match between
// implementations too).  For an active row r with selected id and upstream
// gradient g = grad_logp[r]:
//   d(g * logp[r]) / d x[r, j] = g * (1[j == id] - p_j),  p_j = exp(x[r, j] - lse[r]),
// with lse[r] = x[r, id] - logp[r] recovered from the forward's own output, so
// this pass reads each logits row once and writes each gradient row once.
// Inactive rows get a zero gradient; an active row with an out-of-range id
// gets NaN (fail closed).
//
// Layout: four persistent blocks of 256 threads per SM stride over rows.
// Rows whose input and output start on 16-byte boundaries are swept in
// 8-column groups with 16-byte loads and stores, 32 registers of raw input per
// thread in flight (eight groups of bf16 or four of fp32); the one-hot term is
// applied only in the group that holds the id.  Inactive and out-of-range rows
// are a fill.  Other rows take a plain per-element loop with the same
// arithmetic.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"

namespace lpd {
namespace {

constexpr int kBwdThreads = 256;
constexpr uint32_t kBwdStep = 8 * kBwdThreads;  // columns between a thread's groups

struct BwdArgs {
    const char *x;
    int64_t x_stride;     // bytes
    char *out;
    int64_t out_stride;   // bytes
    int64_t n_rows, vocab;
    const int32_t *ids;
    const uint8_t *mask;
    const float *logp, *grad;
    int vec;              // rows of both tensors are 16-byte aligned
};

template <bool kXBf16>
__device__ __forceinline__ float load_x(const char *row, int64_t j) {
    if constexpr (kXBf16)
        return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(row) + j)) << 16);
    else
        return __ldg(reinterpret_cast<const float *>(row) + j);
}

template <bool kOBf16>
__device__ __forceinline__ void store_out(char *row, int64_t j, float v) {
    if constexpr (kOBf16)
        reinterpret_cast<__nv_bfloat16 *>(row)[j] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(row)[j] = v;
}

// 8 consecutive columns as raw 16-byte words: one for bf16, two for fp32.
template <bool kXBf16>
struct Raw8 {
    uint4 w[kXBf16 ? 1 : 2];
};

// Columns are 32-bit: vocab < 2^31, so a column plus a few sweeps stays below 2^32.
template <bool kXBf16>
__device__ __forceinline__ void load8(const char *xrow, uint32_t c0, Raw8<kXBf16> &r) {
    const uint4 *p = reinterpret_cast<const uint4 *>(xrow + static_cast<size_t>(c0) * (kXBf16 ? 2 : 4));
    r.w[0] = __ldcs(p);
    if constexpr (!kXBf16) r.w[1] = __ldcs(p + 1);
}

template <bool kXBf16>
__device__ __forceinline__ void unpack8(const Raw8<kXBf16> &r, float *x) {
    if constexpr (kXBf16) {
        const uint32_t ws[4] = {r.w[0].x, r.w[0].y, r.w[0].z, r.w[0].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            x[2 * q] = __uint_as_float(ws[q] << 16);
            x[2 * q + 1] = __uint_as_float(ws[q] & 0xffff0000u);
        }
    } else {
        const uint32_t ws[8] = {r.w[0].x, r.w[0].y, r.w[0].z, r.w[0].w, r.w[1].x, r.w[1].y, r.w[1].z, r.w[1].w};
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = __uint_as_float(ws[q]);
    }
}

template <bool kOBf16>
__device__ __forceinline__ void store8(char *orow, uint32_t c0, const float *v) {
    if constexpr (kOBf16) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
            w[q] = *reinterpret_cast<const uint32_t *>(&h);
        }
        __stcs(reinterpret_cast<uint4 *>(orow + static_cast<size_t>(c0) * 2), make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        float4 *p = reinterpret_cast<float4 *>(orow + static_cast<size_t>(c0) * 4);
        __stcs(p, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(p + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
}

// g * (1[j == id] - p_j), p_j = 2^((x_j - lse) log2 e): the one-hot term only
// where the group holds the id.
__device__ __forceinline__ void grad8(const float *x, uint32_t c0, uint32_t id, float lse, float g, float *v) {
    float p[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        p[q] = ex2(__fmul_rn(__fsub_rn(x[q], lse), kLog2e));
        v[q] = __fmul_rn(g, -p[q]);
    }
    const uint32_t j = id - c0;  // wraps for id < c0
    if (j < 8u) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q == j) v[q] = __fmul_rn(g, __fsub_rn(1.f, p[q]));
    }
}

template <bool kXBf16, bool kOBf16>
__global__ void __launch_bounds__(kBwdThreads, 4) backward_kernel(const __grid_constant__ BwdArgs a) {
    constexpr int kGroups = kXBf16 ? 8 : 4;  // groups in flight: 32 registers of raw input
    const int t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < a.n_rows; r += gridDim.x) {
        char *orow = a.out + r * a.out_stride;
        const char *xrow = a.x + r * a.x_stride;
        const bool active = a.mask[r] != 0;
        const int64_t id = active ? a.ids[r] : 0;
        if (!(active && id >= 0 && id < a.vocab)) {
            // inactive rows: 0; an active row with an out-of-range id: NaN
            const float fill = active ? CUDART_NAN_F : 0.f;
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = fill;
            for (int64_t c0 = 8 * t; c0 < a.vocab; c0 += static_cast<int64_t>(kBwdStep)) {
                if (a.vec && c0 + 8 <= a.vocab) {
                    store8<kOBf16>(orow, c0, v);
                } else {
                    for (int q = 0; q < 8 && c0 + q < a.vocab; ++q) store_out<kOBf16>(orow, c0 + q, fill);
                }
            }
            continue;
        }
        const float lse = __fsub_rn(load_x<kXBf16>(xrow, id), a.logp[r]);
        const float g = a.grad[r];
        const uint32_t V = static_cast<uint32_t>(a.vocab), uid = static_cast<uint32_t>(id);
        if (!a.vec) {
            for (int64_t j = t; j < a.vocab; j += kBwdThreads) {
                const float p = ex2(__fmul_rn(__fsub_rn(load_x<kXBf16>(xrow, j), lse), kLog2e));
                store_out<kOBf16>(orow, j, j == id ? __fmul_rn(g, __fsub_rn(1.f, p)) : __fmul_rn(g, -p));
            }
            continue;
        }
        for (uint32_t base = 8 * t; base < V; base += kGroups * kBwdStep) {
            Raw8<kXBf16> raw[kGroups];
#pragma unroll
            for (int gi = 0; gi < kGroups; ++gi) {
                const uint32_t c0 = base + gi * kBwdStep;
                if (c0 + 8 <= V) load8<kXBf16>(xrow, c0, raw[gi]);
            }
#pragma unroll
            for (int gi = 0; gi < kGroups; ++gi) {
                const uint32_t c0 = base + gi * kBwdStep;
                if (c0 >= V) break;
                float x[8], v[8];
                if (c0 + 8 <= V) {
                    unpack8<kXBf16>(raw[gi], x);
                    grad8(x, c0, uid, lse, g, v);
                    store8<kOBf16>(orow, c0, v);
                } else {
                    // the row's last, partial group
#pragma unroll
                    for (int q = 0; q < 8; ++q) x[q] = c0 + q < V ? load_x<kXBf16>(xrow, c0 + q) : 0.f;
                    grad8(x, c0, uid, lse, g, v);
                    for (uint32_t q = 0; q < 8 && c0 + q < V; ++q) store_out<kOBf16>(orow, c0 + q, v[q]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_backward(const void *x, int x_dtype, int64_t x_stride_elems, void *out, int out_dtype,
                            int64_t out_stride_elems, int64_t n_rows, int64_t vocab, const int32_t *ids,
                            const uint8_t *mask, const float *logp, const float *grad, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    BwdArgs a{};
    const bool xb = x_dtype == LPD_BF16, ob = out_dtype == LPD_BF16;
    a.x = static_cast<const char *>(x);
    a.x_stride = x_stride_elems * (xb ? 2 : 4);
    a.out = static_cast<char *>(out);
    a.out_stride = out_stride_elems * (ob ? 2 : 4);
    a.n_rows = n_rows;
    a.vocab = vocab;
    a.ids = ids;
    a.mask = mask;
    a.logp = logp;
    a.grad = grad;
    a.vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (a.x_stride % 16 == 0) &&
            (reinterpret_cast<uintptr_t>(out) % 16 == 0) && (a.out_stride % 16 == 0);
    const int64_t blocks = static_cast<int64_t>(device_sm_count()) * 4;
    const unsigned grid = static_cast<unsigned>(n_rows < blocks ? n_rows : blocks);
    if (xb)
        ob ? backward_kernel<true, true><<<grid, kBwdThreads, 0, stream>>>(a)
           : backward_kernel<true, false><<<grid, kBwdThreads, 0, stream>>>(a);
    else
        ob ? backward_kernel<false, true><<<grid, kBwdThreads, 0, stream>>>(a)
           : backward_kernel<false, false><<<grid, kBwdThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace lpd
