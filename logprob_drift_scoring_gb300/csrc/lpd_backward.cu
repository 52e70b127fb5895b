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
// Layout: four persistent blocks of 256 threads per SM stride over rows; each
// row is swept in 8-column groups, four groups per thread in flight.  Rows whose input and
// output start on 16-byte boundaries use 16-byte loads and stores.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"

namespace lpd {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBwdGroups = 4;  // 8-column groups per thread in flight

struct BwdArgs {
    const char *x;
    int64_t x_stride;     // bytes
    char *out;
    int64_t out_stride;   // bytes
    int64_t n_rows, vocab;
    const int32_t *ids;
    const uint8_t *mask;
    const float *logp, *grad;
    int x_bf16, out_bf16;
    int vec;              // rows of both tensors are 16-byte aligned
};

__device__ __forceinline__ float load_x(const BwdArgs &a, const char *row, int64_t j) {
    if (a.x_bf16)
        return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(row) + j)) << 16);
    return __ldg(reinterpret_cast<const float *>(row) + j);
}

__device__ __forceinline__ void store_out(const BwdArgs &a, char *row, int64_t j, float v) {
    if (a.out_bf16)
        reinterpret_cast<__nv_bfloat16 *>(row)[j] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float *>(row)[j] = v;
}

// One 8-column group: load (vector or scalar), gradient, store.
__device__ __forceinline__ void bwd_load8(const BwdArgs &a, const char *xrow, int64_t c0, bool vec, float *x) {
    if (vec) {
        if (a.x_bf16) {
            const uint4 w = __ldg(reinterpret_cast<const uint4 *>(xrow + c0 * 2));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                x[2 * q] = __uint_as_float(ws[q] << 16);
                x[2 * q + 1] = __uint_as_float(ws[q] & 0xffff0000u);
            }
        } else {
            const float4 w0 = __ldg(reinterpret_cast<const float4 *>(xrow + c0 * 4));
            const float4 w1 = __ldg(reinterpret_cast<const float4 *>(xrow + c0 * 4) + 1);
            x[0] = w0.x; x[1] = w0.y; x[2] = w0.z; x[3] = w0.w;
            x[4] = w1.x; x[5] = w1.y; x[6] = w1.z; x[7] = w1.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = c0 + q < a.vocab ? load_x(a, xrow, c0 + q) : 0.f;
    }
}

__device__ __forceinline__ void bwd_store8(const BwdArgs &a, char *orow, int64_t c0, bool vec, const float *v) {
    if (vec) {
        if (a.out_bf16) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
                w[q] = *reinterpret_cast<const uint32_t *>(&h);
            }
            *reinterpret_cast<uint4 *>(orow + c0 * 2) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            reinterpret_cast<float4 *>(orow + c0 * 4)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4 *>(orow + c0 * 4)[1] = make_float4(v[4], v[5], v[6], v[7]);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (c0 + q < a.vocab) store_out(a, orow, c0 + q, v[q]);
    }
}

// Persistent blocks: block b takes rows b, b + gridDim.x, ...; within a row
// thread t handles 8-column groups at 8 t + 2048 k, four groups per iteration
// with all four loads issued before the arithmetic.  The row prologue (mask,
// id, lse, g) is paid once per row.
__global__ void __launch_bounds__(kBwdThreads, 4) backward_kernel(const __grid_constant__ BwdArgs a) {
    constexpr int64_t kStep = 8 * kBwdThreads;  // columns between a thread's groups
    for (int64_t r = blockIdx.x; r < a.n_rows; r += gridDim.x) {
        char *orow = a.out + r * a.out_stride;
        const char *xrow = a.x + r * a.x_stride;
        const bool active = a.mask[r] != 0;
        const int64_t id = active ? a.ids[r] : 0;
        const bool ok = active && id >= 0 && id < a.vocab;
        float lse = 0.f, g = 0.f;
        if (ok) {
            lse = __fsub_rn(load_x(a, xrow, id), a.logp[r]);
            g = a.grad[r];
        }
        for (int64_t base = 8 * static_cast<int64_t>(threadIdx.x); base < a.vocab; base += kBwdGroups * kStep) {
            float x[kBwdGroups][8];
            if (ok) {
#pragma unroll
                for (int gi = 0; gi < kBwdGroups; ++gi) {
                    const int64_t c0 = base + gi * kStep;
                    if (c0 < a.vocab) bwd_load8(a, xrow, c0, a.vec && c0 + 8 <= a.vocab, x[gi]);
                }
            }
#pragma unroll
            for (int gi = 0; gi < kBwdGroups; ++gi) {
                const int64_t c0 = base + gi * kStep;
                if (c0 >= a.vocab) continue;
                float v[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (!active) {
                        v[q] = 0.f;
                    } else if (!ok) {
                        v[q] = CUDART_NAN_F;
                    } else {
                        const float p = ex2(__fmul_rn(__fsub_rn(x[gi][q], lse), kLog2e));
                        const float onehot = (c0 + q == id) ? 1.f : 0.f;
                        v[q] = __fmul_rn(g, __fsub_rn(onehot, p));
                    }
                }
                bwd_store8(a, orow, c0, a.vec && c0 + 8 <= a.vocab, v);
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
    a.x = static_cast<const char *>(x);
    a.x_bf16 = x_dtype == LPD_BF16;
    a.x_stride = x_stride_elems * (a.x_bf16 ? 2 : 4);
    a.out = static_cast<char *>(out);
    a.out_bf16 = out_dtype == LPD_BF16;
    a.out_stride = out_stride_elems * (a.out_bf16 ? 2 : 4);
    a.n_rows = n_rows;
    a.vocab = vocab;
    a.ids = ids;
    a.mask = mask;
    a.logp = logp;
    a.grad = grad;
    a.vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (a.x_stride % 16 == 0) &&
            (reinterpret_cast<uintptr_t>(out) % 16 == 0) && (a.out_stride % 16 == 0);
    const int64_t blocks = static_cast<int64_t>(device_sm_count()) * 4;
    backward_kernel<<<static_cast<unsigned>(n_rows < blocks ? n_rows : blocks), kBwdThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace lpd
