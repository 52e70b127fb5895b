// Summary of how far one per-token logp result is from another over the
// active rows: each side's largest |b - a| with the lowest row attaining it,
// and how many active rows differ.  Its use on the path is the merge-order
// diagnostic of the vocab-sharded scorer ("[WS2] Framework for ablation
// experiment", LogProb knobs table, row 5: the merge order of the per-shard
// partials is a drift source): a = the fixed global shard order, b = a
// permuted order, both as lpd_score_sharded returns them.
//
// One grid-stride pass over the rows.  A row's |b - a| is formed in fp32,
// which is exact whenever a and b are within a factor of two of each other
// (always the case for two merges of the same row).  The maximum and its
// lowest row travel as one 64-bit key (the value's bits above 2^32 - 1 -
// row, NaN made canonical so every NaN ties and the lowest such row wins);
// keys and counts are combined with integer atomics, so the result does not
// depend on the order in which blocks finish.
#include <cfloat>

#include "lpd_internal.cuh"

namespace lpd {
namespace {

constexpr int kDriftThreads = 256;

__device__ __forceinline__ unsigned long long drift_key(float a, float b, int64_t r) {
    const float d = fabsf(__fsub_rn(b, a));
    const uint32_t bits = isnan(d) ? 0x7fc00000u : __float_as_uint(d);
    return (static_cast<unsigned long long>(bits) << 32) | (0xffffffffull - static_cast<unsigned long long>(r));
}

// a and b are the same number (+0 == -0), or both NaN
__device__ __forceinline__ bool same_number(float a, float b) { return a == b || (isnan(a) && isnan(b)); }

__global__ void __launch_bounds__(kDriftThreads)
    logp_drift_kernel(int64_t n, const float *at, const float *ar, const float *bt, const float *br,
                      const uint8_t *mask, unsigned long long *acc) {
    unsigned long long kt = 0, kr = 0, n_act = 0, n_diff = 0;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kDriftThreads + threadIdx.x; r < n;
         r += static_cast<int64_t>(gridDim.x) * kDriftThreads) {
        if (!mask[r]) continue;
        const float a0 = at[r], b0 = bt[r], a1 = ar[r], b1 = br[r];
        const unsigned long long k0 = drift_key(a0, b0, r), k1 = drift_key(a1, b1, r);
        kt = k0 > kt ? k0 : kt;
        kr = k1 > kr ? k1 : kr;
        n_act += 1;
        n_diff += (same_number(a0, b0) && same_number(a1, b1)) ? 0 : 1;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, kt, off);
        const unsigned long long y = __shfl_xor_sync(0xffffffffu, kr, off);
        kt = x > kt ? x : kt;
        kr = y > kr ? y : kr;
        n_act += __shfl_xor_sync(0xffffffffu, n_act, off);
        n_diff += __shfl_xor_sync(0xffffffffu, n_diff, off);
    }
    __shared__ unsigned long long sh[4][kDriftThreads / 32];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) {
        sh[0][warp] = kt;
        sh[1][warp] = kr;
        sh[2][warp] = n_act;
        sh[3][warp] = n_diff;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kDriftThreads / 32; ++w) {
            kt = sh[0][w] > kt ? sh[0][w] : kt;
            kr = sh[1][w] > kr ? sh[1][w] : kr;
            n_act += sh[2][w];
            n_diff += sh[3][w];
        }
        if (n_act) {
            atomicMax(acc + 0, kt);
            atomicMax(acc + 1, kr);
            atomicAdd(acc + 2, n_act);
            atomicAdd(acc + 3, n_diff);
        }
    }
}

__global__ void logp_drift_finalize_kernel(lpd_logp_drift *d) {
    if (threadIdx.x != 0) return;
    const unsigned long long kt = d->scratch[0], kr = d->scratch[1], n_act = d->scratch[2], n_diff = d->scratch[3];
    d->n_active = static_cast<int64_t>(n_act);
    d->n_differ = static_cast<int64_t>(n_diff);
    if (n_act == 0) {
        d->max_abs_dlogp_train = 0.0;
        d->max_abs_dlogp_rollout = 0.0;
        d->row_train = -1;
        d->row_rollout = -1;
        d->frac_differ = 0.0;
        return;
    }
    d->max_abs_dlogp_train = static_cast<double>(__uint_as_float(static_cast<uint32_t>(kt >> 32)));
    d->max_abs_dlogp_rollout = static_cast<double>(__uint_as_float(static_cast<uint32_t>(kr >> 32)));
    d->row_train = static_cast<int64_t>(0xffffffffull - (kt & 0xffffffffull));
    d->row_rollout = static_cast<int64_t>(0xffffffffull - (kr & 0xffffffffull));
    d->frac_differ = static_cast<double>(n_diff) / static_cast<double>(n_act);
}

}  // namespace

cudaError_t launch_logp_drift(int64_t n_rows, const float *at, const float *ar, const float *bt, const float *br,
                              const uint8_t *mask, lpd_logp_drift *out, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(lpd_logp_drift), stream);
    if (e != cudaSuccess) return e;
    if (n_rows > 0) {
        const int64_t want = (n_rows + kDriftThreads - 1) / kDriftThreads;
        const int64_t cap = static_cast<int64_t>(device_sm_count()) * 4;
        logp_drift_kernel<<<static_cast<unsigned>(want < cap ? want : cap), kDriftThreads, 0, stream>>>(
            n_rows, at, ar, bt, br, mask, reinterpret_cast<unsigned long long *>(out->scratch));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    logp_drift_finalize_kernel<<<1, 32, 0, stream>>>(out);
    return cudaGetLastError();
}

}  // namespace lpd
