// The all-gather of the allgather_logits reduction arm: every shard's columns
// of every row copied into one full row per side ("[WS2] Framework for
// ablation experiment", LogProb knobs table, row 4: reduction topology).
//
// Layout: blocks stride over rows; for each row a block copies each shard's
// piece of both sides.  Where source and destination share their offset
// within 16 bytes (always for shard pieces that start on 16-byte boundaries)
// the middle of the piece moves as streaming 16-byte words, four per thread in
// flight, and the few elements before and after it one by one; otherwise the
// piece is copied element by element.
#include "lpd_internal.cuh"

namespace lpd {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;

struct GatherArgs {
    Segment seg[kMaxSegments];
    int n_seg;
    int64_t n_rows;
    char *dst_t, *dst_r;
    int64_t pitch_t, pitch_r;  // bytes
    int et, er;                // element bytes
};

template <typename E>
__device__ __forceinline__ void copy_elems(char *dst, const char *src, int64_t n) {
    const int t = threadIdx.x;
    E *d = reinterpret_cast<E *>(dst);
    const E *s = reinterpret_cast<const E *>(src);
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst), sa = reinterpret_cast<uintptr_t>(src);
    if ((da & 15) != (sa & 15)) {
        for (int64_t i = t; i < n; i += kGatherThreads) d[i] = s[i];
        return;
    }
    int64_t head = static_cast<int64_t>((16 - (da & 15)) & 15) / static_cast<int64_t>(sizeof(E));
    if (head > n) head = n;
    for (int64_t i = t; i < head; i += kGatherThreads) d[i] = s[i];
    const int64_t nv = (n - head) * static_cast<int64_t>(sizeof(E)) / 16;
    uint4 *d4 = reinterpret_cast<uint4 *>(d + head);
    const uint4 *s4 = reinterpret_cast<const uint4 *>(s + head);
    constexpr int64_t kStride = static_cast<int64_t>(kGatherThreads) * kGatherUnroll;
    for (int64_t base = t; base < nv; base += kStride) {
        uint4 v[kGatherUnroll];
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u)
            if (base + u * kGatherThreads < nv) v[u] = __ldcs(s4 + base + u * kGatherThreads);
#pragma unroll
        for (int u = 0; u < kGatherUnroll; ++u)
            if (base + u * kGatherThreads < nv) __stcs(d4 + base + u * kGatherThreads, v[u]);
    }
    for (int64_t i = head + nv * 16 / static_cast<int64_t>(sizeof(E)) + t; i < n; i += kGatherThreads) d[i] = s[i];
}

__device__ __forceinline__ void copy_piece(char *dst, const char *src, int64_t n, int elt) {
    if (elt == 2)
        copy_elems<unsigned short>(dst, src, n);
    else
        copy_elems<unsigned>(dst, src, n);
}

__global__ void __launch_bounds__(kGatherThreads, 4) gather_shards_kernel(const __grid_constant__ GatherArgs a) {
    for (int64_t r = blockIdx.x; r < a.n_rows; r += gridDim.x) {
        for (int k = 0; k < a.n_seg; ++k) {
            const Segment &sg = a.seg[k];
            copy_piece(a.dst_t + r * a.pitch_t + sg.v_start * a.et, sg.t + r * sg.t_stride, sg.len, a.et);
            copy_piece(a.dst_r + r * a.pitch_r + sg.v_start * a.er, sg.r + r * sg.r_stride, sg.len, a.er);
        }
    }
}

}  // namespace

cudaError_t launch_gather_shards(const Segment *segs, int n_seg, int64_t n_rows, void *dst_t, int64_t pitch_t,
                                 int elt_t, void *dst_r, int64_t pitch_r, int elt_r, cudaStream_t stream) {
    if (n_rows == 0) return cudaSuccess;
    GatherArgs a{};
    for (int k = 0; k < n_seg; ++k) a.seg[k] = segs[k];
    a.n_seg = n_seg;
    a.n_rows = n_rows;
    a.dst_t = static_cast<char *>(dst_t);
    a.dst_r = static_cast<char *>(dst_r);
    a.pitch_t = pitch_t;
    a.pitch_r = pitch_r;
    a.et = elt_t;
    a.er = elt_r;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 8;
    gather_shards_kernel<<<static_cast<unsigned>(n_rows < cap ? n_rows : cap), kGatherThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace lpd
