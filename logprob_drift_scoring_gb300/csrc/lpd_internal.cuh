// Internal definitions shared by the kernels and the C-ABI layer of liblpd.
// Nothing here is part of the public interface (include/lpd.h).
#pragma once

#include <atomic>

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "lpd.h"

namespace lpd {

// ---------------------------------------------------------------- geometry
// The streaming row kernel runs one CTA per SM: W consumer warps plus one
// producer warp.  A tile is 16 * 32 W logical columns of one vocab segment,
// read as four groups of G = 4 * 32 W; consumer thread t owns columns
// [G g + 4t, G g + 4t + 4) of group g = 0..3 of every tile (16 columns per
// thread per tile).  W is 20 (tiles of 10240 columns) in every mode but the
// general transform chain, whose tanh code needs more registers than 21 warps
// leave (the register file allows 80 a thread at up to 6 warps per scheduler)
// and which keeps W = 16 (8192 columns).  These constants fix each row's
// arithmetic order, so they are part of the batch-invariance contract:
// changing them changes results (bitwise), but never makes them depend on the
// batch.
constexpr int kRowPlain = 0, kRowTransform = 1, kRowEntropy = 2, kRowScale = 3, kRowSoftcap = 4;
// Consumer warps W of the single-segment row pass by mode: 23 (with the
// producer, 24 warps: six per SM sub-partition, each at the 80 registers a
// thread that its register file allows), 20 for the reduced soft-cap (no
// faster at 23), 16 for the general transform chain (its larger body needs
// more registers).
__host__ __device__ constexpr int row_warps(int mode) {
    return mode == kRowTransform ? 16 : mode == kRowSoftcap ? 20 : 23;
}
constexpr int kConsumerWarps = 23;               // the largest W: the workspace's warp-state stride
constexpr int kColsPerThread = 16;
constexpr int kMaxSegments = 16;                 // shards per side
constexpr int kRingBytes = 200 * 1024;           // shared-memory staging ring
constexpr int kFinThreads = 256;                 // rows per finalise block
constexpr int kSelThreads = 1024;

constexpr float kLog2e = 1.4426950408889634f;

// Sets a kernel's dynamic shared-memory limit once per device.  `done` holds
// one bit per device id below 64 (the attribute is per device); concurrent
// first calls may both set it, which is harmless.
template <class Kernel>
cudaError_t set_smem_once(Kernel *kern, size_t smem, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// The same with the device's opt-in maximum, for kernels whose shared memory
// per launch depends on the call: the limit never has to move between calls
// (a lower value set by one host thread could fail another's launch).
template <class Kernel>
cudaError_t set_smem_max_once(Kernel *kern, std::atomic<uint64_t> &done) {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && (done.load(std::memory_order_acquire) & (uint64_t{1} << dev))) return cudaSuccess;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    return set_smem_once(kern, static_cast<size_t>(optin), done);
}

// ---------------------------------------------------------------- workspace
// Device workspace carved into fixed regions; every region 256-byte aligned.
struct WsHeader {
    int64_t n_active;
    int64_t reserved[31];
};

struct BlockPartial {  // one finalise block's share of the metrics
    double sum_abs;
    double sum_k3;
    double sum_em1;
    double max_abs;
    int64_t argmax_row;
    int64_t n_clip;
};

struct WsLayout {
    size_t header, rowid, pick, part, dval, keys, blockpart, hist, total;
};

// Bins of the first digit of the |dlogp| radix select (11 bits of the fp32
// pattern: the exponent and four mantissa bits).
constexpr int kKeyHistBins = 2048;

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr WsLayout ws_layout(int64_t n_rows, int n_seg) {
    WsLayout L{};
    size_t off = 0;
    const size_t R = size_t(n_rows);
    L.header = off;    off += align256(sizeof(WsHeader));
    L.rowid = off;     off += align256(R * sizeof(int2));          // (row, token id) of active rows
    L.pick = off;      off += align256(R * sizeof(float2));        // selected logits (train, rollout)
    L.part = off;      off += align256(R * size_t(n_seg) * kConsumerWarps * 2 * sizeof(float4));  // warp states
    L.dval = off;      off += align256(R * sizeof(double));        // dlogp per active row
    L.keys = off;      off += align256(R * sizeof(uint32_t));      // |dlogp| as fp32 bits
    L.blockpart = off; off += align256(((R + kFinThreads - 1) / kFinThreads) * sizeof(BlockPartial));
    L.hist = off;      off += align256(kKeyHistBins * sizeof(uint32_t));  // first-digit histogram of the keys
    L.total = off;
    return L;
}

// ---------------------------------------------------------------- segments
// One vocab segment (a shard, or the whole vocabulary) of both sides.
struct Segment {
    const char *t;      // train base (row 0, local column 0)
    const char *r;      // rollout base
    int64_t t_stride;   // bytes between rows
    int64_t r_stride;
    int64_t v_start;    // global column of local column 0
    int64_t len;        // columns in this segment
};

// Logit transform chain of one side, applied in order to every logit.
struct Xform {
    int n_ops;
    int kind[LPD_MAX_TRANSFORM_OPS];
    float param[LPD_MAX_TRANSFORM_OPS];
};

// A side's chain with at most one soft-cap, in the reduced form the
// kRowSoftcap pass evaluates: x -> softcap_p(x) (when `on`), and the product of
// all the chain's scales applied afterwards through the exponent factor.  A
// scale a before the soft-cap moves behind it, softcap_p(a x) =
// a softcap_{p/a}(x), so p here is the chain's soft-cap divided by the scales
// in front of it.  On |x| < 0.45 p the series p tanh(x / p) = x (1 + u Q(u)),
// u = x^2, runs with the coefficients of its fitted tanh series pre-multiplied
// by the powers of 1/p^2 (q[k] = c_k / p^(2k+2)); beyond, the exponential form.
constexpr int kSoftcapTerms = 4;
struct SoftcapSide {
    int on;                 // 0: no soft-cap on this side (identity)
    float p, r, r2;         // p, 1/p, 1/p^2
    float thr;              // |x| below this is inside the series range for certain
    float q[kSoftcapTerms];
};

struct RowArgs {
    Xform xt, xr;    // train and rollout chains (transform mode only)
    SoftcapSide cap[2];  // train and rollout soft-caps (soft-cap mode only)
    float lt, lr;    // scale-only and soft-cap chains: each side's s log2 e (maxima kept unscaled)
    Segment seg[kMaxSegments];
    int n_seg;
    int64_t vocab;
    const WsHeader *hdr;
    const int2 *rowid;
    float4 *part;
    float2 *pick;
    uint32_t *status;
    int stall;       // tests of the timeout path: CTA 0 withholds its first copy
};

struct FinArgs {
    int n_seg;
    int n_warps;                   // warp states per (row, segment): row_warps of the pass's mode
    int n_perm;                    // 0: no merge-order diagnostic
    int8_t perm[kMaxSegments];
    int topo;                      // LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE or LPD_TOPO_ALLREDUCE_PARTIALS
    float scale_t, scale_r;        // scale-only chains: each side's product of scales (else 1)
    float lg_t, lg_r;              // the row pass's factor to base-2 exponents (s log2 e, else log2 e)
    int n_order;                   // 0: segments reduced in index order
    int8_t order[kMaxSegments];
    int64_t vocab;
    const WsHeader *hdr;
    const int2 *rowid;
    const float4 *part;
    const float2 *pick;
    double *dval;
    uint32_t *keys;
    float *out_lt, *out_lr, *out_d;
    float *out_perm_lt, *out_perm_lr;
    float *out_ent_t, *out_ent_r;  // entropies (entropy mode only)
    uint32_t *status;
};

// ---------------------------------------------------------------- fused head
// Workspace of the fused LM-head path: the common regions (with no per-warp
// states) followed by the dense active hidden rows of both sides and the
// per-(row, vocab tile) partial states.
struct FusedLayout {
    WsLayout base;
    size_t hidden_t, hidden_r, part_a, part_b, total;
    int64_t a_pad;     // rows padded to the 128-row tile
    int n_tiles_n;     // vocab tiles of 256 columns
};

struct FusedCall {
    FusedLayout layout;
    void *workspace;
    const void *hidden_train, *hidden_rollout, *weight;
    int64_t n_rows, hidden, vocab;
    float *out_lt, *out_lr, *out_d;
    uint32_t *status;
    Xform xt, xr;  // logit transform chains (n_ops 0 on both sides: none)
};

FusedLayout fused_layout(int64_t n_rows, int64_t hidden, int64_t vocab);
cudaError_t launch_fused(const FusedCall &c, cudaStream_t stream);

// ---------------------------------------------------------------- launchers
cudaError_t launch_select_active(int64_t n_rows, const uint8_t *mask, const int32_t *ids,
                                 float *out_lt, float *out_lr, float *out_d,
                                 lpd_metrics *metrics, WsHeader *hdr, int2 *rowid,
                                 cudaStream_t stream);
// Consumer warps of the row pass for these segments (the mode's default, or
// for the plain bulk-copy pass over several segments the count whose tiles
// waste the fewest columns on the segments' last tiles: 20, 19 or 16); a
// function of the segment lengths only, so every row keeps its arithmetic in
// any batch.
int row_pass_warps(const Segment *segs, int n_seg, int mode, bool use_tma);
cudaError_t launch_rows(const RowArgs &a, int dtype_t, int dtype_r, bool use_tma, int mode, int warps,
                        cudaStream_t stream);
cudaError_t launch_finalize(const FinArgs &a, int64_t n_rows, cudaStream_t stream);
cudaError_t launch_dlogp_rows(int64_t n_rows, const float *dlogp, const WsHeader *hdr, const int2 *rowid,
                              double *dval, uint32_t *keys, uint32_t *status, cudaStream_t stream);
cudaError_t launch_metrics(int64_t n_rows, double ln_clip_lo, double ln_clip_hi, const WsHeader *hdr,
                           const int2 *rowid, const double *dval, const uint32_t *keys,
                           BlockPartial *bp, uint32_t *hist, lpd_metrics *metrics, cudaStream_t stream);

cudaError_t launch_backward(const void *x, int x_dtype, int64_t x_stride_elems, void *out, int out_dtype,
                            int64_t out_stride_elems, int64_t n_rows, int64_t vocab, const int32_t *ids,
                            const uint8_t *mask, const float *logp, const float *grad, cudaStream_t stream);

// Attention (out, lse) merge: one call of lpd_attn_merge (diag false) or of
// lpd_attn_merge_order_drift (diag true).  Orders are validated permutations.
struct AttnMergeCall {
    const void *parts;
    bool bf16;
    const float *lse;
    int n_parts;
    int64_t n_rows;
    int head_dim;
    int base2;
    const int32_t *order_a, *order_b;   // host, n_parts entries each
    float *out, *out_lse;
    bool diag;
    float *row_dout, *row_dlse;
    lpd_merge_drift *drift;
};
cudaError_t launch_attn_merge(const AttnMergeCall &c, cudaStream_t stream);

// The all-gather of the allgather_logits arm: shard pieces of every row into
// full rows (pitches in bytes).
cudaError_t launch_gather_shards(const Segment *segs, int n_seg, int64_t n_rows, void *dst_t, int64_t pitch_t,
                                 int elt_t, void *dst_r, int64_t pitch_r, int elt_r, cudaStream_t stream);

// Summary of per-token result b against result a over the active rows.
cudaError_t launch_logp_drift(int64_t n_rows, const float *at, const float *ar, const float *bt, const float *br,
                              const uint8_t *mask, lpd_logp_drift *out, cudaStream_t stream);

int device_sm_count();

}  // namespace lpd
