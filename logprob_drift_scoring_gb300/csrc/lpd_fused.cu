// Fused LM-head scoring: the logits x_side[r, v] = sum_k hidden_side[r, k] *
// W[v, k] are produced tile by tile on the tensor cores (tcgen05, fp32
// accumulators in tensor memory) and folded straight into the online
// log-sum-exp state; they are never written to memory.
//
// Method: "[WS2] Framework for ablation experiment", LogProb knobs table, rows
// 9-10 (the head GEMM and its fusion tiling: online softmax over vocab tiles
// with a fixed merge order); "WS2 Cross-Config Logprob Drift Contract",
// "Measurement Contract" (teacher-forced selected-token logp of both sides).
//
// Pipeline (all on the caller's stream):
//   1. gather_hidden_kernel: the active rows of both hidden tensors, in row
//      order, into dense [A_pad, H] buffers (rows past A are zero).
//   2. head_kernel (one CTA per SM, persistent): for each (128-row, 256-vocab)
//      output tile, warp 0 streams 64-wide K blocks of both sides' hidden rows
//      and of W through a 3-stage shared-memory ring with 2-D TMA copies
//      (128-byte swizzle); warp 1 issues tcgen05.mma (kind::f16, bf16 x bf16
//      -> fp32, M=128 N=256 K=16) for both sides against the same W tile, in a
//      fixed K order, into two 256-column accumulators in tensor memory; warps
//      2-17 read the accumulators back (tcgen05.ld), four warps per row, each
//      folding 64 columns of both sides into an online log-sum-exp state
//      (lpd_acc.cuh); the four states are merged in column order and written
//      as that (row, vocab tile)'s partial (in the transform variant each
//      side's logit chain is applied first, lpd_xform.cuh).  The accumulators
//      fill tensor memory, so the next tile's MMAs wait for this drain: four
//      warps per row cut that wait to a quarter, each warp loads both sides'
//      columns before one wait, and each frees its share as soon as its reads
//      are done (the states travel to the row's lead warp through a separate
//      shared-memory buffer).  Tiles are visited in groups of 16 row
//      tiles (2048 tokens) so that the CTAs running together share their W
//      tiles and hidden tiles in L2, and W is read from memory once a group.
//   3. head_finalize_kernel: one warp per active row merges its vocab-tile
//      partials in vocab order (fixed tree) and applies the same fp64 row
//      arithmetic as the unfused path.
// Every row's arithmetic depends only on its own hidden rows, W and the fixed
// tiling (no split-K, no M-dependent choice), so a row scores the same bits in
// any batch.
//
// Every mbarrier wait is bounded; a timeout records LPD_STATUS_TIMEOUT, every
// role leaves its loop, the MMA warp waits (bounded) for its issued MMAs, the
// producer for its issued copies, and tensor memory is freed before exit.
#include <cfloat>
#include <cuda.h>

#include <math_constants.h>

#include "lpd_acc.cuh"
#include "lpd_internal.cuh"
#include "lpd_xform.cuh"

namespace lpd {
namespace {

constexpr int kBM = 128;                       // rows per tile (each side)
constexpr int kBN = 256;                       // vocab columns per tile
constexpr int kBK = 64;                        // K per stage: one 128-byte swizzle row
constexpr int kUmmaK = 16;                     // K per tcgen05.mma (kind::f16)
constexpr int kStages = 3;
constexpr int kATile = kBM * kBK * 2;          // 16 KB
constexpr int kBTile = kBN * kBK * 2;          // 32 KB
constexpr int kStage = 2 * kATile + kBTile;    // 64 KB
constexpr int kEpiSplit = 4;                   // epilogue warps per tensor-memory lane quadrant
constexpr int kEpiWarps = 4 * kEpiSplit;
constexpr int kEpiCols = kBN / kEpiSplit;      // accumulator columns per epilogue warp
constexpr int kHeadThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue warps
constexpr int kGroupM = 16;                    // row tiles per raster group
constexpr uint32_t kTmemCols = 512;            // two 128 x 256 fp32 accumulators
constexpr unsigned long long kWaitLimitNs = 4000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 30;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
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
// Bounded wait; on timeout records LPD_STATUS_TIMEOUT and raises the CTA's
// abort flag.  With honour_abort, also gives up as soon as the flag is raised.
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

// 2-D tiled TMA load of box (x = K element, y = row) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor for a K-major tile written by TMA with the
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row swizzle atoms of 1024 B.
//   bits 0-13  start address >> 4      bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4 (1024 B between 8-row groups)
//   bits 46-48 0b001                   bits 61-63 swizzle mode (2 = 128 B)
__device__ __forceinline__ uint64_t smem_desc_sw128(const void *tile) {
    const uint64_t addr = (smem_u32(tile) & 0x3FFFFu) >> 4;
    return addr | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4)                          // D format: f32
                            | (1u << 7)                        // A format: bf16
                            | (1u << 10)                       // B format: bf16
                            | (static_cast<uint32_t>(kBN >> 3) << 17)
                            | (static_cast<uint32_t>(kBM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every tcgen05.mma this thread issued so far completes.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this warp's 32 accumulator lanes (one row per
// lane), issued without waiting (tmem_wait_ld completes it).
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void unpack16(const uint32_t *r, f2_t *v) {
#pragma unroll
    for (int p = 0; p < 8; ++p) v[p] = f2(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1]));
}

struct HeadMaps {
    CUtensorMap a_t;  // dense active hidden rows, train side
    CUtensorMap a_r;  // rollout side
    CUtensorMap w;    // W [vocab, hidden]
};

struct HeadArgs {
    const WsHeader *hdr;
    const int2 *rowid;
    int64_t vocab;
    int hidden;
    int n_tiles_n;         // ceil(vocab / 256)
    float4 *part_a;        // [A_pad, n_tiles_n] (mt, st, dd, mr)
    float *part_b;         // [A_pad, n_tiles_n] sr
    float2 *pick;          // [A_pad] selected logits
    uint32_t *status;
    Xform xt, xr;          // transform chains (the general-chain kernel only)
    SoftcapSide cap[2];    // reduced soft-caps (the soft-cap kernel only)
    float lt, lr;          // each side's factor to base-2 exponents: s log2 e (scales folded), else log2 e
};

__device__ __forceinline__ void tile_coords(int64_t t, int n_m, int n_n, int &m, int &n) {
    const int64_t per_group = static_cast<int64_t>(kGroupM) * n_n;
    const int g = static_cast<int>(t / per_group);
    const int64_t local = t % per_group;
    const int gm = min(kGroupM, n_m - g * kGroupM);
    m = g * kGroupM + static_cast<int>(local % gm);
    n = static_cast<int>(local / gm);
}

// kChain: 0 no transform; 1 each side's general chain (per-op loop); 2 the
// reduced form of chains with at most one soft-cap per side (the soft-cap on
// each value, the scales folded into the exponent factor); 3 scales only
// (folded into the exponent factor, no per-value work).  The transform runs on
// the accumulator values right after they leave tensor memory, before the
// vocab-tail mask, so the selected logit and the sums see transformed values
// and padding stays -inf; the finalise applies the folded scales in fp64.
template <int kChain>
__global__ void __launch_bounds__(kHeadThreads, 1)
    head_kernel(const __grid_constant__ HeadMaps maps, const __grid_constant__ HeadArgs a) {
    extern __shared__ __align__(1024) char smem_raw[];
    __shared__ uint64_t full[kStages], empty[kStages], tmem_full, tmem_empty, mma_done;
    // a row's column-half states, handed by the other warps of its lane
    // quadrant to the quadrant's lead warp (one phase per tile)
    // two hand-over buffers, used by alternate tiles, each with its own barrier
    // per quadrant, so the lead can free tensor memory before reading them
    __shared__ uint64_t xchg_full[2][4];
    __shared__ float xchg[2][kEpiSplit > 1 ? kEpiSplit - 1 : 1][5][kBM];
    __shared__ uint32_t tmem_base_slot;
    __shared__ int abort_flag;
    __shared__ float4 xf_ops[2 * LPD_MAX_TRANSFORM_OPS];
    // the swizzled tiles need 1024-byte alignment
    char *smem = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_active = a.hdr->n_active;
    const int n_m = static_cast<int>((n_active + kBM - 1) / kBM);
    const int n_n = a.n_tiles_n;
    const int64_t n_tiles = static_cast<int64_t>(n_m) * n_n;
    const int k_blocks = a.hidden / kBK;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&tmem_full, 1);
        mbar_init(&tmem_empty, kEpiWarps);
        mbar_init(&mma_done, 1);
        for (int b = 0; b < 2; ++b)
            for (int q = 0; q < 4; ++q) mbar_init(&xchg_full[b][q], (kEpiSplit - 1) * 32);
        if (kChain == 1) {
            xform_table(a.xt, xf_ops);
            xform_table(a.xr, xf_ops + LPD_MAX_TRANSFORM_OPS);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x) {
                int m, n;
                tile_coords(t, n_m, n_n, m, n);
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const uint32_t s = it % kStages, round = it / kStages;
                    if (round > 0 && !wait_phase(&empty[s], (round - 1) & 1, &abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    char *st = smem + static_cast<size_t>(s) * kStage;
                    mbar_arrive_expect_tx(&full[s], kStage);
                    tma_load_2d(st, &maps.a_t, kb * kBK, m * kBM, &full[s]);
                    tma_load_2d(st + kATile, &maps.a_r, kb * kBK, m * kBM, &full[s]);
                    tma_load_2d(st + 2 * kATile, &maps.w, kb * kBK, n * kBN, &full[s]);
                }
            }
            // every copy issued must land before the CTA exits
            const uint32_t first = it > static_cast<uint32_t>(kStages) ? it - kStages : 0;
            for (uint32_t j = first; j < it; ++j)
                wait_phase(&full[j % kStages], (j / kStages) & 1, &abort_flag, a.status, false);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            uint32_t it = 0, local = 0;
            bool ok = true, issued = false;
            for (int64_t t = blockIdx.x; ok && t < n_tiles; t += gridDim.x, ++local) {
                if (local > 0 && !wait_phase(&tmem_empty, (local - 1) & 1, &abort_flag, a.status)) break;
                tc_fence_after();
                for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                    const uint32_t s = it % kStages, round = it / kStages;
                    if (!wait_phase(&full[s], round & 1, &abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const char *st = smem + static_cast<size_t>(s) * kStage;
                    const uint64_t dt = smem_desc_sw128(st), dr = smem_desc_sw128(st + kATile),
                                   dw = smem_desc_sw128(st + 2 * kATile);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // advancing K by 16 bf16 = 32 bytes inside the swizzle row
                        const uint64_t koff = static_cast<uint64_t>((k * kUmmaK * 2) >> 4);
                        const uint32_t acc = (kb > 0 || k > 0) ? 1u : 0u;
                        umma_bf16(tmem_base, dt + koff, dw + koff, acc);
                        umma_bf16(tmem_base + kBN, dr + koff, dw + koff, acc);
                    }
                    umma_commit(&empty[s]);  // frees the stage once these MMAs have read it
                    issued = true;
                }
                if (ok) umma_commit(&tmem_full);
            }
            // all issued MMAs complete before anyone frees tensor memory
            if (issued) {
                umma_commit(&mma_done);
                wait_phase(&mma_done, 0, &abort_flag, a.status, false);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp w reads tensor-memory lanes [32 (w % 4), +32): one row per lane.
        // The kEpiSplit warps of a quadrant take consecutive kEpiCols-column
        // ranges of the tile, each freeing the accumulators as soon as its own
        // reads are done; the others hand their row states to the lead (split
        // 0) through shared memory (two buffers, alternate tiles), and the lead
        // merges them in column order and writes the tile's partial.
        const int quad = warp & 3;
        const int split = (warp - 2) >> 2;
        const int row_in_tile = quad * 32 + lane;
        const XformView cxt{xf_ops, kChain == 1 ? a.xt.n_ops : 0},
            cxr{xf_ops + LPD_MAX_TRANSFORM_OPS, kChain == 1 ? a.xr.n_ops : 0};
        const float lg_t = kChain >= 2 ? a.lt : kLog2e, lg_r = kChain >= 2 ? a.lr : kLog2e;
        uint32_t local = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++local) {
            const bool ok = wait_phase(&tmem_full, local & 1, &abort_flag, a.status);
            if (__any_sync(0xffffffffu, !ok)) break;
            tc_fence_after();
            int m, n;
            tile_coords(t, n_m, n_n, m, n);
            const int64_t i = static_cast<int64_t>(m) * kBM + row_in_tile;  // active-row index
            const bool valid = i < n_active;
            const int64_t id = valid ? a.rowid[i].y : -1;
            const int64_t c_base = static_cast<int64_t>(n) * kBN;
            Acc2 acc = acc2_init();
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
#pragma unroll 1
            for (int c = split * kEpiCols; c < (split + 1) * kEpiCols; c += 16) {
                f2_t vt[8], vr[8];
                {
                    // both sides' loads in flight together, one wait
                    uint32_t rt[16], rr[16];
                    tmem_ld16_issue(lane_addr + c, rt);
                    tmem_ld16_issue(lane_addr + kBN + c, rr);
                    tmem_wait_ld();
                    unpack16(rt, vt);
                    unpack16(rr, vr);
                }
                if (kChain == 1) {
                    xform16(vt, cxt);
                    xform16(vr, cxr);
                }
                if (kChain == 2) softcap32_u(vt, vr, a.cap[0], a.cap[1]);
                const int64_t col0 = c_base + c;
                if (col0 + 16 > a.vocab) {  // vocab tail: columns past V are not logits
#pragma unroll
                    for (int p = 0; p < 8; ++p) {
                        const bool in0 = col0 + 2 * p < a.vocab, in1 = col0 + 2 * p + 1 < a.vocab;
                        vt[p] = f2(in0 ? f2_lo(vt[p]) : -INFINITY, in1 ? f2_hi(vt[p]) : -INFINITY);
                        vr[p] = f2(in0 ? f2_lo(vr[p]) : -INFINITY, in1 ? f2_hi(vr[p]) : -INFINITY);
                    }
                }
                if (id >= col0 && id < col0 + 16) {
                    const int q = static_cast<int>(id - col0);
                    float xt = f2_lo(vt[0]), xr = f2_lo(vr[0]);
#pragma unroll
                    for (int k = 1; k < 16; ++k) {
                        if (q == k) {
                            xt = (k & 1) ? f2_hi(vt[k >> 1]) : f2_lo(vt[k >> 1]);
                            xr = (k & 1) ? f2_hi(vr[k >> 1]) : f2_lo(vr[k >> 1]);
                        }
                    }
                    a.pick[i] = make_float2(xt, xr);
                }
                accumulate16(vt, vr, acc, lg_t, lg_r);
            }
            Acc r = acc2_fold(acc);
            tc_fence_before();
            __syncwarp();
            // this warp's accumulator reads are complete: its share of tensor
            // memory is free for the next tile's MMAs (the lead included: the
            // hand-over goes through a buffer of its own, see below)
            if (lane == 0) mbar_arrive(&tmem_empty);
            // Hand-over buffer of this tile.  A helper reuses it two tiles later,
            // which needs the MMAs of the tile after this one, which need the
            // lead's free of that tile, which comes after the lead read this one.
            const int xb = static_cast<int>(local & 1);
            if (split > 0) {
                // helper: hand the state over to the quadrant's lead
                float *x = &xchg[xb][split - 1][0][0];
                x[0 * kBM + row_in_tile] = r.mt;
                x[1 * kBM + row_in_tile] = r.st;
                x[2 * kBM + row_in_tile] = r.dd;
                x[3 * kBM + row_in_tile] = r.mr;
                x[4 * kBM + row_in_tile] = r.sr;
                mbar_arrive(&xchg_full[xb][quad]);
                continue;
            }
            if (kEpiSplit > 1) {
                const bool got = wait_phase(&xchg_full[xb][quad], (local >> 1) & 1, &abort_flag, a.status);
                if (__any_sync(0xffffffffu, !got)) break;
#pragma unroll
                for (int h = 0; h < kEpiSplit - 1; ++h) {
                    const float *x = &xchg[xb][h][0][0];
                    Acc o;
                    o.mt = x[0 * kBM + row_in_tile];
                    o.st = x[1 * kBM + row_in_tile];
                    o.dd = x[2 * kBM + row_in_tile];
                    o.mr = x[3 * kBM + row_in_tile];
                    o.sr = x[4 * kBM + row_in_tile];
                    o.ht = o.hr = 0.f;
                    merge_acc<false>(r, o, lg_t, lg_r);
                }
                __syncwarp();
            }
            if (valid) {
                const int64_t o = i * n_n + n;
                a.part_a[o] = make_float4(r.mt, r.st, r.dd, r.mr);
                a.part_b[o] = r.sr;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// Dense copy of the active rows of both hidden tensors ([n_rows, H] bf16) into
// [A_pad, H] buffers; rows from A to the next multiple of 128 are zeroed.
__global__ void __launch_bounds__(256) gather_hidden_kernel(const WsHeader *hdr, const int2 *rowid,
                                                           const uint4 *ht, const uint4 *hr, uint4 *dt, uint4 *dr,
                                                           int vec_per_row) {
    const int64_t n_active = hdr->n_active;
    const int64_t a_pad = (n_active + kBM - 1) / kBM * kBM;
    const int64_t i = blockIdx.x;
    if (i >= a_pad) return;
    uint4 *ot = dt + i * vec_per_row;
    uint4 *orr = dr + i * vec_per_row;
    if (i < n_active) {
        const int64_t r = rowid[i].x;
        const uint4 *st = ht + r * vec_per_row;
        const uint4 *sr = hr + r * vec_per_row;
        for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
            ot[v] = st[v];
            orr[v] = sr[v];
        }
    } else {
        const uint4 z = make_uint4(0, 0, 0, 0);
        for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
            ot[v] = z;
            orr[v] = z;
        }
    }
}

// One warp per active row: lane l folds the row's vocab-tile partials n = l,
// l + 32, ... in order, the warp merges in a fixed butterfly, and lane 0 does
// the fp64 row arithmetic (same formulas as the unfused finalise).
__global__ void __launch_bounds__(256) head_finalize_kernel(const WsHeader *hdr, const int2 *rowid,
                                                           const float4 *part_a, const float *part_b,
                                                           const float2 *pick, int n_n, int64_t vocab,
                                                           float scale_t, float scale_r, float lg_t, float lg_r,
                                                           float *out_lt, float *out_lr, float *out_d,
                                                           double *dval, uint32_t *keys, uint32_t *status) {
    const int64_t n_active = hdr->n_active;
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (i >= n_active) return;
    Acc acc = acc_init();
    for (int n = lane; n < n_n; n += 32) {
        const float4 p = part_a[i * n_n + n];
        Acc o;
        o.mt = p.x;
        o.st = p.y;
        o.dd = p.z;
        o.mr = p.w;
        o.sr = part_b[i * n_n + n];
        o.ht = o.hr = 0.f;
        merge_acc<false>(acc, o, lg_t, lg_r);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Acc o;
        o.mt = __shfl_xor_sync(0xffffffffu, acc.mt, off);
        o.st = __shfl_xor_sync(0xffffffffu, acc.st, off);
        o.dd = __shfl_xor_sync(0xffffffffu, acc.dd, off);
        o.mr = __shfl_xor_sync(0xffffffffu, acc.mr, off);
        o.sr = __shfl_xor_sync(0xffffffffu, acc.sr, off);
        o.ht = o.hr = 0.f;
        merge_acc<false>(acc, o, lg_t, lg_r);
    }
    if (lane != 0) return;
    const int2 rid = rowid[i];
    const int64_t r = rid.x, id = rid.y;
    uint32_t bad = 0;
    double d;
    if (id < 0 || id >= vocab) {
        bad |= LPD_STATUS_TOKEN_OOB;
        d = CUDART_NAN;
        if (out_lt) out_lt[r] = CUDART_NAN_F;
        if (out_lr) out_lr[r] = CUDART_NAN_F;
    } else {
        // folded scales (1 without a chain): lse = s m + ln(sum), x[id] -> s x[id], exact in fp64
        const float2 xs = pick[i];
        const double mt = static_cast<double>(scale_t) * acc.mt, mr = static_cast<double>(scale_r) * acc.mr;
        const double lse_t = mt + log(static_cast<double>(acc.st));
        const double lse_r = mr + log(static_cast<double>(acc.sr));
        const double xt = static_cast<double>(scale_t) * xs.x, xr = static_cast<double>(scale_r) * xs.y;
        const double st = acc.st, sr = acc.sr, dd = acc.dd;
        const double l_ratio = fabs(dd) < 0.5 * st ? log1p(-dd / st) : log(sr / st);
        d = ((xt - xr) - (mt - mr)) + l_ratio;
        if (!(isfinite(lse_t) && isfinite(lse_r) && isfinite(xt) && isfinite(xr))) bad |= LPD_STATUS_NONFINITE;
        if (out_lt) out_lt[r] = static_cast<float>(xt - lse_t);
        if (out_lr) out_lr[r] = static_cast<float>(xr - lse_r);
    }
    if (out_d) out_d[r] = static_cast<float>(d);
    dval[i] = d;
    keys[i] = __float_as_uint(fabsf(static_cast<float>(d)));
    if (bad) atomicOr(status, bad);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// [rows, hidden] bf16 row-major, boxes of 64 (K) x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *ptr, int64_t rows, int64_t hidden, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(hidden), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(hidden) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

FusedLayout fused_layout(int64_t n_rows, int64_t hidden, int64_t vocab) {
    FusedLayout L{};
    const size_t a_pad = static_cast<size_t>((n_rows + kBM - 1) / kBM * kBM);
    const size_t n_n = static_cast<size_t>((vocab + kBN - 1) / kBN);
    const WsLayout base = ws_layout(n_rows, 0);  // no per-warp states: the head kernel writes tile partials
    size_t off = base.total;
    L.base = base;
    L.hidden_t = off;  off += align256(a_pad * static_cast<size_t>(hidden) * 2);
    L.hidden_r = off;  off += align256(a_pad * static_cast<size_t>(hidden) * 2);
    L.part_a = off;    off += align256(a_pad * n_n * sizeof(float4));
    L.part_b = off;    off += align256(a_pad * n_n * sizeof(float));
    L.total = off;
    L.a_pad = static_cast<int64_t>(a_pad);
    L.n_tiles_n = static_cast<int>(n_n);
    return L;
}

cudaError_t launch_fused(const FusedCall &c, cudaStream_t stream) {
    const FusedLayout &L = c.layout;
    char *ws = static_cast<char *>(c.workspace);
    const WsHeader *hdr = reinterpret_cast<const WsHeader *>(ws + L.base.header);
    const int2 *rowid = reinterpret_cast<const int2 *>(ws + L.base.rowid);
    void *ht = ws + L.hidden_t;
    void *hr = ws + L.hidden_r;
    float4 *part_a = reinterpret_cast<float4 *>(ws + L.part_a);
    float *part_b = reinterpret_cast<float *>(ws + L.part_b);
    float2 *pick = reinterpret_cast<float2 *>(ws + L.base.pick);
    if (L.a_pad == 0) return cudaSuccess;

    const int vec_per_row = static_cast<int>(c.hidden * 2 / 16);
    gather_hidden_kernel<<<static_cast<unsigned>(L.a_pad), 256, 0, stream>>>(
        hdr, rowid, static_cast<const uint4 *>(c.hidden_train), static_cast<const uint4 *>(c.hidden_rollout),
        static_cast<uint4 *>(ht), static_cast<uint4 *>(hr), vec_per_row);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    HeadMaps maps;
    if (!make_map(&maps.a_t, ht, L.a_pad, c.hidden, kBM) || !make_map(&maps.a_r, hr, L.a_pad, c.hidden, kBM) ||
        !make_map(&maps.w, c.weight, c.vocab, c.hidden, kBN))
        return cudaErrorInvalidValue;
    HeadArgs a{};
    a.hdr = hdr;
    a.rowid = rowid;
    a.vocab = c.vocab;
    a.hidden = static_cast<int>(c.hidden);
    a.n_tiles_n = L.n_tiles_n;
    a.part_a = part_a;
    a.part_b = part_b;
    a.pick = pick;
    a.status = c.status;
    a.xt = c.xt;
    a.xr = c.xr;
    a.lt = a.lr = kLog2e;
    // the chain's form: none, scales only, at most one soft-cap per side
    // (reduced), or general
    int chain = 0;
    float scale_t = 1.f, scale_r = 1.f;
    if (c.xt.n_ops > 0 || c.xr.n_ops > 0) {
        double post[2];
        chain = 1;
        if (reduce_softcap(c.xt, &a.cap[0], &post[0]) && reduce_softcap(c.xr, &a.cap[1], &post[1])) {
            chain = (a.cap[0].on || a.cap[1].on) ? 2 : 3;
            a.lt = static_cast<float>(post[0] * 1.4426950408889634);
            a.lr = static_cast<float>(post[1] * 1.4426950408889634);
            scale_t = static_cast<float>(post[0]);
            scale_r = static_cast<float>(post[1]);
        }
    }
    const size_t smem = static_cast<size_t>(kStages) * kStage + 1024;
    static std::atomic<uint64_t> configured[4];
    switch (chain) {
        case 0: e = set_smem_once(head_kernel<0>, smem, configured[0]); break;
        case 1: e = set_smem_once(head_kernel<1>, smem, configured[1]); break;
        case 2: e = set_smem_once(head_kernel<2>, smem, configured[2]); break;
        default: e = set_smem_once(head_kernel<3>, smem, configured[3]); break;
    }
    if (e != cudaSuccess) return e;
    switch (chain) {
        case 0: head_kernel<0><<<device_sm_count(), kHeadThreads, smem, stream>>>(maps, a); break;
        case 1: head_kernel<1><<<device_sm_count(), kHeadThreads, smem, stream>>>(maps, a); break;
        case 2: head_kernel<2><<<device_sm_count(), kHeadThreads, smem, stream>>>(maps, a); break;
        default: head_kernel<3><<<device_sm_count(), kHeadThreads, smem, stream>>>(maps, a); break;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const unsigned fin_blocks = static_cast<unsigned>((c.n_rows + 7) / 8);
    head_finalize_kernel<<<fin_blocks, 256, 0, stream>>>(
        hdr, rowid, part_a, part_b, pick, L.n_tiles_n, c.vocab, scale_t, scale_r, a.lt, a.lr, c.out_lt, c.out_lr,
        c.out_d,
        reinterpret_cast<double *>(ws + L.base.dval), reinterpret_cast<uint32_t *>(ws + L.base.keys), c.status);
    return cudaGetLastError();
}

}  // namespace lpd
