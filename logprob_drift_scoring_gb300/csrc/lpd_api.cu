// C ABI of liblpd: host-side validation, workspace carving and the stage
// sequence.  Every argument problem is caught here, before any launch, and
// returned as a negative LPD_ERR_* code (include/lpd.h).  Nothing is allocated:
// the caller passes every buffer, including the workspace.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "lpd_internal.cuh"
#include "lpd_xform.cuh"

namespace lpd {

int device_sm_count() {
    static std::atomic<int> cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

constexpr int64_t kMaxRows = INT32_MAX;   // rows are addressed as int32 in the row list
constexpr int64_t kMaxVocab = INT32_MAX;  // token ids are int32

int elt_bytes(int32_t dtype) { return dtype == LPD_BF16 ? 2 : 4; }
bool valid_dtype(int32_t dtype) { return dtype == LPD_BF16 || dtype == LPD_F32; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_clip(double lo, double hi) {
    if (!std::isfinite(lo) || !std::isfinite(hi) || !(lo > 0.0) || !(lo <= hi)) return LPD_ERR_BAD_CLIP;
    return LPD_OK;
}

int check_rows_vocab(int64_t n_rows, int64_t vocab) {
    if (n_rows < 0 || vocab <= 0) return LPD_ERR_BAD_SIZE;
    if (n_rows > kMaxRows || vocab > kMaxVocab) return LPD_ERR_UNSUPPORTED;
    return LPD_OK;
}

// Elements must sit on their natural boundary (2 bytes for bf16, 4 for fp32).
bool elt_aligned(const void *p, int32_t dtype) {
    return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(elt_bytes(dtype))) == 0;
}

int check_logits(const lpd_logits *x, int64_t n_rows, int64_t vocab) {
    if (!x) return LPD_ERR_NULL_POINTER;
    if (!x->ptr && n_rows > 0) return LPD_ERR_NULL_POINTER;
    if (!valid_dtype(x->dtype)) return LPD_ERR_BAD_DTYPE;
    if (x->row_stride < vocab) return LPD_ERR_BAD_STRIDE;
    if (!elt_aligned(x->ptr, x->dtype)) return LPD_ERR_ALIGNMENT;
    return LPD_OK;
}

int check_workspace(void *ws, size_t bytes, size_t need) {
    if (!ws) return LPD_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LPD_ERR_ALIGNMENT;
    if (bytes < need) return LPD_ERR_WORKSPACE;
    return LPD_OK;
}

struct Ws {
    WsHeader *hdr;
    int2 *rowid;
    float2 *pick;
    float4 *part;
    double *dval;
    uint32_t *keys;
    BlockPartial *blockpart;
    uint32_t *hist;
};

Ws carve(void *base, int64_t n_rows, int n_seg) {
    const WsLayout L = ws_layout(n_rows, n_seg);
    char *b = static_cast<char *>(base);
    return Ws{reinterpret_cast<WsHeader *>(b + L.header),  reinterpret_cast<int2 *>(b + L.rowid),
              reinterpret_cast<float2 *>(b + L.pick),      reinterpret_cast<float4 *>(b + L.part),
              reinterpret_cast<double *>(b + L.dval),      reinterpret_cast<uint32_t *>(b + L.keys),
              reinterpret_cast<BlockPartial *>(b + L.blockpart), reinterpret_cast<uint32_t *>(b + L.hist)};
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? LPD_OK : LPD_ERR_CUDA; }

// A row of a side can stream through the bulk-copy ring when every row
// starts on a 16-byte boundary.
bool rows_aligned(const void *ptr, int64_t stride, int32_t dtype) {
    return aligned16(ptr) && ((stride * elt_bytes(dtype)) % 16) == 0;
}

int run_select(int64_t n_rows, const int32_t *ids, const uint8_t *mask, float *lt, float *lr, float *d,
               lpd_metrics *met, const Ws &w, cudaStream_t s) {
    return cuda_status(launch_select_active(n_rows, mask, ids, lt, lr, d, met, w.hdr, w.rowid, s));
}

// LPD_STALL_ROW_PASS=1 (tests of the timeout path only): the row pass's CTA 0
// withholds its first copy, so that its bounded wait runs out.
bool stall_requested() {
    const char *v = std::getenv("LPD_STALL_ROW_PASS");
    return v && v[0] == '1' && v[1] == '\0';
}

// Stage 2: the streaming row pass, then the per-row finalise.
// Optional extras of the row pass: a transform chain per side, or entropy outputs.
struct RowExtras {
    const Xform *xform = nullptr;       // [2]: train, rollout
    float *ent_t = nullptr, *ent_r = nullptr;
    int topo = LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE;  // how the finalise reduces the segments
    const int32_t *order = nullptr;     // host, n_seg entries: segment reduction order
};

int run_rows(const Segment *segs, int n_seg, int32_t dt, int32_t dr, bool tma, const int32_t *perm, int n_perm,
             int64_t n_rows, int64_t vocab, float *lt, float *lr, float *d, float *plt, float *plr,
             lpd_metrics *met, const Ws &w, cudaStream_t s, const RowExtras &ex = RowExtras{}) {
    if (n_rows == 0) return LPD_OK;
    RowArgs a{};
    int mode = kRowPlain;
    float scale_t = 1.f, scale_r = 1.f, lg_t = kLog2e, lg_r = kLog2e;
    if (ex.xform) {
        a.xt = ex.xform[0];
        a.xr = ex.xform[1];
        mode = kRowTransform;
        // chains made only of scales collapse to one multiply per side
        bool scales_only = true;
        float prod[2] = {1.f, 1.f};
        for (int side = 0; side < 2; ++side)
            for (int k = 0; k < ex.xform[side].n_ops; ++k) {
                if (ex.xform[side].kind[k] != LPD_OP_SCALE) scales_only = false;
                prod[side] *= ex.xform[side].param[k];
            }
        double post[2];
        if (scales_only) {
            // the product of scales rides in each side's exponent factor
            a.lt = static_cast<float>(static_cast<double>(prod[0]) * 1.4426950408889634);
            a.lr = static_cast<float>(static_cast<double>(prod[1]) * 1.4426950408889634);
            scale_t = prod[0];
            scale_r = prod[1];
            lg_t = a.lt;
            lg_r = a.lr;
            mode = kRowScale;
        } else if (reduce_softcap(ex.xform[0], &a.cap[0], &post[0]) &&
                   reduce_softcap(ex.xform[1], &a.cap[1], &post[1])) {
            // one soft-cap per side at most: the soft-cap on each value, the
            // scales (moved behind it) in the exponent factor
            a.lt = static_cast<float>(post[0] * 1.4426950408889634);
            a.lr = static_cast<float>(post[1] * 1.4426950408889634);
            scale_t = static_cast<float>(post[0]);
            scale_r = static_cast<float>(post[1]);
            lg_t = a.lt;
            lg_r = a.lr;
            mode = kRowSoftcap;
        }
    } else if (ex.ent_t || ex.ent_r) {
        mode = kRowEntropy;
    }
    for (int k = 0; k < n_seg; ++k) a.seg[k] = segs[k];
    a.n_seg = n_seg;
    a.vocab = vocab;
    a.hdr = w.hdr;
    a.rowid = w.rowid;
    a.part = w.part;
    a.pick = w.pick;
    a.status = &met->status;
    a.stall = stall_requested() ? 1 : 0;
    const int warps = row_pass_warps(segs, n_seg, mode, tma);
    int rc = cuda_status(launch_rows(a, dt, dr, tma, mode, warps, s));
    if (rc) return rc;
    FinArgs f{};
    f.n_seg = n_seg;
    f.n_warps = warps;
    f.n_perm = n_perm;
    for (int j = 0; j < n_perm; ++j) f.perm[j] = static_cast<int8_t>(perm[j]);
    f.vocab = vocab;
    f.hdr = w.hdr;
    f.rowid = w.rowid;
    f.part = w.part;
    f.pick = w.pick;
    f.dval = w.dval;
    f.keys = w.keys;
    f.out_lt = lt;
    f.out_lr = lr;
    f.out_d = d;
    f.out_perm_lt = plt;
    f.out_perm_lr = plr;
    f.out_ent_t = ex.ent_t;
    f.out_ent_r = ex.ent_r;
    f.topo = ex.topo;
    f.scale_t = scale_t;
    f.scale_r = scale_r;
    f.lg_t = lg_t;
    f.lg_r = lg_r;
    if (ex.order) {
        f.n_order = n_seg;
        for (int j = 0; j < n_seg; ++j) f.order[j] = static_cast<int8_t>(ex.order[j]);
    }
    f.status = &met->status;
    return cuda_status(launch_finalize(f, n_rows, s));
}

// Stage 3: metric terms per block, then the merge and the percentile select.
int run_metrics(int64_t n_rows, double clip_lo, double clip_hi, lpd_metrics *met, const Ws &w, cudaStream_t s) {
    return cuda_status(launch_metrics(n_rows, std::log(clip_lo), std::log(clip_hi), w.hdr, w.rowid, w.dval, w.keys,
                                      w.blockpart, w.hist, met, s));
}

int validate_pair(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows, int64_t vocab) {
    int rc = check_rows_vocab(n_rows, vocab);
    if (rc) return rc;
    if ((rc = check_logits(train, n_rows, vocab))) return rc;
    if ((rc = check_logits(rollout, n_rows, vocab))) return rc;
    return LPD_OK;
}

Segment whole_vocab(const lpd_logits *t, const lpd_logits *r, int64_t vocab) {
    Segment sg{};
    sg.t = static_cast<const char *>(t->ptr);
    sg.r = static_cast<const char *>(r->ptr);
    sg.t_stride = t->row_stride * elt_bytes(t->dtype);
    sg.r_stride = r->row_stride * elt_bytes(r->dtype);
    sg.v_start = 0;
    sg.len = vocab;
    return sg;
}

// A side's chain as the kernel's copy; NULL is the identity.
int to_xform(const lpd_transform *c, Xform *out) {
    *out = Xform{};
    if (!c) return LPD_OK;
    if (c->n_ops < 0 || c->n_ops > LPD_MAX_TRANSFORM_OPS) return LPD_ERR_BAD_TRANSFORM;
    out->n_ops = c->n_ops;
    for (int k = 0; k < c->n_ops; ++k) {
        if (c->kind[k] != LPD_OP_SCALE && c->kind[k] != LPD_OP_SOFTCAP) return LPD_ERR_BAD_TRANSFORM;
        if (!std::isfinite(c->param[k]) || !(c->param[k] > 0.f)) return LPD_ERR_BAD_TRANSFORM;
        out->kind[k] = c->kind[k];
        out->param[k] = c->param[k];
    }
    return LPD_OK;
}

// Exact tiling of [0, vocab) by the shard ranges, in any array order ("fail
// closed on missing vocab-shard bounds"); on success `order` lists the shard
// indices by ascending v_start (the global vocab-shard order).
int check_shards(const lpd_shard *sh, int n, int64_t n_rows, int64_t vocab, int *order) {
    if (!sh) return LPD_ERR_NULL_POINTER;
    for (int k = 0; k < n; ++k) {
        if (!sh[k].ptr && n_rows > 0) return LPD_ERR_NULL_POINTER;
        if (!valid_dtype(sh[k].dtype)) return LPD_ERR_BAD_DTYPE;
        if (sh[k].dtype != sh[0].dtype) return LPD_ERR_BAD_DTYPE;
        if (sh[k].v_start < 0 || sh[k].v_end <= sh[k].v_start || sh[k].v_end > vocab) return LPD_ERR_BAD_SHARDS;
        if (sh[k].row_stride < sh[k].v_end - sh[k].v_start) return LPD_ERR_BAD_STRIDE;
        if (!elt_aligned(sh[k].ptr, sh[k].dtype)) return LPD_ERR_ALIGNMENT;
        order[k] = k;
    }
    std::sort(order, order + n, [&](int x, int y) { return sh[x].v_start < sh[y].v_start; });
    int64_t next = 0;
    for (int j = 0; j < n; ++j) {
        if (sh[order[j]].v_start != next) return LPD_ERR_BAD_SHARDS;
        next = sh[order[j]].v_end;
    }
    return next == vocab ? LPD_OK : LPD_ERR_BAD_SHARDS;
}

// Shared by lpd_attn_merge (diag false: no second order, no drift outputs) and
// lpd_attn_merge_order_drift (diag true: all three drift outputs required).
int attn_merge_impl(const void *out_parts, int32_t parts_dtype, const float *lse_parts, int32_t n_parts,
                    int64_t n_rows, int32_t head_dim, int32_t lse_base2, const int32_t *order_a,
                    const int32_t *order_b, float *out, float *out_lse, float *row_dout, float *row_dlse,
                    lpd_merge_drift *drift, bool diag, void *stream) {
    if (n_rows < 0 || n_rows >= 0xffffffffll || head_dim < 1 || (lse_base2 != 0 && lse_base2 != 1))
        return LPD_ERR_BAD_SIZE;
    if (n_parts < 1 || n_parts > LPD_ATTN_MAX_PARTS) return LPD_ERR_UNSUPPORTED;
    if (!valid_dtype(parts_dtype)) return LPD_ERR_BAD_DTYPE;
    if (diag && (!drift || (n_rows > 0 && (!row_dout || !row_dlse)))) return LPD_ERR_NULL_POINTER;
    if (n_rows > 0 && (!out_parts || !lse_parts || !out || !out_lse)) return LPD_ERR_NULL_POINTER;
    const int64_t row_bytes = static_cast<int64_t>(head_dim) * elt_bytes(parts_dtype);
    if (row_bytes % 16 != 0) return LPD_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(out_parts) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
        reinterpret_cast<uintptr_t>(lse_parts) % 4 || reinterpret_cast<uintptr_t>(out_lse) % 4 ||
        reinterpret_cast<uintptr_t>(row_dout) % 4 || reinterpret_cast<uintptr_t>(row_dlse) % 4 ||
        reinterpret_cast<uintptr_t>(drift) % 8)
        return LPD_ERR_ALIGNMENT;
    // chunk indices are 32-bit: at most 2^32 - 1 16-byte chunks (64 GB) per part
    const int64_t chunks = n_rows * (row_bytes / 16);
    if (chunks >= 0xffffffffll) return LPD_ERR_UNSUPPORTED;
    int32_t ident[LPD_ATTN_MAX_PARTS];
    for (int k = 0; k < n_parts; ++k) ident[k] = k;
    const int32_t *orders[2] = {order_a ? order_a : ident, order_b ? order_b : ident};
    for (const int32_t *o : orders) {
        bool seen[LPD_ATTN_MAX_PARTS] = {false};
        for (int k = 0; k < n_parts; ++k) {
            if (o[k] < 0 || o[k] >= n_parts || seen[o[k]]) return LPD_ERR_BAD_SHARDS;
            seen[o[k]] = true;
        }
    }
    AttnMergeCall c{};
    c.parts = out_parts;
    c.bf16 = parts_dtype == LPD_BF16;
    c.lse = lse_parts;
    c.n_parts = n_parts;
    c.n_rows = n_rows;
    c.head_dim = head_dim;
    c.base2 = lse_base2;
    c.order_a = orders[0];
    c.order_b = orders[1];
    c.out = out;
    c.out_lse = out_lse;
    c.diag = diag;
    c.row_dout = row_dout;
    c.row_dlse = row_dlse;
    c.drift = drift;
    return cuda_status(launch_attn_merge(c, static_cast<cudaStream_t>(stream)));
}

// Shared validation of the sharded entry points: sizes, pointers, both
// sides' shard maps (the same split on each side), and the per-shard segments
// in global vocab order with whether every row can use the bulk-copy ring.
int prepare_shards(const lpd_shard *train, const lpd_shard *rollout, int32_t n_shards, int64_t n_rows,
                   int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask, const lpd_metrics *met,
                   Segment *segs, bool *tma) {
    int rc = check_rows_vocab(n_rows, vocab);
    if (rc) return rc;
    if (n_shards < 1 || n_shards > kMaxSegments) return LPD_ERR_UNSUPPORTED;
    if (!met || ((!token_ids || !action_mask) && n_rows > 0)) return LPD_ERR_NULL_POINTER;
    int ot[kMaxSegments], orr[kMaxSegments];
    if ((rc = check_shards(train, n_shards, n_rows, vocab, ot))) return rc;
    if ((rc = check_shards(rollout, n_shards, n_rows, vocab, orr))) return rc;
    // both sides must use the same split: shard j (in vocab order) covers the
    // same range on each side
    for (int j = 0; j < n_shards; ++j)
        if (train[ot[j]].v_start != rollout[orr[j]].v_start || train[ot[j]].v_end != rollout[orr[j]].v_end)
            return LPD_ERR_BAD_SHARDS;
    *tma = true;
    for (int j = 0; j < n_shards; ++j) {
        const lpd_shard &a = train[ot[j]], &b = rollout[orr[j]];
        segs[j].t = static_cast<const char *>(a.ptr);
        segs[j].r = static_cast<const char *>(b.ptr);
        segs[j].t_stride = a.row_stride * elt_bytes(a.dtype);
        segs[j].r_stride = b.row_stride * elt_bytes(b.dtype);
        segs[j].v_start = a.v_start;
        segs[j].len = a.v_end - a.v_start;
        *tma = *tma && rows_aligned(a.ptr, a.row_stride, a.dtype) && rows_aligned(b.ptr, b.row_stride, b.dtype);
    }
    return LPD_OK;
}

// A host permutation of 0..n-1 (or NULL).
int check_order(const int32_t *order, int n) {
    if (!order) return LPD_OK;
    bool seen[kMaxSegments] = {false};
    for (int j = 0; j < n; ++j) {
        const int k = order[j];
        if (k < 0 || k >= n || seen[k]) return LPD_ERR_BAD_SHARDS;
        seen[k] = true;
    }
    return LPD_OK;
}

// Workspace of the all-gather arm: the single-segment scoring regions, then
// each side's gathered logits with rows padded to 16 bytes.
struct GatherLayout {
    size_t logits_t, logits_r, total;
    int64_t pitch_t, pitch_r;  // bytes
};

GatherLayout gather_layout(int64_t n_rows, int64_t vocab, int32_t dt, int32_t dr) {
    GatherLayout g;
    g.pitch_t = (vocab * elt_bytes(dt) + 15) / 16 * 16;
    g.pitch_r = (vocab * elt_bytes(dr) + 15) / 16 * 16;
    g.logits_t = align256(ws_layout(n_rows, 1).total);
    g.logits_r = align256(g.logits_t + static_cast<size_t>(n_rows) * g.pitch_t);
    g.total = align256(g.logits_r + static_cast<size_t>(n_rows) * g.pitch_r);
    return g;
}

}  // namespace
}  // namespace lpd

using namespace lpd;

extern "C" {

size_t lpd_workspace_size(int32_t kind, int64_t n_rows, int64_t vocab, int32_t n_shards) {
    if (n_rows < 0 || n_rows > kMaxRows) return 0;
    switch (kind) {
        case LPD_KIND_SCORE:
            return ws_layout(n_rows, 1).total;
        case LPD_KIND_SHARDED:
            if (n_shards < 1 || n_shards > kMaxSegments) return 0;
            return ws_layout(n_rows, n_shards).total;
        default:
            (void)vocab;
            return 0;
    }
}

int lpd_backend_info(lpd_backend_info_t *info) {
    if (!info) return LPD_ERR_NULL_POINTER;
    std::memset(info, 0, sizeof(*info));
    std::snprintf(info->backend_id, sizeof info->backend_id, "lpd.sm103a.v1");
    std::snprintf(info->op_name, sizeof info->op_name, "selected_logprob_drift");
    std::snprintf(info->arch, sizeof info->arch, "sm_103a");
    std::snprintf(info->dtypes, sizeof info->dtypes, "bf16,f32");
    info->deterministic = 1;
    info->batch_invariant = 1;
#ifdef __USE_FAST_MATH__
    info->fast_math = 1;
#else
    info->fast_math = 0;
#endif
    info->has_fallback = 0;
    std::snprintf(info->fingerprint, sizeof info->fingerprint, "nvcc %d.%d sm_103a %s %s", __CUDACC_VER_MAJOR__,
                  __CUDACC_VER_MINOR__, __DATE__, __TIME__);
    return LPD_OK;
}

const char *lpd_strerror(int code) {
    switch (code) {
        case LPD_OK: return "success";
        case LPD_ERR_NULL_POINTER: return "a required pointer is NULL";
        case LPD_ERR_BAD_SIZE: return "invalid size (n_rows < 0, vocab <= 0, hidden <= 0 or similar)";
        case LPD_ERR_BAD_DTYPE: return "unsupported or mixed element type";
        case LPD_ERR_BAD_STRIDE: return "row stride smaller than the number of columns";
        case LPD_ERR_BAD_CLIP: return "clip bounds must be finite with 0 < lo <= hi";
        case LPD_ERR_BAD_SHARDS: return "vocab shards do not tile [0, vocab) exactly";
        case LPD_ERR_WORKSPACE: return "workspace missing or smaller than lpd_workspace_size()";
        case LPD_ERR_CUDA: return "a CUDA runtime call failed";
        case LPD_ERR_ALIGNMENT: return "a pointer or stride breaks an alignment rule";
        case LPD_ERR_UNSUPPORTED: return "size outside what this library supports";
        case LPD_ERR_BAD_TRANSFORM: return "transform chain: bad op count, kind or parameter";
        case LPD_ERR_BAD_MEMORY: return "a host-side argument points to device memory";
        case static_cast<int>(LPD_STATUS_TOKEN_OOB): return "status: active token id outside [0, vocab)";
        case static_cast<int>(LPD_STATUS_NONFINITE): return "status: non-finite log-sum-exp or selected logit";
        case static_cast<int>(LPD_STATUS_TIMEOUT): return "status: an internal pipeline wait gave up";
        default: return "unknown code";
    }
}

int lpd_select_active(int64_t n_rows, const int32_t *token_ids, const uint8_t *action_mask, float *out_logp_train,
                      float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (n_rows < 0) return LPD_ERR_BAD_SIZE;
    if (n_rows > kMaxRows) return LPD_ERR_UNSUPPORTED;
    if (!out_metrics || ((!token_ids || !action_mask) && n_rows > 0)) return LPD_ERR_NULL_POINTER;
    int rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0));
    if (rc) return rc;
    const Ws w = carve(workspace, n_rows, 1);
    return run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics, w,
                      static_cast<cudaStream_t>(stream));
}

int lpd_token_logp(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows, int64_t vocab,
                   float *out_logp_train, float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
                   void *workspace, size_t workspace_bytes, void *stream) {
    int rc = validate_pair(train, rollout, n_rows, vocab);
    if (rc) return rc;
    if (!out_metrics) return LPD_ERR_NULL_POINTER;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const Ws w = carve(workspace, n_rows, 1);
    const Segment sg = whole_vocab(train, rollout, vocab);
    const bool tma = rows_aligned(train->ptr, train->row_stride, train->dtype) &&
                     rows_aligned(rollout->ptr, rollout->row_stride, rollout->dtype);
    return run_rows(&sg, 1, train->dtype, rollout->dtype, tma, nullptr, 0, n_rows, vocab, out_logp_train,
                    out_logp_rollout, out_dlogp, nullptr, nullptr, out_metrics, w, static_cast<cudaStream_t>(stream));
}

int lpd_drift_metrics(int64_t n_rows, double clip_lo, double clip_hi, lpd_metrics *out_metrics, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (n_rows < 0) return LPD_ERR_BAD_SIZE;
    if (n_rows > kMaxRows) return LPD_ERR_UNSUPPORTED;
    if (!out_metrics) return LPD_ERR_NULL_POINTER;
    int rc = check_clip(clip_lo, clip_hi);
    if (rc) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const Ws w = carve(workspace, n_rows, 1);
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, static_cast<cudaStream_t>(stream));
}

int lpd_merge_rank_metrics(const lpd_metrics *per_rank, const int64_t *row_offsets, int32_t n_ranks,
                           lpd_metrics *out) {
    if (!per_rank || !out) return LPD_ERR_NULL_POINTER;
    if (n_ranks < 1) return LPD_ERR_BAD_SIZE;
    for (int k = 0; k < n_ranks; ++k)
        if (per_rank[k].n_active < 0) return LPD_ERR_BAD_SIZE;
    lpd_metrics m{};
    m.argmax_row = -1;
    double best = -1.0;
    for (int k = 0; k < n_ranks; ++k) {
        const lpd_metrics &r = per_rank[k];
        m.status |= r.status;
        const int64_t a = r.n_active;
        if (a == 0) continue;
        m.n_active += a;
        const double w = static_cast<double>(a);
        m.ratio0_mean += r.ratio0_mean * w;
        m.clipfrac0 += r.clipfrac0 * w;
        m.approx_kl0 += r.approx_kl0 * w;
        m.mean_abs_dlogp += r.mean_abs_dlogp * w;
        if (r.max_abs_dlogp > best) {  // strict: an earlier rank's rows come first
            best = r.max_abs_dlogp;
            m.max_abs_dlogp = best;
            m.argmax_row = r.argmax_row + (row_offsets ? row_offsets[k] : 0);
        }
    }
    if (m.n_active > 0) {
        const double total = static_cast<double>(m.n_active);
        m.ratio0_mean /= total;
        m.clipfrac0 /= total;
        m.approx_kl0 /= total;
        m.mean_abs_dlogp /= total;
        m.p95_abs_dlogp = m.p99_abs_dlogp = std::nan("");
        m.flags = LPD_FLAG_NO_PERCENTILES;
    } else {
        m.flags = LPD_FLAG_NO_ACTIVE;
    }
    *out = m;
    return LPD_OK;
}

int lpd_drift_metrics_from_dlogp(int64_t n_rows, const float *dlogp, const uint8_t *action_mask, double clip_lo,
                                 double clip_hi, lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    if (n_rows < 0) return LPD_ERR_BAD_SIZE;
    if (n_rows > kMaxRows) return LPD_ERR_UNSUPPORTED;
    if (!out_metrics || (n_rows > 0 && (!dlogp || !action_mask))) return LPD_ERR_NULL_POINTER;
    int rc = check_clip(clip_lo, clip_hi);
    if (rc) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Ws w = carve(workspace, n_rows, 1);
    if ((rc = cuda_status(launch_select_active(n_rows, action_mask, nullptr, nullptr, nullptr, nullptr, out_metrics,
                                               w.hdr, w.rowid, s))))
        return rc;
    if ((rc = cuda_status(launch_dlogp_rows(n_rows, dlogp, w.hdr, w.rowid, w.dval, w.keys, &out_metrics->status, s))))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

int lpd_score(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows, int64_t vocab,
              const int32_t *token_ids, const uint8_t *action_mask, double clip_lo, double clip_hi,
              float *out_logp_train, float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
              void *workspace, size_t workspace_bytes, void *stream) {
    int rc = validate_pair(train, rollout, n_rows, vocab);
    if (rc) return rc;
    if (!out_metrics || ((!token_ids || !action_mask) && n_rows > 0)) return LPD_ERR_NULL_POINTER;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Ws w = carve(workspace, n_rows, 1);
    const Segment sg = whole_vocab(train, rollout, vocab);
    const bool tma = rows_aligned(train->ptr, train->row_stride, train->dtype) &&
                     rows_aligned(rollout->ptr, rollout->row_stride, rollout->dtype);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    if ((rc = run_rows(&sg, 1, train->dtype, rollout->dtype, tma, nullptr, 0, n_rows, vocab, out_logp_train,
                       out_logp_rollout, out_dlogp, nullptr, nullptr, out_metrics, w, s)))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

int lpd_score_host(const lpd_logits *train_host, const lpd_logits *rollout_host, const lpd_logits *train_dev,
                   const lpd_logits *rollout_dev, int64_t n_rows, int64_t vocab, const int32_t *token_ids_host,
                   const uint8_t *action_mask_host, int32_t *token_ids_dev, uint8_t *action_mask_dev, double clip_lo,
                   double clip_hi, float *out_logp_train, float *out_logp_rollout, float *out_dlogp,
                   lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes, int64_t *out_h2d_bytes,
                   void *stream) {
    if (out_h2d_bytes) *out_h2d_bytes = 0;
    int rc = validate_pair(train_host, rollout_host, n_rows, vocab);
    if (rc || (rc = validate_pair(train_dev, rollout_dev, n_rows, vocab))) return rc;
    if (train_host->dtype != train_dev->dtype || rollout_host->dtype != rollout_dev->dtype) return LPD_ERR_BAD_DTYPE;
    if (!out_metrics ||
        ((!token_ids_host || !action_mask_host || !token_ids_dev || !action_mask_dev) && n_rows > 0))
        return LPD_ERR_NULL_POINTER;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    if (n_rows > 0) {
        // the mask is read right here on the host: device memory would fault
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, action_mask_host) == cudaSuccess && pa.type == cudaMemoryTypeDevice)
            return LPD_ERR_BAD_MEMORY;
        cudaGetLastError();  // a failed query leaves no sticky error behind
    }
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    int64_t bytes = 0;
    if (n_rows > 0) {
        const size_t n = static_cast<size_t>(n_rows);
        if ((rc = cuda_status(cudaMemcpyAsync(token_ids_dev, token_ids_host, n * sizeof(int32_t),
                                              cudaMemcpyHostToDevice, s))) ||
            (rc = cuda_status(cudaMemcpyAsync(action_mask_dev, action_mask_host, n, cudaMemcpyHostToDevice, s))))
            return rc;
        bytes += static_cast<int64_t>(n * (sizeof(int32_t) + 1));
        const lpd_logits *side_h[2] = {train_host, rollout_host}, *side_d[2] = {train_dev, rollout_dev};
        for (int64_t r0 = 0; r0 < n_rows;) {
            if (!action_mask_host[r0]) {
                ++r0;
                continue;
            }
            int64_t r1 = r0 + 1;
            while (r1 < n_rows && action_mask_host[r1]) ++r1;
            for (int k = 0; k < 2; ++k) {
                const size_t eb = static_cast<size_t>(elt_bytes(side_h[k]->dtype));
                const size_t ph = static_cast<size_t>(side_h[k]->row_stride) * eb;
                const size_t pd = static_cast<size_t>(side_d[k]->row_stride) * eb;
                const size_t width = static_cast<size_t>(vocab) * eb;
                // the device descriptor names the staging buffer this call fills
                char *dst = static_cast<char *>(const_cast<void *>(side_d[k]->ptr)) + r0 * pd;
                const char *src = static_cast<const char *>(side_h[k]->ptr) + r0 * ph;
                if ((rc = cuda_status(cudaMemcpy2DAsync(dst, pd, src, ph, width, static_cast<size_t>(r1 - r0),
                                                        cudaMemcpyHostToDevice, s))))
                    return rc;
                bytes += static_cast<int64_t>(width) * (r1 - r0);
            }
            r0 = r1;
        }
    }
    if (out_h2d_bytes) *out_h2d_bytes = bytes;
    return lpd_score(train_dev, rollout_dev, n_rows, vocab, token_ids_dev, action_mask_dev, clip_lo, clip_hi,
                     out_logp_train, out_logp_rollout, out_dlogp, out_metrics, workspace, workspace_bytes, stream);
}

int lpd_score_transformed(const lpd_logits *train, const lpd_logits *rollout, const lpd_transform *train_chain,
                          const lpd_transform *rollout_chain, int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                          const uint8_t *action_mask, double clip_lo, double clip_hi, float *out_logp_train,
                          float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics, void *workspace,
                          size_t workspace_bytes, void *stream) {
    int rc = validate_pair(train, rollout, n_rows, vocab);
    if (rc) return rc;
    if (!out_metrics || ((!token_ids || !action_mask) && n_rows > 0)) return LPD_ERR_NULL_POINTER;
    Xform xf[2];
    if ((rc = to_xform(train_chain, &xf[0])) || (rc = to_xform(rollout_chain, &xf[1]))) return rc;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Ws w = carve(workspace, n_rows, 1);
    const Segment sg = whole_vocab(train, rollout, vocab);
    const bool tma = rows_aligned(train->ptr, train->row_stride, train->dtype) &&
                     rows_aligned(rollout->ptr, rollout->row_stride, rollout->dtype);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    RowExtras ex;
    if (xf[0].n_ops > 0 || xf[1].n_ops > 0) ex.xform = xf;
    if ((rc = run_rows(&sg, 1, train->dtype, rollout->dtype, tma, nullptr, 0, n_rows, vocab, out_logp_train,
                       out_logp_rollout, out_dlogp, nullptr, nullptr, out_metrics, w, s, ex)))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

int lpd_score_entropy(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows, int64_t vocab,
                      const int32_t *token_ids, const uint8_t *action_mask, double clip_lo, double clip_hi,
                      float *out_logp_train, float *out_logp_rollout, float *out_dlogp, float *out_entropy_train,
                      float *out_entropy_rollout, lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                      void *stream) {
    int rc = validate_pair(train, rollout, n_rows, vocab);
    if (rc) return rc;
    if (!out_metrics || ((!token_ids || !action_mask) && n_rows > 0)) return LPD_ERR_NULL_POINTER;
    if (!out_entropy_train && !out_entropy_rollout) return LPD_ERR_NULL_POINTER;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_workspace_size(LPD_KIND_SCORE, n_rows, 0, 0))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Ws w = carve(workspace, n_rows, 1);
    const Segment sg = whole_vocab(train, rollout, vocab);
    const bool tma = rows_aligned(train->ptr, train->row_stride, train->dtype) &&
                     rows_aligned(rollout->ptr, rollout->row_stride, rollout->dtype);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    // inactive rows get entropy 0, like the other per-token outputs
    if (out_entropy_train && n_rows > 0 &&
        (rc = cuda_status(cudaMemsetAsync(out_entropy_train, 0, n_rows * sizeof(float), s))))
        return rc;
    if (out_entropy_rollout && n_rows > 0 &&
        (rc = cuda_status(cudaMemsetAsync(out_entropy_rollout, 0, n_rows * sizeof(float), s))))
        return rc;
    RowExtras ex;
    ex.ent_t = out_entropy_train;
    ex.ent_r = out_entropy_rollout;
    if ((rc = run_rows(&sg, 1, train->dtype, rollout->dtype, tma, nullptr, 0, n_rows, vocab, out_logp_train,
                       out_logp_rollout, out_dlogp, nullptr, nullptr, out_metrics, w, s, ex)))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

int lpd_logprob_backward(const lpd_logits *logits, int64_t n_rows, int64_t vocab, const int32_t *token_ids,
                         const uint8_t *action_mask, const float *logp, const float *grad_logp, void *out_dlogits,
                         int32_t out_dtype, int64_t out_row_stride, void *stream) {
    int rc = check_rows_vocab(n_rows, vocab);
    if (rc) return rc;
    if ((rc = check_logits(logits, n_rows, vocab))) return rc;
    if (n_rows > 0 && (!token_ids || !action_mask || !logp || !grad_logp || !out_dlogits))
        return LPD_ERR_NULL_POINTER;
    if (!valid_dtype(out_dtype)) return LPD_ERR_BAD_DTYPE;
    if (out_row_stride < vocab) return LPD_ERR_BAD_STRIDE;
    if (!elt_aligned(out_dlogits, out_dtype)) return LPD_ERR_ALIGNMENT;
    return cuda_status(launch_backward(logits->ptr, logits->dtype, logits->row_stride, out_dlogits, out_dtype,
                                       out_row_stride, n_rows, vocab, token_ids, action_mask, logp, grad_logp,
                                       static_cast<cudaStream_t>(stream)));
}

int lpd_score_sharded(const lpd_shard *train, const lpd_shard *rollout, int32_t n_shards, int64_t n_rows,
                      int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask, double clip_lo,
                      double clip_hi, const int32_t *merge_perm, float *out_logp_train, float *out_logp_rollout,
                      float *out_dlogp, float *out_perm_logp_train, float *out_perm_logp_rollout,
                      lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes, void *stream) {
    Segment segs[kMaxSegments];
    bool tma = true;
    int rc = prepare_shards(train, rollout, n_shards, n_rows, vocab, token_ids, action_mask, out_metrics, segs, &tma);
    if (rc) return rc;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_order(merge_perm, n_shards))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes,
                              lpd_workspace_size(LPD_KIND_SHARDED, n_rows, vocab, n_shards))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Ws w = carve(workspace, n_rows, n_shards);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    if (merge_perm && (out_perm_logp_train || out_perm_logp_rollout)) {
        // zero the diagnostic outputs of inactive rows as stage 1 does for the others
        if (out_perm_logp_train && (rc = cuda_status(cudaMemsetAsync(out_perm_logp_train, 0, n_rows * sizeof(float), s))))
            return rc;
        if (out_perm_logp_rollout && (rc = cuda_status(cudaMemsetAsync(out_perm_logp_rollout, 0, n_rows * sizeof(float), s))))
            return rc;
    }
    if ((rc = run_rows(segs, n_shards, train[0].dtype, rollout[0].dtype, tma, merge_perm, merge_perm ? n_shards : 0,
                       n_rows, vocab, out_logp_train, out_logp_rollout, out_dlogp, out_perm_logp_train,
                       out_perm_logp_rollout, out_metrics, w, s)))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

size_t lpd_topology_workspace_size(int32_t topology, int64_t n_rows, int64_t vocab, int32_t n_shards,
                                   int32_t dtype_train, int32_t dtype_rollout) {
    if (n_rows < 0 || n_rows > kMaxRows || vocab <= 0 || vocab > kMaxVocab || n_shards < 1 ||
        n_shards > kMaxSegments || !valid_dtype(dtype_train) || !valid_dtype(dtype_rollout))
        return 0;
    switch (topology) {
        case LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE:
        case LPD_TOPO_ALLREDUCE_PARTIALS:
            return ws_layout(n_rows, n_shards).total;
        case LPD_TOPO_ALLGATHER_LOGITS: {
            const GatherLayout g = gather_layout(n_rows, vocab, dtype_train, dtype_rollout);
            return g.total;
        }
        default:
            return 0;
    }
}

int lpd_logp_drift_summary(int64_t n_rows, const float *logp_train_a, const float *logp_rollout_a,
                           const float *logp_train_b, const float *logp_rollout_b, const uint8_t *action_mask,
                           lpd_logp_drift *out, void *stream) {
    if (n_rows < 0) return LPD_ERR_BAD_SIZE;
    if (n_rows >= 0xffffffffll) return LPD_ERR_UNSUPPORTED;  // rows travel as 32 bits in the max keys
    if (!out || (n_rows > 0 && (!logp_train_a || !logp_rollout_a || !logp_train_b || !logp_rollout_b ||
                                !action_mask)))
        return LPD_ERR_NULL_POINTER;
    if (reinterpret_cast<uintptr_t>(out) % 8 || reinterpret_cast<uintptr_t>(logp_train_a) % 4 ||
        reinterpret_cast<uintptr_t>(logp_rollout_a) % 4 || reinterpret_cast<uintptr_t>(logp_train_b) % 4 ||
        reinterpret_cast<uintptr_t>(logp_rollout_b) % 4)
        return LPD_ERR_ALIGNMENT;
    return cuda_status(launch_logp_drift(n_rows, logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b,
                                         action_mask, out, static_cast<cudaStream_t>(stream)));
}

int lpd_score_sharded_topology(const lpd_shard *train, const lpd_shard *rollout, int32_t n_shards, int64_t n_rows,
                               int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask, double clip_lo,
                               double clip_hi, int32_t topology, const int32_t *reduce_order, float *out_logp_train,
                               float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics, void *workspace,
                               size_t workspace_bytes, void *stream) {
    if (topology != LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE && topology != LPD_TOPO_ALLREDUCE_PARTIALS &&
        topology != LPD_TOPO_ALLGATHER_LOGITS)
        return LPD_ERR_UNSUPPORTED;
    Segment segs[kMaxSegments];
    bool tma = true;
    int rc = prepare_shards(train, rollout, n_shards, n_rows, vocab, token_ids, action_mask, out_metrics, segs, &tma);
    if (rc) return rc;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if (topology != LPD_TOPO_ALLGATHER_LOGITS && (rc = check_order(reduce_order, n_shards))) return rc;
    const int32_t dt = train[0].dtype, dr = rollout[0].dtype;
    if ((rc = check_workspace(workspace, workspace_bytes,
                              lpd_topology_workspace_size(topology, n_rows, vocab, n_shards, dt, dr))))
        return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (topology == LPD_TOPO_ALLGATHER_LOGITS) {
        // the all-gather: every shard's columns of every row into one full row per side
        const GatherLayout g = gather_layout(n_rows, vocab, dt, dr);
        char *base = static_cast<char *>(workspace);
        char *gt = base + g.logits_t, *gr = base + g.logits_r;
        if ((rc = cuda_status(launch_gather_shards(segs, n_shards, n_rows, gt, g.pitch_t, elt_bytes(dt), gr,
                                                   g.pitch_r, elt_bytes(dr), s))))
            return rc;
        Segment whole{};
        whole.t = gt;
        whole.r = gr;
        whole.t_stride = g.pitch_t;
        whole.r_stride = g.pitch_r;
        whole.v_start = 0;
        whole.len = vocab;
        const Ws w = carve(workspace, n_rows, 1);
        if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp,
                             out_metrics, w, s)))
            return rc;
        if ((rc = run_rows(&whole, 1, dt, dr, true, nullptr, 0, n_rows, vocab, out_logp_train, out_logp_rollout,
                           out_dlogp, nullptr, nullptr, out_metrics, w, s)))
            return rc;
        return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
    }
    const Ws w = carve(workspace, n_rows, n_shards);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    RowExtras ex;
    ex.topo = topology;
    ex.order = reduce_order;
    if ((rc = run_rows(segs, n_shards, dt, dr, tma, nullptr, 0, n_rows, vocab, out_logp_train, out_logp_rollout,
                       out_dlogp, nullptr, nullptr, out_metrics, w, s, ex)))
        return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

int lpd_attn_merge(const void *out_parts, int32_t parts_dtype, const float *lse_parts, int32_t n_parts, int64_t n_rows,
                   int32_t head_dim, int32_t lse_base2, const int32_t *order, float *out, float *out_lse,
                   void *stream) {
    return attn_merge_impl(out_parts, parts_dtype, lse_parts, n_parts, n_rows, head_dim, lse_base2, order, nullptr,
                           out, out_lse, nullptr, nullptr, nullptr, false, stream);
}

int lpd_attn_merge_order_drift(const void *out_parts, int32_t parts_dtype, const float *lse_parts, int32_t n_parts,
                               int64_t n_rows, int32_t head_dim, int32_t lse_base2, const int32_t *order_a,
                               const int32_t *order_b, float *out, float *out_lse, float *row_dout, float *row_dlse,
                               lpd_merge_drift *drift, void *stream) {
    return attn_merge_impl(out_parts, parts_dtype, lse_parts, n_parts, n_rows, head_dim, lse_base2, order_a, order_b,
                           out, out_lse, row_dout, row_dlse, drift, true, stream);
}

size_t lpd_fused_workspace_size(int64_t n_rows, int64_t hidden, int64_t vocab) {
    if (n_rows < 0 || n_rows > kMaxRows || hidden <= 0 || hidden % 64 != 0 || vocab <= 0 || vocab > kMaxVocab)
        return 0;
    return fused_layout(n_rows, hidden, vocab).total;
}

int lpd_score_fused(const void *hidden_train, const void *hidden_rollout, const void *W, int64_t n_rows,
                    int64_t hidden, int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask,
                    double clip_lo, double clip_hi, float *out_logp_train, float *out_logp_rollout,
                    float *out_dlogp, lpd_metrics *out_metrics, void *workspace, size_t workspace_bytes,
                    void *stream) {
    return lpd_score_fused_transformed(hidden_train, hidden_rollout, W, nullptr, nullptr, n_rows, hidden, vocab,
                                       token_ids, action_mask, clip_lo, clip_hi, out_logp_train, out_logp_rollout,
                                       out_dlogp, out_metrics, workspace, workspace_bytes, stream);
}

int lpd_score_fused_transformed(const void *hidden_train, const void *hidden_rollout, const void *W,
                                const lpd_transform *train_chain, const lpd_transform *rollout_chain,
                                int64_t n_rows, int64_t hidden, int64_t vocab, const int32_t *token_ids,
                                const uint8_t *action_mask, double clip_lo, double clip_hi, float *out_logp_train,
                                float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
                                void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_rows_vocab(n_rows, vocab);
    if (rc) return rc;
    if (hidden <= 0) return LPD_ERR_BAD_SIZE;
    if (hidden % 64 != 0 || hidden > (1 << 20)) return LPD_ERR_ALIGNMENT;
    if (!out_metrics || !W || ((!token_ids || !action_mask || !hidden_train || !hidden_rollout) && n_rows > 0))
        return LPD_ERR_NULL_POINTER;
    if (!aligned16(hidden_train) || !aligned16(hidden_rollout) || !aligned16(W)) return LPD_ERR_ALIGNMENT;
    if ((rc = check_clip(clip_lo, clip_hi))) return rc;
    if ((rc = check_workspace(workspace, workspace_bytes, lpd_fused_workspace_size(n_rows, hidden, vocab))))
        return rc;
    Xform xt, xr;
    if ((rc = to_xform(train_chain, &xt)) || (rc = to_xform(rollout_chain, &xr))) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    FusedCall c{};
    c.xt = xt;
    c.xr = xr;
    c.layout = fused_layout(n_rows, hidden, vocab);
    c.workspace = workspace;
    c.hidden_train = hidden_train;
    c.hidden_rollout = hidden_rollout;
    c.weight = W;
    c.n_rows = n_rows;
    c.hidden = hidden;
    c.vocab = vocab;
    c.out_lt = out_logp_train;
    c.out_lr = out_logp_rollout;
    c.out_d = out_dlogp;
    c.status = &out_metrics->status;
    const Ws w = carve(workspace, n_rows, 0);
    if ((rc = run_select(n_rows, token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                         w, s)))
        return rc;
    if ((rc = cuda_status(launch_fused(c, s)))) return rc;
    return run_metrics(n_rows, clip_lo, clip_hi, out_metrics, w, s);
}

}  // extern "C"
