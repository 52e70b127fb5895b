// lpd_score_noalloc: lpd_score for callers that cannot allocate device memory.
//
// Some callers of a scorer like this one have no way to obtain device memory
// of their own: a hook running inside another engine whose caching allocator
// owns the whole device (a raw cudaMalloc there bypasses its memory accounting
// and can fail or fragment its pool), or a plugin host that hands its plugins
// only a stream and the tensors to work on.  Such callers still pass inputs
// and outputs, but cannot pass the workspace lpd_score needs.  This entry
// point supplies that workspace from a fixed-size array of device memory that
// the library itself declares at file scope and that every GPU loading the
// library holds until the process exits.
//
// The pages describe no such entry point; it exists only for the reason above.
//
// Set-up: the first call on each device, with that device current, looks up
// the array's device address (cudaGetSymbolAddress); that first call should
// therefore come before any stream capture on that device.  Later calls reuse
// the cached address as long as the device's context is the same one: the
// cache is keyed on the context's unique id, so after a device reset (a new
// primary context, into which the library's module is loaded afresh, possibly
// at another address) the next call looks the address up again instead of
// writing through a stale pointer.  Calls allocate nothing (no cudaMalloc,
// cudaFree or allocating library routine).
//
// Sharing: every call on a device uses the same array, and the array keeps
// whatever the previous call left there.  Nothing in it needs to start at zero:
// within one call every region of the workspace is written before it is read.
// Two calls whose work overlaps on the GPU (different streams, or different
// host threads without ordering) race on the array and give wrong results;
// order them on one stream, or use lpd_score with separate workspaces.
#include <cuda.h>

#include <mutex>

#include "lpd_internal.cuh"

namespace {

constexpr size_t kScratchBytes = lpd::ws_layout(LPD_NOALLOC_MAX_ROWS, 1).total;
constexpr int kMaxDevices = 64;

// The workspace of lpd_score for up to LPD_NOALLOC_MAX_ROWS rows.  In host
// code this name is only a stand-in for the device array; its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Per device: the id of the context the address was looked up in, and the
// address.  Guarded by g_lock (host threads may make their first call on a
// device at the same time).
struct ScratchSlot {
    unsigned long long ctx_id;
    void *addr;
};
ScratchSlot g_slot[kMaxDevices] = {};
std::mutex g_lock;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// The CUDA driver API's cuCtxGetCurrent and cuCtxGetId, fetched once through
// the runtime (the library links only the CUDA runtime).
bool driver_ctx_fns(CtxGetCurrentFn *get_current, CtxGetIdFn *get_id) {
    static CtxGetCurrentFn s_cur = nullptr;
    static CtxGetIdFn s_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            s_cur = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            s_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    *get_current = s_cur;
    *get_id = s_id;
    return s_cur != nullptr && s_id != nullptr;
}

// Unique id of the context current on this thread (the one the runtime uses
// for the current device); 0 when none is current yet.
int current_ctx_id(unsigned long long *id) {
    CtxGetCurrentFn get_current;
    CtxGetIdFn get_id;
    if (!driver_ctx_fns(&get_current, &get_id)) return LPD_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return LPD_ERR_CUDA;
    *id = 0;
    if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return LPD_ERR_CUDA;
    return LPD_OK;
}

// Device address of g_scratch in the current device's context, looked up once
// per context.
int scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LPD_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LPD_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    int rc = current_ctx_id(&id);
    if (rc != LPD_OK) return rc;
    std::lock_guard<std::mutex> hold(g_lock);
    if (id != 0 && g_slot[dev].ctx_id == id && g_slot[dev].addr != nullptr) {
        *out = g_slot[dev].addr;
        return LPD_OK;
    }
    // first call in this context (or no context yet: the lookup creates the
    // device's primary context and makes it current)
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return LPD_ERR_CUDA;
    if (id == 0 && ((rc = current_ctx_id(&id)) != LPD_OK || id == 0)) return rc != LPD_OK ? rc : LPD_ERR_CUDA;
    g_slot[dev].ctx_id = id;
    g_slot[dev].addr = p;
    *out = p;
    return LPD_OK;
}

}  // namespace

extern "C" int lpd_score_noalloc(const lpd_logits *train, const lpd_logits *rollout, int64_t n_rows,
                                 int64_t vocab, const int32_t *token_ids, const uint8_t *action_mask,
                                 double clip_lo, double clip_hi, float *out_logp_train,
                                 float *out_logp_rollout, float *out_dlogp, lpd_metrics *out_metrics,
                                 void *stream) {
    if (n_rows < 0) return LPD_ERR_BAD_SIZE;
    if (n_rows > LPD_NOALLOC_MAX_ROWS) return LPD_ERR_UNSUPPORTED;  // the array is sized for this many rows
    void *ws = nullptr;
    const int rc = scratch_on_current_device(&ws);
    if (rc != LPD_OK) return rc;
    return lpd_score(train, rollout, n_rows, vocab, token_ids, action_mask, clip_lo, clip_hi, out_logp_train,
                     out_logp_rollout, out_dlogp, out_metrics, ws, kScratchBytes, stream);
}
