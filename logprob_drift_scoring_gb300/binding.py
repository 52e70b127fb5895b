"""Thin Python binding of liblpd (include/lpd.h): same names, marshalling only.

Every function here converts torch tensors to the C structs and pointers of
the C ABI and calls the library; all arithmetic runs in the CUDA kernels.
There is no CPU or library fallback: if liblpd.so cannot be loaded (or
built), importing the binding fails.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

from . import _build

# ---- constants (mirror include/lpd.h) --------------------------------------
LPD_BF16, LPD_F32 = 0, 1
LPD_OK = 0
LPD_ERR_NULL_POINTER = -1
LPD_ERR_BAD_SIZE = -2
LPD_ERR_BAD_DTYPE = -3
LPD_ERR_BAD_STRIDE = -4
LPD_ERR_BAD_CLIP = -5
LPD_ERR_BAD_SHARDS = -6
LPD_ERR_WORKSPACE = -7
LPD_ERR_CUDA = -8
LPD_ERR_ALIGNMENT = -9
LPD_ERR_UNSUPPORTED = -10
LPD_ERR_BAD_TRANSFORM = -11
LPD_ERR_BAD_MEMORY = -12
LPD_OP_SCALE, LPD_OP_SOFTCAP = 1, 2
LPD_STATUS_TOKEN_OOB = 1
LPD_STATUS_NONFINITE = 2
LPD_STATUS_TIMEOUT = 4
LPD_FLAG_NO_ACTIVE = 1
LPD_FLAG_NO_PERCENTILES = 2
LPD_KIND_SCORE, LPD_KIND_SHARDED = 0, 1
LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE, LPD_TOPO_ALLREDUCE_PARTIALS, LPD_TOPO_ALLGATHER_LOGITS = 0, 1, 2
TOPOLOGIES = {"allgather_partials_fixed_merge": 0, "allreduce_partials": 1, "allgather_logits": 2}


class LpdLogits(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("row_stride", ctypes.c_int64)]


class LpdShard(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("row_stride", ctypes.c_int64), ("v_start", ctypes.c_int64), ("v_end", ctypes.c_int64)]


class LpdTransform(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("kind", ctypes.c_int32 * 4), ("param", ctypes.c_float * 4)]


def transform_struct(ops):
    """lpd_transform from [(kind, param), ...] applied in order; None for the identity."""
    if ops is None:
        return None
    t = LpdTransform()
    t.n_ops = len(ops)
    for i, (k, p) in enumerate(ops):
        t.kind[i] = k
        t.param[i] = p
    return t


class LpdMetrics(ctypes.Structure):
    _fields_ = [("n_active", ctypes.c_int64), ("argmax_row", ctypes.c_int64), ("flags", ctypes.c_uint32),
                ("status", ctypes.c_uint32), ("ratio0_mean", ctypes.c_double), ("clipfrac0", ctypes.c_double),
                ("approx_kl0", ctypes.c_double), ("mean_abs_dlogp", ctypes.c_double),
                ("p95_abs_dlogp", ctypes.c_double), ("p99_abs_dlogp", ctypes.c_double),
                ("max_abs_dlogp", ctypes.c_double)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class LpdBackendInfo(ctypes.Structure):
    _fields_ = [("backend_id", ctypes.c_char * 32), ("op_name", ctypes.c_char * 48), ("arch", ctypes.c_char * 16),
                ("dtypes", ctypes.c_char * 32), ("deterministic", ctypes.c_int32),
                ("batch_invariant", ctypes.c_int32), ("fast_math", ctypes.c_int32),
                ("has_fallback", ctypes.c_int32), ("fingerprint", ctypes.c_char * 96)]


METRICS_BYTES = ctypes.sizeof(LpdMetrics)


class LpdMergeDrift(ctypes.Structure):
    _fields_ = [("max_abs_dout", ctypes.c_double), ("max_abs_dlse", ctypes.c_double),
                ("row_dout", ctypes.c_int64), ("row_dlse", ctypes.c_int64), ("scratch", ctypes.c_uint64 * 2)]

    def as_dict(self) -> dict:
        return {"max_abs_dout": self.max_abs_dout, "max_abs_dlse": self.max_abs_dlse,
                "row_dout": self.row_dout, "row_dlse": self.row_dlse}


MERGE_DRIFT_BYTES = ctypes.sizeof(LpdMergeDrift)


class LpdLogpDrift(ctypes.Structure):
    _fields_ = [("max_abs_dlogp_train", ctypes.c_double), ("max_abs_dlogp_rollout", ctypes.c_double),
                ("row_train", ctypes.c_int64), ("row_rollout", ctypes.c_int64), ("n_active", ctypes.c_int64),
                ("n_differ", ctypes.c_int64), ("frac_differ", ctypes.c_double), ("scratch", ctypes.c_uint64 * 4)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_ if name != "scratch"}


LOGP_DRIFT_BYTES = ctypes.sizeof(LpdLogpDrift)

# every symbol include/lpd.h declares
EXPORTED = ("lpd_workspace_size", "lpd_backend_info", "lpd_strerror", "lpd_score", "lpd_score_host",
            "lpd_select_active",
            "lpd_token_logp", "lpd_drift_metrics", "lpd_score_sharded", "lpd_score_noalloc",
            "lpd_fused_workspace_size", "lpd_score_fused", "lpd_score_fused_transformed", "lpd_score_transformed",
            "lpd_score_entropy", "lpd_logprob_backward", "lpd_attn_merge", "lpd_attn_merge_order_drift",
            "lpd_topology_workspace_size", "lpd_score_sharded_topology", "lpd_drift_metrics_from_dlogp",
            "lpd_logp_drift_summary", "lpd_merge_rank_metrics")
LPD_NOALLOC_MAX_ROWS = 32768
LPD_ATTN_MAX_PARTS = 64


class LpdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib().lpd_strerror(code).decode()} (code {code})")


_LIB: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    """The loaded liblpd.so (built in-tree on first use if nvcc is present)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(str(path))
        P, I32, I64, SZ, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_double
        L.lpd_workspace_size.restype = SZ
        L.lpd_workspace_size.argtypes = [I32, I64, I64, I32]
        L.lpd_backend_info.restype = ctypes.c_int
        L.lpd_backend_info.argtypes = [P]
        L.lpd_strerror.restype = ctypes.c_char_p
        L.lpd_strerror.argtypes = [ctypes.c_int]
        L.lpd_score.restype = ctypes.c_int
        L.lpd_score.argtypes = [P, P, I64, I64, P, P, D, D, P, P, P, P, P, SZ, P]
        L.lpd_select_active.restype = ctypes.c_int
        L.lpd_select_active.argtypes = [I64, P, P, P, P, P, P, P, SZ, P]
        L.lpd_token_logp.restype = ctypes.c_int
        L.lpd_token_logp.argtypes = [P, P, I64, I64, P, P, P, P, P, SZ, P]
        L.lpd_drift_metrics.restype = ctypes.c_int
        L.lpd_drift_metrics.argtypes = [I64, D, D, P, P, SZ, P]
        L.lpd_score_sharded.restype = ctypes.c_int
        L.lpd_score_sharded.argtypes = [P, P, I32, I64, I64, P, P, D, D, P, P, P, P, P, P, P, P, SZ, P]
        L.lpd_fused_workspace_size.restype = SZ
        L.lpd_fused_workspace_size.argtypes = [I64, I64, I64]
        L.lpd_score_fused.restype = ctypes.c_int
        L.lpd_score_fused.argtypes = [P, P, P, I64, I64, I64, P, P, D, D, P, P, P, P, P, SZ, P]
        L.lpd_score_fused_transformed.restype = ctypes.c_int
        L.lpd_score_fused_transformed.argtypes = [P, P, P, P, P, I64, I64, I64, P, P, D, D, P, P, P, P, P, SZ, P]
        L.lpd_score_host.restype = ctypes.c_int
        L.lpd_score_host.argtypes = [P, P, P, P, I64, I64, P, P, P, P, D, D, P, P, P, P, P, SZ, P, P]
        L.lpd_score_transformed.restype = ctypes.c_int
        L.lpd_score_transformed.argtypes = [P, P, P, P, I64, I64, P, P, D, D, P, P, P, P, P, SZ, P]
        L.lpd_score_entropy.restype = ctypes.c_int
        L.lpd_score_entropy.argtypes = [P, P, I64, I64, P, P, D, D, P, P, P, P, P, P, P, SZ, P]
        L.lpd_logprob_backward.restype = ctypes.c_int
        L.lpd_logprob_backward.argtypes = [P, I64, I64, P, P, P, P, P, I32, I64, P]
        L.lpd_score_noalloc.restype = ctypes.c_int
        L.lpd_score_noalloc.argtypes = [P, P, I64, I64, P, P, D, D, P, P, P, P, P]
        L.lpd_drift_metrics_from_dlogp.restype = ctypes.c_int
        L.lpd_drift_metrics_from_dlogp.argtypes = [I64, P, P, D, D, P, P, SZ, P]
        L.lpd_topology_workspace_size.restype = SZ
        L.lpd_topology_workspace_size.argtypes = [I32, I64, I64, I32, I32, I32]
        L.lpd_score_sharded_topology.restype = ctypes.c_int
        L.lpd_score_sharded_topology.argtypes = [P, P, I32, I64, I64, P, P, D, D, I32, P, P, P, P, P, P, SZ, P]
        L.lpd_attn_merge.restype = ctypes.c_int
        L.lpd_attn_merge.argtypes = [P, I32, P, I32, I64, I32, I32, P, P, P, P]
        L.lpd_attn_merge_order_drift.restype = ctypes.c_int
        L.lpd_attn_merge_order_drift.argtypes = [P, I32, P, I32, I64, I32, I32, P, P, P, P, P, P, P, P]
        L.lpd_logp_drift_summary.restype = ctypes.c_int
        L.lpd_merge_rank_metrics.restype = ctypes.c_int
        L.lpd_merge_rank_metrics.argtypes = [P, P, I32, P]
        L.lpd_logp_drift_summary.argtypes = [I64, P, P, P, P, P, P, P]
        _LIB = L
    return _LIB


# ---- marshalling helpers ----------------------------------------------------

def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _dtype_code(t) -> int:
    import torch

    if t.dtype == torch.bfloat16:
        return LPD_BF16
    if t.dtype == torch.float32:
        return LPD_F32
    return 99  # rejected by the library with LPD_ERR_BAD_DTYPE


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def logits_struct(t) -> LpdLogits:
    """lpd_logits for a 2-D tensor with unit column stride (rows may be padded)."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError("logits must be 2-D with contiguous columns")
    return LpdLogits(t.data_ptr(), _dtype_code(t), 0, t.stride(0))


def shard_array(shards, v_ranges):
    arr = (LpdShard * len(shards))()
    for i, (t, (v0, v1)) in enumerate(zip(shards, v_ranges)):
        if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
            raise ValueError("shard logits must be 2-D with contiguous columns")
        arr[i] = LpdShard(t.data_ptr(), _dtype_code(t), 0, t.stride(0), int(v0), int(v1))
    return arr


def _check(rc: int, where: str) -> None:
    if rc != LPD_OK:
        raise LpdError(rc, where)


# ---- the C ABI, one Python function per entry point ---------------------------

def lpd_workspace_size(kind: int, n_rows: int, vocab: int = 0, n_shards: int = 0) -> int:
    return int(lib().lpd_workspace_size(kind, n_rows, vocab, n_shards))


def lpd_backend_info() -> dict:
    info = LpdBackendInfo()
    _check(lib().lpd_backend_info(ctypes.byref(info)), "lpd_backend_info")
    out = {}
    for name, _ in info._fields_:
        v = getattr(info, name)
        out[name] = v.decode() if isinstance(v, bytes) else v
    return out


def lpd_strerror(code: int) -> str:
    return lib().lpd_strerror(code).decode()


def lpd_score(train, rollout, token_ids, action_mask, clip_lo, clip_hi, out_logp_train, out_logp_rollout,
              out_dlogp, out_metrics, workspace, stream=None) -> None:
    t, r = logits_struct(train), logits_struct(rollout)
    rc = lib().lpd_score(ctypes.byref(t), ctypes.byref(r), train.shape[0], train.shape[1], _ptr(token_ids),
                         _ptr(action_mask), float(clip_lo), float(clip_hi), _ptr(out_logp_train),
                         _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics), _ptr(workspace),
                         workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(rc, "lpd_score")


def lpd_score_host(train_host, rollout_host, token_ids_host, action_mask_host, clip_lo, clip_hi, train_dev,
                   rollout_dev, token_ids_dev, action_mask_dev, out_logp_train, out_logp_rollout, out_dlogp,
                   out_metrics, workspace, stream=None) -> int:
    """lpd_score_host: host tensors in, device staging and outputs; returns
    the bytes copied to the device."""
    th, rh = logits_struct(train_host), logits_struct(rollout_host)
    td, rd = logits_struct(train_dev), logits_struct(rollout_dev)
    copied = ctypes.c_int64(0)
    rc = lib().lpd_score_host(ctypes.byref(th), ctypes.byref(rh), ctypes.byref(td), ctypes.byref(rd),
                              train_host.shape[0], train_host.shape[1], _ptr(token_ids_host), _ptr(action_mask_host),
                              _ptr(token_ids_dev), _ptr(action_mask_dev), float(clip_lo), float(clip_hi),
                              _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics),
                              _ptr(workspace), workspace.numel() if workspace is not None else 0,
                              ctypes.byref(copied), _stream(stream))
    _check(rc, "lpd_score_host")
    return int(copied.value)


def lpd_score_transformed(train, rollout, train_ops, rollout_ops, token_ids, action_mask, clip_lo, clip_hi,
                          out_logp_train, out_logp_rollout, out_dlogp, out_metrics, workspace, stream=None) -> None:
    t, r = logits_struct(train), logits_struct(rollout)
    ct, cr = transform_struct(train_ops), transform_struct(rollout_ops)
    rc = lib().lpd_score_transformed(ctypes.byref(t), ctypes.byref(r), ctypes.byref(ct) if ct else None,
                                     ctypes.byref(cr) if cr else None, train.shape[0], train.shape[1],
                                     _ptr(token_ids), _ptr(action_mask), float(clip_lo), float(clip_hi),
                                     _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics),
                                     _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "lpd_score_transformed")


def lpd_score_entropy(train, rollout, token_ids, action_mask, clip_lo, clip_hi, out_logp_train, out_logp_rollout,
                      out_dlogp, out_entropy_train, out_entropy_rollout, out_metrics, workspace, stream=None) -> None:
    t, r = logits_struct(train), logits_struct(rollout)
    rc = lib().lpd_score_entropy(ctypes.byref(t), ctypes.byref(r), train.shape[0], train.shape[1], _ptr(token_ids),
                                 _ptr(action_mask), float(clip_lo), float(clip_hi), _ptr(out_logp_train),
                                 _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_entropy_train),
                                 _ptr(out_entropy_rollout), _ptr(out_metrics), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check(rc, "lpd_score_entropy")


def lpd_logprob_backward(logits, token_ids, action_mask, logp, grad_logp, out_dlogits, stream=None) -> None:
    x = logits_struct(logits)
    if out_dlogits.dim() != 2 or (out_dlogits.shape[1] > 1 and out_dlogits.stride(1) != 1):
        raise ValueError("out_dlogits must be 2-D with contiguous columns")
    rc = lib().lpd_logprob_backward(ctypes.byref(x), logits.shape[0], logits.shape[1], _ptr(token_ids),
                                    _ptr(action_mask), _ptr(logp), _ptr(grad_logp), _ptr(out_dlogits),
                                    _dtype_code(out_dlogits), out_dlogits.stride(0), _stream(stream))
    _check(rc, "lpd_logprob_backward")


def lpd_select_active(token_ids, action_mask, out_logp_train, out_logp_rollout, out_dlogp, out_metrics, workspace,
                      stream=None) -> None:
    n = action_mask.shape[0]
    rc = lib().lpd_select_active(n, _ptr(token_ids), _ptr(action_mask), _ptr(out_logp_train), _ptr(out_logp_rollout),
                                 _ptr(out_dlogp), _ptr(out_metrics), _ptr(workspace), workspace.numel(),
                                 _stream(stream))
    _check(rc, "lpd_select_active")


def lpd_token_logp(train, rollout, out_logp_train, out_logp_rollout, out_dlogp, out_metrics, workspace,
                   stream=None) -> None:
    t, r = logits_struct(train), logits_struct(rollout)
    rc = lib().lpd_token_logp(ctypes.byref(t), ctypes.byref(r), train.shape[0], train.shape[1],
                              _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics),
                              _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "lpd_token_logp")


def lpd_drift_metrics(n_rows, clip_lo, clip_hi, out_metrics, workspace, stream=None) -> None:
    rc = lib().lpd_drift_metrics(n_rows, float(clip_lo), float(clip_hi), _ptr(out_metrics), _ptr(workspace),
                                 workspace.numel(), _stream(stream))
    _check(rc, "lpd_drift_metrics")


def lpd_score_sharded(train_shards, rollout_shards, v_ranges, token_ids, action_mask, clip_lo, clip_hi,
                      merge_perm, out_logp_train, out_logp_rollout, out_dlogp, out_perm_logp_train,
                      out_perm_logp_rollout, out_metrics, workspace, stream=None) -> None:
    ts, rs = shard_array(train_shards, v_ranges), shard_array(rollout_shards, v_ranges)
    n_rows = train_shards[0].shape[0]
    vocab = max(v1 for _, v1 in v_ranges)
    perm = None
    if merge_perm is not None:
        perm = (ctypes.c_int32 * len(merge_perm))(*[int(k) for k in merge_perm])
    rc = lib().lpd_score_sharded(ts, rs, len(train_shards), n_rows, vocab, _ptr(token_ids), _ptr(action_mask),
                                 float(clip_lo), float(clip_hi), perm, _ptr(out_logp_train), _ptr(out_logp_rollout),
                                 _ptr(out_dlogp), _ptr(out_perm_logp_train), _ptr(out_perm_logp_rollout),
                                 _ptr(out_metrics), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "lpd_score_sharded")


def lpd_drift_metrics_from_dlogp(dlogp, action_mask, clip_lo, clip_hi, out_metrics, workspace, stream=None) -> None:
    rc = lib().lpd_drift_metrics_from_dlogp(dlogp.shape[0], _ptr(dlogp), _ptr(action_mask), float(clip_lo),
                                            float(clip_hi), _ptr(out_metrics), _ptr(workspace), workspace.numel(),
                                            _stream(stream))
    _check(rc, "lpd_drift_metrics_from_dlogp")


def drift_metrics_from_dlogp(dlogp, action_mask, clip=(0.8, 1.2), stream=None) -> dict:
    """The metrics record of given per-token dlogp (float32, device) over the active rows."""
    import torch

    dev = dlogp.device
    met = torch.empty(METRICS_BYTES, dtype=torch.uint8, device=dev)
    ws = torch.empty(lpd_workspace_size(LPD_KIND_SCORE, dlogp.shape[0]), dtype=torch.uint8, device=dev)
    lpd_drift_metrics_from_dlogp(dlogp, action_mask, clip[0], clip[1], met, ws, stream)
    return read_metrics(met)


def lpd_topology_workspace_size(topology: int, n_rows: int, vocab: int, n_shards: int, dtype_train: int,
                                dtype_rollout: int) -> int:
    return int(lib().lpd_topology_workspace_size(topology, n_rows, vocab, n_shards, dtype_train, dtype_rollout))


def lpd_score_sharded_topology(train_shards, rollout_shards, v_ranges, token_ids, action_mask, clip_lo, clip_hi,
                               topology, reduce_order, out_logp_train, out_logp_rollout, out_dlogp, out_metrics,
                               workspace, stream=None) -> None:
    ts, rs = shard_array(train_shards, v_ranges), shard_array(rollout_shards, v_ranges)
    n_rows = train_shards[0].shape[0]
    vocab = max(v1 for _, v1 in v_ranges)
    order = None
    if reduce_order is not None:
        order = (ctypes.c_int32 * len(reduce_order))(*[int(k) for k in reduce_order])
    rc = lib().lpd_score_sharded_topology(ts, rs, len(train_shards), n_rows, vocab, _ptr(token_ids),
                                          _ptr(action_mask), float(clip_lo), float(clip_hi), int(topology), order,
                                          _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp),
                                          _ptr(out_metrics), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "lpd_score_sharded_topology")


def lpd_fused_workspace_size(n_rows: int, hidden: int, vocab: int) -> int:
    return int(lib().lpd_fused_workspace_size(n_rows, hidden, vocab))


def lpd_score_fused(hidden_train, hidden_rollout, W, token_ids, action_mask, clip_lo, clip_hi, out_logp_train,
                    out_logp_rollout, out_dlogp, out_metrics, workspace, stream=None) -> None:
    n_rows, hidden = hidden_train.shape
    rc = lib().lpd_score_fused(_ptr(hidden_train), _ptr(hidden_rollout), _ptr(W), n_rows, hidden, W.shape[0],
                               _ptr(token_ids), _ptr(action_mask), float(clip_lo), float(clip_hi),
                               _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics),
                               _ptr(workspace), workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(rc, "lpd_score_fused")


def lpd_score_fused_transformed(hidden_train, hidden_rollout, W, train_ops, rollout_ops, token_ids, action_mask,
                                clip_lo, clip_hi, out_logp_train, out_logp_rollout, out_dlogp, out_metrics, workspace,
                                stream=None) -> None:
    n_rows, hidden = hidden_train.shape
    ct, cr = transform_struct(train_ops), transform_struct(rollout_ops)
    rc = lib().lpd_score_fused_transformed(
        _ptr(hidden_train), _ptr(hidden_rollout), _ptr(W), ctypes.byref(ct) if ct else None,
        ctypes.byref(cr) if cr else None, n_rows, hidden, W.shape[0], _ptr(token_ids), _ptr(action_mask),
        float(clip_lo), float(clip_hi), _ptr(out_logp_train), _ptr(out_logp_rollout), _ptr(out_dlogp),
        _ptr(out_metrics), _ptr(workspace), workspace.numel() if workspace is not None else 0, _stream(stream))
    _check(rc, "lpd_score_fused_transformed")


def lpd_score_noalloc(train, rollout, token_ids, action_mask, clip_lo, clip_hi, out_logp_train, out_logp_rollout,
                      out_dlogp, out_metrics, stream=None) -> None:
    """lpd_score with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory; n_rows <= 32768)."""
    t, r = logits_struct(train), logits_struct(rollout)
    rc = lib().lpd_score_noalloc(ctypes.byref(t), ctypes.byref(r), train.shape[0], train.shape[1], _ptr(token_ids),
                                 _ptr(action_mask), float(clip_lo), float(clip_hi), _ptr(out_logp_train),
                                 _ptr(out_logp_rollout), _ptr(out_dlogp), _ptr(out_metrics), _stream(stream))
    _check(rc, "lpd_score_noalloc")


def _order(order, n_parts):
    if order is None:
        return None
    order = [int(k) for k in order]
    if len(order) != n_parts:
        raise ValueError(f"order has {len(order)} entries for {n_parts} parts")
    return (ctypes.c_int32 * n_parts)(*order)


def _parts_shape(out_parts, lse_parts):
    if out_parts.dim() != 3 or not out_parts.is_contiguous() or not lse_parts.is_contiguous():
        raise ValueError("out_parts must be a dense [K, n_rows, head_dim] tensor and lse_parts dense [K, n_rows]")
    K, n, d = out_parts.shape
    if tuple(lse_parts.shape) != (K, n):
        raise ValueError("lse_parts must be [K, n_rows]")
    return K, n, d


def lpd_attn_merge(out_parts, lse_parts, order, out, out_lse, lse_base2=False, stream=None) -> None:
    K, n, d = _parts_shape(out_parts, lse_parts)
    rc = lib().lpd_attn_merge(_ptr(out_parts), _dtype_code(out_parts), _ptr(lse_parts), K, n, d, int(bool(lse_base2)),
                              _order(order, K), _ptr(out), _ptr(out_lse), _stream(stream))
    _check(rc, "lpd_attn_merge")


def lpd_attn_merge_order_drift(out_parts, lse_parts, order_a, order_b, out, out_lse, row_dout, row_dlse, drift,
                               lse_base2=False, stream=None) -> None:
    K, n, d = _parts_shape(out_parts, lse_parts)
    rc = lib().lpd_attn_merge_order_drift(_ptr(out_parts), _dtype_code(out_parts), _ptr(lse_parts), K, n, d,
                                          int(bool(lse_base2)), _order(order_a, K), _order(order_b, K), _ptr(out),
                                          _ptr(out_lse), _ptr(row_dout), _ptr(row_dlse), _ptr(drift), _stream(stream))
    _check(rc, "lpd_attn_merge_order_drift")


def lpd_logp_drift_summary(logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b, action_mask, out,
                           stream=None) -> None:
    """Merge-order drift summary of per-token result b against result a over
    the active rows (device float32 [n] each, uint8 mask, out: a device buffer
    of LOGP_DRIFT_BYTES)."""
    n = action_mask.shape[0]
    for x in (logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b):
        if x.shape[0] != n:
            raise ValueError("per-token results and mask must have the same length")
    rc = lib().lpd_logp_drift_summary(n, _ptr(logp_train_a), _ptr(logp_rollout_a), _ptr(logp_train_b),
                                      _ptr(logp_rollout_b), _ptr(action_mask), _ptr(out), _stream(stream))
    _check(rc, "lpd_logp_drift_summary")


# ---- convenience: allocate with torch, call, read back ------------------------

def read_merge_drift(buf) -> dict:
    """Copy a device lpd_merge_drift record (uint8 tensor) to the host as a dict."""
    host = buf.detach().to("cpu", copy=True).numpy().tobytes()
    return LpdMergeDrift.from_buffer_copy(host).as_dict()


def attn_merge(out_parts, lse_parts, order=None, lse_base2=False, stream=None):
    """Merged (out [n, d] f32, lse [n] f32) of K partials, allocated with torch."""
    import torch

    K, n, d = _parts_shape(out_parts, lse_parts)
    out = torch.empty((n, d), dtype=torch.float32, device=out_parts.device)
    lse = torch.empty((n,), dtype=torch.float32, device=out_parts.device)
    lpd_attn_merge(out_parts, lse_parts, order, out, lse, lse_base2, stream)
    return out, lse


def attn_merge_order_drift(out_parts, lse_parts, order_a=None, order_b=None, lse_base2=False, stream=None):
    """(out, lse, row_dout, row_dlse, summary dict) of the order_a vs order_b merge."""
    import torch

    K, n, d = _parts_shape(out_parts, lse_parts)
    dev = out_parts.device
    out = torch.empty((n, d), dtype=torch.float32, device=dev)
    lse = torch.empty((n,), dtype=torch.float32, device=dev)
    rdo = torch.empty((n,), dtype=torch.float32, device=dev)
    rdl = torch.empty((n,), dtype=torch.float32, device=dev)
    drift = torch.empty(MERGE_DRIFT_BYTES, dtype=torch.uint8, device=dev)
    lpd_attn_merge_order_drift(out_parts, lse_parts, order_a, order_b, out, lse, rdo, rdl, drift, lse_base2, stream)
    return out, lse, rdo, rdl, read_merge_drift(drift)


def read_logp_drift(buf) -> dict:
    """Copy a device lpd_logp_drift record (uint8 tensor) to the host as a dict."""
    host = buf.detach().to("cpu", copy=True).numpy().tobytes()
    return LpdLogpDrift.from_buffer_copy(host).as_dict()


def logp_drift_summary(logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b, action_mask, stream=None) -> dict:
    """lpd_logp_drift_summary with a torch-allocated record, read back as a dict."""
    import torch

    out = torch.empty(LOGP_DRIFT_BYTES, dtype=torch.uint8, device=action_mask.device)
    lpd_logp_drift_summary(logp_train_a, logp_rollout_a, logp_train_b, logp_rollout_b, action_mask, out, stream)
    return read_logp_drift(out)


def merge_rank_metrics(per_rank: list[dict], row_offsets: list[int] | None = None) -> dict:
    """lpd_merge_rank_metrics (a host call) on metrics records given as dicts
    in rank order; returns the merged record as a dict."""
    n = len(per_rank)
    arr = (LpdMetrics * max(n, 1))()
    for k, rec in enumerate(per_rank):
        for name, _ in LpdMetrics._fields_:
            setattr(arr[k], name, rec.get(name, 0))
    offs = None if row_offsets is None else (ctypes.c_int64 * max(n, 1))(*[int(o) for o in row_offsets])
    out = LpdMetrics()
    rc = lib().lpd_merge_rank_metrics(ctypes.addressof(arr), None if offs is None else ctypes.addressof(offs), n,
                                      ctypes.addressof(out))
    _check(rc, "lpd_merge_rank_metrics")
    return out.as_dict()


def read_metrics(buf) -> dict:
    """Copy a device lpd_metrics record (uint8 tensor) to the host as a dict."""
    host = buf.detach().to("cpu", copy=True).numpy().tobytes()
    return LpdMetrics.from_buffer_copy(host).as_dict()


def score_fused(hidden_train, hidden_rollout, W, token_ids, action_mask, clip=(0.8, 1.2), stream=None,
                train_ops=None, rollout_ops=None):
    """Allocate outputs and workspace with torch, run lpd_score_fused (or
    lpd_score_fused_transformed when a chain is given)."""
    import torch

    dev = hidden_train.device
    n = hidden_train.shape[0]
    outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
    met = torch.empty(METRICS_BYTES, dtype=torch.uint8, device=dev)
    ws = torch.empty(lpd_fused_workspace_size(n, hidden_train.shape[1], W.shape[0]), dtype=torch.uint8, device=dev)
    if train_ops is None and rollout_ops is None:
        lpd_score_fused(hidden_train, hidden_rollout, W, token_ids, action_mask, clip[0], clip[1], *outs, met, ws,
                        stream=stream)
    else:
        lpd_score_fused_transformed(hidden_train, hidden_rollout, W, train_ops, rollout_ops, token_ids, action_mask,
                                    clip[0], clip[1], *outs, met, ws, stream=stream)
    return ScoreResult(outs[0], outs[1], outs[2], read_metrics(met))


@dataclass
class ScoreResult:
    logp_train: object
    logp_rollout: object
    dlogp: object
    metrics: dict


def score(train, rollout, token_ids, action_mask, clip=(0.8, 1.2), stream=None, train_ops=None,
          rollout_ops=None) -> ScoreResult:
    """Allocate outputs and workspace with torch on the logits' device, run
    lpd_score (or lpd_score_transformed when a chain is given), and return
    per-token tensors plus the metrics as a dict."""
    import torch

    dev = train.device
    n = train.shape[0]
    outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
    met = torch.empty(METRICS_BYTES, dtype=torch.uint8, device=dev)
    ws = torch.empty(lpd_workspace_size(LPD_KIND_SCORE, n), dtype=torch.uint8, device=dev)
    if train_ops is None and rollout_ops is None:
        lpd_score(train, rollout, token_ids, action_mask, clip[0], clip[1], *outs, met, ws, stream=stream)
    else:
        lpd_score_transformed(train, rollout, train_ops, rollout_ops, token_ids, action_mask, clip[0], clip[1],
                              *outs, met, ws, stream=stream)
    return ScoreResult(outs[0], outs[1], outs[2], read_metrics(met))


def score_sharded_topology(train_shards, rollout_shards, v_ranges, token_ids, action_mask, topology,
                           reduce_order=None, clip=(0.8, 1.2), stream=None) -> ScoreResult:
    """lpd_score_sharded_topology with torch-allocated outputs and workspace."""
    import torch

    dev = token_ids.device
    n = token_ids.shape[0]
    vocab = max(v1 for _, v1 in v_ranges)
    outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
    met = torch.empty(METRICS_BYTES, dtype=torch.uint8, device=dev)
    nbytes = lpd_topology_workspace_size(topology, n, vocab, len(train_shards), _dtype_code(train_shards[0]),
                                         _dtype_code(rollout_shards[0]))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    lpd_score_sharded_topology(train_shards, rollout_shards, v_ranges, token_ids, action_mask, clip[0], clip[1],
                               topology, reduce_order, *outs, met, ws, stream)
    return ScoreResult(*outs, read_metrics(met))
