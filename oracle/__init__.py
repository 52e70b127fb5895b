"""Float64 CPU oracle for selected-token logprob drift scoring.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this module.  The product path
(``logprob_drift_scoring_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``lpd_oracle.c`` (plain serial C, double precision),
compiled here with gcc and called through ctypes.  This module only marshals
numpy arrays; it adds no arithmetic of its own.  bf16 tensors are passed as
``numpy.uint16`` arrays holding the raw bf16 bits.

Sources: "WS2 Cross-Config Logprob Drift Contract" (sections "Measurement
Contract" and "Diagnostics"); "[WS2] Framework for ablation experiment"
(LogProb knobs table, rows 3-5 and 8-10).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from dataclasses import dataclass
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
SOURCE = _HERE / "lpd_oracle.c"
BUILD_DIR = _HERE / "_build"

BF16, F32 = 0, 1
STATUS_TOKEN_OOB = 1
STATUS_NONFINITE = 2
FLAG_NO_ACTIVE = 1


class Metrics(ctypes.Structure):
    _fields_ = [
        ("n_active", ctypes.c_int64),
        ("argmax_row", ctypes.c_int64),
        ("flags", ctypes.c_uint32),
        ("status", ctypes.c_uint32),
        ("ratio0_mean", ctypes.c_double),
        ("clipfrac0", ctypes.c_double),
        ("approx_kl0", ctypes.c_double),
        ("mean_abs_dlogp", ctypes.c_double),
        ("p95_abs_dlogp", ctypes.c_double),
        ("p99_abs_dlogp", ctypes.c_double),
        ("max_abs_dlogp", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class LogpDrift(ctypes.Structure):
    _fields_ = [
        ("max_abs_dlogp_train", ctypes.c_double),
        ("max_abs_dlogp_rollout", ctypes.c_double),
        ("row_train", ctypes.c_int64),
        ("row_rollout", ctypes.c_int64),
        ("n_active", ctypes.c_int64),
        ("n_differ", ctypes.c_int64),
        ("frac_differ", ctypes.c_double),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class Shard(ctypes.Structure):
    _fields_ = [
        ("ptr", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("pad_", ctypes.c_int32),
        ("stride", ctypes.c_int64),
        ("v_start", ctypes.c_int64),
        ("v_end", ctypes.c_int64),
    ]


OP_SCALE, OP_SOFTCAP = 1, 2


class Transform(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("kind", ctypes.c_int32 * 4), ("param", ctypes.c_float * 4)]


def transform(ops) -> Transform | None:
    """ops: list of (kind, param) applied in order; None or [] is the identity."""
    if not ops:
        return None
    t = Transform()
    t.n_ops = len(ops)
    for i, (k, p) in enumerate(ops):
        t.kind[i] = k
        t.param[i] = p
    return t


def compile_oracle(source: Path | str = SOURCE, out: Path | None = None) -> Path:
    """Compile the oracle C source to a shared object (gcc -O2, no fast-math)."""
    source = Path(source)
    text = source.read_bytes()
    tag = hashlib.sha1(text).hexdigest()[:12]
    if out is None:
        BUILD_DIR.mkdir(exist_ok=True)
        out = BUILD_DIR / f"liblpd_oracle_{tag}.so"
    if not out.exists():
        tmp = out.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             str(source), "-o", str(tmp), "-lm"],
            check=True,
        )
        os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P, I64, I32, U32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_double
    lib.lpdo_score.restype = U32
    lib.lpdo_score.argtypes = [P, I32, I64, P, I32, I64, I64, I64, P, P, D, D, P, P, P, P]
    lib.lpdo_score_rows.restype = U32
    lib.lpdo_score_rows.argtypes = [P, I32, I64, P, I32, I64, I64, P, P, I64, P, P, P]
    lib.lpdo_row_logp.restype = U32
    lib.lpdo_row_logp.argtypes = [P, I32, I64, I64, P]
    lib.lpdo_partial.restype = None
    lib.lpdo_partial.argtypes = [P, I32, I64, I64, P, P]
    lib.lpdo_metrics_from_dlogp.restype = None
    lib.lpdo_metrics_from_dlogp.argtypes = [P, P, I64, D, D, P]
    lib.lpdo_check_tiling.restype = ctypes.c_int
    lib.lpdo_check_tiling.argtypes = [P, ctypes.c_int, I64]
    lib.lpdo_score_sharded.restype = U32
    lib.lpdo_score_sharded.argtypes = [P, P, ctypes.c_int, P, I64, I64, P, P, D, D, P, P, P, P]
    lib.lpdo_head_logits.restype = None
    lib.lpdo_head_logits.argtypes = [P, P, I64, I64, P]
    lib.lpdo_score_transformed.restype = U32
    lib.lpdo_score_transformed.argtypes = [P, I32, I64, P, I32, I64, P, P, I64, I64, P, P, D, D, P, P, P, P]
    lib.lpdo_row_entropy.restype = D
    lib.lpdo_row_entropy.argtypes = [P, I32, I64]
    lib.lpdo_entropy.restype = None
    lib.lpdo_entropy.argtypes = [P, I32, I64, P, I32, I64, I64, I64, P, P, P]
    lib.lpdo_logprob_backward_row.restype = None
    lib.lpdo_logprob_backward_row.argtypes = [P, I32, I64, I64, D, P]
    lib.lpdo_attn_merge.restype = None
    lib.lpdo_attn_merge.argtypes = [P, P, ctypes.c_int, I64, ctypes.c_int, ctypes.c_int, P, P, P]
    lib.lpdo_score_head_rows.restype = U32
    lib.lpdo_score_head_rows.argtypes = [P, P, P, I64, I64, P, P, I64, P, P, P]
    lib.lpdo_logp_drift.restype = None
    lib.lpdo_logp_drift.argtypes = [I64, P, P, P, P, P, P]
    return lib


_LIB: ctypes.CDLL | None = None


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library.  With ``path`` given,
    load that build instead of the default one (used by the mutation tests)."""
    global _LIB
    if path is not None:
        return _bind(ctypes.CDLL(str(path)))
    if _LIB is None:
        _LIB = _bind(ctypes.CDLL(str(compile_oracle())))
    return _LIB


# ---------------------------------------------------------------- helpers

def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _logits_arg(x: np.ndarray):
    """(array, dtype code, row stride in elements) for a 2-D logits array whose
    rows may be padded (row stride >= vocab) but whose columns are contiguous."""
    if x.dtype == np.uint16:
        code = BF16
    elif x.dtype == np.float32:
        code = F32
    else:
        raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {x.dtype}")
    if x.ndim != 2 or x.strides[1] != x.itemsize:
        raise ValueError("logits must be 2-D with contiguous columns")
    return x, code, x.strides[0] // x.itemsize


@dataclass
class Result:
    logp_train: np.ndarray
    logp_rollout: np.ndarray
    dlogp: np.ndarray
    status: int
    metrics: dict | None = None


def score(train, rollout, token_ids, mask, clip_lo=0.8, clip_hi=1.2, lib=None) -> Result:
    """Score every row of both sides and the drift metrics over active rows."""
    lib = lib or load()
    t, tc, ts = _logits_arg(train)
    r, rc, rs = _logits_arg(rollout)
    n_rows, vocab = t.shape[0], t.shape[1]
    assert r.shape == t.shape
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    lt, lr, d = (np.zeros(n_rows) for _ in range(3))
    met = Metrics()
    st = lib.lpdo_score(_ptr(t), tc, ts, _ptr(r), rc, rs, n_rows, vocab, _ptr(ids), _ptr(m8),
                        float(clip_lo), float(clip_hi), _ptr(lt), _ptr(lr), _ptr(d),
                        ctypes.addressof(met))
    return Result(lt, lr, d, int(st), met.as_dict())


def score_rows(train, rollout, token_ids, rows, lib=None) -> Result:
    """Score only the listed rows (no metrics)."""
    lib = lib or load()
    t, tc, ts = _logits_arg(train)
    r, rc, rs = _logits_arg(rollout)
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    sel = np.ascontiguousarray(rows, dtype=np.int64)
    n = sel.shape[0]
    lt, lr, d = (np.zeros(n) for _ in range(3))
    st = lib.lpdo_score_rows(_ptr(t), tc, ts, _ptr(r), rc, rs, t.shape[1], _ptr(ids), _ptr(sel), n,
                             _ptr(lt), _ptr(lr), _ptr(d))
    return Result(lt, lr, d, int(st))


def row_logp(row, token_id: int, lib=None) -> tuple[float, int]:
    """logp of one 1-D row and the status bits it raises."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    code = BF16 if row.dtype == np.uint16 else F32
    assert row.dtype in (np.uint16, np.float32)
    out = ctypes.c_double()
    st = lib.lpdo_row_logp(_ptr(row), code, row.shape[0], int(token_id), ctypes.addressof(out))
    return out.value, int(st)


def partial(row, c0: int, c1: int, lib=None) -> tuple[float, float]:
    """(max, sum exp(x - max)) over columns [c0, c1) of one 1-D row."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    code = BF16 if row.dtype == np.uint16 else F32
    m, s = ctypes.c_double(), ctypes.c_double()
    lib.lpdo_partial(_ptr(row), code, int(c0), int(c1), ctypes.addressof(m), ctypes.addressof(s))
    return m.value, s.value


def metrics(dlogp, mask, clip_lo=0.8, clip_hi=1.2, lib=None) -> dict:
    """Drift diagnostics from a per-row dlogp vector and the active mask."""
    lib = lib or load()
    d = np.ascontiguousarray(dlogp, dtype=np.float64)
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    met = Metrics()
    lib.lpdo_metrics_from_dlogp(_ptr(d), _ptr(m8), d.shape[0], float(clip_lo), float(clip_hi),
                                ctypes.addressof(met))
    return met.as_dict()


def _shard_array(shards, v_ranges):
    arr = (Shard * len(shards))()
    keep = []
    for i, (x, (v0, v1)) in enumerate(zip(shards, v_ranges)):
        a, code, stride = _logits_arg(x)
        keep.append(a)
        arr[i] = Shard(a.ctypes.data, code, 0, stride, int(v0), int(v1))
    return arr, keep


def check_tiling(v_ranges, vocab: int, lib=None) -> bool:
    lib = lib or load()
    arr = (Shard * max(len(v_ranges), 1))()
    for i, (v0, v1) in enumerate(v_ranges):
        arr[i] = Shard(None, BF16, 0, 0, int(v0), int(v1))
    return lib.lpdo_check_tiling(ctypes.addressof(arr), len(v_ranges), int(vocab)) == 0


def score_sharded(train_shards, rollout_shards, v_ranges, token_ids, mask, order=None,
                  clip_lo=0.8, clip_hi=1.2, lib=None) -> Result:
    """Vocab-sharded scoring: per-shard partials merged in ``order`` (a list of
    shard indices; default ascending vocab position)."""
    lib = lib or load()
    n = len(v_ranges)
    if order is None:
        order = sorted(range(n), key=lambda i: v_ranges[i][0])
    order = np.ascontiguousarray(order, dtype=np.int32)
    ts, keep_t = _shard_array(train_shards, v_ranges)
    rs, keep_r = _shard_array(rollout_shards, v_ranges)
    n_rows = train_shards[0].shape[0]
    vocab = max(v1 for _, v1 in v_ranges)
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    lt, lr, d = (np.zeros(n_rows) for _ in range(3))
    met = Metrics()
    st = lib.lpdo_score_sharded(ctypes.addressof(ts), ctypes.addressof(rs), n, _ptr(order), n_rows,
                                vocab, _ptr(ids), _ptr(m8), float(clip_lo), float(clip_hi),
                                _ptr(lt), _ptr(lr), _ptr(d), ctypes.addressof(met))
    del keep_t, keep_r
    return Result(lt, lr, d, int(st), met.as_dict())


def head_logits(h, W, lib=None) -> np.ndarray:
    """Double-precision logits of one hidden vector through the head W."""
    lib = lib or load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    x = np.zeros(W.shape[0])
    lib.lpdo_head_logits(_ptr(h), _ptr(W), W.shape[1], W.shape[0], _ptr(x))
    return x


def score_head_rows(hidden_t, hidden_r, W, token_ids, rows, lib=None) -> Result:
    """LM-head scoring of the listed rows (logits materialised in double)."""
    lib = lib or load()
    ht = np.ascontiguousarray(hidden_t, dtype=np.uint16)
    hr = np.ascontiguousarray(hidden_r, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    sel = np.ascontiguousarray(rows, dtype=np.int64)
    n = sel.shape[0]
    lt, lr, d = (np.zeros(n) for _ in range(3))
    st = lib.lpdo_score_head_rows(_ptr(ht), _ptr(hr), _ptr(W), W.shape[1], W.shape[0], _ptr(ids),
                                  _ptr(sel), n, _ptr(lt), _ptr(lr), _ptr(d))
    return Result(lt, lr, d, int(st))


def score_transformed(train, rollout, token_ids, mask, train_ops=None, rollout_ops=None, clip_lo=0.8,
                      clip_hi=1.2, lib=None) -> Result:
    """score() with an ordered chain of logit transforms per side."""
    lib = lib or load()
    t, tc, ts = _logits_arg(train)
    r, rc, rs = _logits_arg(rollout)
    n_rows, vocab = t.shape[0], t.shape[1]
    ids = np.ascontiguousarray(token_ids, dtype=np.int32)
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    ct, cr = transform(train_ops), transform(rollout_ops)
    lt, lr, d = (np.zeros(n_rows) for _ in range(3))
    met = Metrics()
    st = lib.lpdo_score_transformed(_ptr(t), tc, ts, _ptr(r), rc, rs,
                                    ctypes.addressof(ct) if ct else None, ctypes.addressof(cr) if cr else None,
                                    n_rows, vocab, _ptr(ids), _ptr(m8), float(clip_lo), float(clip_hi),
                                    _ptr(lt), _ptr(lr), _ptr(d), ctypes.addressof(met))
    return Result(lt, lr, d, int(st), met.as_dict())


def row_entropy(row, lib=None) -> float:
    """Entropy of the softmax of one 1-D row."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    code = BF16 if row.dtype == np.uint16 else F32
    return float(lib.lpdo_row_entropy(_ptr(row), code, row.shape[0]))


def entropy(train, rollout, mask, lib=None):
    """Per-row entropies of both sides (0 where inactive)."""
    lib = lib or load()
    t, tc, ts = _logits_arg(train)
    r, rc, rs = _logits_arg(rollout)
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    et, er = np.zeros(t.shape[0]), np.zeros(t.shape[0])
    lib.lpdo_entropy(_ptr(t), tc, ts, _ptr(r), rc, rs, t.shape[0], t.shape[1], _ptr(m8), _ptr(et), _ptr(er))
    return et, er


def logprob_backward_row(row, token_id: int, grad: float, lib=None) -> np.ndarray:
    """grad * d logp[token_id] / d logits for one 1-D row, in double."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    code = BF16 if row.dtype == np.uint16 else F32
    out = np.zeros(row.shape[0])
    lib.lpdo_logprob_backward_row(_ptr(row), code, row.shape[0], int(token_id), float(grad), _ptr(out))
    return out


def attn_merge(out_parts, lse_parts, order=None, lse_base2=False, lib=None):
    """Merge partial attention results: out_parts [K, n, d] f32, lse_parts
    [K, n] f32, parts visited in ``order``.  Returns (out [n, d], lse [n])."""
    lib = lib or load()
    o = np.ascontiguousarray(out_parts, dtype=np.float32)
    l = np.ascontiguousarray(lse_parts, dtype=np.float32)
    K, n, d = o.shape
    order = np.ascontiguousarray(range(K) if order is None else order, dtype=np.int32)
    out = np.zeros((n, d))
    lse = np.zeros(n)
    lib.lpdo_attn_merge(_ptr(o), _ptr(l), K, n, d, int(bool(lse_base2)), _ptr(order), _ptr(out), _ptr(lse))
    return out, lse


def logp_drift(a_train, a_rollout, b_train, b_rollout, mask, lib=None) -> dict:
    """Summary of how far per-token result b is from result a (float32
    arrays, e.g. a permuted against the fixed shard merge order) over the
    active rows: each side's max |b - a| with its lowest row, and the count and
    fraction of active rows where they differ."""
    lib = lib or load()
    arrs = [np.ascontiguousarray(x, dtype=np.float32) for x in (a_train, a_rollout, b_train, b_rollout)]
    m8 = np.ascontiguousarray(mask, dtype=np.uint8)
    n = m8.shape[0]
    assert all(x.shape == (n,) for x in arrs)
    out = LogpDrift()
    lib.lpdo_logp_drift(n, *(_ptr(x) for x in arrs), _ptr(m8), ctypes.addressof(out))
    return out.as_dict()
