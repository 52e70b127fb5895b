"""Shared test helpers: tensor <-> numpy marshalling for the oracle, and the
parity bars.

Tolerances are the ones the scorer's specification fixes: per-token logp
within 1e-4 absolute; approx_kl0 and mean_abs_dlogp within 1e-4 relative;
p95/p99/max |dlogp| within 1e-4 absolute; active counts, token selection and
the batch-invariance controls bit-exact.  ratio0_mean has no stated bar; it is
the mean of exp(dlogp) ("Diagnostics": ratio0 = exp(dlogp)), whose error is
the mean of exp(dlogp) * (error of dlogp), i.e. about 1e-7 of the ratio
itself, so (1e-6 + the largest per-token dlogp error observed against the
oracle) x max(1, ratio0_mean) is used; the per-token error is itself held to
the logp bar.  clipfrac0 must match exactly
except for tokens whose oracle dlogp lies within 1e-9 of ln(lo) or ln(hi),
where the two sides may legitimately decide differently (1e-6 when the
reference is the oracle's metric function applied to the GPU's own fp32
per-token dlogp, whose rounding is ~6e-8 relative).
"""
from __future__ import annotations

import math

import numpy as np

LOGP_ATOL = 1e-4
REL_TOL = 1e-4
PCT_ATOL = 1e-4
RATIO_ATOL = 1e-6
CLIP_AMBIGUITY = 1e-9


def to_oracle(t) -> np.ndarray:
    """Host numpy view for the oracle: bf16 as uint16 bits, fp32 as float32.
    Keeps the row stride of a column slice of a wider tensor."""
    import torch

    if t.dtype == torch.bfloat16:
        base = t.detach().cpu()
        return base.view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def assert_metrics_match(gpu: dict, ref: dict, ref_dlogp=None, mask=None, clip=(0.8, 1.2),
                         ambiguity=CLIP_AMBIGUITY, dlogp_err=0.0):
    assert gpu["status"] == ref["status"], (gpu["status"], ref["status"])
    assert gpu["n_active"] == ref["n_active"]
    assert gpu["flags"] == ref["flags"]
    if ref["n_active"] == 0:
        for k in ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp", "p95_abs_dlogp",
                  "p99_abs_dlogp", "max_abs_dlogp"):
            assert gpu[k] == 0.0
        assert gpu["argmax_row"] == -1
        return
    for k in ("approx_kl0", "mean_abs_dlogp"):
        tol = REL_TOL * abs(ref[k]) + 1e-300
        assert abs(gpu[k] - ref[k]) <= tol, (k, gpu[k], ref[k], abs(gpu[k] - ref[k]) / max(abs(ref[k]), 1e-300))
    for k in ("p95_abs_dlogp", "p99_abs_dlogp", "max_abs_dlogp"):
        assert abs(gpu[k] - ref[k]) <= PCT_ATOL, (k, gpu[k], ref[k])
    ratio_tol = (RATIO_ATOL + 1.01 * dlogp_err) * max(1.0, abs(ref["ratio0_mean"]))
    assert abs(gpu["ratio0_mean"] - ref["ratio0_mean"]) <= ratio_tol, (gpu["ratio0_mean"], ref["ratio0_mean"])
    # clip decisions: exact unless the oracle value sits on a boundary
    n_amb = 0
    if ref_dlogp is not None:
        d = np.asarray(ref_dlogp)[np.asarray(mask) != 0]
        lo, hi = math.log(clip[0]), math.log(clip[1])
        n_amb = int(np.sum((np.abs(d - lo) < ambiguity) | (np.abs(d - hi) < ambiguity)))
    diff = abs(gpu["clipfrac0"] - ref["clipfrac0"]) * ref["n_active"]
    assert diff <= n_amb + 1e-6, (gpu["clipfrac0"], ref["clipfrac0"], n_amb)
    # worst token: the GPU's choice must be a valid argmax of the oracle |d|
    if ref_dlogp is not None:
        r = gpu["argmax_row"]
        assert mask[r] != 0
        assert abs(abs(ref_dlogp[r]) - ref["max_abs_dlogp"]) <= PCT_ATOL
    else:
        assert gpu["argmax_row"] == ref["argmax_row"]


def metrics_abs_close(a: dict, b: dict, keys=("approx_kl0", "mean_abs_dlogp")):
    return all(abs(a[k] - b[k]) <= REL_TOL * abs(b[k]) for k in keys)
