"""lpd_score_noalloc: lpd_score for callers that cannot allocate device memory.

Callers running inside another engine whose allocator owns the device, or
plugins that receive only a stream and tensors, cannot pass lpd_score a
workspace.  lpd_score_noalloc uses an array of device memory built into the
library instead.  These tests call it through the C ABI and compare it with
lpd_score (which gets a workspace allocated here) on two calls in a row, so the
second call runs on scratch that still holds the first call's contents.

This file is collected last on purpose; it also passes when run alone in a
fresh process (the first call on the device does the one-time set-up).
"""
import ctypes

import numpy as np
import pytest

from logprob_drift_scoring_gb300 import binding as B
from tests.helpers import LOGP_ATOL, PCT_ATOL, RATIO_ATOL, REL_TOL


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    # checked on the host before the GPU is touched
    t = B.LpdLogits(0x7F0000000000, B.LPD_BF16, 0, 16)
    rc = B.lib().lpd_score_noalloc(ctypes.byref(t), ctypes.byref(t), B.LPD_NOALLOC_MAX_ROWS + 1, 16,
                                   0x7F0000000000, 0x7F0000000000, 0.8, 1.2, None, None, None,
                                   0x7F0000000000, None)
    assert rc == B.LPD_ERR_UNSUPPORTED


def _compare(got, want):
    for a, b in zip(got[:3], want[:3]):
        a = a.cpu().numpy().astype(np.float64)
        b = b.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(a - b)) <= LOGP_ATOL
    gm, wm = got[3], want[3]
    assert gm["status"] == wm["status"] == 0
    assert gm["n_active"] == wm["n_active"] and gm["flags"] == wm["flags"]
    assert gm["argmax_row"] == wm["argmax_row"]
    for k in ("approx_kl0", "mean_abs_dlogp"):
        assert abs(gm[k] - wm[k]) <= REL_TOL * abs(wm[k])
    for k in ("p95_abs_dlogp", "p99_abs_dlogp", "max_abs_dlogp"):
        assert abs(gm[k] - wm[k]) <= PCT_ATOL
    assert abs(gm["ratio0_mean"] - wm["ratio0_mean"]) <= RATIO_ATOL * max(1.0, abs(wm["ratio0_mean"]))
    assert gm["clipfrac0"] == wm["clipfrac0"]


@pytest.mark.gpu
def test_noalloc_matches_lpd_score_on_two_calls_in_a_row():
    import torch

    from logprob_drift_scoring_gb300 import workloads as W

    dev = "cuda"
    cases = [
        W.synthetic(3000, 20000, seed=41, device=dev),                                   # bf16 / bf16
        W.synthetic(700, 9000, seed=42, device=dev, dtype_rollout=torch.float32,       # mixed dtypes, fewer rows:
                    rollout_noise=0.3),                                                 # stale scratch beyond row 700
    ]
    for w in cases:
        n = w.n_rows
        want = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
        outs = [torch.full((n,), float("nan"), dtype=torch.float32, device=dev) for _ in range(3)]
        met = torch.zeros(B.METRICS_BYTES, dtype=torch.uint8, device=dev)
        B.lpd_score_noalloc(w.train, w.rollout, w.token_ids, w.action_mask, w.clip[0], w.clip[1], *outs, met)
        torch.cuda.synchronize()
        _compare((*outs, B.read_metrics(met)), (want.logp_train, want.logp_rollout, want.dlogp, want.metrics))
