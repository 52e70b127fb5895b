"""lpd_merge_rank_metrics (a host call of the library; no GPU): per-rank
metric records combined in rank order ("WS2 Cross-Config Logprob Drift
Contract", "Diagnostics": the same metrics per rank and globally)."""
import math

import pytest

from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300.ranks import merge_rank_metrics


def _rec(n, argmax, mx, ratio=1.0, clip=0.0, kl=0.0, mabs=0.0, status=0):
    return dict(n_active=n, argmax_row=argmax, flags=0 if n else B.LPD_FLAG_NO_ACTIVE, status=status,
                ratio0_mean=ratio, clipfrac0=clip, approx_kl0=kl, mean_abs_dlogp=mabs, p95_abs_dlogp=0.5,
                p99_abs_dlogp=0.7, max_abs_dlogp=mx)


def test_weighted_means_worst_token_and_offsets():
    per_rank = [_rec(3, 2, 0.5, ratio=1.5, clip=1 / 3, kl=0.25, mabs=0.125),
                _rec(0, -1, 0.0, status=B.LPD_STATUS_TOKEN_OOB),
                _rec(5, 4, 0.75, ratio=0.5, clip=0.0, kl=0.5, mabs=0.25),
                _rec(2, 0, 0.75, ratio=1.0, clip=0.5, kl=1.0, mabs=1.0)]   # ties rank 2's max: rank 2 keeps it
    m = merge_rank_metrics(per_rank, [0, 10, 10, 30])
    assert m["n_active"] == 10 and m["status"] == B.LPD_STATUS_TOKEN_OOB
    assert m["ratio0_mean"] == (3 * 1.5 + 5 * 0.5 + 2 * 1.0) / 10
    assert m["clipfrac0"] == (3 * (1 / 3) + 2 * 0.5) / 10
    assert m["approx_kl0"] == (3 * 0.25 + 5 * 0.5 + 2 * 1.0) / 10
    assert m["mean_abs_dlogp"] == (3 * 0.125 + 5 * 0.25 + 2 * 1.0) / 10
    assert m["max_abs_dlogp"] == 0.75 and m["argmax_row"] == 14
    assert m["flags"] == B.LPD_FLAG_NO_PERCENTILES
    assert math.isnan(m["p95_abs_dlogp"]) and math.isnan(m["p99_abs_dlogp"])


def test_no_offsets_and_nothing_active():
    m = merge_rank_metrics([_rec(2, 1, 0.25), _rec(1, 0, 0.5)])
    assert m["argmax_row"] == 0 and m["max_abs_dlogp"] == 0.5
    z = merge_rank_metrics([_rec(0, -1, 0.0), _rec(0, -1, 0.0)])
    assert z["n_active"] == 0 and z["flags"] == B.LPD_FLAG_NO_ACTIVE and z["argmax_row"] == -1
    assert all(z[k] == 0.0 for k in ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp", "max_abs_dlogp"))


def test_validation():
    with pytest.raises(B.LpdError):
        merge_rank_metrics([])
    with pytest.raises(B.LpdError):
        merge_rank_metrics([_rec(-1, 0, 0.0)])
    out = B.LpdMetrics()
    import ctypes
    assert B.lib().lpd_merge_rank_metrics(None, None, 1, ctypes.addressof(out)) == B.LPD_ERR_NULL_POINTER
