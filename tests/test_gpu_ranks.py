"""Data-parallel ranks emulated on one GPU ("WS2 Cross-Config Logprob Drift
Contract", "Diagnostics": the same metrics per rank and globally): rows split
into logical ranks, each scored on its own, then merged in rank order (needs
a GPU).

Bars: a row's results do not depend on which rank scored it (bitwise); the
host merge of the per-rank records gives the whole batch's count and worst
token exactly and its means within 1e-12 relative (one more rounding per
rank); the metrics of the gathered per-token values
(lpd_drift_metrics_from_dlogp) match the oracle's metric function on the same
float32 values with the scorer's bars, and the whole batch's percentiles
within 1e-4.
"""
import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from logprob_drift_scoring_gb300.ranks import merge_rank_metrics
from tests.helpers import PCT_ATOL, assert_metrics_match

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_logical_ranks_merge_to_the_whole_batch():
    w = W.synthetic(1000, 20000, seed=61, device=DEV, active_prob=0.85, rollout_noise=5e-3)
    bounds = [(0, 317), (317, 700), (700, 1000)]
    whole = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
    per_rank, d_parts, m_parts = [], [], []
    for k, (a, b) in enumerate(bounds):
        res = B.score(w.train[a:b], w.rollout[a:b], w.token_ids[a:b], w.action_mask[a:b], w.clip)
        rec = dict(res.metrics)
        rec["rank"] = k
        per_rank.append(rec)
        d_parts.append(res.dlogp)
        m_parts.append(w.action_mask[a:b])
    torch.cuda.synchronize()
    d_all, m_all = torch.cat(d_parts), torch.cat(m_parts)
    # which rank scored a row does not change its bits
    assert torch.equal(d_all, whole.dlogp)

    merged = merge_rank_metrics(per_rank, [a for a, _ in bounds])
    wm = whole.metrics
    assert merged["n_active"] == wm["n_active"] == int(w.action_mask.sum().item())
    assert merged["argmax_row"] == wm["argmax_row"] and merged["max_abs_dlogp"] == wm["max_abs_dlogp"]
    for key in ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp"):
        assert abs(merged[key] - wm[key]) <= 1e-12 * max(1.0, abs(wm[key])), key
    assert [p["n_active"] for p in per_rank] == [int(w.action_mask[a:b].sum().item()) for a, b in bounds]

    union = B.drift_metrics_from_dlogp(d_all, m_all, w.clip)
    mask = m_all.cpu().numpy()
    d64 = d_all.cpu().numpy().astype(np.float64)
    ref = oracle.metrics(d64, mask, *w.clip)
    ref["status"] = 0
    assert_metrics_match(union, ref, d64, mask, w.clip, ambiguity=1e-6)
    for key in ("p95_abs_dlogp", "p99_abs_dlogp", "max_abs_dlogp"):
        assert abs(union[key] - wm[key]) <= PCT_ATOL
    assert union["argmax_row"] == wm["argmax_row"]


def test_metrics_from_dlogp_edge_cases():
    n = 300
    d = torch.randn(n, device=DEV) * 1e-3
    mask = torch.zeros(n, dtype=torch.uint8, device=DEV)
    met = B.drift_metrics_from_dlogp(d, mask)
    assert met["n_active"] == 0 and met["flags"] == B.LPD_FLAG_NO_ACTIVE and met["argmax_row"] == -1
    mask[::3] = 1
    d[6] = float("nan")          # active
    d[7] = float("inf")          # inactive: never read
    met = B.drift_metrics_from_dlogp(d, mask)
    assert met["status"] & B.LPD_STATUS_NONFINITE
    assert met["n_active"] == 100
    mask[6] = 0
    met = B.drift_metrics_from_dlogp(d, mask)
    assert met["status"] == 0
    ref = oracle.metrics(d.cpu().numpy().astype(np.float64), mask.cpu().numpy(), 0.8, 1.2)
    ref["status"] = 0
    assert_metrics_match(met, ref, d.cpu().numpy().astype(np.float64), mask.cpu().numpy(), ambiguity=1e-6)
    empty = torch.empty(0, device=DEV)
    met = B.drift_metrics_from_dlogp(empty, torch.empty(0, dtype=torch.uint8, device=DEV))
    assert met["n_active"] == 0
