"""lpd_score_host: logits in host memory, only the active rows copied to the
device (needs a GPU).

Bars: the results equal lpd_score on the same logits already on the device,
bit for bit (the same kernels read the same rows); the inactive rows of the
device staging buffers are neither copied nor read (they are filled with NaN
first, stay NaN, and the results do not change); the reported byte count is
the active rows' bytes of both sides plus the ids and the mask.
"""
import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import LOGP_ATOL, assert_metrics_match, to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host_copy(x, pad=0, pinned=True):
    """x on the host, optionally with `pad` extra columns per stored row."""
    buf = torch.empty((x.shape[0], x.shape[1] + pad), dtype=x.dtype, pin_memory=pinned)
    buf[:, :x.shape[1]] = x.cpu()
    return buf[:, :x.shape[1]]


def _staging(x, pad=0):
    buf = torch.full((x.shape[0], x.shape[1] + pad), float("nan"), dtype=x.dtype, device=DEV)
    return buf[:, :x.shape[1]]


def _run_host(w, host_pad=0, dev_pad=0, pinned=True):
    n = w.n_rows
    th, rh = _host_copy(w.train, host_pad, pinned), _host_copy(w.rollout, host_pad, pinned)
    ids_h = w.token_ids.cpu().pin_memory() if pinned else w.token_ids.cpu()
    mask_h = w.action_mask.cpu().pin_memory() if pinned else w.action_mask.cpu()
    td, rd = _staging(w.train, dev_pad), _staging(w.rollout, dev_pad)
    ids_d = torch.full((n,), -7, dtype=torch.int32, device=DEV)
    mask_d = torch.full((n,), 3, dtype=torch.uint8, device=DEV)
    outs = [torch.empty(n, device=DEV) for _ in range(3)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    copied = B.lpd_score_host(th, rh, ids_h, mask_h, *w.clip, td, rd, ids_d, mask_d, *outs, met, ws)
    torch.cuda.synchronize()
    return outs, B.read_metrics(met), copied, td, rd, mask_h


def _check(w, **kw):
    outs, met, copied, td, rd, mask_h = _run_host(w, **kw)
    ref = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
    torch.cuda.synchronize()
    for a, b in zip(outs, (ref.logp_train, ref.logp_rollout, ref.dlogp)):
        assert torch.equal(a, b)
    assert met == ref.metrics
    act = mask_h.numpy() != 0
    n_act = int(act.sum())
    row_bytes = w.vocab * (w.train.element_size() + w.rollout.element_size())
    assert copied == n_act * row_bytes + w.n_rows * 5
    sel = torch.as_tensor(act, device=DEV)
    # active rows staged exactly, inactive rows never written
    assert torch.equal(td[sel], w.train[sel]) and torch.equal(rd[sel], w.rollout[sel])
    if n_act < w.n_rows:
        assert torch.all(torch.isnan(td[~sel].float())) and torch.all(torch.isnan(rd[~sel].float()))
    return outs, met


def test_response_spans_bitwise_and_against_oracle():
    # prompt / response / right padding per sequence, as in RL batches
    batch, seq = 3, 1200
    w = W.synthetic(batch * seq, 9000, seed=5, device=DEV, active_prob=1.0)
    t = torch.arange(seq, device=DEV)[None, :]
    prompt = torch.tensor([[256], [700], [1000]], device=DEV)
    pad = torch.tensor([[0], [300], [100]], device=DEV)
    w.action_mask = ((t >= prompt) & (t < seq - pad)).reshape(-1).to(torch.uint8)
    outs, met = _check(w)
    mask = w.action_mask.cpu().numpy()
    ref = oracle.score(to_oracle(w.train), to_oracle(w.rollout), w.token_ids.cpu().numpy(), mask)
    act = mask != 0
    for got, want in zip(outs, (ref.logp_train, ref.logp_rollout, ref.dlogp)):
        assert np.max(np.abs(got.cpu().numpy().astype(np.float64)[act] - want[act])) <= LOGP_ATOL
    assert_metrics_match(met, ref.metrics, ref.dlogp, mask)


@pytest.mark.parametrize("active", [0.0, 0.35, 1.0])
def test_scattered_masks(active):
    # Bernoulli masks: many runs of active rows, each its own copy
    w = W.synthetic(500, 7001, seed=int(active * 10) + 1, device=DEV, active_prob=active)
    _check(w)


def test_padded_strides_and_mixed_dtypes():
    w = W.synthetic(300, 5003, seed=9, device=DEV, dtype_rollout=torch.float32, active_prob=0.6)
    _check(w, host_pad=13, dev_pad=5)


def test_pageable_host_memory():
    w = W.synthetic(200, 4096, seed=10, device=DEV, active_prob=0.7)
    _check(w, pinned=False)


def test_zero_rows():
    w = W.synthetic(0, 1000, seed=11, device=DEV)
    outs, met, copied, *_ = _run_host(w)
    assert copied == 0 and met["n_active"] == 0 and met["flags"] == B.LPD_FLAG_NO_ACTIVE


def test_device_mask_is_refused():
    # the host reads the mask during the call: device memory there is an
    # argument error, reported before anything is copied
    w = W.synthetic(50, 3000, seed=13, device=DEV)
    th, rh = _host_copy(w.train), _host_copy(w.rollout)
    td, rd = _staging(w.train), _staging(w.rollout)
    ids_h = w.token_ids.cpu()
    outs = [torch.empty(50, device=DEV) for _ in range(3)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, 50), dtype=torch.uint8, device=DEV)
    with pytest.raises(RuntimeError, match="device memory"):
        B.lpd_score_host(th, rh, ids_h, w.action_mask, *w.clip, td, rd, torch.empty_like(w.token_ids),
                         torch.empty_like(w.action_mask), *outs, met, ws)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(td.float()))  # nothing was copied
