"""Fused LM-head path against the float64 oracle (needs a GPU).

The oracle materialises x = h W^T in double (every bf16 x bf16 product is
exact in double) and applies the plain definition; the GPU never materialises
the logits.  Bars as in tests/helpers.py.
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


def run(w, ht=None, hr=None, ids=None, mask=None):
    res = B.score_fused(w.hidden_train if ht is None else ht, w.hidden_rollout if hr is None else hr, w.weight,
                        w.token_ids if ids is None else ids, w.action_mask if mask is None else mask, w.clip)
    torch.cuda.synchronize()
    return res


def oracle_rows(w, rows):
    return oracle.score_head_rows(to_oracle(w.hidden_train), to_oracle(w.hidden_rollout), to_oracle(w.weight),
                                  w.token_ids.cpu().numpy(), rows)


@pytest.mark.parametrize("rows,hidden,vocab,active", [
    (40, 64, 300, 1.0),        # one row tile, two vocab tiles (ragged), K = one stage
    (200, 128, 1000, 0.8),     # two row tiles (ragged), four vocab tiles (ragged), masked rows
    (300, 512, 5000, 0.9),     # several K blocks per tile and many vocab tiles
    (129, 256, 256, 1.0),      # exactly one vocab tile, one row past a tile
])
def test_fused_vs_oracle(rows, hidden, vocab, active):
    w = W.head(rows, hidden, vocab, seed=rows + hidden, device=DEV, active_prob=active)
    res = run(w)
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    ref = oracle_rows(w, act)
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout),
                      (res.dlogp, ref.dlogp)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g[act] - want)) <= LOGP_ATOL
    assert np.all(res.dlogp.cpu().numpy()[mask == 0] == 0)
    d = np.zeros(rows)
    d[act] = ref.dlogp
    met = oracle.metrics(d, mask, *w.clip)
    met["status"] = 0
    assert_metrics_match(res.metrics, met, d, mask, w.clip)


def test_fused_identical_inputs_exact_zero():
    w = W.head(150, 128, 700, seed=3, device=DEV)
    res = run(w, hr=w.hidden_train)
    assert torch.all(res.dlogp == 0)
    assert torch.equal(res.logp_train, res.logp_rollout)
    assert res.metrics["approx_kl0"] == 0.0 and res.metrics["ratio0_mean"] == 1.0


def test_fused_batch_composition_bitwise():
    w = W.head(140, 256, 1300, seed=5, device=DEV)
    full = run(w)
    for start, total, off in ((0, 1, 0), (17, 7, 3), (100, 40, 33), (5, 300, 200)):
        k = min(total - off, 7 if total > 1 else 1)
        sel = slice(start, start + k)
        g = torch.Generator(device=DEV).manual_seed(start)
        ht = torch.randn((total, w.hidden), generator=g, device=DEV).to(torch.bfloat16)
        hr = torch.randn((total, w.hidden), generator=g, device=DEV).to(torch.bfloat16)
        ids = torch.randint(0, w.vocab, (total,), generator=g, device=DEV, dtype=torch.int32)
        mask = torch.ones(total, dtype=torch.uint8, device=DEV)
        ht[off:off + k] = w.hidden_train[sel]
        hr[off:off + k] = w.hidden_rollout[sel]
        ids[off:off + k] = w.token_ids[sel]
        res = run(w, ht, hr, ids, mask)
        for a, b in ((res.logp_train, full.logp_train), (res.logp_rollout, full.logp_rollout),
                     (res.dlogp, full.dlogp)):
            assert torch.equal(a[off:off + k], b[sel])


def test_fused_matches_unfused_on_materialised_logits():
    # the fused path and the streaming path agree on the same logits to the
    # logp bar (the streaming path reads fp32 logits materialised here)
    w = W.head(96, 256, 3000, seed=7, device=DEV)
    res = run(w)
    xt = (w.hidden_train.float() @ w.weight.float().T).contiguous()
    xr = (w.hidden_rollout.float() @ w.weight.float().T).contiguous()
    ref = B.score(xt, xr, w.token_ids, w.action_mask)
    torch.cuda.synchronize()
    for a, b in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout)):
        assert torch.max(torch.abs(a - b)).item() <= LOGP_ATOL


def test_full_size_fused_sampled_rows():
    w = W.fused(device=DEV)
    res = run(w)
    assert res.metrics["n_active"] == w.n_rows and res.metrics["status"] == 0
    rows = np.array([0, 1, 127, 128, 8191, 16383])
    sel = torch.as_tensor(rows, device=DEV)
    sub = W.HeadWorkload("sub", w.hidden_train[sel], w.hidden_rollout[sel], w.weight, w.token_ids[sel],
                         w.action_mask[sel])
    ref = oracle_rows(sub, np.arange(rows.size))
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout),
                      (res.dlogp, ref.dlogp)):
        g = got[sel].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g - want)) <= LOGP_ATOL
    d = res.dlogp.cpu().numpy().astype(np.float64)
    prop = oracle.metrics(d, np.ones(w.n_rows, np.uint8), *w.clip)
    prop["status"] = 0
    assert_metrics_match(res.metrics, prop, d, np.ones(w.n_rows, np.uint8), w.clip, ambiguity=1e-6)


# ---- transform chains in the fused epilogue ("[WS2] Framework for ablation
# experiment", LogProb knobs table, row 7) ------------------------------------
SCALE, SOFTCAP = B.LPD_OP_SCALE, B.LPD_OP_SOFTCAP


def oracle_rows_transformed(w, rows, train_ops, rollout_ops):
    """The oracle's double-precision head logits of the listed rows, rounded
    once to float32 (the oracle's transformed scorer reads bf16 or float32
    logits; the rounding, 2^-24 relative, is far below the logp bar), through
    each side's chain and the plain definition."""
    ht, hr, wt = to_oracle(w.hidden_train), to_oracle(w.hidden_rollout), to_oracle(w.weight)
    xt = np.stack([oracle.head_logits(ht[r], wt) for r in rows]).astype(np.float32)
    xr = np.stack([oracle.head_logits(hr[r], wt) for r in rows]).astype(np.float32)
    ids = w.token_ids.cpu().numpy()[rows]
    return oracle.score_transformed(xt, xr, ids, np.ones(len(rows), np.uint8), train_ops, rollout_ops, *w.clip)


CHAINS = [
    ([(SCALE, 1 / 0.7)], [(SCALE, 1 / 0.7)]),                      # temperature on both sides
    ([(SOFTCAP, 0.5)], [(SOFTCAP, 0.5)]),                          # soft-cap in its exponential range
    ([(SCALE, 30.0), (SOFTCAP, 10.0)], [(SCALE, 30.0), (SOFTCAP, 10.0)]),  # both tanh ranges
    ([], [(SCALE, 1 / 0.7)]),                                      # temperature on one side only
    ([(SCALE, 2.0), (SOFTCAP, 1.0)], [(SOFTCAP, 1.0), (SCALE, 2.0)]),     # order mismatch
]


@pytest.mark.parametrize("train_ops,rollout_ops", CHAINS)
@pytest.mark.parametrize("rows,hidden,vocab,active", [
    (40, 64, 300, 1.0),        # ragged last vocab tile: padding must stay out after the chain
    (200, 256, 1000, 0.8),     # two row tiles (ragged), masked rows
    (130, 512, 2600, 0.9),
])
def test_fused_transform_vs_oracle(train_ops, rollout_ops, rows, hidden, vocab, active):
    w = W.head(rows, hidden, vocab, seed=rows + vocab, device=DEV, active_prob=active)
    res = B.score_fused(w.hidden_train, w.hidden_rollout, w.weight, w.token_ids, w.action_mask, w.clip,
                        train_ops=train_ops, rollout_ops=rollout_ops)
    torch.cuda.synchronize()
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    ref = oracle_rows_transformed(w, act, train_ops, rollout_ops)
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout),
                      (res.dlogp, ref.dlogp)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g[act] - want)) <= LOGP_ATOL
    assert np.all(res.dlogp.cpu().numpy()[mask == 0] == 0)
    d = np.zeros(rows)
    d[act] = ref.dlogp
    d_err = float(np.max(np.abs(res.dlogp.cpu().numpy().astype(np.float64)[act] - ref.dlogp)))
    met = oracle.metrics(d, mask, *w.clip)
    met["status"] = 0
    assert_metrics_match(res.metrics, met, d, mask, w.clip, dlogp_err=d_err)


def test_fused_transform_matches_streaming_transform():
    # same chain on the fused path and on the streaming path over float32
    # logits materialised here: the two agree to the logp bar
    w = W.head(96, 256, 3000, seed=9, device=DEV)
    ops_t, ops_r = [(SCALE, 20.0), (SOFTCAP, 8.0)], [(SOFTCAP, 8.0), (SCALE, 20.0)]
    res = B.score_fused(w.hidden_train, w.hidden_rollout, w.weight, w.token_ids, w.action_mask, w.clip,
                        train_ops=ops_t, rollout_ops=ops_r)
    xt = (w.hidden_train.float() @ w.weight.float().T).contiguous()
    xr = (w.hidden_rollout.float() @ w.weight.float().T).contiguous()
    ref = B.score(xt, xr, w.token_ids, w.action_mask, w.clip, train_ops=ops_t, rollout_ops=ops_r)
    torch.cuda.synchronize()
    for a, b in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout), (res.dlogp, ref.dlogp)):
        assert torch.max(torch.abs(a - b)).item() <= LOGP_ATOL


def test_fused_same_chain_identical_inputs_exact_zero():
    w = W.head(150, 128, 700, seed=11, device=DEV)
    ops = [(SOFTCAP, 0.3), (SCALE, 1.7)]
    res = B.score_fused(w.hidden_train, w.hidden_train, w.weight, w.token_ids, w.action_mask, w.clip,
                        train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    assert torch.all(res.dlogp == 0) and torch.equal(res.logp_train, res.logp_rollout)
    assert res.metrics["approx_kl0"] == 0.0


def test_fused_empty_chains_are_the_plain_kernel():
    w = W.head(100, 128, 900, seed=13, device=DEV)
    plain = run(w)
    ident = B.score_fused(w.hidden_train, w.hidden_rollout, w.weight, w.token_ids, w.action_mask, w.clip,
                          train_ops=[], rollout_ops=[])
    torch.cuda.synchronize()
    for a, b in ((plain.logp_train, ident.logp_train), (plain.dlogp, ident.dlogp)):
        assert torch.equal(a, b)


@pytest.mark.slow
def test_full_size_fused_transform_sampled_rows():
    w = W.fused(device=DEV)
    ops = [(SOFTCAP, 30.0), (SCALE, 1 / 0.7)]
    res = B.score_fused(w.hidden_train, w.hidden_rollout, w.weight, w.token_ids, w.action_mask, w.clip,
                        train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    assert res.metrics["status"] == 0 and res.metrics["n_active"] == w.n_rows
    rows = np.array([0, 127, 128, 16383])
    sel = torch.as_tensor(rows, device=DEV)
    sub = W.HeadWorkload("sub", w.hidden_train[sel], w.hidden_rollout[sel], w.weight, w.token_ids[sel],
                         w.action_mask[sel])
    ref = oracle_rows_transformed(sub, np.arange(rows.size), ops, ops)
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout), (res.dlogp, ref.dlogp)):
        assert np.max(np.abs(got[sel].cpu().numpy().astype(np.float64) - want)) <= LOGP_ATOL
