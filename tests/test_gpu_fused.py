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


def _embed_head(w, sel, k, n_left, n_before, n_after, n_right, seed):
    """A batch holding the rows ``sel`` (k of them) of w after n_before active
    garbage rows (so the picked rows start at compacted position n_before and
    may straddle a 128-row tile), with n_after active garbage rows after them,
    and n_left / n_right inactive garbage rows at the two ends.  Returns the
    batch and the batch position of the first picked row."""
    total = n_left + n_before + k + n_after + n_right
    g = torch.Generator(device=DEV).manual_seed(seed)
    ht = torch.randn((total, w.hidden), generator=g, device=DEV).to(torch.bfloat16)
    hr = torch.randn((total, w.hidden), generator=g, device=DEV).to(torch.bfloat16)
    ids = torch.randint(0, w.vocab, (total,), generator=g, device=DEV, dtype=torch.int32)
    mask = torch.ones(total, dtype=torch.uint8, device=DEV)
    mask[:n_left] = 0
    mask[total - n_right:] = 0
    off = n_left + n_before
    ht[off:off + k] = w.hidden_train[sel]
    hr[off:off + k] = w.hidden_rollout[sel]
    ids[off:off + k] = w.token_ids[sel]
    return ht, hr, ids, mask, off


# (first picked row, k, inactive left pad, active rows before, active rows
# after, inactive right pad): batches of 1, 7 and 64, placed at the start of a
# tile, at its last row, across the boundary between the first and second
# 128-row tiles, and behind left and right padding
HEAD_PLACEMENTS = [(0, 1, 0, 0, 0, 0), (5, 1, 3, 127, 0, 2), (9, 1, 0, 128, 40, 0), (0, 7, 0, 0, 0, 0),
                   (7, 7, 2, 125, 0, 5), (20, 7, 9, 60, 100, 0), (0, 64, 0, 0, 0, 0), (0, 64, 4, 100, 30, 11),
                   (0, 64, 0, 250, 0, 1)]


def _head_batch_controls(w, full, picked, seed):
    for j0, k, n_left, n_before, n_after, n_right in HEAD_PLACEMENTS:
        sel = picked[j0:j0 + k]
        ht, hr, ids, mask, off = _embed_head(w, sel, k, n_left, n_before, n_after, n_right, seed + j0 + 3 * k)
        res = run(w, ht, hr, ids, mask)
        for a, b in ((res.logp_train, full.logp_train), (res.logp_rollout, full.logp_rollout),
                     (res.dlogp, full.dlogp)):
            assert torch.equal(a[off:off + k], b[sel]), (j0, k, n_left, n_before, n_after, n_right)


def test_fused_batch_composition_bitwise():
    w = W.head(300, 256, 1300, seed=5, device=DEV)
    full = run(w)
    picked = torch.arange(10, 74, device=DEV)
    _head_batch_controls(w, full, picked, seed=5)


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


@pytest.mark.slow
def test_full_size_fused_rows_and_batch_control():
    """The fused LM-head workload itself (16384 tokens x H = 4096, W [151936,
    4096]): 128 rows, one in every 128-row tile at a different position,
    against the oracle's double-precision head on all host cores; then the
    batch-composition control at this shape (every tile runs all 64 K blocks
    of H = 4096): 64 rows rescored at batch 1, 7 and 64, across tile
    boundaries and behind padding, bitwise equal to the full batch."""
    from oracle import stream

    w = W.fused(device=DEV)
    res = run(w)
    assert res.metrics["n_active"] == w.n_rows and res.metrics["status"] == 0
    n_tiles = w.n_rows // 128
    rows = np.array([128 * j + (37 * j) % 128 for j in range(n_tiles)])
    rows[0], rows[-1] = 0, w.n_rows - 1
    ref = stream.score_head_rows_parallel(to_oracle(w.hidden_train), to_oracle(w.hidden_rollout),
                                          to_oracle(w.weight), w.token_ids.cpu().numpy(), rows)
    sel = torch.as_tensor(rows, device=DEV)
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout),
                      (res.dlogp, ref.dlogp)):
        g = got[sel].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g - want)) <= LOGP_ATOL
    # the metrics over all 16384 tokens: the oracle's metric function of the
    # GPU's per-token dlogp (the oracle's head costs ~2 s of one core per row)
    d = res.dlogp.cpu().numpy().astype(np.float64)
    prop = oracle.metrics(d, np.ones(w.n_rows, np.uint8), *w.clip)
    prop["status"] = 0
    assert_metrics_match(res.metrics, prop, d, np.ones(w.n_rows, np.uint8), w.clip, ambiguity=1e-6)
    rng = np.random.default_rng(19)
    picked = torch.as_tensor(np.sort(rng.choice(w.n_rows, size=64, replace=False)), device=DEV)
    _head_batch_controls(w, res, picked, seed=23)
    del w, res
    torch.cuda.empty_cache()


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
    # two soft-caps per side: the general per-op chain in the epilogue
    ([(SOFTCAP, 3.0), (SCALE, 1.5), (SOFTCAP, 4.0)], [(SOFTCAP, 3.0), (SCALE, 1.5), (SOFTCAP, 4.0)]),
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
