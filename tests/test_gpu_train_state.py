"""Entropy and the logprob gradient ("[WS2] Framework for ablation
experiment", LogProb knobs table, row 11) against the float64 oracle (needs a
GPU)."""
import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
ENT_ATOL = 1e-4


def score_entropy(w, train=None, rollout=None):
    train = w.train if train is None else train
    rollout = w.rollout if rollout is None else rollout
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(5)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    B.lpd_score_entropy(train, rollout, w.token_ids, w.action_mask, *w.clip, *outs, met, ws)
    torch.cuda.synchronize()
    return outs, B.read_metrics(met)


@pytest.mark.parametrize("rows,vocab,dr,pad", [
    (200, 3 * 8192 + 520, torch.bfloat16, 0),
    (150, 12805, torch.bfloat16, 3),
    (120, 9000, torch.float32, 0),
    (60, 151936, torch.bfloat16, 0),
    (80, 7, torch.bfloat16, 0),
    (90, 11776 + 8, torch.float32, 0),   # one full tile and an 8-column ragged one
])
def test_entropy_vs_oracle(rows, vocab, dr, pad):
    w = W.synthetic(rows, vocab, seed=rows + vocab, device=DEV, dtype_rollout=dr, row_pad=pad, spike_frac=0.1)
    (lt, lr, d, et, er), met = score_entropy(w)
    mask = w.action_mask.cpu().numpy()
    ref_t, ref_r = oracle.entropy(to_oracle(w.train), to_oracle(w.rollout), mask)
    act = mask != 0
    for got, want in ((et, ref_t), (er, ref_r)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g[act] - want[act])) <= ENT_ATOL
        assert np.all(g[~act] == 0)
    # the scoring outputs are the plain pass's, bit for bit
    plain = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
    torch.cuda.synchronize()
    for a, b in ((lt, plain.logp_train), (lr, plain.logp_rollout), (d, plain.dlogp)):
        assert torch.equal(a, b)
    assert met == plain.metrics


@pytest.mark.parametrize("rows,vocab,dr,pad", [
    (24, 151936, torch.bfloat16, 0),     # bulk-copy path, ragged last tile
    (24, 2 * 11776, torch.bfloat16, 0),  # whole tiles only: every column on the unclamped path
    (24, 12805, torch.float32, 3),       # unaligned rows: plain loads
])
def test_entropy_with_neg_inf_logits(rows, vocab, dr, pad):
    """-inf logits inside full tiles (a masked vocabulary): their softmax terms
    are 0 and add nothing to the entropy.  Rows without -inf give the same bits
    as in a batch with no -inf at all."""
    w = W.synthetic(rows, vocab, seed=vocab + 1, device=DEV, dtype_rollout=dr, row_pad=pad, active_prob=1.0)
    g = torch.Generator().manual_seed(11)
    tr, ro = w.train.clone(), w.rollout.clone()
    ninf = float("-inf")
    scatter = torch.rand(vocab, generator=g) < 0.1
    tr[0, scatter.to(DEV)] = ninf                         # scattered, train side
    ro[1, : vocab // 2] = ninf                            # a leading block, rollout side
    tr[2, vocab // 3: vocab // 3 + 5000] = ninf           # a middle block, both sides
    ro[2, vocab // 3: vocab // 3 + 5000] = ninf
    keep = torch.zeros(vocab, dtype=torch.bool)
    keep[torch.randint(0, vocab, (40,), generator=g)] = True
    tr[3, ~keep.to(DEV)] = ninf                           # all but a few columns
    ro[3, ~keep.to(DEV)] = ninf
    tr[4, -1] = ninf                                      # the last column only
    for r in range(5):                                    # selected tokens stay finite
        c = int(w.token_ids[r])
        tr[r, c], ro[r, c] = w.train[r, c], w.rollout[r, c]
    (lt, lr, d, et, er), met = score_entropy(w, tr, ro)
    mask = w.action_mask.cpu().numpy()
    ref_t, ref_r = oracle.entropy(to_oracle(tr), to_oracle(ro), mask)
    for got, want in ((et, ref_t), (er, ref_r)):
        gn = got.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(gn)) and np.max(np.abs(gn - want)) <= ENT_ATOL
    plain = B.score(tr, ro, w.token_ids, w.action_mask, w.clip)
    torch.cuda.synchronize()
    for a, b in ((lt, plain.logp_train), (lr, plain.logp_rollout), (d, plain.dlogp)):
        assert torch.equal(a, b)
    (_, _, _, et0, er0), _ = score_entropy(w)
    assert torch.equal(et[5:], et0[5:]) and torch.equal(er[5:], er0[5:])


def test_entropy_closed_forms():
    vocab = 5000
    u = torch.full((40, vocab), 1.5, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros(40, dtype=torch.int32, device=DEV)
    mask = torch.ones(40, dtype=torch.uint8, device=DEV)
    w = W.Workload("u", u, u, ids, mask, vocab)
    (_, _, _, et, er), _ = score_entropy(w)
    assert torch.max(torch.abs(et.double() - np.log(vocab))).item() <= ENT_ATOL
    assert torch.equal(et, er)
    peaked = torch.zeros((8, vocab), dtype=torch.float32, device=DEV)
    peaked[:, 11] = 80.0
    w2 = W.Workload("p", peaked, peaked, ids[:8], mask[:8], vocab)
    (_, _, _, e2, _), _ = score_entropy(w2)
    assert torch.all(e2.abs() <= ENT_ATOL)


@pytest.mark.parametrize("rows,vocab,dt,out_dtype,pad", [
    (64, 3 * 2048 + 40, torch.bfloat16, torch.float32, 0),
    (64, 5000, torch.float32, torch.float32, 3),
    (48, 1001, torch.bfloat16, torch.float32, 0),     # rows not 16-byte aligned: scalar path
    (64, 20000, torch.bfloat16, torch.bfloat16, 0),
])
def test_backward_vs_oracle(rows, vocab, dt, out_dtype, pad):
    w = W.synthetic(rows, vocab, seed=rows * 7 + vocab, device=DEV, dtype_train=dt, row_pad=pad, active_prob=0.8)
    res = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
    g = torch.Generator(device=DEV).manual_seed(5)
    grad = torch.randn(rows, generator=g, device=DEV)
    out = torch.full((rows, vocab), float("nan"), dtype=out_dtype, device=DEV)
    B.lpd_logprob_backward(w.train, w.token_ids, w.action_mask, res.logp_train, grad, out)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    x = to_oracle(w.train)
    mask = w.action_mask.cpu().numpy()
    ids = w.token_ids.cpu().numpy()
    gr = grad.double().cpu().numpy()
    for r in range(rows):
        if not mask[r]:
            assert np.all(got[r] == 0)
            continue
        want = oracle.logprob_backward_row(np.ascontiguousarray(x[r]), int(ids[r]), float(gr[r]))
        tol = 1e-5 * abs(gr[r]) + (2.0 ** -8 * np.abs(want) if out_dtype == torch.bfloat16 else 0.0)
        assert np.all(np.abs(got[r] - want) <= tol + 1e-12), r
        if out_dtype == torch.float32:
            assert abs(got[r].sum()) <= 1e-4 * abs(gr[r]) + 1e-9


def test_backward_oob_id_is_nan():
    w = W.synthetic(10, 3000, seed=9, device=DEV, active_prob=1.0)
    res = B.score(w.train, w.rollout, w.token_ids, w.action_mask)
    ids = w.token_ids.clone()
    ids[3] = 3000
    out = torch.zeros((10, 3000), dtype=torch.float32, device=DEV)
    B.lpd_logprob_backward(w.train, ids, w.action_mask, res.logp_train, torch.ones(10, device=DEV), out)
    torch.cuda.synchronize()
    assert torch.all(torch.isnan(out[3])) and not torch.any(torch.isnan(out[2]))


@pytest.mark.slow
def test_full_size_entropy_and_backward():
    """The Qwen workload (32768 rows x 151936, bf16 both sides) in the launch
    configurations the benchmark times: every active row's two entropies
    against the oracle (all host cores); the gradient of 256 active rows
    against the oracle's, and inactive gradient rows all zero."""
    from oracle import stream

    w = W.qwen(device=DEV)
    (lt, _, _, et, er), met = score_entropy(w)
    assert met["status"] == 0
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    ref_t, ref_r = stream.entropy_rows_device(w.train, w.rollout, act)
    assert np.max(np.abs(et.cpu().numpy().astype(np.float64)[act] - ref_t)) <= ENT_ATOL
    assert np.max(np.abs(er.cpu().numpy().astype(np.float64)[act] - ref_r)) <= ENT_ATOL
    assert np.all(et.cpu().numpy()[mask == 0] == 0) and np.all(er.cpu().numpy()[mask == 0] == 0)
    g = torch.Generator(device=DEV).manual_seed(22)
    grad = torch.randn(w.n_rows, generator=g, device=DEV)
    out = torch.empty((w.n_rows, w.vocab), dtype=torch.bfloat16, device=DEV)
    B.lpd_logprob_backward(w.train, w.token_ids, w.action_mask, lt, grad, out)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(21).choice(act, size=256, replace=False))
    want = stream.backward_rows_device(w.train, w.token_ids, grad, rows)
    got = out[torch.as_tensor(rows, device=DEV)].double().cpu().numpy()
    gr = np.abs(grad.double().cpu().numpy()[rows])[:, None]
    assert np.all(np.abs(got - want) <= 1e-5 * gr + 2.0 ** -8 * np.abs(want) + 1e-12)
    for r in np.flatnonzero(mask == 0)[:4]:
        assert torch.all(out[int(r)] == 0)
