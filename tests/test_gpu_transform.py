"""Vocab padding policies and the logit transform chain ("[WS2] Framework
for ablation experiment", LogProb knobs table, rows 2 and 7) against the
float64 oracle (needs a GPU)."""
import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import LOGP_ATOL, assert_metrics_match, to_oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE, SOFTCAP = B.LPD_OP_SCALE, B.LPD_OP_SOFTCAP


def _check(w, train_ops, rollout_ops, train=None, rollout=None):
    train = w.train if train is None else train
    rollout = w.rollout if rollout is None else rollout
    res = B.score(train, rollout, w.token_ids, w.action_mask, w.clip, train_ops=train_ops, rollout_ops=rollout_ops)
    torch.cuda.synchronize()
    mask = w.action_mask.cpu().numpy()
    ref = oracle.score_transformed(to_oracle(train), to_oracle(rollout), w.token_ids.cpu().numpy(), mask,
                                   train_ops, rollout_ops, *w.clip)
    act = mask != 0
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout),
                      (res.dlogp, ref.dlogp)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g[act] - want[act])) <= LOGP_ATOL
    # transformed logits are formed in fp32, so per-token dlogp carries their
    # rounding; the ratio mean is held to that per-token error
    d_err = float(np.max(np.abs(res.dlogp.cpu().numpy().astype(np.float64)[act] - ref.dlogp[act]))) if act.any() else 0.0
    assert_metrics_match(res.metrics, ref.metrics, ref.dlogp, mask, w.clip, dlogp_err=d_err)
    return res, ref


@pytest.mark.parametrize("train_ops,rollout_ops", [
    ([(SCALE, 1 / 0.7)], [(SCALE, 1 / 0.7)]),                       # same temperature both sides
    ([(SOFTCAP, 30.0)], [(SOFTCAP, 30.0)]),                         # soft-cap
    ([(SOFTCAP, 30.0), (SCALE, 1 / 0.7)], [(SOFTCAP, 30.0), (SCALE, 1 / 0.7)]),
    ([], [(SCALE, 1 / 0.7)]),                                       # temperature applied on one side only
    ([(SCALE, 1 / 0.7), (SOFTCAP, 30.0)], [(SOFTCAP, 30.0), (SCALE, 1 / 0.7)]),  # order mismatch
    # two soft-caps, and a soft-cap far from 1: the general per-op pass
    ([(SOFTCAP, 30.0), (SCALE, 2.0), (SOFTCAP, 25.0)], [(SOFTCAP, 30.0), (SCALE, 2.0), (SOFTCAP, 25.0)]),
    ([(SOFTCAP, 3e4)], [(SCALE, 1 / 0.7), (SOFTCAP, 5.0)]),
])
@pytest.mark.parametrize("shape", [(300, 3 * 8192 + 520, 0), (150, 12805, 3), (200, 5000, 0)])
def test_transform_chain_vs_oracle(train_ops, rollout_ops, shape):
    rows, vocab, pad = shape
    w = W.synthetic(rows, vocab, seed=rows + vocab, device=DEV, row_pad=pad, spike_frac=0.05, spike=40.0)
    _check(w, train_ops, rollout_ops)


@pytest.mark.parametrize("dt,dr", [(torch.bfloat16, torch.float32), (torch.float32, torch.bfloat16),
                                   (torch.float32, torch.float32)])
@pytest.mark.parametrize("ops", [[(SOFTCAP, 30.0), (SCALE, 1 / 0.7)],                   # reduced soft-cap pass
                                 [(SOFTCAP, 30.0), (SCALE, 1 / 0.7), (SOFTCAP, 40.0)],  # general pass
                                 [(SCALE, 1 / 0.7)]])                                    # scales only
@pytest.mark.parametrize("vocab,pad", [(3 * 10240 + 520, 0), (12805, 3)])
def test_transform_chain_mixed_dtypes_vs_oracle(dt, dr, ops, vocab, pad):
    # every dtype pairing of each chain form, on 16-byte aligned rows (bulk
    # copies, full and ragged tiles) and on rows that are not (plain loads)
    w = W.synthetic(120, vocab, seed=vocab + pad, device=DEV, dtype_train=dt, dtype_rollout=dr, row_pad=pad,
                    spike_frac=0.05, spike=40.0)
    _check(w, ops, ops)


def test_reduced_pass_side_without_cap_keeps_huge_logits():
    """A soft-cap on the train side only: the rollout side runs the identity
    series, whose x^3 would overflow above ~7e12, so such values must take the
    slow path (which leaves that side alone).  Huge values of both signs and
    -inf on both sides; per-token logp against the oracle within 1e-4 plus
    float32 rounding of the value itself (a logp near -1e30 carries ulps of
    1e23), and no NaN anywhere (the drift metrics of such rows are infinite on
    both sides, so they are not compared)."""
    w = W.synthetic(64, 3000, seed=37, device=DEV, active_prob=1.0)
    t, r = w.train.float().contiguous(), w.rollout.float().contiguous()
    g = torch.Generator(device=DEV).manual_seed(38)
    for x in (t, r):
        rows = torch.randint(0, 64, (20,), generator=g, device=DEV)
        cols = torch.randint(0, 3000, (20,), generator=g, device=DEV)
        x[rows, cols] = torch.tensor([1e13, -1e13, 3e30, -3e30, float("-inf")] * 4, device=DEV)
    ids = torch.remainder(w.token_ids, 3000)
    sel = torch.arange(64, device=DEV)
    mask = (torch.isfinite(t[sel, ids.long()]) & torch.isfinite(r[sel, ids.long()])).to(torch.uint8)
    ops_t, ops_r = [(SOFTCAP, 30.0), (SCALE, 1 / 0.7)], [(SCALE, 1 / 0.7)]
    res = B.score(t, r, ids, mask, train_ops=ops_t, rollout_ops=ops_r)
    torch.cuda.synchronize()
    m = mask.cpu().numpy()
    ref = oracle.score_transformed(t.cpu().numpy(), r.cpu().numpy(), ids.cpu().numpy(), m, ops_t, ops_r)
    act = m != 0
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout)):
        gn = got.cpu().numpy().astype(np.float64)
        assert not np.any(np.isnan(gn))
        assert np.all(np.abs(gn[act] - want[act]) <= LOGP_ATOL + 2.0 ** -22 * np.abs(want[act]))


def test_identity_chain_is_bitwise_lpd_score():
    w = W.synthetic(250, 20000, seed=31, device=DEV)
    plain = B.score(w.train, w.rollout, w.token_ids, w.action_mask)
    ident = B.score(w.train, w.rollout, w.token_ids, w.action_mask, train_ops=[], rollout_ops=[])
    torch.cuda.synchronize()
    for a, b in ((plain.logp_train, ident.logp_train), (plain.dlogp, ident.dlogp)):
        assert torch.equal(a, b)


def test_same_chain_both_sides_keeps_identical_rows_at_zero():
    w = W.synthetic(120, 9000, seed=32, device=DEV)
    ops = [(SOFTCAP, 20.0), (SCALE, 1.3)]
    res = B.score(w.train, w.train, w.token_ids, w.action_mask, train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    assert torch.all(res.dlogp == 0) and res.metrics["approx_kl0"] == 0.0


@pytest.mark.parametrize("policy", ["mask", "include"])
def test_vocab_padding_policies(policy):
    # padded vocab: 12288 columns stored, the first 12000 are the real vocabulary;
    # "mask" scores with vocab = 12000 and the padding never enters the LSE,
    # "include" scores all 12288 columns (pad rows initialised to 0 here)
    real, padded = 12000, 12288
    base = W.synthetic(160, padded, seed=33, device=DEV)
    train = base.train.clone()
    rollout = base.rollout.clone()
    train[:, real:] = 0.0
    rollout[:, real:] = 0.0
    ids = torch.remainder(base.token_ids, real)
    vocab = real if policy == "mask" else padded
    w = W.Workload("pad", train[:, :vocab], rollout[:, :vocab], ids, base.action_mask, vocab)
    res, ref = _check(w, None, None)
    # the two policies differ by exactly the padding's probability mass
    if policy == "include":
        other = oracle.score(to_oracle(train[:, :real]), to_oracle(rollout[:, :real]), ids.cpu().numpy(),
                             base.action_mask.cpu().numpy())
        act = base.action_mask.cpu().numpy() != 0
        assert np.all(ref.logp_train[act] < other.logp_train[act])


@pytest.mark.parametrize("ops", [
    [(SOFTCAP, 30.0)],                                  # the reduced single soft-cap pass
    [(SCALE, 0.5), (SOFTCAP, 15.0), (SCALE, 2.0)],      # the same function, scales moved behind the cap
    [(SOFTCAP, 30.0), (SOFTCAP, 1e6)],                  # general per-op pass (the second cap moves f < 1e-8)
])
def test_softcap_tanh_accuracy_per_value(ops):
    """Rows [a, 0] under soft-cap 30: logp of column 0 is -log(1 + exp(-f(a)))
    with f(a) = 30 tanh(a / 30), whose sensitivity to f is at most 1.  The
    kernel's own tanh must keep f within a few ulp: the bar is 8 ulp of
    max(1, |f|) plus the float32 rounding of logp itself.  The values cover
    both forms of the tanh (|a| < 18 and beyond), the switch point, tiny and
    saturating arguments and +-inf.  Each chain computes the same f, on the
    reduced soft-cap pass or on the general one."""
    a = np.concatenate([np.linspace(-200, 200, 4001), 18 + np.linspace(-1e-3, 1e-3, 201),
                        -18 + np.linspace(-1e-3, 1e-3, 201), [1e-30, -1e-30, 1e-7, 3e3, -3e3, np.inf, -np.inf]])
    a = a.astype(np.float32)
    n = a.size
    x = np.zeros((n, 2), np.float32)
    x[:, 0] = a
    t = torch.from_numpy(x).to(DEV)
    ids = torch.zeros(n, dtype=torch.int32, device=DEV)
    mask = torch.ones(n, dtype=torch.uint8, device=DEV)
    res = B.score(t, t, ids, mask, train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    ref = oracle.score_transformed(x, x, np.zeros(n, np.int32), np.ones(n, np.uint8), ops, ops, 0.8, 1.2)
    got = res.logp_train.cpu().numpy().astype(np.float64)
    f = 30.0 * np.tanh(a.astype(np.float64) / 30.0)
    tol = 8 * 2.0 ** -24 * np.maximum(1.0, np.abs(f)) + 2.0 ** -24 * np.maximum(1.0, np.abs(ref.logp_train))
    err = np.abs(got - ref.logp_train)
    assert np.all(err <= tol), (float(a[np.argmax(err - tol)]), float(np.max(err - tol)))


@pytest.mark.parametrize("sigma", [20.0, 3.0])
@pytest.mark.parametrize("ops", [[(SOFTCAP, 30.0), (SCALE, 1 / 0.7)],                # reduced soft-cap pass
                                 [(SOFTCAP, 30.0), (SCALE, 1 / 0.7), (SOFTCAP, 40.0)]])  # general pass
def test_softcap_load_paths_agree_bitwise(ops, sigma):
    # logits spread over both forms of the tanh within the same warps (sigma
    # 20), or all in the series range so that whole warps take the packed
    # series (sigma 3), stored with 16-byte aligned rows (bulk-copy ring) and
    # with an odd row stride (plain loads, one value at a time): identical bits
    base = W.synthetic(40, 3 * 4096 + 517, seed=19, device=DEV, row_pad=3, active_prob=1.0, sigma=sigma)
    aligned = B.score(base.train, base.rollout, base.token_ids, base.action_mask, train_ops=ops, rollout_ops=ops)
    t2, r2 = base.train.contiguous(), base.rollout.contiguous()
    assert (t2.stride(0) * 2) % 16 != 0
    generic = B.score(t2, r2, base.token_ids, base.action_mask, train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    for a, b in ((aligned.logp_train, generic.logp_train), (aligned.logp_rollout, generic.logp_rollout),
                 (aligned.dlogp, generic.dlogp)):
        assert torch.equal(a, b)


@pytest.mark.slow
@pytest.mark.parametrize("ops", [[(SOFTCAP, 30.0), (SCALE, 1 / 0.7)], [(SCALE, 1 / 0.7)],
                                 [(SOFTCAP, 30.0), (SCALE, 1 / 0.7), (SOFTCAP, 40.0)]])
def test_full_size_transform_every_active_row(ops):
    """The Qwen workload with the chains the benchmark times (soft-cap then
    temperature on the reduced soft-cap pass, temperature alone on the
    scale-only pass, and a two-cap chain on the general pass): every active row
    against the oracle on all host cores, the metrics against the oracle's
    metric function of the oracle's own per-token dlogp."""
    from oracle import stream

    w = W.qwen(device=DEV)
    res = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip, train_ops=ops, rollout_ops=ops)
    torch.cuda.synchronize()
    assert res.metrics["status"] == 0
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    ref = stream.score_transformed_rows_device(w.train, w.rollout, w.token_ids, act, ops, ops)
    errs = []
    for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout), (res.dlogp, ref.dlogp)):
        g = got.cpu().numpy().astype(np.float64)
        errs.append(float(np.max(np.abs(g[act] - want))))
    assert max(errs) <= LOGP_ATOL, errs
    d = np.zeros(mask.size)
    d[act] = ref.dlogp
    ref_m = oracle.metrics(d, mask, *w.clip)
    ref_m["status"] = ref.status
    assert_metrics_match(res.metrics, ref_m, d, mask, w.clip, dlogp_err=errs[2])
    del w, res
    torch.cuda.empty_cache()
