"""The reduction-topology arms of the vocab-sharded path ("[WS2] Framework for
ablation experiment", LogProb knobs table, row 4) against the float64 oracle
and against each other (needs a GPU).

All three arms compute the same logp exactly, so the oracle is the plain
definition (lpd score of the concatenated logits).  Bars:
  allgather_partials_fixed_merge  bitwise lpd_score_sharded (its main result,
      or its permuted-merge result for a given order);
  allgather_logits                bitwise lpd_score on the concatenated rows;
  allreduce_partials              per-token logp within 1e-4 (the scorer's
      bar); per-token dlogp within 6e-6 of the oracle.  Each side's lse here
      comes from its own fp32 sums, and dlogp is the difference of the two
      sides' logp with no exact-difference carry, so the two sides' sum errors
      add up instead of cancelling.  Per side, a shard's sum passes through at
      most about 45 fp32 roundings in sequence (a thread's running sum over
      the tiles of a row, the warp butterfly, the merge of 16 warp states),
      then the reduction adds one rescale (ex2, below 2^-22) and one addition
      per shard: below 3e-6 relative, so 6e-6 for the difference.  The
      metrics equal the oracle's metric function applied to this arm's own
      per-token dlogp.
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
FIXED, ALLREDUCE, ALLGATHER = (B.LPD_TOPO_ALLGATHER_PARTIALS_FIXED_MERGE, B.LPD_TOPO_ALLREDUCE_PARTIALS,
                               B.LPD_TOPO_ALLGATHER_LOGITS)
ALLREDUCE_D_ATOL = 6e-6


def _split(base, bounds, pad=0, rollout_dtype=None):
    def piece(x, a, b):
        if pad:
            wide = torch.full((x.shape[0], b - a + pad), float("nan"), dtype=x.dtype, device=DEV)
            wide[:, :b - a] = x[:, a:b]
            return wide[:, :b - a]
        return x[:, a:b].contiguous()

    r = base.rollout if rollout_dtype is None else base.rollout.to(rollout_dtype)
    ts = [piece(base.train, a, b) for a, b in bounds]
    rs = [piece(r, a, b) for a, b in bounds]
    return W.Workload("sh", ts, rs, base.token_ids, base.action_mask, base.vocab, v_ranges=list(bounds))


def _arm(w, topo, order=None):
    res = B.score_sharded_topology(w.train, w.rollout, w.v_ranges, w.token_ids, w.action_mask, topo, order)
    torch.cuda.synchronize()
    return res


def _sharded(w, perm=None):
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(5)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SHARDED, n, w.vocab, len(w.v_ranges)), dtype=torch.uint8,
                     device=DEV)
    B.lpd_score_sharded(w.train, w.rollout, w.v_ranges, w.token_ids, w.action_mask, 0.8, 1.2, perm, *outs, met, ws)
    torch.cuda.synchronize()
    return outs, B.read_metrics(met)


LAYOUTS = {
    "four_equal": ([(0, 4096), (4096, 8192), (8192, 12288), (12288, 16384)], 0, None),
    "ragged_padded": ([(0, 1000), (1000, 9000), (9000, 9001), (9001, 12003)], 5, None),
    "mixed_dtype": ([(0, 3001), (3001, 7000)], 0, torch.float32),
    # 16-byte multiples on both sides: the -inf tail copies with mixed dtypes
    "mixed_dtype_filled_tails": ([(0, 4096), (4096, 9000), (9000, 9016)], 0, torch.float32),
    "one_shard": ([(0, 5000)], 0, None),
}


@pytest.mark.parametrize("name", sorted(LAYOUTS))
def test_arms_against_oracle_and_each_other(name):
    bounds, pad, rdt = LAYOUTS[name]
    base = W.synthetic(150, bounds[-1][1], seed=len(bounds) * 7 + pad, device=DEV, active_prob=0.8,
                       rollout_noise=3e-3)
    w = _split(base, bounds, pad, rdt)
    mask = w.action_mask.cpu().numpy()
    act = mask != 0
    full_r = base.rollout if rdt is None else base.rollout.to(rdt)
    ref = oracle.score(to_oracle(base.train), to_oracle(full_r), base.token_ids.cpu().numpy(), mask)
    order = list(range(len(bounds)))[::-1]

    # fixed merge: lpd_score_sharded's result, bit for bit (in shard order and reversed)
    (lt, lr, d, plt, plr), met = _sharded(w, order)
    fx = _arm(w, FIXED)
    assert torch.equal(fx.logp_train, lt) and torch.equal(fx.logp_rollout, lr) and torch.equal(fx.dlogp, d)
    assert fx.metrics == met
    fxo = _arm(w, FIXED, order)
    assert torch.equal(fxo.logp_train, plt) and torch.equal(fxo.logp_rollout, plr)

    # all-gather of the logits: lpd_score on the concatenated rows, bit for bit
    ag = _arm(w, ALLGATHER)
    whole = B.score(base.train, full_r, base.token_ids, base.action_mask)
    torch.cuda.synchronize()
    for a, b in ((ag.logp_train, whole.logp_train), (ag.logp_rollout, whole.logp_rollout),
                 (ag.dlogp, whole.dlogp)):
        assert torch.equal(a, b)
    assert ag.metrics == whole.metrics
    assert_metrics_match(ag.metrics, ref.metrics, ref.dlogp, mask)

    # all-reduce of the partials, in shard order and reversed
    for o in (None, order):
        ar = _arm(w, ALLREDUCE, o)
        lt_a, lr_a, d_a = (x.cpu().numpy().astype(np.float64) for x in (ar.logp_train, ar.logp_rollout, ar.dlogp))
        assert np.all(lt_a[~act] == 0) and np.all(d_a[~act] == 0)
        assert np.max(np.abs(lt_a[act] - ref.logp_train[act])) <= LOGP_ATOL
        assert np.max(np.abs(lr_a[act] - ref.logp_rollout[act])) <= LOGP_ATOL
        assert np.max(np.abs(d_a[act] - ref.dlogp[act])) <= ALLREDUCE_D_ATOL
        prop = oracle.metrics(d_a, mask, 0.8, 1.2)
        prop["status"] = 0
        assert_metrics_match(ar.metrics, prop, d_a, mask, ambiguity=1e-6)


def test_allreduce_of_identical_sides_gives_exact_zero():
    # both sides' lse come out of the same arithmetic, so their difference is 0
    base = W.synthetic(64, 9000, seed=3, device=DEV, active_prob=1.0)
    w = _split(base, [(0, 2000), (2000, 9000)])
    w.rollout = w.train
    ar = _arm(w, ALLREDUCE, [1, 0])
    assert torch.all(ar.dlogp == 0)
    assert ar.metrics["approx_kl0"] == 0.0 and ar.metrics["ratio0_mean"] == 1.0


def test_arms_edge_cases():
    base = W.synthetic(40, 3000, seed=4, device=DEV, active_prob=0.0)
    w = _split(base, [(0, 1000), (1000, 3000)])
    for topo in (FIXED, ALLREDUCE, ALLGATHER):
        res = _arm(w, topo)
        assert res.metrics["n_active"] == 0 and res.metrics["flags"] == B.LPD_FLAG_NO_ACTIVE
        assert torch.all(res.dlogp == 0)
    # an out-of-range id on an active row fails closed in every arm
    base = W.synthetic(20, 3000, seed=5, device=DEV, active_prob=1.0)
    base.token_ids[3] = 3000
    w = _split(base, [(0, 1000), (1000, 3000)])
    for topo in (FIXED, ALLREDUCE, ALLGATHER):
        res = _arm(w, topo)
        assert res.metrics["status"] & B.LPD_STATUS_TOKEN_OOB
        assert torch.isnan(res.logp_train[3])
    # zero rows
    empty = W.synthetic(0, 3000, seed=6, device=DEV)
    w = _split(empty, [(0, 1000), (1000, 3000)])
    for topo in (FIXED, ALLREDUCE, ALLGATHER):
        assert _arm(w, topo).metrics["n_active"] == 0


@pytest.mark.slow
def test_full_size_arms_every_row():
    """The 4-way vocab split of 32768 rows x 151936 in the benchmark's launch
    configuration; every row of each arm against the oracle (all host cores).
    The fixed-merge and all-gather arms keep the exact-difference carry, so
    their metrics are held to the oracle's metric function of the oracle's own
    dlogp; the all-reduce arm's dlogp carries up to 6e-6 of independent sum
    rounding per token (module docstring), which alone moves approx_kl0 of this
    workload (|dlogp| ~ 1e-3) by more than 1e-4 relative, so its metrics are
    held to the oracle's metric function of its own per-token dlogp."""
    from oracle import stream

    w = W.sharded(device=DEV)
    rows = np.arange(w.n_rows)
    ref = stream.score_sharded_rows_device(w.train, w.rollout, w.v_ranges, w.token_ids, rows)
    mask = w.action_mask.cpu().numpy()
    ref_m = oracle.metrics(ref.dlogp, mask, *w.clip)
    ref_m["status"] = ref.status
    results = {}
    for topo in (FIXED, ALLREDUCE, ALLGATHER):
        res = _arm(w, topo)
        assert res.metrics["status"] == 0 and res.metrics["n_active"] == w.n_rows
        for got, want in ((res.logp_train, ref.logp_train), (res.logp_rollout, ref.logp_rollout)):
            assert np.max(np.abs(got.cpu().numpy().astype(np.float64) - want)) <= LOGP_ATOL
        d = res.dlogp.cpu().numpy().astype(np.float64)
        d_err = float(np.max(np.abs(d - ref.dlogp)))
        if topo == ALLREDUCE:
            assert d_err <= ALLREDUCE_D_ATOL
            prop = oracle.metrics(d, mask, *w.clip)
            prop["status"] = 0
            assert_metrics_match(res.metrics, prop, d, mask, w.clip, ambiguity=1e-6)
        else:
            assert d_err <= LOGP_ATOL
            assert_metrics_match(res.metrics, ref_m, ref.dlogp, mask, w.clip, dlogp_err=d_err)
        results[topo] = res
    # the arms move the same numbers: topology drift is rounding only
    for topo in (ALLREDUCE, ALLGATHER):
        assert torch.max(torch.abs(results[topo].dlogp - results[FIXED].dlogp)).item() <= 2 * ALLREDUCE_D_ATOL
