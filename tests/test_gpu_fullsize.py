"""Full-size parity, end to end, against the float64 oracle (needs a GPU).

For the Qwen3-8B-vocab (8 x 4096 rows, V = 151936, bf16/bf16), Llama-vocab
(64 x 1024 rows, V = 128256, bf16/fp32) and vocab-sharded (4 x 37984
columns, 32768 rows) workloads, EVERY active row is scored by the oracle
(serial float64 C, spread over all host cores by oracle/stream.py, which
only schedules), and:
  * each per-token logp_train, logp_rollout and dlogp is within 1e-4 of the
    oracle's ("WS2 Cross-Config Logprob Drift Contract", "Measurement
    Contract");
  * the GPU's metric record is held to the oracle's metric function applied to
    the ORACLE's own dlogp ("Diagnostics"): approx_kl0 and mean_abs_dlogp
    within 1e-4 relative, p95/p99/max within 1e-4, counts and the worst token
    exact, clipfrac0 exact but for tokens within 1e-9 of a clip bound;
  * the batch-composition control ("Attention Debug Matrix", "Metrics", C1)
    runs at the workload's own shape and dtypes: 64 of its rows, rescored
    alone, seven at a time and all at once, at shifted offsets inside batches
    padded with inactive garbage rows on either side, give bitwise the logp and
    dlogp they got in the full batch.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from oracle import stream
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import LOGP_ATOL, assert_metrics_match

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _per_token_and_metrics(got, mask, ref, clip):
    """got: (logp_t, logp_r, dlogp) device tensors over all rows; ref: the
    oracle's Result over the active rows in row order."""
    act = np.flatnonzero(mask)
    errs = []
    for g, want in zip(got, (ref.logp_train, ref.logp_rollout, ref.dlogp)):
        gn = g.cpu().numpy().astype(np.float64)
        assert np.all(gn[mask == 0] == 0)
        e = float(np.max(np.abs(gn[act] - want))) if act.size else 0.0
        errs.append(e)
    assert max(errs) <= LOGP_ATOL, errs
    d_full = np.zeros(mask.size)
    d_full[act] = ref.dlogp
    ref_m = oracle.metrics(d_full, mask, *clip)
    ref_m["status"] = ref.status
    return d_full, ref_m, errs


def _embed(rows_t, rows_r, ids, n_total, offset, seed):
    """The given rows at [offset, offset + k) of a batch of n_total rows whose
    other rows are inactive garbage (padding on either side)."""
    k, V = rows_t.shape
    g = torch.Generator(device=DEV).manual_seed(seed)
    t = (100 * torch.randn((n_total, V), generator=g, device=DEV)).to(rows_t.dtype)
    r = (100 * torch.randn((n_total, V), generator=g, device=DEV)).to(rows_r.dtype)
    i = torch.randint(-5, V + 5, (n_total,), generator=g, device=DEV, dtype=torch.int32)
    m = torch.zeros(n_total, dtype=torch.uint8, device=DEV)
    t[offset:offset + k] = rows_t
    r[offset:offset + k] = rows_r
    i[offset:offset + k] = ids
    m[offset:offset + k] = 1
    return t, r, i, m


# (first picked row, batch size k, total rows, offset): batch 1 at both ends,
# batches of 7 with left padding, right padding and both, batch 64 in the middle
PLACEMENTS = [(0, 1, 1, 0), (63, 1, 5, 4), (9, 1, 3, 1), (0, 7, 7, 0), (7, 7, 20, 13), (30, 7, 9, 0),
              (57, 7, 40, 17), (0, 64, 64, 0), (0, 64, 200, 77)]


def _batch_controls(score_fn, take, full, picked, seed):
    """score_fn(t, r, ids, mask) -> (lt, lr, d); take(sl) -> (rows_t, rows_r, ids)
    of the picked rows sl; full: (lt, lr, d) of the whole batch."""
    ref = [x[picked] for x in full]
    for j0, k, total, off in PLACEMENTS:
        rt, rr, ids = take(slice(j0, j0 + k))
        got = score_fn(*_embed(rt, rr, ids, total, off, seed + 7 * j0 + k))
        for a, b in zip(got, ref):
            assert torch.equal(a[off:off + k], b[j0:j0 + k]), (j0, k, total, off)


def _score(t, r, i, m):
    res = B.score(t, r, i, m)
    torch.cuda.synchronize()
    return res.logp_train, res.logp_rollout, res.dlogp


@pytest.mark.parametrize("name", ["qwen", "llama"])
def test_full_size_every_active_row(name):
    w = (W.qwen if name == "qwen" else W.llama)(device=DEV)
    res = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
    torch.cuda.synchronize()
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    assert res.metrics["n_active"] == act.size and res.metrics["status"] == 0
    t0 = time.perf_counter()
    ref = stream.score_rows_device(w.train, w.rollout, w.token_ids, act)
    print(f"\n{name}: oracle over {act.size} active rows on {stream.host_threads()} threads: "
          f"{time.perf_counter() - t0:.1f} s")
    assert ref.status == 0
    got = (res.logp_train, res.logp_rollout, res.dlogp)
    d_full, ref_m, errs = _per_token_and_metrics(got, mask, ref, w.clip)
    print(f"{name}: max |err| logp_t {errs[0]:.2e} logp_r {errs[1]:.2e} dlogp {errs[2]:.2e}; "
          f"approx_kl0 rel {abs(res.metrics['approx_kl0'] - ref_m['approx_kl0']) / ref_m['approx_kl0']:.2e}, "
          f"mean_abs rel {abs(res.metrics['mean_abs_dlogp'] - ref_m['mean_abs_dlogp']) / ref_m['mean_abs_dlogp']:.2e}")
    assert_metrics_match(res.metrics, ref_m, d_full, mask, w.clip, dlogp_err=errs[2])
    # batch-composition control at this shape and these dtypes
    rng = np.random.default_rng(17)
    picked = torch.as_tensor(np.sort(rng.choice(act, size=64, replace=False)), device=DEV)
    _batch_controls(_score, lambda sl: (w.train[picked[sl]], w.rollout[picked[sl]], w.token_ids[picked[sl]]),
                    got, picked, seed=101)
    del w, res
    torch.cuda.empty_cache()


def _sharded(w, perm=None, t=None, r=None, ids=None, mask=None):
    t = w.train if t is None else t
    r = w.rollout if r is None else r
    ids = w.token_ids if ids is None else ids
    mask = w.action_mask if mask is None else mask
    n = ids.shape[0]
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(5)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SHARDED, n, w.vocab, len(w.v_ranges)), dtype=torch.uint8,
                     device=DEV)
    B.lpd_score_sharded(t, r, w.v_ranges, ids, mask, *w.clip, perm, *outs, met, ws)
    torch.cuda.synchronize()
    return outs, B.read_metrics(met)


def test_full_size_sharded_every_row():
    w = W.sharded(device=DEV)
    perm = [2, 0, 3, 1]
    (lt, lr, d, plt, plr), met = _sharded(w, perm)
    mask = w.action_mask.cpu().numpy()
    act = np.flatnonzero(mask)
    assert met["n_active"] == act.size and met["status"] == 0
    t0 = time.perf_counter()
    ref = stream.score_sharded_rows_device(w.train, w.rollout, w.v_ranges, w.token_ids, act)
    print(f"\nsharded: oracle over {act.size} rows on {stream.host_threads()} threads: "
          f"{time.perf_counter() - t0:.1f} s")
    assert ref.status == 0
    d_full, ref_m, errs = _per_token_and_metrics((lt, lr, d), mask, ref, w.clip)
    assert_metrics_match(met, ref_m, d_full, mask, w.clip, dlogp_err=errs[2])
    # the permuted-order merge is a diagnostic: still within the logp bar, and
    # its GPU summary equals the oracle's summary of the same per-token values
    for g, want in ((plt, ref.logp_train), (plr, ref.logp_rollout)):
        assert np.max(np.abs(g.cpu().numpy().astype(np.float64)[act] - want)) <= LOGP_ATOL
    summ = B.logp_drift_summary(lt, lr, plt, plr, w.action_mask)
    want = oracle.logp_drift(lt.cpu().numpy(), lr.cpu().numpy(), plt.cpu().numpy(), plr.cpu().numpy(), mask)
    assert summ == want, (summ, want)
    print(f"sharded merge order {perm}: max |dlogp| train {summ['max_abs_dlogp_train']:.2e} rollout "
          f"{summ['max_abs_dlogp_rollout']:.2e}, rows differing {summ['frac_differ']:.4f}")
    # batch-composition control on the sharded layout: picked rows of every
    # shard embedded in small batches, both the fixed and the permuted results
    rng = np.random.default_rng(18)
    picked = torch.as_tensor(np.sort(rng.choice(act, size=64, replace=False)), device=DEV)
    full = (lt, lr, d, plt, plr)
    ref_rows = [x[picked] for x in full]
    for j0, k, total, off in PLACEMENTS:
        sl = picked[j0:j0 + k]
        ts, rs = [], []
        for s, (x, y) in enumerate(zip(w.train, w.rollout)):
            t_e, r_e, ids, m = _embed(x[sl], y[sl], w.token_ids[sl], total, off, 300 + 7 * j0 + k + s)
            ts.append(t_e)
            rs.append(r_e)
        (a_lt, a_lr, a_d, a_plt, a_plr), _ = _sharded(w, perm, ts, rs, ids, m)
        for a, b in zip((a_lt, a_lr, a_d, a_plt, a_plr), ref_rows):
            assert torch.equal(a[off:off + k], b[j0:j0 + k]), (j0, k, total, off)
    del w
    torch.cuda.empty_cache()
