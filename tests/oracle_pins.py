"""Pins for the float64 oracle: checks against facts that the pages and the
mathematics fix, independent of the oracle's own code.

Each pin is a function ``pin_*(lib)`` that raises ``AssertionError`` when the
oracle library ``lib`` disagrees with the fact.  ``test_oracle_pins.py`` runs
them against the real oracle; ``test_oracle_mutants.py`` runs them against
deliberately broken copies of the oracle and requires each copy to fail at
least one pin.

Facts used (no pin re-types the oracle's formula):
  * closed forms: uniform logits give logp = -ln V; V = 1 gives 0; V = 2 gives
    -log1p(exp(x_other - x_id));
  * brute force in 50-digit decimal arithmetic on rows of V <= 16;
  * invariants: probabilities sum to one; shifting every logit by a constant
    changes nothing; a -inf logit is the same as a missing column;
  * a library routine: scipy's log_softmax in float64;
  * the metric definitions of the Diagnostics table ("WS2 Cross-Config
    Logprob Drift Contract", section "Diagnostics") evaluated on hand-built
    dlogp vectors in decimal arithmetic, percentiles by their counting
    definition and by numpy's inverted-CDF percentile;
  * the zero-update expectation (same page, section "Primary Failure Signal"):
    identical train and rollout inputs give dlogp = 0, ratio0 = 1,
    approx_kl0 = 0 exactly;
  * the masking rule (section "Measurement Contract"): inactive rows never
    influence any aggregate;
  * item B1 of the roadmap: zero active tokens and worst-token metadata;
  * the shard rules of the LogProb knobs table ("[WS2] Framework for ablation
    experiment", rows 3-5 and 8): exact tiling, single-owner gather, merge
    result independent of the shard split up to rounding.
"""
from __future__ import annotations

import json
import math
from decimal import Decimal, getcontext
from pathlib import Path

import numpy as np

import oracle

getcontext().prec = 50


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even) and return the raw bits."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def dec_logp(row_vals, idx) -> Decimal:
    """log softmax of one row in 50-digit decimal arithmetic."""
    vals = [Decimal(float(v)) for v in row_vals]
    total = sum((v.exp() for v in vals), Decimal(0))
    return vals[idx] - total.ln()


def _close(a, b, tol, what=""):
    assert abs(a - b) <= tol, f"{what}: {a!r} vs {b!r} (|diff| {abs(a - b):.3e} > {tol:.1e})"


# --------------------------------------------------------------- logp pins

def pin_uniform_minus_log_v(lib):
    for vocab in (1, 2, 3, 7, 1000, 151936):
        for c in (0.0, -3.5, 80.0):
            row = np.full(vocab, c, dtype=np.float32)
            lp, st = oracle.row_logp(row, vocab // 2, lib=lib)
            assert st == 0
            _close(lp, -math.log(vocab), 1e-13 * max(1.0, abs(c)) + 1e-15, f"uniform V={vocab} c={c}")
            lpb, _ = oracle.row_logp(bf16_bits(row), vocab - 1, lib=lib)
            _close(lpb, -math.log(vocab), 1e-13 * max(1.0, abs(c)) + 1e-15, f"uniform bf16 V={vocab}")


def pin_single_token_vocab(lib):
    for c in (0.0, 5.25, -1e30):
        lp, st = oracle.row_logp(np.array([c], dtype=np.float32), 0, lib=lib)
        assert st == 0 and lp == 0.0, (c, lp)


def pin_two_token_closed_form(lib):
    rng = np.random.default_rng(11)
    for _ in range(50):
        x = rng.normal(0, 4, size=2).astype(np.float32)
        for i in (0, 1):
            lp, _ = oracle.row_logp(x, i, lib=lib)
            other = float(x[1 - i]) - float(x[i])
            want = -math.log1p(math.exp(other)) if other < 30 else -other - math.log1p(math.exp(-other))
            _close(lp, want, 1e-14, "V=2")


def pin_brute_force_decimal(lib):
    rng = np.random.default_rng(12)
    for vocab in (3, 5, 8, 16):
        for _ in range(6):
            raw = rng.normal(0, 3, size=vocab).astype(np.float32)
            for arr in (raw, bf16_bits(raw)):
                vals = arr if arr.dtype == np.float32 else bf16_to_f32(arr)
                idx = int(rng.integers(0, vocab))
                lp, _ = oracle.row_logp(arr, idx, lib=lib)
                _close(lp, float(dec_logp(vals, idx)), 1e-13, f"decimal V={vocab}")


def pin_probabilities_sum_to_one(lib):
    rng = np.random.default_rng(13)
    for vocab in (10, 257):
        x = bf16_bits(rng.normal(0, 3, size=vocab).astype(np.float32))
        total = math.fsum(math.exp(oracle.row_logp(x, j, lib=lib)[0]) for j in range(vocab))
        _close(total, 1.0, 1e-12, "sum of probabilities")


def pin_shift_invariance(lib):
    rng = np.random.default_rng(14)
    x = (rng.integers(-8192, 8192, size=300) / 1024.0).astype(np.float32)  # exact in fp32
    for c in (64.0, -256.0):
        xs = (x + np.float32(c)).astype(np.float32)
        assert np.all(xs.astype(np.float64) == x.astype(np.float64) + c)
        for idx in (0, 17, 299):
            a, _ = oracle.row_logp(x, idx, lib=lib)
            b, _ = oracle.row_logp(xs, idx, lib=lib)
            _close(a, b, 1e-12, "shift")


def pin_library_log_softmax(lib):
    from scipy.special import log_softmax

    rng = np.random.default_rng(15)
    x = rng.normal(0, 3, size=(4, 5000)).astype(np.float32)
    x[1, 123] += 15.0
    ref = log_softmax(x.astype(np.float64), axis=1)
    for r in range(4):
        for idx in (0, 123, 4999):
            lp, _ = oracle.row_logp(x[r], idx, lib=lib)
            _close(lp, ref[r, idx], 1e-11, "scipy log_softmax")


def pin_neg_inf_is_missing_column(lib):
    rng = np.random.default_rng(16)
    x = rng.normal(0, 2, size=40).astype(np.float32)
    y = x.copy()
    y[[3, 30]] = -np.inf
    keep = np.array([j for j in range(40) if j not in (3, 30)])
    for idx in (0, 20, 39):
        a, st = oracle.row_logp(y, idx, lib=lib)
        assert st == 0
        b, _ = oracle.row_logp(np.ascontiguousarray(x[keep]), int(np.searchsorted(keep, idx)), lib=lib)
        _close(a, b, 1e-14, "-inf column")


def pin_selected_index_and_bf16_widening(lib):
    # logits 0, 1, 2, ... (exact in bf16): logp(j) differs from logp(0) by exactly j
    x = np.arange(12, dtype=np.float32)
    for arr in (x, bf16_bits(x)):
        base, _ = oracle.row_logp(arr, 0, lib=lib)
        for j in (1, 5, 11):
            lp, _ = oracle.row_logp(arr, j, lib=lib)
            _close(lp - base, float(j), 1e-12, "selected index")
        _close(base, float(dec_logp(x, 0)), 1e-13, "bf16 widening")


# --------------------------------------------------------------- metric pins

def _dec_metrics(d, lo, hi):
    """The Diagnostics table, evaluated in decimal on the active values."""
    n = len(d)
    ds = [Decimal(float(v)) for v in d]
    ratio = [v.exp() for v in ds]
    return {
        "ratio0_mean": float(sum(ratio) / n),
        "approx_kl0": float(sum(r - 1 - v for r, v in zip(ratio, ds)) / n),
        "mean_abs_dlogp": float(sum(abs(v) for v in ds) / n),
        "clipfrac0": sum(1 for r in ratio if r < Decimal(lo) or r > Decimal(hi)) / n,
    }


def _nearest_rank_by_counting(values, p):
    """Smallest v among the values with #{x <= v} >= p*A/100."""
    a = len(values)
    best = None
    for v in values:
        if sum(1 for x in values if x <= v) * 100 >= p * a:
            if best is None or v < best:
                best = v
    return best


def pin_metrics_decimal(lib):
    rng = np.random.default_rng(21)
    for n in (1, 2, 5, 37, 200):
        d = rng.normal(0, 0.3, size=n) * rng.choice([1e-6, 1e-2, 1.0], size=n)
        d[0] = 0.9  # ratio above 1.2 -> clipped
        mask = np.ones(n, dtype=np.uint8)
        got = oracle.metrics(d, mask, 0.8, 1.2, lib=lib)
        want = _dec_metrics(d, 0.8, 1.2)
        for k in ("ratio0_mean", "mean_abs_dlogp"):
            _close(got[k], want[k], 1e-14, k)
        _close(got["approx_kl0"], want["approx_kl0"], 1e-13 * max(want["approx_kl0"], 1e-300), "approx_kl0")
        assert got["clipfrac0"] == want["clipfrac0"], (got["clipfrac0"], want["clipfrac0"])
        assert got["n_active"] == n
        # the same values with inactive rows interleaved: only active rows count
        full = np.concatenate([d, rng.normal(0, 5, size=n)])
        fmask = np.concatenate([mask, np.zeros(n, np.uint8)])
        order = rng.permutation(2 * n)
        got2 = oracle.metrics(full[order], fmask[order], 0.8, 1.2, lib=lib)
        for k in ("ratio0_mean", "mean_abs_dlogp", "clipfrac0"):
            _close(got2[k], want[k], 1e-14, "masked " + k)
        assert got2["n_active"] == n


def pin_constant_dlogp(lib):
    for c in (-0.25, 1e-3, 3e-8, 0.5):
        d = np.full(9, c)
        got = oracle.metrics(d, np.ones(9, np.uint8), 0.8, 1.2, lib=lib)
        dc = Decimal(c)
        k3 = float(dc.exp() - 1 - dc)
        # expm1(c) - c in double cancels: the error is a few ulps of c, not of the result
        _close(got["approx_kl0"], k3, 4 * abs(c) * 2.0**-52 + 1e-15 * k3, "k3(c)")
        _close(got["ratio0_mean"], float(dc.exp()), 1e-15, "ratio0")
        assert got["mean_abs_dlogp"] == abs(c)
        assert got["p95_abs_dlogp"] == got["p99_abs_dlogp"] == got["max_abs_dlogp"] == abs(c)


def pin_percentiles_definition(lib):
    rng = np.random.default_rng(22)
    for n in list(range(1, 41)) + [97, 100, 101, 199, 200]:
        d = rng.normal(0, 1, size=n)
        if n > 4:
            d[:3] = d[3]  # ties
        absd = np.abs(d)
        got = oracle.metrics(d, np.ones(n, np.uint8), 0.8, 1.2, lib=lib)
        for p, key in ((95, "p95_abs_dlogp"), (99, "p99_abs_dlogp"), (100, "max_abs_dlogp")):
            want = _nearest_rank_by_counting(list(absd), p)
            assert got[key] == want, (n, key, got[key], want)
            assert got[key] == np.percentile(absd, p, method="inverted_cdf")


def pin_clipfrac_constructed(lib):
    # ratios 0.5, 1, 2, 0.9, 1.1, 0.79, 1.21: four are outside [0.8, 1.2]
    d = np.log(np.array([0.5, 1.0, 2.0, 0.9, 1.1, 0.79, 1.21]))
    got = oracle.metrics(d, np.ones(7, np.uint8), 0.8, 1.2, lib=lib)
    assert got["clipfrac0"] == 4 / 7, got["clipfrac0"]
    # a ratio equal to a bound counts as inside: choose bounds that are exp of the data
    d2 = np.array([-0.5, 0.0, 0.25])
    got2 = oracle.metrics(d2, np.ones(3, np.uint8), math.exp(-0.5), math.exp(0.25), lib=lib)
    assert got2["clipfrac0"] == 0.0, got2["clipfrac0"]
    got3 = oracle.metrics(d2, np.ones(3, np.uint8), math.exp(-0.5) * (1 + 1e-12), 2.0, lib=lib)
    assert got3["clipfrac0"] == 1 / 3


def pin_argmax_lowest_row(lib):
    d = np.array([0.1, -0.7, 0.3, 0.7, -0.7, 0.2])
    mask = np.array([1, 0, 1, 1, 1, 1], np.uint8)
    got = oracle.metrics(d, mask, 0.8, 1.2, lib=lib)
    assert got["argmax_row"] == 3 and got["max_abs_dlogp"] == 0.7, got
    mask[1] = 1
    assert oracle.metrics(d, mask, 0.8, 1.2, lib=lib)["argmax_row"] == 1


def pin_zero_active(lib):
    got = oracle.metrics(np.array([1.0, -2.0]), np.zeros(2, np.uint8), 0.8, 1.2, lib=lib)
    assert got["n_active"] == 0 and got["flags"] & oracle.FLAG_NO_ACTIVE and got["argmax_row"] == -1
    for k in ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp", "p95_abs_dlogp",
              "p99_abs_dlogp", "max_abs_dlogp"):
        assert got[k] == 0.0


# ------------------------------------------------------- whole-scoring pins

def _case(n_rows, vocab, seed, dtype="bf16"):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2, size=(n_rows, vocab)).astype(np.float32)
    r = t + rng.normal(0, 0.05, size=t.shape).astype(np.float32)
    if dtype == "bf16":
        t, r = bf16_bits(t), bf16_bits(r)
    ids = rng.integers(0, vocab, size=n_rows).astype(np.int32)
    mask = (rng.random(n_rows) < 0.7).astype(np.uint8)
    mask[0] = 1
    return t, r, ids, mask


GOLDEN = Path(__file__).resolve().parent / "golden"


def pin_zero_update_expectation(lib):
    expect = json.loads((GOLDEN / "zero_update_expectation.json").read_text())["expect_when_inputs_identical"]
    t, _, ids, mask = _case(30, 50, 31)
    res = oracle.score(t, t, ids, mask, lib=lib)
    assert res.status == 0
    assert np.all(res.dlogp == expect["dlogp"])
    for k, v in expect.items():
        if k != "dlogp":
            assert res.metrics[k] == v, (k, res.metrics[k], v)
    # bf16 against its exact fp32 upcast is the same input
    up = np.ascontiguousarray(bf16_to_f32(t))
    res2 = oracle.score(t, up, ids, mask, lib=lib)
    assert np.all(res2.dlogp == 0.0)


def pin_dlogp_sign_and_values(lib):
    t, r, ids, mask = _case(12, 9, 32, dtype="f32")
    res = oracle.score(t, r, ids, mask, lib=lib)
    for i in np.flatnonzero(mask):
        lt = float(dec_logp(t[i], ids[i]))
        lr = float(dec_logp(r[i], ids[i]))
        _close(res.logp_train[i], lt, 1e-13, "logp_train")
        _close(res.logp_rollout[i], lr, 1e-13, "logp_rollout")
        _close(res.dlogp[i], lt - lr, 1e-13, "dlogp = train - rollout")
    assert np.all(res.dlogp[mask == 0] == 0.0)


def pin_masked_rows_never_read(lib):
    t, r, ids, mask = _case(40, 33, 33, dtype="f32")
    base = oracle.score(t, r, ids, mask, lib=lib)
    t2, r2, ids2 = t.copy(), r.copy(), ids.copy()
    off = mask == 0
    t2[off] = np.nan
    r2[off, 0] = np.inf
    ids2[off] = -5
    res = oracle.score(t2, r2, ids2, mask, lib=lib)
    assert res.status == 0
    assert res.metrics == base.metrics
    active = mask == 1
    assert np.array_equal(res.dlogp[active], base.dlogp[active])


def pin_active_token_count(lib):
    t, r, ids, mask = _case(50, 7, 34)
    res = oracle.score(t, r, ids, mask, lib=lib)
    assert res.metrics["n_active"] == int(mask.sum())


def pin_bad_rows_flagged(lib):
    t, r, ids, mask = _case(6, 10, 35, dtype="f32")
    mask[:] = 1
    ids2 = ids.copy()
    ids2[2] = 10
    assert oracle.score(t, r, ids2, mask, lib=lib).status == oracle.STATUS_TOKEN_OOB
    ids2[2] = -1
    assert oracle.score(t, r, ids2, mask, lib=lib).status == oracle.STATUS_TOKEN_OOB
    t2 = t.copy()
    t2[4, 3] = np.nan
    assert oracle.score(t2, r, ids, mask, lib=lib).status == oracle.STATUS_NONFINITE
    t3 = t.copy()
    t3[1, :] = -np.inf
    assert oracle.score(t3, r, ids, mask, lib=lib).status == oracle.STATUS_NONFINITE


def pin_padded_row_stride(lib):
    t, r, ids, mask = _case(8, 20, 36, dtype="f32")
    base = oracle.score(t, r, ids, mask, lib=lib)
    wide = np.full((8, 27), 99.0, dtype=np.float32)
    wide[:, :20] = t
    res = oracle.score(wide[:, :20], r, ids, mask, lib=lib)
    assert np.array_equal(res.dlogp, base.dlogp)


# -------------------------------------------------------------- shard pins

def _split(x, bounds):
    return [np.ascontiguousarray(x[:, a:b]) for a, b in bounds]


def pin_sharded_equals_unsharded(lib):
    t, r, ids, mask = _case(20, 64, 41)
    base = oracle.score(t, r, ids, mask, lib=lib)
    for bounds in ([(0, 64)], [(0, 16), (16, 32), (32, 48), (48, 64)], [(0, 5), (5, 63), (63, 64)]):
        res = oracle.score_sharded(_split(t, bounds), _split(r, bounds), bounds, ids, mask, lib=lib)
        assert res.status == 0
        np.testing.assert_allclose(res.logp_train, base.logp_train, rtol=0, atol=1e-12)
        np.testing.assert_allclose(res.dlogp, base.dlogp, rtol=0, atol=1e-12)
        perm = list(range(len(bounds)))[::-1]
        res2 = oracle.score_sharded(_split(t, bounds), _split(r, bounds), bounds, ids, mask, order=perm, lib=lib)
        np.testing.assert_allclose(res2.logp_rollout, base.logp_rollout, rtol=0, atol=1e-12)


def pin_shard_tiling_rules(lib):
    assert oracle.check_tiling([(0, 10), (10, 20)], 20, lib=lib)
    assert oracle.check_tiling([(10, 20), (0, 10)], 20, lib=lib)
    assert not oracle.check_tiling([(0, 10), (11, 20)], 20, lib=lib)   # gap
    assert not oracle.check_tiling([(0, 11), (10, 20)], 20, lib=lib)   # overlap
    assert not oracle.check_tiling([(0, 10), (10, 21)], 20, lib=lib)   # past the vocab
    assert not oracle.check_tiling([(0, 10)], 20, lib=lib)             # short
    assert not oracle.check_tiling([(0, 10), (5, 15)], 20, lib=lib)    # overlap hides a gap
    assert not oracle.check_tiling([], 20, lib=lib)


# --------------------------------------------------------------- head pins

def pin_head_logits_matmul(lib):
    from scipy.special import log_softmax

    rng = np.random.default_rng(51)
    hidden, vocab = 24, 40
    h = bf16_bits(rng.normal(0, 1, size=(3, hidden)).astype(np.float32))
    W = bf16_bits(rng.normal(0, 0.5, size=(vocab, hidden)).astype(np.float32))
    ref = bf16_to_f32(h).astype(np.float64) @ bf16_to_f32(W).astype(np.float64).T
    for i in range(3):
        x = oracle.head_logits(h[i], W, lib=lib)
        np.testing.assert_allclose(x, ref[i], rtol=1e-13, atol=1e-13)
    h2 = bf16_bits(bf16_to_f32(h) + rng.normal(0, 0.1, size=h.shape).astype(np.float32))
    ids = rng.integers(0, vocab, size=3).astype(np.int32)
    res = oracle.score_head_rows(h, h2, W, ids, [0, 2], lib=lib)
    ref2 = bf16_to_f32(h2).astype(np.float64) @ bf16_to_f32(W).astype(np.float64).T
    for k, i in enumerate((0, 2)):
        _close(res.logp_train[k], log_softmax(ref[i])[ids[i]], 1e-12, "head logp train")
        _close(res.logp_rollout[k], log_softmax(ref2[i])[ids[i]], 1e-12, "head logp rollout")


# ----------------------------------------------------- transform-chain pins

def _dec_tanh(y: Decimal) -> Decimal:
    e = (2 * y).exp()
    return (e - 1) / (e + 1)


def _dec_chain(x, ops):
    v = Decimal(float(x))
    for kind, p in ops:
        p = Decimal(float(np.float32(p)))
        v = v * p if kind == oracle.OP_SCALE else p * _dec_tanh(v / p)
    return v


def _dec_logp_chain(row, idx, ops):
    vals = [_dec_chain(x, ops) for x in row]
    total = sum((v.exp() for v in vals), Decimal(0))
    return vals[idx] - total.ln()


def pin_transform_identity_is_plain(lib):
    t, r, ids, mask = _case(25, 40, 61, dtype="f32")
    a = oracle.score(t, r, ids, mask, lib=lib)
    b = oracle.score_transformed(t, r, ids, mask, [], None, lib=lib)
    assert np.array_equal(a.dlogp, b.dlogp) and a.metrics == b.metrics


def pin_transform_scale_closed_form(lib):
    rng = np.random.default_rng(62)
    for s in (0.5, 1.25, 2.0):
        x = rng.normal(0, 3, size=(6, 2)).astype(np.float32)
        ids = np.zeros(6, np.int32)
        res = oracle.score_transformed(x, x, ids, np.ones(6, np.uint8), [(oracle.OP_SCALE, s)], None, lib=lib)
        for i in range(6):
            want = -math.log1p(math.exp(s * (float(x[i, 1]) - float(x[i, 0]))))
            _close(res.logp_train[i], want, 1e-13, "scaled V=2")
            _close(res.logp_rollout[i], float(dec_logp(x[i], 0)), 1e-13, "unscaled side")
    u = np.full((2, 500), 1.75, np.float32)
    res = oracle.score_transformed(u, u, np.array([3, 7], np.int32), np.ones(2, np.uint8),
                                   [(oracle.OP_SCALE, 1 / 0.7)], None, lib=lib)
    _close(res.logp_train[0], -math.log(500), 1e-13, "temperature on uniform")


def pin_transform_softcap_and_order_decimal(lib):
    rng = np.random.default_rng(63)
    x = (rng.normal(0, 20, size=(4, 12))).astype(np.float32)
    x[0, 3] = 1e4
    x[1, 5] = -1e4
    ids = rng.integers(0, 12, size=4).astype(np.int32)
    chains = ([(oracle.OP_SOFTCAP, 30.0)], [(oracle.OP_SCALE, 2.0), (oracle.OP_SOFTCAP, 15.0)],
              [(oracle.OP_SOFTCAP, 15.0), (oracle.OP_SCALE, 2.0)])
    got = []
    for ops in chains:
        res = oracle.score_transformed(x, x, ids, np.ones(4, np.uint8), ops, None, lib=lib)
        for i in range(4):
            _close(res.logp_train[i], float(_dec_logp_chain(x[i], int(ids[i]), ops)), 1e-12, f"chain {ops}")
        got.append(res.logp_train.copy())
    assert not np.allclose(got[1], got[2]), "chain order must matter"


def pin_transform_per_side(lib):
    rng = np.random.default_rng(64)
    x = rng.normal(0, 3, size=(5, 9)).astype(np.float32)
    ids = rng.integers(0, 9, size=5).astype(np.int32)
    ops = [(oracle.OP_SCALE, 1 / 0.7)]
    res = oracle.score_transformed(x, x, ids, np.ones(5, np.uint8), None, ops, lib=lib)
    for i in range(5):
        want = dec_logp(x[i], int(ids[i])) - _dec_logp_chain(x[i], int(ids[i]), ops)
        _close(res.dlogp[i], float(want), 1e-12, "train plain, rollout tempered")


# ------------------------------------------------- entropy and backward pins

def pin_entropy_closed_forms(lib):
    for vocab in (1, 2, 7, 1000):
        _close(oracle.row_entropy(np.full(vocab, 2.5, np.float32), lib=lib), math.log(vocab), 1e-12, "uniform H")
    rng = np.random.default_rng(71)
    for _ in range(10):
        x = rng.normal(0, 3, size=2).astype(np.float32)
        p = 1.0 / (1.0 + math.exp(float(x[1]) - float(x[0])))
        want = -(p * math.log(p) + (1 - p) * math.log(1 - p)) if 0 < p < 1 else 0.0
        _close(oracle.row_entropy(x, lib=lib), want, 1e-12, "two-token H")
    peaked = np.zeros(50, np.float32)
    peaked[7] = 80.0
    assert 0.0 <= oracle.row_entropy(peaked, lib=lib) < 1e-30


def pin_entropy_decimal(lib):
    rng = np.random.default_rng(72)
    for vocab in (3, 9, 16):
        x = rng.normal(0, 3, size=vocab).astype(np.float32)
        vals = [Decimal(float(v)) for v in x]
        z = sum((v.exp() for v in vals), Decimal(0))
        h = -sum(((v.exp() / z) * (v - z.ln()) for v in vals), Decimal(0))
        _close(oracle.row_entropy(x, lib=lib), float(h), 1e-12, "decimal H")


def pin_backward_finite_differences(lib):
    rng = np.random.default_rng(73)
    x = rng.normal(0, 2, size=12)
    idx, grad, eps = 5, -0.75, 1e-6

    def logp(v):
        return float(dec_logp(v, idx))

    g = oracle.logprob_backward_row(x.astype(np.float32), idx, grad, lib=lib)
    xf = x.astype(np.float32).astype(np.float64)
    for j in range(12):
        hi, lo = xf.copy(), xf.copy()
        hi[j] += eps
        lo[j] -= eps
        fd = grad * (logp(hi) - logp(lo)) / (2 * eps)
        _close(g[j], fd, 1e-8, f"d logp / d x_{j}")
    _close(float(np.sum(g)), 0.0, 1e-14, "gradient sums to zero")


def pin_backward_uniform(lib):
    vocab, idx, grad = 40, 3, 2.0
    g = oracle.logprob_backward_row(np.zeros(vocab, np.float32), idx, grad, lib=lib)
    for j in range(vocab):
        want = grad * ((1.0 if j == idx else 0.0) - 1.0 / vocab)
        _close(g[j], want, 1e-15, "uniform gradient")


# ------------------------------------------------------ attention merge pins

def _attention_split(rng, n, d, n_keys, bounds):
    """Softmax attention of n queries over n_keys keys, computed whole and per
    key block (each block's own normalised output and natural-log lse)."""
    q = rng.normal(0, 1, size=(n, d))
    k = rng.normal(0, 1, size=(n_keys, d))
    v = rng.normal(0, 1, size=(n_keys, d))
    s = q @ k.T / math.sqrt(d)
    full_lse = np.log(np.sum(np.exp(s), axis=1))
    full_out = np.exp(s - full_lse[:, None]) @ v
    outs, lses = [], []
    for a, b in bounds:
        sb = s[:, a:b]
        lb = np.log(np.sum(np.exp(sb), axis=1))
        outs.append(np.exp(sb - lb[:, None]) @ v[a:b])
        lses.append(lb)
    return full_out, full_lse, np.array(outs, np.float32), np.array(lses, np.float32)


def pin_attn_merge_equals_unsplit_attention(lib):
    rng = np.random.default_rng(81)
    full_out, full_lse, outs, lses = _attention_split(rng, 6, 8, 40, [(0, 9), (9, 25), (25, 40)])
    for order in ([0, 1, 2], [2, 0, 1]):
        out, lse = oracle.attn_merge(outs, lses, order, lib=lib)
        np.testing.assert_allclose(out, full_out, rtol=0, atol=2e-6)     # parts are stored in fp32
        np.testing.assert_allclose(lse, full_lse, rtol=0, atol=2e-6)


def pin_attn_merge_closed_forms(lib):
    rng = np.random.default_rng(82)
    outs = rng.normal(0, 1, size=(1, 5, 4)).astype(np.float32)
    lses = rng.normal(0, 1, size=(1, 5)).astype(np.float32)
    out, lse = oracle.attn_merge(outs, lses, lib=lib)                        # one part: identity
    assert np.array_equal(out, outs[0].astype(np.float64)) and np.array_equal(lse, lses[0].astype(np.float64))
    outs = rng.normal(0, 1, size=(4, 3, 2)).astype(np.float32)
    lses = np.full((4, 3), 1.5, np.float32)
    out, lse = oracle.attn_merge(outs, lses, lib=lib)                        # equal lse: plain mean
    np.testing.assert_allclose(out, outs.astype(np.float64).mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, 1.5 + math.log(4), rtol=0, atol=1e-14)
    out2, lse2 = oracle.attn_merge(outs, lses / np.float32(math.log(2)), lse_base2=True, lib=lib)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-6)
    np.testing.assert_allclose(lse2 * math.log(2), lse, rtol=0, atol=1e-6)


def pin_attn_merge_masked_parts(lib):
    # causal split: the last key block lies after every query, so its part saw
    # no keys (lse -inf, out left as NaN by the backend); merging the remaining
    # parts must still equal unsplit attention over the keys that exist
    rng = np.random.default_rng(83)
    full_out, full_lse, outs, lses = _attention_split(rng, 4, 8, 30, [(0, 12), (12, 30)])
    outs = np.concatenate([outs, np.full((1, 4, 8), np.nan, np.float32)])
    lses = np.concatenate([lses, np.full((1, 4), -np.inf, np.float32)])
    for order in ([0, 1, 2], [2, 1, 0]):
        out, lse = oracle.attn_merge(outs, lses, order, lib=lib)
        np.testing.assert_allclose(out, full_out, rtol=0, atol=2e-6)
        np.testing.assert_allclose(lse, full_lse, rtol=0, atol=2e-6)
    # a row that no part saw: out 0, lse -inf
    out, lse = oracle.attn_merge(np.full((2, 1, 3), np.nan, np.float32), np.full((2, 1), -np.inf, np.float32), lib=lib)
    assert np.array_equal(out, np.zeros((1, 3))) and lse[0] == -np.inf



# ---- merge-order drift summary ("[WS2] Framework for ablation experiment",
# LogProb knobs table, row 5: the merge order of the shard partials as a drift
# source).  Hand-built result pairs whose summary is known by construction.

def pin_logp_drift_identical_and_empty(lib):
    rng = np.random.default_rng(91)
    a_t = rng.normal(-12, 1, 40).astype(np.float32)
    a_r = rng.normal(-12, 1, 40).astype(np.float32)
    mask = (rng.random(40) < 0.7).astype(np.uint8)
    mask[:3] = 0
    s = oracle.logp_drift(a_t, a_r, a_t.copy(), a_r.copy(), mask, lib=lib)
    first = int(np.flatnonzero(mask)[0])
    assert s["max_abs_dlogp_train"] == 0.0 and s["max_abs_dlogp_rollout"] == 0.0
    assert s["row_train"] == first and s["row_rollout"] == first          # every active row ties at 0
    assert s["n_active"] == int(mask.sum()) and s["n_differ"] == 0 and s["frac_differ"] == 0.0
    s0 = oracle.logp_drift(a_t, a_r, a_t, a_r, np.zeros(40, np.uint8), lib=lib)
    assert s0 == {"max_abs_dlogp_train": 0.0, "max_abs_dlogp_rollout": 0.0, "row_train": -1, "row_rollout": -1,
                  "n_active": 0, "n_differ": 0, "frac_differ": 0.0}


def pin_logp_drift_constructed(lib):
    n = 12
    a_t = np.full(n, -10.0, np.float32)
    a_r = np.full(n, -11.0, np.float32)
    b_t, b_r = a_t.copy(), a_r.copy()
    mask = np.ones(n, np.uint8)
    b_t[2] = -10.25          # |d| 0.25
    b_t[5] = -9.5            # |d| 0.5, first of a tie
    b_t[9] = -10.5           # |d| 0.5, the tie's later row
    b_t[7] = -13.0           # |d| 3, but the row is masked out
    mask[7] = 0
    b_r[4] = -11.0 + 2.0 ** -20   # one float32 step apart: a tiny but real difference
    a_r[6], b_r[6] = 0.0, -0.0    # +0 and -0 are the same number
    s = oracle.logp_drift(a_t, a_r, b_t, b_r, mask, lib=lib)
    assert s["max_abs_dlogp_train"] == 0.5 and s["row_train"] == 5
    assert s["max_abs_dlogp_rollout"] == 2.0 ** -20 and s["row_rollout"] == 4
    assert s["n_active"] == n - 1
    assert s["n_differ"] == 4                               # rows 2, 4, 5, 9
    assert s["frac_differ"] == 4 / (n - 1)
    # differing on the rollout side only still counts the row
    s2 = oracle.logp_drift(a_t, a_r, a_t, b_r, mask, lib=lib)
    assert s2["n_differ"] == 1 and s2["max_abs_dlogp_train"] == 0.0


def pin_logp_drift_nan_ranks_highest(lib):
    a = np.array([-1.0, -2.0, np.nan, -4.0, np.nan], np.float32)
    b = np.array([-1.5, -2.0, np.nan, -9.0, -5.0], np.float32)
    mask = np.ones(5, np.uint8)
    s = oracle.logp_drift(a, a, b, b, mask, lib=lib)
    assert math.isnan(s["max_abs_dlogp_train"]) and s["row_train"] == 2    # lowest NaN row, above |d| = 5
    # two NaNs are the same result; NaN against a number is a difference
    assert s["n_differ"] == 3                                               # rows 0, 3, 4
    mask[2] = 0
    s2 = oracle.logp_drift(a, a, b, b, mask, lib=lib)
    assert math.isnan(s2["max_abs_dlogp_train"]) and s2["row_train"] == 4


def pin_logp_drift_of_shard_merge_orders(lib):
    # the exact logp does not depend on the merge order: in double, the fixed
    # and permuted merges agree to rounding, so their float32 results differ
    # by at most one float32 step
    rng = np.random.default_rng(92)
    V, bounds = 3000, [(0, 700), (700, 701), (701, 2500), (2500, 3000)]
    x = bf16_bits(rng.normal(0, 3, size=(30, V)).astype(np.float32))
    y = bf16_bits(rng.normal(0, 3, size=(30, V)).astype(np.float32))
    ids = rng.integers(0, V, 30).astype(np.int32)
    mask = np.ones(30, np.uint8)
    ts = [np.ascontiguousarray(x[:, a:b]) for a, b in bounds]
    rs = [np.ascontiguousarray(y[:, a:b]) for a, b in bounds]
    fixed = oracle.score_sharded(ts, rs, bounds, ids, mask, lib=lib)
    perm = oracle.score_sharded(ts, rs, bounds, ids, mask, order=[3, 1, 0, 2], lib=lib)
    f = [v.astype(np.float32) for v in (fixed.logp_train, fixed.logp_rollout, perm.logp_train, perm.logp_rollout)]
    s = oracle.logp_drift(*f, mask, lib=lib)
    step = float(np.max(np.spacing(np.abs(f[0]))))
    assert s["n_active"] == 30 and s["max_abs_dlogp_train"] <= step and s["max_abs_dlogp_rollout"] <= step


ALL_PINS = {name: fn for name, fn in sorted(globals().items()) if name.startswith("pin_")}
