"""CUDA path against the float64 oracle, through the C ABI (needs a GPU).

Bars (see tests/helpers.py): per-token logp within 1e-4 absolute, approx_kl0
and mean_abs_dlogp within 1e-4 relative, percentiles within 1e-4 absolute,
counts and selection exact, batch-invariance controls bitwise.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import LOGP_ATOL, assert_metrics_match, to_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda"


def run(train, rollout, ids, mask, clip=(0.8, 1.2)):
    res = B.score(train, rollout, ids, mask, clip)
    torch.cuda.synchronize()
    return res


def oracle_score(train, rollout, ids, mask, clip=(0.8, 1.2)):
    return oracle.score(to_oracle(train), to_oracle(rollout), ids.cpu().numpy(), mask.cpu().numpy(), *clip)


def check_against_oracle(w, clip=(0.8, 1.2)):
    res = run(w.train, w.rollout, w.token_ids, w.action_mask, clip)
    ref = oracle_score(w.train, w.rollout, w.token_ids, w.action_mask, clip)
    mask = w.action_mask.cpu().numpy()
    lt, lr, d = (x.cpu().numpy().astype(np.float64) for x in (res.logp_train, res.logp_rollout, res.dlogp))
    act = mask != 0
    assert np.all(lt[~act] == 0) and np.all(lr[~act] == 0) and np.all(d[~act] == 0)
    if act.any():
        assert np.max(np.abs(lt[act] - ref.logp_train[act])) <= LOGP_ATOL
        assert np.max(np.abs(lr[act] - ref.logp_rollout[act])) <= LOGP_ATOL
        assert np.max(np.abs(d[act] - ref.dlogp[act])) <= LOGP_ATOL
    assert_metrics_match(res.metrics, ref.metrics, ref.dlogp, mask, clip)
    return res, ref


# ------------------------------------------------------------------ parity

def test_tiny_config_vs_oracle():
    w = W.tiny(device=DEV)
    res, ref = check_against_oracle(w)
    assert res.metrics["n_active"] == int(w.action_mask.sum())
    # the tiny drift is ~1e-3: dlogp itself must be far better than the logp bar
    act = w.action_mask.cpu().numpy() != 0
    err = np.abs(res.dlogp.cpu().numpy()[act] - ref.dlogp[act])
    assert err.max() <= 1e-6, err.max()


CASES = {
    # name: (rows, vocab, dtype_t, dtype_r, kwargs)
    "bf16_3tiles_ragged_tma": (300, 3 * 4096 + 520, torch.bfloat16, torch.bfloat16, {}),
    "bf16_unaligned_rows_generic": (257, 3 * 4096 + 517, torch.bfloat16, torch.bfloat16, {}),
    "bf16_padded_rows_tma_subvector_tail": (130, 3 * 4096 + 517, torch.bfloat16, torch.bfloat16, dict(row_pad=3)),
    "mixed_bf16_f32": (200, 9000, torch.bfloat16, torch.float32, {}),
    "mixed_f32_bf16_one_tile": (150, 4096, torch.float32, torch.bfloat16, {}),
    "f32_f32_vocab5": (90, 5, torch.float32, torch.float32, {}),
    "bf16_vocab1": (40, 1, torch.bfloat16, torch.bfloat16, {}),
    "bf16_vocab2": (40, 2, torch.bfloat16, torch.bfloat16, {}),
    "bf16_vocab7_generic": (40, 7, torch.bfloat16, torch.bfloat16, {}),
    "many_rows_small_vocab": (5000, 256, torch.bfloat16, torch.bfloat16, {}),
    "spiky_wide": (64, 151936, torch.bfloat16, torch.bfloat16, dict(spike_frac=0.2)),
    "independent_rollout_clipping": (400, 2000, torch.bfloat16, torch.bfloat16, dict(rollout_noise=0.4)),
    "f32_unaligned_generic": (100, 4097, torch.float32, torch.float32, {}),
    "f32_vocab5_padded_tma_tail": (90, 5, torch.float32, torch.float32, dict(row_pad=3)),
    "bf16_vocab7_padded_tma_tail": (40, 7, torch.bfloat16, torch.bfloat16, dict(row_pad=1)),
    # past 2^22 columns: column indices and byte offsets well beyond 32-bit
    # products of the per-tile arithmetic; ids near both ends come from the
    # uniform draw plus the spikes
    "huge_vocab_mixed": (6, (1 << 22) + 123, torch.bfloat16, torch.float32, dict(spike_frac=0.5)),
    # 300 000 rows: many grid-stride passes per CTA and a percentile select
    # over ~270 000 keys
    "many_rows_vocab16": (300_000, 16, torch.bfloat16, torch.bfloat16, {}),
    # around the plain pass's 11 776-column tile (23 consumer warps x 512):
    # exactly one tile, one column past two tiles, one column short of a tile
    "bf16_one_full_tile": (120, 11776, torch.bfloat16, torch.bfloat16, {}),
    "bf16_two_tiles_plus_one": (120, 2 * 11776 + 1, torch.bfloat16, torch.bfloat16, {}),
    "mixed_one_tile_minus_one": (100, 11775, torch.bfloat16, torch.float32, {}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_parity_synthetic(name):
    rows, vocab, dt, dr, kw = CASES[name]
    w = W.synthetic(rows, vocab, seed=zlib.crc32(name.encode()) % 1000, device=DEV, dtype_train=dt, dtype_rollout=dr, **kw)
    res, ref = check_against_oracle(w)
    if name == "independent_rollout_clipping":
        assert ref.metrics["clipfrac0"] > 0.05


# --------------------------------------------------------- bitwise controls

def test_identical_inputs_give_exact_zeros():
    w = W.synthetic(300, 5000, seed=5, device=DEV)
    res = run(w.train, w.train, w.token_ids, w.action_mask)
    assert torch.all(res.dlogp == 0)
    assert torch.equal(res.logp_train, res.logp_rollout)
    m = res.metrics
    assert m["ratio0_mean"] == 1.0 and m["approx_kl0"] == 0.0 and m["clipfrac0"] == 0.0
    assert m["mean_abs_dlogp"] == m["p95_abs_dlogp"] == m["p99_abs_dlogp"] == m["max_abs_dlogp"] == 0.0


def test_bf16_against_its_fp32_upcast_is_bitwise_zero():
    w = W.synthetic(200, 12808, seed=6, device=DEV)
    up = w.train.float().contiguous()
    res = run(w.train, up, w.token_ids, w.action_mask)
    assert torch.all(res.dlogp == 0)
    assert torch.equal(res.logp_train, res.logp_rollout)


def test_constant_shift_gives_exact_zero():
    # a rollout that is the train logits plus a constant has the same
    # distribution: logp is identical and dlogp must be exactly zero
    # (values on a 1/16 grid in [-8, 8): exact in bf16, and exact after the shift)
    w = W.synthetic(120, 3 * 4096 + 520, seed=14, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(14)
    grid = torch.randint(-127, 128, (w.n_rows, w.vocab), generator=g, device=DEV).float() / 16
    train = grid.to(torch.bfloat16)
    assert torch.equal(train.float(), grid)
    shifted = (grid + 0.75).contiguous()
    assert torch.equal(shifted - 0.75, grid)
    res = run(train, shifted, w.token_ids, w.action_mask)
    assert torch.all(res.dlogp == 0)
    m = res.metrics
    assert m["approx_kl0"] == 0.0 and m["mean_abs_dlogp"] == 0.0 and m["ratio0_mean"] == 1.0
    ref = oracle_score(train, shifted, w.token_ids, w.action_mask)
    assert np.max(np.abs(ref.dlogp)) < 1e-12


def _embed(rows_t, rows_r, ids, n_total, offset, seed):
    """Place the given rows at [offset, offset+k) of a bigger batch whose other
    rows are inactive garbage (padding on either side)."""
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


def test_batch_composition_control_bitwise():
    base = W.synthetic(64, 3 * 4096 + 520, seed=7, device=DEV, active_prob=1.0)
    full = run(base.train, base.rollout, base.token_ids, base.action_mask)
    outs = (full.logp_train, full.logp_rollout, full.dlogp)
    # batch of 1, each row alone at a different offset
    for j in (0, 5, 63):
        t, r, i, m = _embed(base.train[j:j + 1], base.rollout[j:j + 1], base.token_ids[j:j + 1], 3, j % 3, j)
        res = run(t, r, i, m)
        off = j % 3
        for a, b in zip((res.logp_train, res.logp_rollout, res.dlogp), outs):
            assert torch.equal(a[off:off + 1], b[j:j + 1])
    # batches of 7 at shifted offsets with left and right padding
    for start, total, off in ((0, 7, 0), (10, 20, 13), (57, 9, 2), (30, 160, 100)):
        sl = slice(start, start + 7)
        t, r, i, m = _embed(base.train[sl], base.rollout[sl], base.token_ids[sl], total, off, start)
        res = run(t, r, i, m)
        for a, b in zip((res.logp_train, res.logp_rollout, res.dlogp), outs):
            assert torch.equal(a[off:off + 7], b[sl])
    # batch of 64 inside a larger batch
    t, r, i, m = _embed(base.train, base.rollout, base.token_ids, 200, 77, 99)
    res = run(t, r, i, m)
    for a, b in zip((res.logp_train, res.logp_rollout, res.dlogp), outs):
        assert torch.equal(a[77:141], b)


def test_load_path_does_not_change_bits():
    # same rows stored with 16-byte aligned rows (bulk-copy ring) and with an
    # odd row stride (plain loads): identical results
    base = W.synthetic(50, 3 * 4096 + 517, seed=8, device=DEV, row_pad=3, active_prob=1.0)
    aligned = run(base.train, base.rollout, base.token_ids, base.action_mask)
    t2 = base.train.contiguous()   # stride 12805 elements: rows not 16-byte aligned
    r2 = base.rollout.contiguous()
    assert (t2.stride(0) * 2) % 16 != 0
    generic = run(t2, r2, base.token_ids, base.action_mask)
    for a, b in zip((aligned.logp_train, aligned.logp_rollout, aligned.dlogp),
                    (generic.logp_train, generic.logp_rollout, generic.dlogp)):
        assert torch.equal(a, b)


def test_run_to_run_bitwise():
    w = W.synthetic(700, 20000, seed=9, device=DEV)
    a = run(w.train, w.rollout, w.token_ids, w.action_mask)
    b = run(w.train, w.rollout, w.token_ids, w.action_mask)
    for x, y in zip((a.logp_train, a.logp_rollout, a.dlogp), (b.logp_train, b.logp_rollout, b.dlogp)):
        assert torch.equal(x, y)
    assert a.metrics == b.metrics


# ------------------------------------------------------------------- edges

def test_zero_rows():
    t = torch.empty((0, 100), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(0, dtype=torch.int32, device=DEV)
    mask = torch.empty(0, dtype=torch.uint8, device=DEV)
    res = run(t, t, ids, mask)
    m = res.metrics
    assert m["n_active"] == 0 and m["flags"] == B.LPD_FLAG_NO_ACTIVE and m["status"] == 0
    assert m["argmax_row"] == -1 and m["max_abs_dlogp"] == 0.0


def test_all_masked():
    w = W.synthetic(100, 3000, seed=10, device=DEV)
    mask = torch.zeros_like(w.action_mask)
    res, ref = check_against_oracle(W.Workload("m", w.train, w.rollout, w.token_ids, mask, w.vocab))
    assert res.metrics["n_active"] == 0 and res.metrics["flags"] == B.LPD_FLAG_NO_ACTIVE
    assert torch.all(res.dlogp == 0)


def test_token_out_of_range():
    w = W.synthetic(50, 1000, seed=11, device=DEV, active_prob=1.0)
    ids = w.token_ids.clone()
    ids[7] = 1000
    res = run(w.train, w.rollout, ids, w.action_mask)
    assert res.metrics["status"] == B.LPD_STATUS_TOKEN_OOB
    assert torch.isnan(res.logp_train[7]) and torch.isnan(res.dlogp[7])
    ids[7] = -3
    assert run(w.train, w.rollout, ids, w.action_mask).metrics["status"] == B.LPD_STATUS_TOKEN_OOB
    # the same bad id on an inactive row is never looked at
    mask = w.action_mask.clone()
    mask[7] = 0
    res2 = run(w.train, w.rollout, ids, mask)
    assert res2.metrics["status"] == 0


def test_nonfinite_logits():
    w = W.synthetic(20, 5000, seed=12, device=DEV, active_prob=1.0)
    t = w.train.clone()
    t[3, 100] = float("nan")
    assert run(t, w.rollout, w.token_ids, w.action_mask).metrics["status"] == B.LPD_STATUS_NONFINITE
    t = w.train.clone()
    t[4, :] = float("-inf")
    assert run(t, w.rollout, w.token_ids, w.action_mask).metrics["status"] == B.LPD_STATUS_NONFINITE
    # -inf columns elsewhere are fine and agree with the oracle
    t = w.train.clone()
    cols = (w.token_ids[5].item() + 1) % 5000
    t[5, cols] = float("-inf")
    t[6, 4999] = float("-inf")
    w2 = W.Workload("ninf", t, w.rollout, w.token_ids, w.action_mask, w.vocab)
    res, ref = check_against_oracle(w2)
    assert res.metrics["status"] == 0
    # garbage in inactive rows changes nothing
    mask = w.action_mask.clone()
    mask[9] = 0
    t = w.train.clone()
    t[9] = float("nan")
    res3 = run(t, w.rollout, w.token_ids, mask)
    assert res3.metrics["status"] == 0


def test_stage_entry_points_equal_lpd_score():
    w = W.synthetic(333, 7000, seed=13, device=DEV)
    full = run(w.train, w.rollout, w.token_ids, w.action_mask)
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(3)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    B.lpd_select_active(w.token_ids, w.action_mask, *outs, met, ws)
    B.lpd_token_logp(w.train, w.rollout, *outs, met, ws)
    B.lpd_drift_metrics(n, 0.8, 1.2, met, ws)
    torch.cuda.synchronize()
    for a, b in zip(outs, (full.logp_train, full.logp_rollout, full.dlogp)):
        assert torch.equal(a, b)
    assert B.read_metrics(met) == full.metrics


# ------------------------------------------------------------------ sharded

def _sharded_call(w, perm=None):
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(5)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SHARDED, n, w.vocab, len(w.v_ranges)), dtype=torch.uint8,
                     device=DEV)
    B.lpd_score_sharded(w.train, w.rollout, w.v_ranges, w.token_ids, w.action_mask, 0.8, 1.2, perm, *outs, met, ws)
    torch.cuda.synchronize()
    return outs, B.read_metrics(met)


def _small_sharded(bounds, rows=120, seed=20):
    base = W.synthetic(rows, bounds[-1][1], seed=seed, device=DEV)
    ts = [base.train[:, a:b].contiguous() for a, b in bounds]
    rs = [base.rollout[:, a:b].contiguous() for a, b in bounds]
    return base, W.Workload("sh", ts, rs, base.token_ids, base.action_mask, base.vocab, v_ranges=list(bounds))


@pytest.mark.parametrize("bounds", [
    [(0, 4096), (4096, 8192), (8192, 12288), (12288, 16384)],
    [(0, 1000), (1000, 9000), (9000, 9001), (9001, 12000)],
    [(0, 5000)],
    # the maximum of 16 shards, uneven, one of a single column
    [(a, b) for a, b in zip([0, 700, 701, 2000, 2100, 4097, 5000, 6000, 6001, 7000, 8192, 9000, 10001, 11000, 12000,
                             13000], [700, 701, 2000, 2100, 4097, 5000, 6000, 6001, 7000, 8192, 9000, 10001, 11000,
                                      12000, 13000, 14001])],
    # segment lengths that make the multi-segment pass take 23 consumer warps:
    # whole 11 776-column tiles, then ragged last tiles padded by -inf copies
    [(0, 23552), (23552, 47104)],
    [(0, 22776), (22776, 45552)],
])
def test_sharded_vs_oracle(bounds):
    base, w = _small_sharded(bounds)
    perm = list(range(len(bounds)))[::-1]
    (lt, lr, d, plt, plr), met = _sharded_call(w, perm)
    mask = w.action_mask.cpu().numpy()
    ref = oracle.score_sharded([to_oracle(x) for x in w.train], [to_oracle(x) for x in w.rollout], w.v_ranges,
                               w.token_ids.cpu().numpy(), mask)
    ref_p = oracle.score_sharded([to_oracle(x) for x in w.train], [to_oracle(x) for x in w.rollout], w.v_ranges,
                                 w.token_ids.cpu().numpy(), mask, order=perm)
    act = mask != 0
    for got, want in ((lt, ref.logp_train), (lr, ref.logp_rollout), (d, ref.dlogp),
                      (plt, ref_p.logp_train), (plr, ref_p.logp_rollout)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.max(np.abs(g[act] - want[act])) <= LOGP_ATOL
        assert np.all(g[~act] == 0)
    assert_metrics_match(met, ref.metrics, ref.dlogp, mask)
    # the fixed-order result is bitwise repeatable
    (lt2, _, d2, _, _), met2 = _sharded_call(w, perm)
    assert torch.equal(lt, lt2) and torch.equal(d, d2) and met == met2
    # array order of the shards does not matter (merge order is vocab order)
    rev = W.Workload("rev", w.train[::-1], w.rollout[::-1], w.token_ids, w.action_mask, w.vocab,
                     v_ranges=w.v_ranges[::-1])
    (lt3, _, d3, _, _), _ = _sharded_call(rev)
    assert torch.equal(lt, lt3) and torch.equal(d, d3)


def _summary_vs_oracle(a_t, a_r, b_t, b_r, mask):
    """GPU lpd_logp_drift_summary against the oracle's summary of the same
    float32 values: equal field by field (|b - a| of two floats within a factor
    of two is exact in fp32, so even the maxima agree bitwise)."""
    got = B.logp_drift_summary(a_t, a_r, b_t, b_r, mask)
    want = oracle.logp_drift(*(x.cpu().numpy() for x in (a_t, a_r, b_t, b_r)), mask.cpu().numpy())
    for k, v in want.items():
        g = got[k]
        assert (np.isnan(g) and np.isnan(v)) if isinstance(v, float) and np.isnan(v) else g == v, (k, g, v)
    return got


@pytest.mark.parametrize("bounds,perm", [
    ([(0, 4096), (4096, 8192), (8192, 12288), (12288, 16384)], [3, 2, 1, 0]),
    ([(0, 1000), (1000, 9000), (9000, 9001), (9001, 12000)], [2, 0, 3, 1]),
    ([(0, 5000)], [0]),
])
def test_shard_merge_order_summary(bounds, perm):
    """The merge-order diagnostic's summary ("[WS2] Framework for ablation
    experiment", LogProb knobs table, row 5): the GPU summary of the fixed
    against the permuted per-token result equals the oracle's summary of the
    same values, and, both orders being within the logp bar of the oracle's
    fixed-order and permuted-order results, the largest drift is within twice
    the bar; a single shard, or the identity order, drifts by exactly 0."""
    base, w = _small_sharded(bounds, rows=300, seed=31)
    (lt, lr, d, plt, plr), met = _sharded_call(w, perm)
    s = _summary_vs_oracle(lt, lr, plt, plr, w.action_mask)
    assert s["n_active"] == met["n_active"]
    mask = w.action_mask.cpu().numpy()
    ref = oracle.score_sharded([to_oracle(x) for x in w.train], [to_oracle(x) for x in w.rollout], w.v_ranges,
                               w.token_ids.cpu().numpy(), mask)
    ref_p = oracle.score_sharded([to_oracle(x) for x in w.train], [to_oracle(x) for x in w.rollout], w.v_ranges,
                                 w.token_ids.cpu().numpy(), mask, order=perm)
    exact = oracle.logp_drift(*(v.astype(np.float32) for v in (ref.logp_train, ref.logp_rollout, ref_p.logp_train,
                                                                ref_p.logp_rollout)), mask)
    assert exact["max_abs_dlogp_train"] <= 1e-5 and exact["max_abs_dlogp_rollout"] <= 1e-5
    assert s["max_abs_dlogp_train"] <= 2 * LOGP_ATOL and s["max_abs_dlogp_rollout"] <= 2 * LOGP_ATOL
    if perm == sorted(perm):
        assert s["n_differ"] == 0 and s["max_abs_dlogp_train"] == 0.0 and s["max_abs_dlogp_rollout"] == 0.0


def test_logp_drift_summary_edges():
    g = torch.Generator(device=DEV).manual_seed(32)
    n = 70000
    a_t = -12 + torch.randn(n, generator=g, device=DEV)
    a_r = -12 + torch.randn(n, generator=g, device=DEV)
    b_t, b_r = a_t.clone(), a_r.clone()
    mask = (torch.rand(n, generator=g, device=DEV) < 0.8).to(torch.uint8)
    # planted differences: a tie on the train side (lowest row wins), a bigger
    # one on a masked row, one float32 step, +0 / -0, and NaN pairs
    b_t[[100, 200, 60000]] += torch.tensor([0.5, 0.25, 0.5], device=DEV)
    mask[[100, 200, 60000]] = 1
    b_t[300] += 4.0
    mask[300] = 0
    b_r[5] = torch.nextafter(a_r[5], torch.tensor(0.0, device=DEV))
    mask[5] = 1
    a_r[7], b_r[7] = 0.0, -0.0
    s = _summary_vs_oracle(a_t, a_r, b_t, b_r, mask)
    assert s["row_train"] == 100 and s["n_differ"] == 4
    # a NaN pair (both results NaN: the same) still ranks above every number
    a_t[40000] = b_t[40000] = float("nan")
    mask[40000] = 1
    s = _summary_vs_oracle(a_t, a_r, b_t, b_r, mask)
    assert np.isnan(s["max_abs_dlogp_train"]) and s["row_train"] == 40000 and s["n_differ"] == 4
    # nothing active, and no rows at all
    _summary_vs_oracle(a_t, a_r, b_t, b_r, torch.zeros_like(mask))
    e = torch.empty(0, device=DEV)
    s = _summary_vs_oracle(e, e, e, e, torch.empty(0, dtype=torch.uint8, device=DEV))
    assert s["row_train"] == -1 and s["n_active"] == 0 and s["frac_differ"] == 0.0


# ------------------------------------------------------------- timeouts

def test_stalled_pipeline_times_out_cleanly(monkeypatch):
    """LPD_STALL_ROW_PASS=1 makes one CTA of the row pass withhold its first
    copy (a barrier nothing completes): the call returns after the bounded
    waits with LPD_STATUS_TIMEOUT set instead of hanging, and the next call on
    the same context scores normally."""
    w = W.synthetic(600, 3 * 8192 + 96, seed=91, device=DEV, active_prob=1.0)
    assert (w.train.stride(0) * 2) % 16 == 0   # rows take the bulk-copy ring, whose waits are bounded
    monkeypatch.setenv("LPD_STALL_ROW_PASS", "1")
    res = run(w.train, w.rollout, w.token_ids, w.action_mask)
    assert res.metrics["status"] & B.LPD_STATUS_TIMEOUT
    monkeypatch.delenv("LPD_STALL_ROW_PASS")
    check_against_oracle(w)


def test_drift_metrics_repeated_on_one_workspace():
    """The staged calls, then the metrics stage twice more on the same
    workspace (its select histogram is rebuilt each call) and once with other
    clip bounds: the same record each time at the same bounds, and the oracle's
    metrics at the others."""
    w = W.synthetic(20000, 3000, seed=41, device=DEV, rollout_noise=0.3)
    n = w.n_rows
    lt, lr, d = (torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(3))
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    B.lpd_select_active(w.token_ids, w.action_mask, lt, lr, d, met, ws)
    B.lpd_token_logp(w.train, w.rollout, lt, lr, d, met, ws)
    B.lpd_drift_metrics(n, 0.8, 1.2, met, ws)
    torch.cuda.synchronize()
    first = B.read_metrics(met)
    B.lpd_drift_metrics(n, 0.8, 1.2, met, ws)
    B.lpd_drift_metrics(n, 0.8, 1.2, met, ws)
    torch.cuda.synchronize()
    assert B.read_metrics(met) == first
    B.lpd_drift_metrics(n, 0.5, 1.5, met, ws)
    torch.cuda.synchronize()
    other = B.read_metrics(met)
    mask = w.action_mask.cpu().numpy()
    ref = oracle_score(w.train, w.rollout, w.token_ids, w.action_mask, clip=(0.5, 1.5))
    assert_metrics_match(other, ref.metrics, ref.dlogp, mask, (0.5, 1.5))
    assert other["p95_abs_dlogp"] == first["p95_abs_dlogp"] and other["clipfrac0"] < first["clipfrac0"]
