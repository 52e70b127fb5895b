"""The multi-core oracle runner (oracle/stream.py) only schedules: split over
host threads and chunks, every row must come out bit for bit what the serial
oracle gives, in the order of the listed rows."""
import numpy as np
import torch

import oracle
from oracle import stream
from logprob_drift_scoring_gb300 import workloads as W
from tests.helpers import to_oracle


def _same(a, b):
    assert a.status == b.status
    for x, y in ((a.logp_train, b.logp_train), (a.logp_rollout, b.logp_rollout), (a.dlogp, b.dlogp)):
        assert np.array_equal(x, y)


def test_threaded_rows_equal_serial_rows():
    w = W.synthetic(90, 777, seed=3, device="cpu", dtype_rollout=torch.float32)
    rows = np.array([5, 0, 89, 17, 17, 40, 3] + list(range(50, 80)))
    want = oracle.score_rows(to_oracle(w.train), to_oracle(w.rollout), w.token_ids.numpy(), rows)
    got = stream.score_rows_device(w.train, w.rollout, w.token_ids, rows, chunk=7, threads=4)
    _same(got, want)
    got2 = stream.score_rows_parallel(to_oracle(w.train), to_oracle(w.rollout), w.token_ids.numpy(), rows,
                                      chunk=5, threads=3)
    _same(got2, want)


def test_threaded_rows_report_status():
    w = W.synthetic(20, 64, seed=4, device="cpu")
    ids = w.token_ids.clone()
    ids[13] = 64  # out of range
    rows = np.arange(20)
    got = stream.score_rows_device(w.train, w.rollout, ids, rows, chunk=3, threads=2)
    assert got.status == oracle.STATUS_TOKEN_OOB and np.isnan(got.logp_train[13])


def test_threaded_sharded_equal_serial_sharded():
    base = W.synthetic(40, 1000, seed=5, device="cpu", active_prob=1.0)
    bounds = [(0, 300), (300, 301), (301, 1000)]
    ts = [base.train[:, a:b].contiguous() for a, b in bounds]
    rs = [base.rollout[:, a:b].contiguous() for a, b in bounds]
    rows = np.array([39, 2, 7, 8, 9, 10, 11, 30])
    for order in (None, [2, 0, 1]):
        want = oracle.score_sharded([to_oracle(x[rows]) for x in ts], [to_oracle(x[rows]) for x in rs], bounds,
                                    base.token_ids.numpy()[rows], np.ones(rows.size, np.uint8), order=order)
        got = stream.score_sharded_rows_device(ts, rs, bounds, base.token_ids, rows, order=order, chunk=3,
                                               threads=3)
        _same(got, want)


def test_threaded_head_rows_equal_serial():
    w = W.head(12, 32, 50, seed=6, device="cpu")
    ht, hr, wt = to_oracle(w.hidden_train), to_oracle(w.hidden_rollout), to_oracle(w.weight)
    rows = np.array([11, 0, 4, 5, 6])
    want = oracle.score_head_rows(ht, hr, wt, w.token_ids.numpy(), rows)
    got = stream.score_head_rows_parallel(ht, hr, wt, w.token_ids.numpy(), rows, chunk=2, threads=3)
    _same(got, want)


def test_threaded_transformed_equal_serial():
    w = W.synthetic(33, 500, seed=7, device="cpu", sigma=20.0, active_prob=1.0)
    ops_t, ops_r = [(oracle.OP_SOFTCAP, 30.0), (oracle.OP_SCALE, 1.4)], [(oracle.OP_SCALE, 0.5)]
    rows = np.array([32, 1, 2, 3, 10, 20])
    want = oracle.score_transformed(to_oracle(w.train[rows]), to_oracle(w.rollout[rows]), w.token_ids.numpy()[rows],
                                    np.ones(rows.size, np.uint8), ops_t, ops_r)
    got = stream.score_transformed_rows_device(w.train, w.rollout, w.token_ids, rows, ops_t, ops_r, chunk=4,
                                               threads=2)
    _same(got, want)


def test_threaded_entropy_and_backward_equal_serial():
    w = W.synthetic(20, 300, seed=8, device="cpu", active_prob=1.0)
    rows = np.array([19, 0, 5, 6, 7])
    et, er = oracle.entropy(to_oracle(w.train[rows]), to_oracle(w.rollout[rows]), np.ones(rows.size, np.uint8))
    gt, gr = stream.entropy_rows_device(w.train, w.rollout, rows, chunk=2, threads=3)
    assert np.array_equal(gt, et) and np.array_equal(gr, er)
    grad = torch.linspace(-2, 2, 20)
    got = stream.backward_rows_device(w.train, w.token_ids, grad, rows, chunk=2, threads=2)
    x = to_oracle(w.train)
    for j, r in enumerate(rows):
        want = oracle.logprob_backward_row(np.ascontiguousarray(x[r]), int(w.token_ids[r]), float(grad[r]))
        assert np.array_equal(got[j], want)


def test_threaded_attention_merge_equals_serial():
    a = W.attn_partials(40, 3, 8, 5, seed=9, device="cpu", masked_fill=float("nan"))
    parts, lse = a.out_parts.numpy(), a.lse_parts.numpy()
    want = oracle.attn_merge(parts, lse, [4, 0, 3, 1, 2])
    got = stream.attn_merge_parallel(parts, lse, [4, 0, 3, 1, 2], chunk=7, threads=3)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
