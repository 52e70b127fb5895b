"""Multi-rank host logic on CPU with the gloo backend (world size 2).

Each rank scores its own contiguous rows (here with the oracle, since these
processes have no GPU), exchanges only its metric record, and the merged
record must equal the single-process metrics over all rows; the bench's
max-over-ranks timing helper is checked the same way.
"""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _data(n_rows=300, vocab=500):
    from tests.oracle_pins import bf16_bits

    rng = np.random.default_rng(77)
    t = rng.normal(0, 3, size=(n_rows, vocab)).astype(np.float32)
    r = t + rng.normal(0, 0.05, size=t.shape).astype(np.float32)
    ids = rng.integers(0, vocab, size=n_rows).astype(np.int32)
    mask = (rng.random(n_rows) < 0.8).astype(np.uint8)
    return bf16_bits(t), bf16_bits(r), ids, mask


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import oracle
    import torch

    from logprob_drift_scoring_gb300.ranks import gather_rank_metrics, gather_rank_rows, merge_rank_metrics

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    t, r, ids, mask = _data()
    rows = np.array_split(np.arange(t.shape[0]), world)[rank]
    lo = int(rows[0])
    local = oracle.score(np.ascontiguousarray(t[rows]), np.ascontiguousarray(r[rows]), ids[rows], mask[rows])
    per_rank = gather_rank_metrics(local.metrics, rank_meta={"row_offset": lo})
    merged = merge_rank_metrics(per_rank, [p["row_offset"] for p in per_rank])
    tmax = bench.barrier_max(float(rank + 1), world)
    # rows of every rank in rank order: first the real split's dlogp, then
    # deliberately uneven sizes (rank k holds 3 + 4k rows)
    d_all, m_all = gather_rank_rows(torch.from_numpy(local.dlogp.astype(np.float32)),
                                    torch.from_numpy(mask[rows].copy()))
    n_k = 3 + 4 * rank
    u_d, u_m = gather_rank_rows(torch.arange(n_k, dtype=torch.float32) + 100 * rank,
                                (torch.arange(n_k) % 2).to(torch.uint8))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"per_rank": per_rank, "merged": merged, "tmax": tmax, "d_all": d_all.tolist(),
                   "m_all": m_all.tolist(), "u_d": u_d.tolist(), "u_m": u_m.tolist()}, f)
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_metrics_merge_and_timing(tmp_path):
    import oracle

    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{k}.json")) for k in range(world)]
    t, r, ids, mask = _data()
    whole = oracle.score(t, r, ids, mask).metrics
    for k in range(world):
        assert res[k]["tmax"] == 2.0
        assert [p["rank"] for p in res[k]["per_rank"]] == [0, 1]
        m = res[k]["merged"]
        assert m["n_active"] == whole["n_active"] == int(mask.sum())
        assert m["argmax_row"] == whole["argmax_row"]
        assert m["max_abs_dlogp"] == whole["max_abs_dlogp"]
        for key in ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp"):
            assert abs(m[key] - whole[key]) <= 1e-12 * max(1.0, abs(whole[key])), key
    # the per-rank view keeps each rank's own active count
    counts = [p["n_active"] for p in res[0]["per_rank"]]
    halves = np.array_split(np.arange(len(mask)), world)
    assert counts == [int(mask[h].sum()) for h in halves]
    # gathered rows: the union in rank order, identical on every rank; its
    # metrics (percentiles included) are those of the whole batch
    whole_d = oracle.score(t, r, ids, mask).dlogp.astype(np.float32)
    for k in range(world):
        assert np.array_equal(np.array(res[k]["d_all"], np.float32), whole_d)
        assert np.array_equal(np.array(res[k]["m_all"], np.uint8), mask)
        assert res[k]["u_d"] == [0.0, 1.0, 2.0] + [100.0 + i for i in range(7)]
        assert res[k]["u_m"] == [0, 1, 0] + [i % 2 for i in range(7)]
    union = oracle.metrics(np.array(res[0]["d_all"], np.float64), mask, 0.8, 1.2)
    ref = oracle.metrics(whole_d.astype(np.float64), mask, 0.8, 1.2)
    for key in ("p95_abs_dlogp", "p99_abs_dlogp", "max_abs_dlogp", "approx_kl0", "n_active", "argmax_row"):
        assert union[key] == ref[key], key
