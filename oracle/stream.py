"""The float64 oracle over large, device-resident workloads, on all host cores.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline and reference legs of ``bench.py`` may import this module.

Scheduling only, no arithmetic: the listed rows of the input tensors are
copied to host memory chunk by chunk (``torch`` is used for the device-to-host
copy and nothing else), and a pool of host threads runs the oracle's serial
C on each chunk.  ctypes releases the GIL for the duration of every C call, so
the chunks run in parallel; each row still goes through exactly the serial
float64 code of ``oracle.score_rows`` / ``oracle.score_sharded`` /
``oracle.score_head_rows``, and the results are put back in the order of the
listed rows.  Host memory in flight is bounded by ``2 * threads`` chunks.
"""
from __future__ import annotations

import os
from collections import deque
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import (Result, attn_merge, entropy, load, logprob_backward_row, score_head_rows, score_rows,
               score_sharded, score_transformed)


def host_threads(threads: int | None = None) -> int:
    """Worker threads to use: all host cores unless told otherwise."""
    return max(1, int(threads) if threads else (os.cpu_count() or 1))


def _host(t) -> np.ndarray:
    """Host numpy copy of a tensor for the oracle (bf16 as uint16 bits)."""
    import torch

    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().contiguous().numpy()


def _run_chunks(chunks, work, threads: int | None):
    """work(payload) for every (key, payload) that ``chunks`` yields, on a
    bounded pool; returns {key: result}.  The generator (device copies) runs on
    the calling thread while the pool scores earlier chunks."""
    n = host_threads(threads)
    out = {}
    with ThreadPoolExecutor(max_workers=n) as pool:
        pending = deque()
        for key, payload in chunks:
            pending.append((key, pool.submit(work, payload)))
            while len(pending) >= 2 * n:
                k, f = pending.popleft()
                out[k] = f.result()
        while pending:
            k, f = pending.popleft()
            out[k] = f.result()
    return out


def _concat(parts: list[Result]) -> Result:
    status = 0
    for p in parts:
        status |= p.status
    return Result(np.concatenate([p.logp_train for p in parts]) if parts else np.zeros(0),
                  np.concatenate([p.logp_rollout for p in parts]) if parts else np.zeros(0),
                  np.concatenate([p.dlogp for p in parts]) if parts else np.zeros(0), status)


def score_rows_device(train, rollout, token_ids, rows, chunk: int = 64, threads: int | None = None) -> Result:
    """oracle.score_rows of the listed rows of device (or host) tensors
    train/rollout [R, V] and token_ids [R]; per-row results in ``rows`` order."""
    import torch

    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dev = train.device
    ids_all = token_ids.detach().cpu().numpy().astype(np.int32)

    def chunks():
        for c in range(0, rows.size, chunk):
            sel_np = rows[c:c + chunk]
            sel = torch.as_tensor(sel_np, device=dev)
            yield c, (_host(train.index_select(0, sel)), _host(rollout.index_select(0, sel)), ids_all[sel_np])

    def work(p):
        t, r, ids = p
        return score_rows(t, r, ids, np.arange(t.shape[0]), lib=lib)

    res = _run_chunks(chunks(), work, threads)
    return _concat([res[k] for k in sorted(res)])


def score_transformed_rows_device(train, rollout, token_ids, rows, train_ops=None, rollout_ops=None,
                                  chunk: int = 64, threads: int | None = None) -> Result:
    """oracle.score_transformed of the listed rows (every listed row active),
    each side through its chain of logit transforms."""
    import torch

    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dev = train.device
    ids_all = token_ids.detach().cpu().numpy().astype(np.int32)

    def chunks():
        for c in range(0, rows.size, chunk):
            sel_np = rows[c:c + chunk]
            sel = torch.as_tensor(sel_np, device=dev)
            yield c, (_host(train.index_select(0, sel)), _host(rollout.index_select(0, sel)), ids_all[sel_np])

    def work(p):
        t, r, ids = p
        return score_transformed(t, r, ids, np.ones(ids.size, np.uint8), train_ops, rollout_ops, lib=lib)

    res = _run_chunks(chunks(), work, threads)
    return _concat([res[k] for k in sorted(res)])


def score_sharded_rows_device(train_shards, rollout_shards, v_ranges, token_ids, rows, order=None,
                              chunk: int = 64, threads: int | None = None) -> Result:
    """oracle.score_sharded of the listed rows (every listed row active),
    shards merged in ``order`` (default: ascending vocab position)."""
    import torch

    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dev = train_shards[0].device
    ids_all = token_ids.detach().cpu().numpy().astype(np.int32)

    def chunks():
        for c in range(0, rows.size, chunk):
            sel_np = rows[c:c + chunk]
            sel = torch.as_tensor(sel_np, device=dev)
            yield c, ([_host(x.index_select(0, sel)) for x in train_shards],
                      [_host(x.index_select(0, sel)) for x in rollout_shards], ids_all[sel_np])

    def work(p):
        ts, rs, ids = p
        return score_sharded(ts, rs, v_ranges, ids, np.ones(ids.size, np.uint8), order=order, lib=lib)

    res = _run_chunks(chunks(), work, threads)
    return _concat([res[k] for k in sorted(res)])


def score_head_rows_parallel(hidden_train, hidden_rollout, weight, token_ids, rows, chunk: int = 4,
                             threads: int | None = None) -> Result:
    """oracle.score_head_rows (logits materialised in double) of the listed
    rows; host arrays (bf16 bits as uint16), rows split over host threads."""
    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)

    def chunks():
        for c in range(0, rows.size, chunk):
            yield c, rows[c:c + chunk]

    def work(sel):
        return score_head_rows(hidden_train, hidden_rollout, weight, token_ids, sel, lib=lib)

    res = _run_chunks(chunks(), work, threads)
    return _concat([res[k] for k in sorted(res)])


def score_rows_parallel(train, rollout, token_ids, rows, chunk: int = 64, threads: int | None = None) -> Result:
    """oracle.score_rows of host arrays with the listed rows split over host
    threads."""
    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)

    def chunks():
        for c in range(0, rows.size, chunk):
            yield c, rows[c:c + chunk]

    def work(sel):
        return score_rows(train, rollout, token_ids, sel, lib=lib)

    res = _run_chunks(chunks(), work, threads)
    return _concat([res[k] for k in sorted(res)])


def entropy_rows_device(train, rollout, rows, chunk: int = 64, threads: int | None = None):
    """oracle.entropy of the listed rows (every listed row active): the two
    sides' softmax entropies, in ``rows`` order."""
    import torch

    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dev = train.device

    def chunks():
        for c in range(0, rows.size, chunk):
            sel = torch.as_tensor(rows[c:c + chunk], device=dev)
            yield c, (_host(train.index_select(0, sel)), _host(rollout.index_select(0, sel)))

    def work(p):
        t, r = p
        return entropy(t, r, np.ones(t.shape[0], np.uint8), lib=lib)

    res = _run_chunks(chunks(), work, threads)
    keys = sorted(res)
    if not keys:
        return np.zeros(0), np.zeros(0)
    return np.concatenate([res[k][0] for k in keys]), np.concatenate([res[k][1] for k in keys])


def backward_rows_device(logits, token_ids, grad, rows, chunk: int = 8, threads: int | None = None):
    """oracle.logprob_backward_row of each listed row (grad[r] * d logp / d
    logits), as a [len(rows), V] float64 array in ``rows`` order."""
    import torch

    lib = load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    dev = logits.device
    ids = token_ids.detach().cpu().numpy().astype(np.int64)
    g = grad.detach().double().cpu().numpy()

    def chunks():
        for c in range(0, rows.size, chunk):
            sel_np = rows[c:c + chunk]
            yield c, (_host(logits.index_select(0, torch.as_tensor(sel_np, device=dev))), sel_np)

    def work(p):
        x, sel_np = p
        return np.stack([logprob_backward_row(np.ascontiguousarray(x[j]), int(ids[r]), float(g[r]), lib=lib)
                         for j, r in enumerate(sel_np)])

    res = _run_chunks(chunks(), work, threads)
    keys = sorted(res)
    return np.concatenate([res[k] for k in keys]) if keys else np.zeros((0, logits.shape[1]))


def attn_merge_parallel(out_parts, lse_parts, order=None, lse_base2=False, chunk: int = 4096,
                        threads: int | None = None):
    """oracle.attn_merge of host arrays ([K, n, d], [K, n]) with the rows split
    into chunks over host threads; (out [n, d], lse [n]) in row order."""
    lib = load()
    n = lse_parts.shape[1]

    def chunks():
        for c in range(0, n, chunk):
            yield c, (out_parts[:, c:c + chunk], lse_parts[:, c:c + chunk])   # views; copied by the worker

    def work(p):
        o, l = p
        return attn_merge(np.ascontiguousarray(o), np.ascontiguousarray(l), order, lse_base2, lib=lib)

    res = _run_chunks(chunks(), work, threads)
    keys = sorted(res)
    if not keys:
        return np.zeros((0, out_parts.shape[2])), np.zeros(0)
    return np.concatenate([res[k][0] for k in keys]), np.concatenate([res[k][1] for k in keys])
