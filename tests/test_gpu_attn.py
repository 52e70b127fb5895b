"""Attention (out, lse) merge and its merge-order diagnostic ("Attention Debug
Matrix", row A7 merge_order; "[WS2] Framework for ablation experiment",
Attention knobs table, rows 6-7) against the float64 oracle (needs a GPU).

Tolerance.  The merge folds K parts in fp32: per part one weight
exp(lse_k - m) from ex2.approx (relative error below 2^-22) of an argument
rounded once or twice, and one fused multiply-add per column; the final
division and log add one rounding each.  Summed over K parts that stays below
(8K + 4) * 2^-24 of the largest |out_k| of the row for out, and
(8K + 8) * 2^-24 * max(1, |lse|) for lse.
"""
import numpy as np
import pytest
import torch

import oracle
from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


def _rows(w, rows):
    if rows is None:
        return w.out_parts, w.lse_parts
    idx = torch.as_tensor(rows, device=w.out_parts.device)
    return w.out_parts[:, idx], w.lse_parts[:, idx]


def _oracle(w, order=None, rows=None):
    parts, lse = _rows(w, rows)
    return oracle.attn_merge(parts.float().cpu().numpy(), lse.cpu().numpy(), order, lse_base2=w.lse_base2)


def _row_scale(w, rows=None):
    """Largest |out_k| over the parts that saw keys, per row."""
    parts, lse = _rows(w, rows)
    parts = parts.float()
    keyed = torch.isfinite(lse)
    mag = torch.where(keyed[:, :, None], parts.abs(), torch.zeros_like(parts)).amax(dim=(0, 2))
    return mag.cpu().numpy().astype(np.float64)


def _assert_close(w, got_out, got_lse, order=None, rows=None):
    want_out, want_lse = _oracle(w, order, rows)
    K = w.n_parts
    go = got_out.cpu().numpy().astype(np.float64)
    gl = got_lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        go, gl = go[rows], gl[rows]
    dead = want_lse == -np.inf
    assert np.array_equal(gl[dead], want_lse[dead])                  # rows no part saw
    assert np.all(go[dead] == 0.0)
    live = ~dead
    tol_o = (8 * K + 4) * U * _row_scale(w, rows)[live]
    err_o = np.max(np.abs(go[live] - want_out[live]), axis=1) if live.any() else np.zeros(0)
    assert np.all(err_o <= tol_o), float(np.max(err_o - tol_o))
    tol_l = (8 * K + 8) * U * np.maximum(1.0, np.abs(want_lse[live]))
    assert np.all(np.abs(gl[live] - want_lse[live]) <= tol_l)


@pytest.mark.parametrize("T,H,d,K,dtype,base2", [
    (37, 3, 128, 5, torch.float32, False),      # ragged last block, 32 chunks per row
    (61, 2, 80, 7, torch.float32, False),       # 20 chunks per row: rows straddle blocks
    (50, 4, 64, 8, torch.bfloat16, False),      # bf16 partial state, 8 chunks per row
    (300, 2, 8, 3, torch.bfloat16, False),      # one chunk per row: 128 rows per block
    (40, 2, 128, 6, torch.float32, True),       # base-2 lse
    (33, 2, 4, 1, torch.float32, False),        # one part
    (130, 1, 16, 64, torch.float32, False),     # the most parts
    (11, 2, 16, 20, torch.float32, False),      # looped part count, two chunks per thread
    (7, 1, 16, 32, torch.bfloat16, False),      # the most parts with two chunks per thread
    (9, 3, 8, 33, torch.bfloat16, True),        # one chunk per row, looped part count
    (4000, 16, 128, 8, torch.float32, False),   # more tiles than resident blocks: persistent loop
    (3000, 8, 64, 12, torch.bfloat16, False),   # the same with a looped part count
])
def test_merge_matches_oracle(T, H, d, K, dtype, base2):
    w = W.attn_partials(T, H, d, K, seed=T + K, device=DEV, dtype=dtype, lse_base2=base2,
                        masked_fill=float("nan"))
    rng = np.random.default_rng(T)
    for order in (None, list(range(K))[::-1], list(rng.permutation(K))):
        out, lse = B.attn_merge(w.out_parts, w.lse_parts, order, lse_base2=base2)
        torch.cuda.synchronize()
        _assert_close(w, out, lse, order)


def test_merge_rows_no_part_saw():
    w = W.attn_partials(20, 2, 32, 4, seed=9, device=DEV, masked_fill=float("nan"))
    w.lse_parts[:, 5] = -float("inf")
    w.lse_parts[:, 17] = -float("inf")
    w.out_parts[:, 5] = float("nan")
    out, lse = B.attn_merge(w.out_parts, w.lse_parts)
    torch.cuda.synchronize()
    assert lse[5].item() == -float("inf") and lse[17].item() == -float("inf")
    assert torch.all(out[5] == 0) and torch.all(out[17] == 0)
    _assert_close(w, out, lse)


def test_one_part_is_the_identity_and_equal_parts_average_exactly():
    w = W.attn_partials(64, 2, 32, 1, seed=10, device=DEV, causal=False)
    out, lse = B.attn_merge(w.out_parts, w.lse_parts)
    torch.cuda.synchronize()
    assert torch.equal(out, w.out_parts[0]) and torch.equal(lse, w.lse_parts[0])
    # four identical parts: acc = 4 o and s = 4 exactly, so out = o bitwise
    parts = w.out_parts.expand(4, -1, -1).contiguous()
    lses = w.lse_parts.expand(4, -1).contiguous()
    out, lse = B.attn_merge(parts, lses, [2, 0, 3, 1])
    torch.cuda.synchronize()
    assert torch.equal(out, w.out_parts[0])
    want = (w.lse_parts[0].double() + np.log(4.0)).cpu().numpy()
    assert np.max(np.abs(lse.cpu().numpy() - want)) <= 2 * U * np.max(np.abs(want))


def test_order_names_the_visit_sequence():
    # permuting the stored parts and the order together visits the same data in
    # the same sequence, so the result is bitwise the same
    w = W.attn_partials(45, 3, 64, 6, seed=11, device=DEV)
    order = [3, 0, 5, 1, 4, 2]
    pi = [2, 5, 0, 4, 1, 3]                     # stored part j = original part pi[j]
    inv = np.argsort(pi)
    parts = w.out_parts[pi].contiguous()
    lses = w.lse_parts[pi].contiguous()
    a = B.attn_merge(w.out_parts, w.lse_parts, order)
    b = B.attn_merge(parts, lses, [int(inv[k]) for k in order])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_merge_is_batch_invariant_and_deterministic():
    w = W.attn_partials(200, 4, 128, 8, seed=12, device=DEV)
    full = B.attn_merge(w.out_parts, w.lse_parts, [7, 1, 3, 5, 0, 2, 4, 6])
    again = B.attn_merge(w.out_parts, w.lse_parts, [7, 1, 3, 5, 0, 2, 4, 6])
    lo, hi = 123, 517
    part = B.attn_merge(w.out_parts[:, lo:hi].contiguous(), w.lse_parts[:, lo:hi].contiguous(),
                        [7, 1, 3, 5, 0, 2, 4, 6])
    torch.cuda.synchronize()
    assert torch.equal(full[0], again[0]) and torch.equal(full[1], again[1])
    assert torch.equal(full[0][lo:hi], part[0]) and torch.equal(full[1][lo:hi], part[1])


def _summary(rdo, rdl):
    rdo = rdo.cpu().numpy()
    rdl = rdl.cpu().numpy()
    return {"max_abs_dout": float(rdo.max()), "row_dout": int(np.argmax(rdo)),
            "max_abs_dlse": float(rdl.max()), "row_dlse": int(np.argmax(rdl))}


@pytest.mark.parametrize("T,H,d,K,dtype", [
    (37, 3, 128, 5, torch.float32),
    (61, 2, 80, 7, torch.float32),
    (50, 4, 64, 8, torch.bfloat16),
    (130, 1, 16, 64, torch.float32),
    (11, 2, 16, 20, torch.float32),
    (300, 2, 8, 3, torch.bfloat16),
    (4000, 16, 128, 8, torch.float32),
])
def test_order_drift_is_the_difference_of_the_two_merges(T, H, d, K, dtype):
    w = W.attn_partials(T, H, d, K, seed=T * K, device=DEV, dtype=dtype, masked_fill=float("nan"))
    order_a = list(range(K))
    order_b = list(np.random.default_rng(K).permutation(K))
    out, lse, rdo, rdl, summ = B.attn_merge_order_drift(w.out_parts, w.lse_parts, order_a, order_b)
    oa, la = B.attn_merge(w.out_parts, w.lse_parts, order_a)
    ob, lb = B.attn_merge(w.out_parts, w.lse_parts, order_b)
    torch.cuda.synchronize()
    assert torch.equal(out, oa) and torch.equal(lse, la)          # order_a result, bitwise
    assert torch.equal(rdo, (oa - ob).abs().amax(dim=1))
    same = la == lb
    assert torch.equal(rdl, torch.where(same, torch.zeros_like(la), (la - lb).abs()))
    assert summ == _summary(rdo, rdl)
    # each order is within the merge bound of the exact result, so the drift is too
    _assert_close(w, ob, lb, order_b)
    bound = 2 * (8 * K + 4) * U * _row_scale(w)
    assert np.all(rdo.cpu().numpy() <= bound)


def test_order_drift_degenerate_cases():
    w = W.attn_partials(50, 2, 32, 4, seed=13, device=DEV)
    out, lse, rdo, rdl, summ = B.attn_merge_order_drift(w.out_parts, w.lse_parts, [1, 3, 0, 2], [1, 3, 0, 2])
    torch.cuda.synchronize()
    assert torch.all(rdo == 0) and torch.all(rdl == 0)
    assert summ == {"max_abs_dout": 0.0, "max_abs_dlse": 0.0, "row_dout": 0, "row_dlse": 0}
    empty = W.attn_partials(0, 2, 32, 4, seed=13, device=DEV)
    *_, summ = B.attn_merge_order_drift(empty.out_parts, empty.lse_parts, None, [3, 2, 1, 0])
    torch.cuda.synchronize()
    assert summ == {"max_abs_dout": 0.0, "max_abs_dlse": 0.0, "row_dout": -1, "row_dlse": -1}
    out, lse = B.attn_merge(empty.out_parts, empty.lse_parts)
    assert out.numel() == 0 and lse.numel() == 0


@pytest.mark.slow
def test_full_size_merge_and_drift_on_sampled_rows():
    """The 8-way causal split of 32768 tokens x 32 heads, head_dim 128, in the
    launch configuration the benchmark times; sampled rows against the oracle."""
    w = W.attn(device=DEV)
    rows = np.sort(np.random.default_rng(14).choice(w.n_rows, size=1500, replace=False))
    rows = np.concatenate([rows, [0, 31, w.n_rows - 1]])
    order_b = [7, 6, 5, 4, 3, 2, 1, 0]
    out, lse, rdo, rdl, summ = B.attn_merge_order_drift(w.out_parts, w.lse_parts, None, order_b)
    torch.cuda.synchronize()
    _assert_close(w, out, lse, None, rows)
    ob, lb = B.attn_merge(w.out_parts, w.lse_parts, order_b)
    torch.cuda.synchronize()
    _assert_close(w, ob, lb, order_b, rows)
    assert torch.equal(rdo, (out - ob).abs().amax(dim=1))
    assert summ == _summary(rdo, rdl)
