"""Each plausible mistake in the oracle must fail at least one pin.

A mutant is the oracle's C source with one textual change (a dropped term, a
wrong sign, a wrong index, an off-by-one rank, a swapped operand).  It is
compiled into a temporary library and the whole pin suite runs against it.
The real oracle file is never modified.
"""
import subprocess
import sys
from pathlib import Path

import pytest

import oracle

MUTANTS = {
    "exp_sign": ("s += exp(logit_at(row, dtype, j) - m);", "s += exp(logit_at(row, dtype, j) + m);"),
    "lse_sign": ("return m + log(s);", "return m - log(s);"),
    "lse_drop_max": ("return m + log(s);", "return log(s);"),
    "logp_operands": ("*logp_out = xs - lse;", "*logp_out = lse - xs;"),
    "selected_index": ("double xs = logit_at(row, dtype, id);", "double xs = logit_at(row, dtype, 0);"),
    "dlogp_sign": ("dlogp[r] = logp_train[r] - logp_rollout[r];", "dlogp[r] = logp_rollout[r] - logp_train[r];"),
    "bf16_widening": ("uint32_t bits = (uint32_t)((const uint16_t *)row)[j] << 16;",
                      "uint32_t bits = (uint32_t)((const uint16_t *)row)[j] << 15;"),
    "max_skipped": ("if (x > m)\n            m = x;", "if (x < m)\n            m = x;"),
    "rank_floor": ("int64_t k95 = (95 * a + 99) / 100", "int64_t k95 = (95 * a) / 100 + (a < 20)"),
    "rank_off_by_one": ("out->p99_abs_dlogp = absd[k99 - 1];", "out->p99_abs_dlogp = absd[k99 < a ? k99 : a - 1];"),
    "clip_inclusive": ("if (ratio < clip_lo || ratio > clip_hi)", "if (ratio <= clip_lo || ratio >= clip_hi)"),
    "clip_one_sided": ("if (ratio < clip_lo || ratio > clip_hi)", "if (ratio > clip_hi)"),
    "k3_sign": ("sum_k3 += expm1(x) - x;", "sum_k3 += expm1(x) + x;"),
    "k3_dropped_one": ("sum_k3 += expm1(x) - x;", "sum_k3 += exp(x) - x;"),
    "argmax_ties_high": ("if (fabs(x) > best) {", "if (fabs(x) >= best) {"),
    "mask_ignored_count": ("a += mask[r] != 0;", "a += 1;"),
    "mask_ignored_rows": ("        if (!mask[r])\n            continue;\n        double x = d[r];",
                          "        double x = d[r];"),
    "mean_abs_denominator": ("out->mean_abs_dlogp = sum_abs / (double)a;",
                             "out->mean_abs_dlogp = sum_abs / (double)n_rows;"),
    "ratio_mean_log": ("double ratio = exp(x);                 /* ratio0 */",
                       "double ratio = 1.0 + x;                 /* ratio0 */"),
    "shard_merge_rescale": ("s = (m == -INFINITY ? 0.0 : s * exp(m - mn))",
                            "s = (m == -INFINITY ? 0.0 : s * exp(mn - m))"),
    "shard_owner_offset": ("xs = logit_at(row, k->dtype, id - k->v_start);",
                           "xs = logit_at(row, k->dtype, id);"),
    "tiling_overlap_unchecked": ("if (sh[i].v_start < sh[j].v_end && sh[j].v_start < sh[i].v_end)",
                                 "if (0)"),
    "head_transposed": ("const uint16_t *w = W + (size_t)v * (size_t)hidden;",
                        "const uint16_t *w = W + (size_t)v;"),
    "oob_unchecked": ("    if (id < 0 || id >= vocab) {\n        *logp_out = NAN;\n        return LPDO_STATUS_TOKEN_OOB;\n    }\n    double m, s;",
                      "    double m, s;"),
    "chain_scale_divides": ("x = x * p;", "x = x / p;"),
    "chain_softcap_no_outer": ("x = p * tanh(x / p);", "x = tanh(x / p);"),
    "chain_reversed": ("for (int k = 0; k < c->n_ops; ++k) {\n        double p = (double)c->param[k];",
                       "for (int k = c->n_ops - 1; k >= 0; --k) {\n        double p = (double)c->param[k];"),
    "chain_skips_selected": ("double xs = apply_chain(c, logit_at(row, dtype, id));",
                             "double xs = logit_at(row, dtype, id);"),
    "chain_wrong_side": ("token_ids[r], rollout_chain, &logp_rollout[r]);", "token_ids[r], train_chain, &logp_rollout[r]);"),
    "entropy_sign": ("    return lse - px;\n}", "    return px - lse;\n}"),
    "entropy_drops_lse": ("    return lse - px;\n}", "    return -px;\n}"),
    "backward_onehot_dropped": ("out[j] = grad * ((j == id ? 1.0 : 0.0) - p);", "out[j] = grad * (0.0 - p);"),
    "backward_sign": ("out[j] = grad * ((j == id ? 1.0 : 0.0) - p);", "out[j] = grad * (p - (j == id ? 1.0 : 0.0));"),
    "attn_weight_sign": ("double w = exp(l - lse);", "double w = exp(lse - l);"),
    "attn_base2_unconverted": ("            if (lse_base2)\n                l *= ln2;\n            double w", "            double w"),
    "attn_masked_part_read": ("            if (l == -INFINITY)\n                continue;\n            if (lse_base2)\n                l *= ln2;\n            double w",
                              "            if (lse_base2)\n                l *= ln2;\n            double w"),
    "drift_ties_high": ("    return diff > best;\n}", "    return diff >= best;\n}"),
    "drift_mask_ignored": ("        if (!mask[r])\n            continue;\n        double dt", "        double dt"),
    "drift_nan_ignored": ("    if (isnan(diff))\n        return 1;", "    if (isnan(diff))\n        return 0;"),
    "drift_frac_denominator": ("(double)out->n_differ / (double)out->n_active", "(double)out->n_differ / (double)n_rows"),
    "drift_one_side": ("if (!same_number(a_t[r], b_t[r]) || !same_number(a_r[r], b_r[r]))",
                       "if (!same_number(a_t[r], b_t[r]))"),
    "drift_nan_pairs_differ": ("    if (isnan(a) && isnan(b))\n        return 1;", "    if (isnan(a) && isnan(b))\n        return 0;"),
    "nonfinite_unflagged": ("return (isfinite(lse) && isfinite(xs)) ? 0u : LPDO_STATUS_NONFINITE;\n}\n\nstatic int",
                            "return 0u;\n}\n\nstatic int"),
}


_CHILD = """
import sys
sys.path.insert(0, sys.argv[1])
import oracle
from tests.oracle_pins import ALL_PINS
lib = oracle.load(sys.argv[2])
failed = []
for name, pin in ALL_PINS.items():
    try:
        pin(lib)
    except Exception:
        failed.append(name)
print("FAILED:" + ",".join(failed))
"""


def _run_pins_in_child(lib_path):
    """Run every pin against the library at lib_path in a fresh process, so a
    mutant that reads out of bounds and crashes (or hangs) cannot take the test
    run down.  Returns (crashed_or_hung, failed pin names)."""
    root = str(Path(__file__).resolve().parent.parent)
    try:
        proc = subprocess.run([sys.executable, "-c", _CHILD, root, str(lib_path)],
                              capture_output=True, text=True, timeout=60)
    except subprocess.TimeoutExpired:  # a mutant that corrupts memory may hang instead of crashing
        return True, []
    if proc.returncode < 0:  # killed by a signal (e.g. an out-of-bounds read)
        return True, []
    assert proc.returncode == 0, proc.stderr[-2000:]
    line = [ln for ln in proc.stdout.splitlines() if ln.startswith("FAILED:")][-1]
    return False, [n for n in line[len("FAILED:"):].split(",") if n]


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tmp_path):
    src = oracle.SOURCE.read_text()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1, f"mutation site for {mutant} not found"
    mutated = tmp_path / "lpd_oracle_mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib_path = oracle.compile_oracle(mutated, tmp_path / "liblpd_oracle_mutant.so")
    crashed, failed = _run_pins_in_child(lib_path)
    assert crashed or failed, f"mutant {mutant!r} passed every pin"


def test_unmutated_oracle_passes_in_child(tmp_path):
    crashed, failed = _run_pins_in_child(oracle.compile_oracle())
    assert not crashed and not failed, failed
