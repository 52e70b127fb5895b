"""The page-fixed facts under tests/golden/ against the oracle's and the
C ABI's metric records (CPU only)."""
import ctypes
import json
from pathlib import Path

import numpy as np

import oracle
from logprob_drift_scoring_gb300 import binding as B

GOLDEN = Path(__file__).resolve().parent / "golden"


def test_every_diagnostic_is_reported():
    table = json.loads((GOLDEN / "diagnostics_table.json").read_text())
    c_fields = {name for name, _ in B.LpdMetrics._fields_}
    o_fields = {name for name, _ in oracle.Metrics._fields_}
    for field in table["record_fields"]:
        assert field in c_fields and field in o_fields, field
    for metric in table["metrics"]:
        assert any(f.startswith(metric) for f in c_fields), metric


def test_metric_records_have_the_same_layout():
    assert [f for f, _ in B.LpdMetrics._fields_] == [f for f, _ in oracle.Metrics._fields_]
    assert ctypes.sizeof(B.LpdMetrics) == ctypes.sizeof(oracle.Metrics)


def test_zero_update_fixture_on_the_oracle():
    expect = json.loads((GOLDEN / "zero_update_expectation.json").read_text())["expect_when_inputs_identical"]
    rng = np.random.default_rng(3)
    x = rng.normal(0, 3, size=(20, 300)).astype(np.float32)
    ids = rng.integers(0, 300, size=20).astype(np.int32)
    res = oracle.score(x, x, ids, np.ones(20, np.uint8))
    for k, v in expect.items():
        if k != "dlogp":
            assert res.metrics[k] == v
