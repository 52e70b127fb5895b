"""The C ABI without a GPU: the library loads, exports every symbol that
include/lpd.h declares, and rejects invalid arguments on the host with the
documented codes before launching anything."""
import ctypes
import re
from pathlib import Path

import pytest

from logprob_drift_scoring_gb300 import binding as B

HEADER = Path(__file__).resolve().parent.parent / "include" / "lpd.h"


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(lpd_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    names = declared_functions()
    assert set(names) == set(B.EXPORTED), names
    for name in names:
        assert hasattr(lib, name), name


def test_struct_sizes_match_header_layout():
    assert ctypes.sizeof(B.LpdLogits) == 24
    assert ctypes.sizeof(B.LpdShard) == 40
    assert ctypes.sizeof(B.LpdMetrics) == 80
    assert ctypes.sizeof(B.LpdBackendInfo) == 32 + 48 + 16 + 32 + 16 + 96
    assert ctypes.sizeof(B.LpdMergeDrift) == 48
    assert ctypes.sizeof(B.LpdLogpDrift) == 7 * 8 + 32


def test_backend_info():
    info = B.lpd_backend_info()
    assert info["backend_id"] == "lpd.sm103a.v1"
    assert info["op_name"] == "selected_logprob_drift"
    assert info["arch"] == "sm_103a"
    assert info["deterministic"] == 1 and info["batch_invariant"] == 1
    assert info["fast_math"] == 0 and info["has_fallback"] == 0
    assert "nvcc" in info["fingerprint"]


def test_strerror_covers_every_code():
    header = (Path(__file__).resolve().parents[1] / "include" / "lpd.h").read_text()
    codes = [int(c) for c in re.findall(r"#define LPD_ERR_\w+ \((-\d+)\)", header)]
    assert len(codes) >= 12 and len(set(codes)) == len(codes)
    for code in [0] + codes:
        assert B.lpd_strerror(code) != "unknown code", code
    for bit in (B.LPD_STATUS_TOKEN_OOB, B.LPD_STATUS_NONFINITE, B.LPD_STATUS_TIMEOUT):
        assert B.lpd_strerror(bit).startswith("status")
    assert B.lpd_strerror(12345) == "unknown code"


def test_workspace_size():
    small = B.lpd_workspace_size(B.LPD_KIND_SCORE, 10)
    big = B.lpd_workspace_size(B.LPD_KIND_SCORE, 100000)
    assert 0 < small < big and small % 256 == 0 and big % 256 == 0
    assert B.lpd_workspace_size(B.LPD_KIND_SCORE, 0) > 0
    assert B.lpd_workspace_size(B.LPD_KIND_SCORE, -1) == 0
    assert B.lpd_workspace_size(B.LPD_KIND_SHARDED, 100, 1000, 4) > B.lpd_workspace_size(B.LPD_KIND_SCORE, 100)
    assert B.lpd_workspace_size(B.LPD_KIND_SHARDED, 100, 1000, 0) == 0
    assert B.lpd_workspace_size(B.LPD_KIND_SHARDED, 100, 1000, 17) == 0
    assert B.lpd_workspace_size(99, 100) == 0


# Fake device addresses: validation must reject these calls before any launch.
FAKE = 0x7F0000000000
WS_OK = FAKE + 0x100000


def _call_score(t=None, r=None, n_rows=8, vocab=16, ids=FAKE, mask=FAKE, lo=0.8, hi=1.2, met=FAKE,
                ws=WS_OK, ws_bytes=1 << 20):
    lib = B.lib()
    t = t if t is not None else B.LpdLogits(FAKE, B.LPD_BF16, 0, vocab)
    r = r if r is not None else B.LpdLogits(FAKE, B.LPD_F32, 0, vocab)
    return lib.lpd_score(ctypes.byref(t) if t != "null" else None, ctypes.byref(r), n_rows, vocab, ids, mask,
                         lo, hi, None, None, None, met, ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(t="null"), B.LPD_ERR_NULL_POINTER),
    (dict(t=B.LpdLogits(None, B.LPD_BF16, 0, 16)), B.LPD_ERR_NULL_POINTER),
    (dict(ids=None), B.LPD_ERR_NULL_POINTER),
    (dict(mask=None), B.LPD_ERR_NULL_POINTER),
    (dict(met=None), B.LPD_ERR_NULL_POINTER),
    (dict(n_rows=-1), B.LPD_ERR_BAD_SIZE),
    (dict(vocab=0), B.LPD_ERR_BAD_SIZE),
    (dict(vocab=1 << 31), B.LPD_ERR_UNSUPPORTED),
    (dict(t=B.LpdLogits(FAKE, 7, 0, 16)), B.LPD_ERR_BAD_DTYPE),
    (dict(r=B.LpdLogits(FAKE, B.LPD_F32, 0, 15)), B.LPD_ERR_BAD_STRIDE),
    (dict(t=B.LpdLogits(FAKE + 1, B.LPD_BF16, 0, 16)), B.LPD_ERR_ALIGNMENT),
    (dict(r=B.LpdLogits(FAKE + 2, B.LPD_F32, 0, 16)), B.LPD_ERR_ALIGNMENT),
    (dict(lo=1.3, hi=1.2), B.LPD_ERR_BAD_CLIP),
    (dict(lo=0.0), B.LPD_ERR_BAD_CLIP),
    (dict(lo=-0.5), B.LPD_ERR_BAD_CLIP),
    (dict(hi=float("inf")), B.LPD_ERR_BAD_CLIP),
    (dict(lo=float("nan")), B.LPD_ERR_BAD_CLIP),
    (dict(ws=None), B.LPD_ERR_WORKSPACE),
    (dict(ws_bytes=16), B.LPD_ERR_WORKSPACE),
    (dict(ws=WS_OK + 8), B.LPD_ERR_ALIGNMENT),
])
def test_score_rejects_invalid_arguments(kwargs, code):
    assert _call_score(**kwargs) == code


def _call_sharded(shards_t, shards_r, vocab=100, perm=None, n_rows=4):
    lib = B.lib()
    n = len(shards_t)
    ts = (B.LpdShard * n)(*shards_t)
    rs = (B.LpdShard * n)(*shards_r)
    p = (ctypes.c_int32 * n)(*perm) if perm is not None else None
    return lib.lpd_score_sharded(ts, rs, n, n_rows, vocab, FAKE, FAKE, 0.8, 1.2, p, None, None, None, None, None,
                                 FAKE, WS_OK, 1 << 24, None)


def _sh(v0, v1, dtype=B.LPD_BF16, stride=None):
    return B.LpdShard(FAKE, dtype, 0, stride if stride is not None else v1 - v0, v0, v1)


@pytest.mark.parametrize("t,r,perm,code", [
    ([_sh(0, 50), _sh(51, 100)], [_sh(0, 50), _sh(51, 100)], None, B.LPD_ERR_BAD_SHARDS),        # gap
    ([_sh(0, 51), _sh(50, 100)], [_sh(0, 51), _sh(50, 100)], None, B.LPD_ERR_BAD_SHARDS),        # overlap
    ([_sh(0, 50), _sh(25, 75)], [_sh(0, 50), _sh(25, 75)], None, B.LPD_ERR_BAD_SHARDS),          # overlap hides gap
    ([_sh(0, 50), _sh(50, 101)], [_sh(0, 50), _sh(50, 101)], None, B.LPD_ERR_BAD_SHARDS),        # past vocab
    ([_sh(0, 50)], [_sh(0, 50)], None, B.LPD_ERR_BAD_SHARDS),                                   # short
    ([_sh(0, 50), _sh(50, 100)], [_sh(0, 40), _sh(40, 100)], None, B.LPD_ERR_BAD_SHARDS),        # sides differ
    ([_sh(0, 50), _sh(50, 100, B.LPD_F32)], [_sh(0, 50), _sh(50, 100)], None, B.LPD_ERR_BAD_DTYPE),
    ([_sh(0, 50), _sh(50, 100, stride=49)], [_sh(0, 50), _sh(50, 100)], None, B.LPD_ERR_BAD_STRIDE),
    ([_sh(0, 50), _sh(50, 100)], [_sh(0, 50), _sh(50, 100)], [0, 0], B.LPD_ERR_BAD_SHARDS),      # not a permutation
    ([_sh(0, 50), _sh(50, 100)], [_sh(0, 50), _sh(50, 100)], [0, 2], B.LPD_ERR_BAD_SHARDS),
])
def test_sharded_rejects_bad_maps(t, r, perm, code):
    assert _call_sharded(t, r, perm=perm) == code


def test_sharded_shard_count_limits():
    assert _call_sharded([], [], vocab=100) == B.LPD_ERR_UNSUPPORTED
    many = [_sh(k, k + 1) for k in range(17)]
    assert _call_sharded(many, many, vocab=17) == B.LPD_ERR_UNSUPPORTED


def test_stage_entry_points_validate():
    lib = B.lib()
    assert lib.lpd_select_active(-1, FAKE, FAKE, None, None, None, FAKE, WS_OK, 1 << 20, None) == B.LPD_ERR_BAD_SIZE
    assert lib.lpd_select_active(4, None, FAKE, None, None, None, FAKE, WS_OK, 1 << 20, None) == B.LPD_ERR_NULL_POINTER
    assert lib.lpd_drift_metrics(4, 1.0, 0.5, FAKE, WS_OK, 1 << 20, None) == B.LPD_ERR_BAD_CLIP
    assert lib.lpd_drift_metrics(4, 0.8, 1.2, None, WS_OK, 1 << 20, None) == B.LPD_ERR_NULL_POINTER
    t = B.LpdLogits(FAKE, B.LPD_BF16, 0, 10)
    assert lib.lpd_token_logp(ctypes.byref(t), ctypes.byref(t), 4, 11, None, None, None, FAKE, WS_OK, 1 << 20,
                              None) == B.LPD_ERR_BAD_STRIDE


def _call_fused(ht=FAKE, hr=FAKE, W=FAKE, n_rows=8, hidden=128, vocab=100, ws=WS_OK, ws_bytes=1 << 30, lo=0.8):
    return B.lib().lpd_score_fused(ht, hr, W, n_rows, hidden, vocab, FAKE, FAKE, lo, 1.2, None, None, None, FAKE,
                                   ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(hidden=0), B.LPD_ERR_BAD_SIZE),
    (dict(hidden=100), B.LPD_ERR_ALIGNMENT),
    (dict(ht=FAKE + 8), B.LPD_ERR_ALIGNMENT),
    (dict(W=FAKE + 2), B.LPD_ERR_ALIGNMENT),
    (dict(W=None), B.LPD_ERR_NULL_POINTER),
    (dict(hr=None), B.LPD_ERR_NULL_POINTER),
    (dict(vocab=0), B.LPD_ERR_BAD_SIZE),
    (dict(n_rows=-3), B.LPD_ERR_BAD_SIZE),
    (dict(lo=-1.0), B.LPD_ERR_BAD_CLIP),
    (dict(ws_bytes=1024), B.LPD_ERR_WORKSPACE),
])
def test_fused_rejects_invalid_arguments(kwargs, code):
    assert _call_fused(**kwargs) == code


def test_fused_workspace_size():
    assert B.lpd_fused_workspace_size(100, 100, 1000) == 0          # hidden not a multiple of 64
    small = B.lpd_fused_workspace_size(100, 128, 1000)
    assert small > 0 and small % 256 == 0
    # dense hidden copies dominate: 2 sides x 128 padded rows x 4096 x 2 B
    assert B.lpd_fused_workspace_size(128, 4096, 1000) >= 2 * 128 * 4096 * 2


BAD_CHAINS = [
    [(3, 1.0)],                      # unknown kind
    [(B.LPD_OP_SCALE, 0.0)],         # non-positive
    [(B.LPD_OP_SCALE, -2.0)],
    [(B.LPD_OP_SOFTCAP, float("inf"))],
    [(B.LPD_OP_SOFTCAP, float("nan"))],
]


@pytest.mark.parametrize("ops", BAD_CHAINS)
def test_transform_chain_rejected(ops):
    t = B.LpdLogits(FAKE, B.LPD_BF16, 0, 16)
    c = B.transform_struct(ops)
    rc = B.lib().lpd_score_transformed(ctypes.byref(t), ctypes.byref(t), None, ctypes.byref(c), 8, 16, FAKE, FAKE,
                                       0.8, 1.2, None, None, None, FAKE, WS_OK, 1 << 20, None)
    assert rc == B.LPD_ERR_BAD_TRANSFORM


@pytest.mark.parametrize("ops", BAD_CHAINS)
def test_fused_transform_chain_rejected(ops):
    c = B.transform_struct(ops)
    lib = B.lib()
    rc = lib.lpd_score_fused_transformed(FAKE, FAKE, FAKE, ctypes.byref(c), None, 8, 128, 100, FAKE, FAKE, 0.8, 1.2,
                                         None, None, None, FAKE, WS_OK, 1 << 30, None)
    assert rc == B.LPD_ERR_BAD_TRANSFORM
    # the fused-path argument checks still come first for the transformed entry
    rc = lib.lpd_score_fused_transformed(FAKE, FAKE, FAKE, ctypes.byref(c), None, 8, 100, 100, FAKE, FAKE, 0.8, 1.2,
                                         None, None, None, FAKE, WS_OK, 1 << 30, None)
    assert rc == B.LPD_ERR_ALIGNMENT


def test_transform_chain_too_long():
    t = B.LpdLogits(FAKE, B.LPD_BF16, 0, 16)
    c = B.transform_struct([(B.LPD_OP_SCALE, 1.0)] * 4)
    c.n_ops = 5
    rc = B.lib().lpd_score_transformed(ctypes.byref(t), ctypes.byref(t), ctypes.byref(c), None, 8, 16, FAKE, FAKE,
                                       0.8, 1.2, None, None, None, FAKE, WS_OK, 1 << 20, None)
    assert rc == B.LPD_ERR_BAD_TRANSFORM


def test_entropy_and_backward_validation():
    lib = B.lib()
    t = B.LpdLogits(FAKE, B.LPD_BF16, 0, 16)
    assert lib.lpd_score_entropy(ctypes.byref(t), ctypes.byref(t), 8, 16, FAKE, FAKE, 0.8, 1.2, None, None, None,
                                 None, None, FAKE, WS_OK, 1 << 20, None) == B.LPD_ERR_NULL_POINTER
    args = dict(n=8, v=16, ids=FAKE, mask=FAKE, logp=FAKE, grad=FAKE, out=FAKE, dt=B.LPD_F32, stride=16)

    def call(**kw):
        a = {**args, **kw}
        return lib.lpd_logprob_backward(ctypes.byref(t), a["n"], a["v"], a["ids"], a["mask"], a["logp"], a["grad"],
                                        a["out"], a["dt"], a["stride"], None)
    assert call(out=None) == B.LPD_ERR_NULL_POINTER
    assert call(grad=None) == B.LPD_ERR_NULL_POINTER
    assert call(dt=5) == B.LPD_ERR_BAD_DTYPE
    assert call(stride=15) == B.LPD_ERR_BAD_STRIDE
    assert call(out=FAKE + 2) == B.LPD_ERR_ALIGNMENT
    assert call(v=0) == B.LPD_ERR_BAD_SIZE


def _call_merge(parts=FAKE, dtype=B.LPD_F32, lse=FAKE, K=4, n=8, d=128, base2=0, order_a=None, order_b=None,
                out=FAKE, out_lse=FAKE, rdo=FAKE, rdl=FAKE, drift=FAKE, diag=True):
    lib = B.lib()
    oa = None if order_a is None else (ctypes.c_int32 * len(order_a))(*order_a)
    ob = None if order_b is None else (ctypes.c_int32 * len(order_b))(*order_b)
    if diag:
        return lib.lpd_attn_merge_order_drift(parts, dtype, lse, K, n, d, base2, oa, ob, out, out_lse, rdo, rdl,
                                              drift, None)
    return lib.lpd_attn_merge(parts, dtype, lse, K, n, d, base2, oa, out, out_lse, None)


@pytest.mark.parametrize("diag", [False, True])
@pytest.mark.parametrize("kwargs,code", [
    (dict(n=-1), B.LPD_ERR_BAD_SIZE),
    (dict(n=0xFFFFFFFF), B.LPD_ERR_BAD_SIZE),
    (dict(d=0), B.LPD_ERR_BAD_SIZE),
    (dict(base2=2), B.LPD_ERR_BAD_SIZE),
    (dict(K=0), B.LPD_ERR_UNSUPPORTED),
    (dict(K=B.LPD_ATTN_MAX_PARTS + 1), B.LPD_ERR_UNSUPPORTED),
    (dict(n=1 << 30, d=64), B.LPD_ERR_UNSUPPORTED),           # 2^34 chunks in one part
    (dict(dtype=7), B.LPD_ERR_BAD_DTYPE),
    (dict(parts=None), B.LPD_ERR_NULL_POINTER),
    (dict(lse=None), B.LPD_ERR_NULL_POINTER),
    (dict(out=None), B.LPD_ERR_NULL_POINTER),
    (dict(out_lse=None), B.LPD_ERR_NULL_POINTER),
    (dict(d=6), B.LPD_ERR_ALIGNMENT),                       # 24-byte rows
    (dict(dtype=B.LPD_BF16, d=12), B.LPD_ERR_ALIGNMENT),    # 24-byte rows
    (dict(parts=FAKE + 8), B.LPD_ERR_ALIGNMENT),
    (dict(out=FAKE + 4), B.LPD_ERR_ALIGNMENT),
    (dict(lse=FAKE + 2), B.LPD_ERR_ALIGNMENT),
    (dict(order_a=[0, 1, 1, 3]), B.LPD_ERR_BAD_SHARDS),
    (dict(order_a=[0, 1, 2, 4]), B.LPD_ERR_BAD_SHARDS),
    (dict(order_a=[0, 1, 2, -1]), B.LPD_ERR_BAD_SHARDS),
])
def test_attn_merge_rejects_invalid_arguments(kwargs, code, diag):
    assert _call_merge(diag=diag, **kwargs) == code


@pytest.mark.parametrize("kwargs,code", [
    (dict(drift=None), B.LPD_ERR_NULL_POINTER),
    (dict(drift=None, n=0), B.LPD_ERR_NULL_POINTER),
    (dict(rdo=None), B.LPD_ERR_NULL_POINTER),
    (dict(rdl=None), B.LPD_ERR_NULL_POINTER),
    (dict(rdo=FAKE + 2), B.LPD_ERR_ALIGNMENT),
    (dict(drift=FAKE + 4), B.LPD_ERR_ALIGNMENT),
    (dict(order_b=[3, 2, 2, 0]), B.LPD_ERR_BAD_SHARDS),
])
def test_attn_merge_drift_rejects_invalid_arguments(kwargs, code):
    assert _call_merge(**kwargs) == code


def test_attn_merge_binding_checks_shapes():
    torch = pytest.importorskip("torch")
    parts = torch.zeros((2, 3, 8))
    with pytest.raises(ValueError):
        B.attn_merge(parts, torch.zeros((3, 2)))
    with pytest.raises(ValueError):
        B.attn_merge(parts, torch.zeros((2, 3)), order=[0])


def _call_topology(shards_t, shards_r, topology=B.LPD_TOPO_ALLREDUCE_PARTIALS, order=None, n_rows=8, vocab=100,
                   ws=WS_OK, ws_bytes=1 << 24):
    lib = B.lib()
    n = len(shards_t)
    ts = (B.LpdShard * n)(*shards_t)
    rs = (B.LpdShard * n)(*shards_r)
    o = (ctypes.c_int32 * len(order))(*order) if order is not None else None
    return lib.lpd_score_sharded_topology(ts, rs, n, n_rows, vocab, FAKE, FAKE, 0.8, 1.2, topology, o, None, None,
                                          None, FAKE, ws, ws_bytes, None)


@pytest.mark.parametrize("topology", [0, 1, 2])
@pytest.mark.parametrize("t,r,order,code", [
    ([_sh(0, 50), _sh(51, 100)], [_sh(0, 50), _sh(51, 100)], None, B.LPD_ERR_BAD_SHARDS),        # gap
    ([_sh(0, 50), _sh(50, 100)], [_sh(0, 40), _sh(40, 100)], None, B.LPD_ERR_BAD_SHARDS),        # sides differ
    ([_sh(0, 50), _sh(50, 100, B.LPD_F32)], [_sh(0, 50), _sh(50, 100)], None, B.LPD_ERR_BAD_DTYPE),
    ([_sh(0, 50), _sh(50, 100, stride=49)], [_sh(0, 50), _sh(50, 100)], None, B.LPD_ERR_BAD_STRIDE),
])
def test_topology_rejects_bad_maps(t, r, order, code, topology):
    assert _call_topology(t, r, topology, order) == code


def test_topology_rejects_bad_order_topology_and_workspace():
    t = [_sh(0, 50), _sh(50, 100)]
    for topo in (0, 1):
        assert _call_topology(t, t, topo, [1, 1]) == B.LPD_ERR_BAD_SHARDS
        assert _call_topology(t, t, topo, [0, 2]) == B.LPD_ERR_BAD_SHARDS
    assert _call_topology(t, t, 3) == B.LPD_ERR_UNSUPPORTED
    assert _call_topology(t, t, -1) == B.LPD_ERR_UNSUPPORTED
    need = B.lpd_topology_workspace_size(2, 8, 100, 2, B.LPD_BF16, B.LPD_BF16)
    assert _call_topology(t, t, 2, ws_bytes=need - 1) == B.LPD_ERR_WORKSPACE
    assert _call_topology(t, t, 1, ws=WS_OK + 8) == B.LPD_ERR_ALIGNMENT     # not 256-byte aligned


def test_topology_workspace_size():
    part = B.lpd_topology_workspace_size(B.LPD_TOPO_ALLREDUCE_PARTIALS, 100, 1000, 4, B.LPD_BF16, B.LPD_BF16)
    assert part == B.lpd_workspace_size(B.LPD_KIND_SHARDED, 100, 1000, 4)
    assert B.lpd_topology_workspace_size(0, 100, 1000, 4, B.LPD_BF16, B.LPD_F32) == part
    gather = B.lpd_topology_workspace_size(B.LPD_TOPO_ALLGATHER_LOGITS, 100, 1000, 4, B.LPD_BF16, B.LPD_F32)
    # both sides' rows (padded to 16 bytes) on top of a single-segment scoring workspace
    assert gather >= B.lpd_workspace_size(B.LPD_KIND_SCORE, 100) + 100 * 2000 + 100 * 4000
    assert gather % 256 == 0
    assert B.lpd_topology_workspace_size(5, 100, 1000, 4, B.LPD_BF16, B.LPD_BF16) == 0
    assert B.lpd_topology_workspace_size(0, 100, 1000, 0, B.LPD_BF16, B.LPD_BF16) == 0
    assert B.lpd_topology_workspace_size(0, 100, 1000, 4, 9, B.LPD_BF16) == 0


@pytest.mark.parametrize("kwargs,code", [
    (dict(n=-1), B.LPD_ERR_BAD_SIZE),
    (dict(d=None), B.LPD_ERR_NULL_POINTER),
    (dict(m=None), B.LPD_ERR_NULL_POINTER),
    (dict(met=None), B.LPD_ERR_NULL_POINTER),
    (dict(lo=1.3), B.LPD_ERR_BAD_CLIP),
    (dict(ws=None), B.LPD_ERR_WORKSPACE),
    (dict(ws_bytes=16), B.LPD_ERR_WORKSPACE),
])
def test_metrics_from_dlogp_validation(kwargs, code):
    a = dict(n=8, d=FAKE, m=FAKE, lo=0.8, hi=1.2, met=FAKE, ws=WS_OK, ws_bytes=1 << 20)
    a.update(kwargs)
    rc = B.lib().lpd_drift_metrics_from_dlogp(a["n"], a["d"], a["m"], a["lo"], a["hi"], a["met"], a["ws"],
                                              a["ws_bytes"], None)
    assert rc == code


def _call_host(th=None, rh=None, td=None, rd=None, n_rows=8, vocab=16, ids_dev=FAKE, lo=0.8, ws_bytes=1 << 20):
    t = B.LpdLogits(FAKE, B.LPD_BF16, 0, 16)
    th, rh, td, rd = (x if x is not None else t for x in (th, rh, td, rd))
    copied = ctypes.c_int64(-1)
    rc = B.lib().lpd_score_host(ctypes.byref(th), ctypes.byref(rh), ctypes.byref(td), ctypes.byref(rd), n_rows,
                                vocab, FAKE, FAKE, ids_dev, FAKE, lo, 1.2, None, None, None, FAKE, WS_OK, ws_bytes,
                                ctypes.byref(copied), None)
    return rc, copied.value


@pytest.mark.parametrize("kwargs,code", [
    (dict(td=B.LpdLogits(FAKE, B.LPD_F32, 0, 16)), B.LPD_ERR_BAD_DTYPE),        # device dtype != host dtype
    (dict(rh=B.LpdLogits(FAKE, B.LPD_F32, 0, 16)), B.LPD_ERR_BAD_DTYPE),
    (dict(rd=B.LpdLogits(FAKE, B.LPD_BF16, 0, 15)), B.LPD_ERR_BAD_STRIDE),      # staging row shorter than vocab
    (dict(th=B.LpdLogits(None, B.LPD_BF16, 0, 16)), B.LPD_ERR_NULL_POINTER),
    (dict(ids_dev=None), B.LPD_ERR_NULL_POINTER),
    (dict(lo=2.0), B.LPD_ERR_BAD_CLIP),
    (dict(ws_bytes=16), B.LPD_ERR_WORKSPACE),
    (dict(n_rows=-1), B.LPD_ERR_BAD_SIZE),
])
def test_score_host_rejects_invalid_arguments(kwargs, code):
    rc, copied = _call_host(**kwargs)
    assert rc == code
    assert copied == 0  # nothing was copied


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lpd.h"

int main(void) {
    lpd_backend_info_t info;
    lpd_logits t;
    lpd_metrics *met = (lpd_metrics *)0x1000;
    int rc;
    if (lpd_backend_info(&info) != LPD_OK || strcmp(info.backend_id, "lpd.sm103a.v1") != 0) return 1;
    if (lpd_backend_info(NULL) != LPD_ERR_NULL_POINTER) return 2;
    if (lpd_workspace_size(LPD_KIND_SCORE, 1000, 0, 0) == 0) return 3;
    memset(&t, 0, sizeof t);
    t.dtype = LPD_BF16;
    t.row_stride = 10;
    /* vocab 11 > row_stride 10: refused on the host, nothing launched */
    rc = lpd_score(&t, &t, 4, 11, NULL, NULL, 0.8, 1.2, NULL, NULL, NULL, met, NULL, 0, NULL);
    if (rc != LPD_ERR_NULL_POINTER && rc != LPD_ERR_BAD_STRIDE) return 4;
    printf("%s|%s|%d\n", info.op_name, lpd_strerror(LPD_ERR_BAD_STRIDE), (int)sizeof(lpd_metrics));
    return 0;
}
"""


@pytest.mark.parametrize("kwargs,code", [
    (dict(n=-1), B.LPD_ERR_BAD_SIZE),
    (dict(n=0xFFFFFFFF), B.LPD_ERR_UNSUPPORTED),
    (dict(at=None), B.LPD_ERR_NULL_POINTER),
    (dict(br=None), B.LPD_ERR_NULL_POINTER),
    (dict(m=None), B.LPD_ERR_NULL_POINTER),
    (dict(out=None), B.LPD_ERR_NULL_POINTER),
    (dict(n=0, out=None), B.LPD_ERR_NULL_POINTER),
    (dict(out=FAKE + 4), B.LPD_ERR_ALIGNMENT),
    (dict(bt=FAKE + 2), B.LPD_ERR_ALIGNMENT),
])
def test_logp_drift_summary_validation(kwargs, code):
    a = dict(n=8, at=FAKE, ar=FAKE, bt=FAKE, br=FAKE, m=FAKE, out=FAKE)
    a.update(kwargs)
    rc = B.lib().lpd_logp_drift_summary(a["n"], a["at"], a["ar"], a["bt"], a["br"], a["m"], a["out"], None)
    assert rc == code


def test_header_is_plain_c_and_links(tmp_path):
    """include/lpd.h compiles as strict C99 and a C program links against
    liblpd.so and calls it (host-side entry points only: no GPU needed)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from logprob_drift_scoring_gb300 import _build

    lib = _build.LIB
    src = tmp_path / "use_lpd.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "use_lpd"
    inc = Path(__file__).resolve().parents[1] / "include"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{inc}", str(src), str(lib),
           f"-Wl,-rpath,{lib.parent}", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    name, msg, size = out.stdout.strip().split("|")
    assert name == "selected_logprob_drift" and msg == B.lib().lpd_strerror(B.LPD_ERR_BAD_STRIDE).decode()
    assert int(size) == ctypes.sizeof(B.LpdMetrics)
