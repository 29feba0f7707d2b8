"""The C-ABI library on the host: it loads, exports what include/*.h declare,
and its plan validation and argument checks behave as the pages require.

No compute call is made here; every case is rejected (or answered) on the
host before the library touches a GPU, so these run on a CPU-only machine.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle_pins
from oracle import tp_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tp.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300",
                         reason="libtp.so not built (python tensor_sharded_linear_tp_gb300/build.py)")

REASON_TO_STATUS = {"OK": "TP_OK", O.INVALID_ARG: "TP_ERR_INVALID_ARG",
                    O.HEADS_NOT_DIVISIBLE: "TP_ERR_HEADS_NOT_DIVISIBLE",
                    O.SPLIT_NOT_DIVISIBLE: "TP_ERR_SPLIT_NOT_DIVISIBLE", O.SPLIT_SUM: "TP_ERR_SPLIT_SUM",
                    O.NOT_WHOLE_HEADS: "TP_ERR_NOT_WHOLE_HEADS"}


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"TP_API\s+[\w\s\*]+?\b(tp_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("tp_validate", "tp_shard_shape", "tp_plan_shard", "tp_linear_colwise", "tp_linear_rowwise",
                     "tp_rowwise_workspace_bytes", "tp_combine", "tp_last_error", "tp_device_status", "tp_st_open",
                     "tp_st_plan_shard_ranks"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tp.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"libtp.so does not export {name}"
    assert set(declared_functions()) == set(tp.EXPORTED)
    assert tp.tp_abi_version() >= 100


def test_status_names_match_header():
    text = open(HEADER).read()
    enum = re.findall(r"(TP_(?:OK|ERR_\w+))\s*=\s*(\d+)", text)
    for name, value in enum:
        assert tp.tp_status_name(int(value)) == name
        assert tp.STATUS_NAMES[int(value)] == name


def _status_of(fn, *a, **kw):
    try:
        fn(*a, **kw)
        return "TP_OK"
    except tp.TPError as e:
        return e.name


def test_validate_matches_golden_table():
    for style, r, c, p, h, d, sizes, expected in oracle_pins.read_plan_fixture():
        got = _status_of(tp.tp_validate, r, c, style, p, h, d, sizes)
        assert got == REASON_TO_STATUS[expected], (style, r, c, p, h, d, sizes, got)


def test_validate_agrees_with_oracle_on_random_plans():
    rng = np.random.default_rng(3)
    for _ in range(3000):
        style = ["colwise", "rowwise"][rng.integers(2)]
        p = int(rng.integers(-1, 10))
        h = int(rng.choice([0, 4, 6, 12, 24, 48]))
        d = int(rng.choice([0, 0, 8, 16]))
        nb = int(rng.integers(0, 5))
        sizes = [int(rng.integers(0, 7)) * int(rng.choice([1, 8, 16])) for _ in range(nb)] or None
        dim = sum(sizes) if sizes and rng.random() < 0.8 else int(rng.integers(0, 200))
        other = int(rng.integers(0, 50))
        rows, cols = (dim, other) if style == "colwise" else (other, dim)
        try:
            O.check_plan(rows, cols, style, p, num_heads=h, head_dim=d, splits=sizes)
            want = "TP_OK"
        except O.PlanRejected as e:
            want = REASON_TO_STATUS[e.reason]
        got = _status_of(tp.tp_validate, rows, cols, style, p, h, d, sizes)
        assert got == want, (style, rows, cols, p, h, d, sizes)


def test_shard_shape():
    assert tp.tp_shard_shape(9216, 3072, "colwise", 4, [3072] * 3) == (2304, 3072)
    assert tp.tp_shard_shape(3072, 3072, "rowwise", 4) == (3072, 768)
    assert tp.tp_shard_shape(36864, 6144, "colwise", 4, [18432, 18432]) == (9216, 6144)
    assert tp.tp_shard_shape(6144, 18432, "rowwise", 4) == (6144, 4608)
    assert tp.tp_shard_shape(0, 16, "colwise", 2) == (0, 16)
    with pytest.raises(tp.TPError) as e:
        tp.tp_shard_shape(10, 16, "colwise", 4)
    assert e.value.name == "TP_ERR_SPLIT_NOT_DIVISIBLE"


def test_last_error_message():
    with pytest.raises(tp.TPError) as e:
        tp.tp_validate(18432, 6144, "colwise", 5, 48, 128, [6144] * 3)
    assert e.value.name == "TP_ERR_HEADS_NOT_DIVISIBLE"
    assert "num_heads=48" in str(e.value) and "tp_degree=5" in str(e.value)
    tp.tp_validate(18432, 6144, "colwise", 4, 48, 128, [6144] * 3)
    assert tp.tp_last_error() == ""


def test_workspace_bytes():
    # p partials of T x N fp32 (rounded up to 256 B) plus one int counter per 128 x 128 output block.
    p, T, N = 4, 4096, 3072
    part = p * T * N * 4
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "workspace") == ((part + 255) // 256) * 256 + 32 * 24 * 4
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "accum") == 0
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "none") == 0
    assert tp.tp_rowwise_workspace_bytes(p, 0, N, "workspace") == 0


# --- faults injected on the host: each call must be refused before any device work --------------------

FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case below fails validation first


def _plan_shard_raw(rows, cols, style, p, rank, splits=None, heads=0, hd=0, w=FAKE, out=FAKE):
    arr, n = (None, 0) if not splits else ((ctypes.c_int64 * len(splits))(*splits), len(splits))
    return tp.STATUS_NAMES[tp.lib.tp_plan_shard(w, rows, cols, tp.STYLES[style], p, rank, arr, n, heads, hd, out,
                                                None)]


def test_plan_shard_rejects_bad_plans_before_copying():
    assert _plan_shard_raw(18432, 6144, "colwise", 5, 0, [6144] * 3, 48, 128) == "TP_ERR_HEADS_NOT_DIVISIBLE"
    assert _plan_shard_raw(18432, 6144, "colwise", 7, 0, [6144] * 3, 48, 128) == "TP_ERR_HEADS_NOT_DIVISIBLE"
    assert _plan_shard_raw(16, 8, "colwise", 2, 2) == "TP_ERR_INVALID_ARG"        # rank >= tp
    assert _plan_shard_raw(16, 8, "colwise", 2, -1) == "TP_ERR_INVALID_ARG"
    assert _plan_shard_raw(16, 8, "colwise", 0, 0) == "TP_ERR_INVALID_ARG"
    assert _plan_shard_raw(8, 16, "colwise", 2, 0, [3, 5]) == "TP_ERR_SPLIT_NOT_DIVISIBLE"
    assert _plan_shard_raw(8, 16, "colwise", 2, 0, [2, 4]) == "TP_ERR_SPLIT_SUM"
    assert _plan_shard_raw(16, 8, "colwise", 2, 0, w=0) == "TP_ERR_INVALID_ARG"   # NULL weight
    assert _plan_shard_raw(16, 8, "colwise", 2, 0, out=0) == "TP_ERR_INVALID_ARG"
    assert _plan_shard_raw(0, 8, "colwise", 2, 1, w=0, out=0) == "TP_OK"          # empty shard: nothing to do


def _shard_request(rows, cols, style, p, splits=None, heads=0, hd=0, rank_begin=0, rank_count=None, w=FAKE, keep=None):
    rc = p - rank_begin if rank_count is None else rank_count
    sp = (ctypes.c_int64 * len(splits))(*splits) if splits else None
    n_outs = min(max(1, rc), 16)   # a refused request reads none of them
    outs = (ctypes.c_void_p * n_outs)(*([FAKE] * n_outs))
    if keep is not None:
        keep += [sp, outs]
    return tp.ShardRequest(w, rows, cols, tp.STYLES[style], p, rank_begin, rc, sp, len(splits) if splits else 0,
                           heads, hd, outs)


def test_plan_shard_many_checks_every_request_first():
    keep = []
    good = _shard_request(16, 8, "colwise", 2, keep=keep)
    bad = _shard_request(18432, 6144, "colwise", 5, [6144] * 3, 48, 128, keep=keep)
    arr = (tp.ShardRequest * 3)(good, good, bad)
    st = tp.lib.tp_plan_shard_many(arr, 3, None)
    assert tp.STATUS_NAMES[st] == "TP_ERR_HEADS_NOT_DIVISIBLE"
    assert "request 2" in tp.tp_last_error()
    arr = (tp.ShardRequest * 2)(good, _shard_request(8, 16, "colwise", 2, [2, 4], keep=keep))
    assert tp.STATUS_NAMES[tp.lib.tp_plan_shard_many(arr, 2, None)] == "TP_ERR_SPLIT_SUM"
    assert tp.STATUS_NAMES[tp.lib.tp_plan_shard_many(arr, -1, None)] == "TP_ERR_INVALID_ARG"
    assert tp.STATUS_NAMES[tp.lib.tp_plan_shard_many(arr, 65, None)] == "TP_ERR_UNSUPPORTED"
    assert tp.STATUS_NAMES[tp.lib.tp_plan_shard_many(None, 2, None)] == "TP_ERR_INVALID_ARG"
    # A rank range whose end would overflow an int is refused, not wrapped around.
    huge = (tp.ShardRequest * 1)(_shard_request(16, 8, "colwise", 2, rank_begin=1, rank_count=2 ** 31 - 1,
                                                keep=keep))
    assert tp.STATUS_NAMES[tp.lib.tp_plan_shard_many(huge, 1, None)] == "TP_ERR_INVALID_ARG"
    assert tp.lib.tp_plan_shard_many(None, 0, None) == 0
    # Requests with nothing to copy pass without touching memory.
    empty = (tp.ShardRequest * 2)(_shard_request(0, 8, "colwise", 2, w=0, keep=keep),
                                  _shard_request(16, 8, "colwise", 2, rank_count=0, w=0, keep=keep))
    assert tp.lib.tp_plan_shard_many(empty, 2, None) == 0


def _colwise_raw(p=2, T=64, K=256, N_r=512, act="none", ldy=0, x=FAKE, w=FAKE, y=FAKE):
    ws = (ctypes.c_void_p * max(p, 1))(*([w] * max(p, 1)))
    ys = (ctypes.c_void_p * max(p, 1))(*([y] * max(p, 1)))
    return tp.STATUS_NAMES[tp.lib.tp_linear_colwise(x, ws, None, tp.ACTS[act], p, T, K, N_r, ys, ldy, None)]


def test_colwise_argument_checks():
    assert _colwise_raw(p=0) == "TP_ERR_INVALID_ARG"
    assert _colwise_raw(p=17) == "TP_ERR_UNSUPPORTED"
    assert _colwise_raw(K=100) == "TP_ERR_ALIGNMENT"                 # 200-byte rows are not 16-byte multiples
    assert _colwise_raw(N_r=36) == "TP_ERR_ALIGNMENT"
    assert _colwise_raw(act="swiglu", N_r=33) == "TP_ERR_INVALID_ARG"  # cannot split into gate/up halves
    assert _colwise_raw(act="swiglu", N_r=34) == "TP_ERR_ALIGNMENT"    # halves of 17 columns
    assert _colwise_raw(ldy=100) == "TP_ERR_INVALID_ARG"             # ldy below the output width
    assert _colwise_raw(x=FAKE + 8) == "TP_ERR_ALIGNMENT"
    assert _colwise_raw(x=0) == "TP_ERR_INVALID_ARG"
    assert _colwise_raw(K=0) == "TP_ERR_INVALID_ARG"
    assert _colwise_raw(T=0, x=0, w=0, y=0) == "TP_OK"               # empty: enqueues nothing
    assert _colwise_raw(T=-1) == "TP_ERR_INVALID_ARG"


def _rowwise_raw(p=2, T=64, K=512, N=256, mode="accum", ws=None, ws_bytes=0, out=FAKE, x=FAKE, w=FAKE):
    xs = (ctypes.c_void_p * max(p, 1))(*([x] * max(p, 1)))
    wsh = (ctypes.c_void_p * max(p, 1))(*([w] * max(p, 1)))
    return tp.STATUS_NAMES[tp.lib.tp_linear_rowwise(xs, wsh, None, p, T, K, N, tp.REDUCE_MODES[mode], ws, ws_bytes,
                                                    out, None)]


def test_rowwise_argument_checks():
    assert _rowwise_raw(p=0) == "TP_ERR_INVALID_ARG"
    assert _rowwise_raw(p=17) == "TP_ERR_UNSUPPORTED"
    assert _rowwise_raw(K=12) == "TP_ERR_ALIGNMENT"
    assert _rowwise_raw(N=12) == "TP_ERR_ALIGNMENT"
    assert _rowwise_raw(mode="workspace") == "TP_ERR_WORKSPACE"       # no workspace given
    need = tp.tp_rowwise_workspace_bytes(2, 64, 256, "workspace")
    assert _rowwise_raw(mode="workspace", ws=FAKE, ws_bytes=need - 1) == "TP_ERR_WORKSPACE"
    assert _rowwise_raw(out=0) == "TP_ERR_INVALID_ARG"
    assert _rowwise_raw(T=0, out=0, x=0, w=0) == "TP_OK"


def test_combine_argument_checks():
    parts = (ctypes.c_void_p * 2)(FAKE, FAKE)
    assert tp.STATUS_NAMES[tp.lib.tp_combine(7, parts, 2, 4, 8, FAKE, None)] == "TP_ERR_INVALID_ARG"
    assert tp.STATUS_NAMES[tp.lib.tp_combine(0, parts, 0, 4, 8, FAKE, None)] == "TP_ERR_INVALID_ARG"
    assert tp.STATUS_NAMES[tp.lib.tp_combine(0, parts, 17, 4, 8, FAKE, None)] == "TP_ERR_UNSUPPORTED"
    assert tp.STATUS_NAMES[tp.lib.tp_combine(0, parts, 2, 0, 8, 0, None)] == "TP_OK"
    nulls = (ctypes.c_void_p * 2)(FAKE, None)
    assert tp.STATUS_NAMES[tp.lib.tp_combine(0, nulls, 2, 4, 8, FAKE, None)] == "TP_ERR_INVALID_ARG"


def test_tile_wait_limit_round_trips_on_the_host():
    # Host-side setting only (read by later launches); 0 restores the 2 s default.
    assert tp.tp_tile_wait_limit_ns() == 2_000_000_000
    try:
        tp.tp_set_tile_wait_limit_ns(12345)
        assert tp.tp_tile_wait_limit_ns() == 12345
    finally:
        tp.tp_set_tile_wait_limit_ns(0)
    assert tp.tp_tile_wait_limit_ns() == 2_000_000_000


def test_noalloc_scratch_size_matches_the_header():
    # The binding's constant is the header's #define, not a second copy that could drift.
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "tp.h")).read()
    m = re.search(r"#define TP_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", hdr)
    assert m is not None
    assert tp.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_colwise_chunked_flag_checks():
    # TP_ACCUM_CHUNKED is accepted with TP_ACT_NONE only; other bits are not activations.
    ws = (ctypes.c_void_p * 2)(*([FAKE] * 2))
    ys = (ctypes.c_void_p * 2)(*([FAKE] * 2))
    call = lambda code: tp.STATUS_NAMES[tp.lib.tp_linear_colwise(FAKE, ws, None, code, 2, 64, 256, 512, ys, 0,  # noqa
                                                                   None)]
    assert call(tp.ACTS["gelu_tanh"] | tp.ACCUM_CHUNKED) == "TP_ERR_UNSUPPORTED"
    assert call(tp.ACTS["swiglu"] | tp.ACCUM_CHUNKED) == "TP_ERR_UNSUPPORTED"
    assert call(0x200) == "TP_ERR_INVALID_ARG"
    assert tp.ACCUM_CHUNKED == 0x100
