"""Parity of the CUDA path (through the C-ABI) with the CPU oracle.

Extraction and gathers are compared bit for bit; products of integer-valued
inputs are exact in fp32 and are compared bit for bit too; everything else is
held to the tolerance in ``tolerance.py``.  Small shapes span several 128 x 256
tiles with ragged tails; the full-size workloads are checked on a seeded
sample of token rows, which the oracle computes exactly.
"""
import numpy as np
import pytest
import torch

import tp_inputs
from oracle import tp_oracle as O
from tolerance import assert_close

pytestmark = pytest.mark.gpu

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")

DEV = "cuda"


def dev(bits):
    return tp.bf16_from_bits(bits, DEV)


def pinned(bits):
    t = tp.bf16_from_bits(bits)
    p = torch.empty(t.shape, dtype=torch.bfloat16, pin_memory=True)
    p.copy_(t)
    return p


def host_bits(t):
    torch.cuda.synchronize()
    return tp.bits_from_bf16(t)


def f64(t):
    torch.cuda.synchronize()
    return O.bf16_to_f64(tp.bits_from_bf16(t))


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    tp.tp_device_status()   # raises if any kernel gave up on a bounded wait


# ----------------------------------------------------------------------------- extraction

EXTRACT_CASES = [
    # (rows, cols, style, tp, splits, heads, head_dim)
    (96, 64, "colwise", 2, None, 0, 0),
    (18, 24, "colwise", 2, [2, 2, 2, 6, 6], 0, 0),          # [1,1,1,3,3] fused QKV+gate+up
    (48, 40, "colwise", 4, [24, 24], 0, 0),                 # gate/up [1,1]
    (3 * 96, 64, "colwise", 3, [96, 96, 96], 12, 8),        # QKV, whole heads
    (40, 96, "rowwise", 4, None, 0, 0),
    (24, 96, "rowwise", 2, [32, 64], 0, 0),                 # packed rowwise [inner, mlp_hidden]
    (33, 48, "rowwise", 3, None, 0, 0),                     # 32-byte windows of odd row counts
    (10, 20, "rowwise", 2, None, 0, 0),                     # 20-byte rows: 2-byte path
    (14, 6, "colwise", 2, None, 0, 0),                      # 12-byte rows: 2-byte path
    (0, 16, "colwise", 2, None, 0, 0),                      # empty
]


@pytest.mark.parametrize("case", EXTRACT_CASES, ids=lambda c: f"{c[2]}-{c[0]}x{c[1]}-tp{c[3]}-{c[4]}")
@pytest.mark.parametrize("source", ["device", "pinned_host"])
def test_extract_bit_exact(case, source):
    rows, cols, style, p, splits, h, d = case
    w = tp_inputs.random_bits(100, rows * 1000 + cols, (rows, cols))   # any 16-bit pattern, NaN payloads too
    src = dev(w) if source == "device" else pinned(w)
    for r in range(p):
        out = tp.tp_plan_shard(src, style, p, r, splits, h, d, device=DEV)
        exp = O.shard(w, style, p, r, splits, num_heads=h, head_dim=d)
        got = host_bits(out)
        assert got.shape == exp.shape and np.array_equal(got, exp), (case, r)


@pytest.mark.parametrize("source", ["device", "pinned_host"])
def test_extract_all_ranks_one_launch(source):
    # 3 packed blocks x 8 ranks = 24 segments in one launch; 16 blocks x 8 ranks spills past 64 segments.
    for rows, cols, style, p, splits in ((3 * 64, 48, "colwise", 8, [64, 64, 64]), (128, 24, "colwise", 8, [8] * 16),
                                         (16, 64, "rowwise", 8, [32, 32])):
        w = tp_inputs.random_bits(105, rows + cols, (rows, cols))
        src = dev(w) if source == "device" else pinned(w)
        outs = tp.tp_plan_shard_ranks(src, style, p, fused_splits=splits, device=DEV)
        for r in range(p):
            assert np.array_equal(host_bits(outs[r]), O.shard(w, style, p, r, splits)), (rows, r)
        mid = tp.tp_plan_shard_ranks(src, style, p, 2, 3, fused_splits=splits, device=DEV)
        for i in range(3):
            assert np.array_equal(host_bits(mid[i]), O.shard(w, style, p, 2 + i, splits))
    with pytest.raises(tp.TPError) as e:
        tp.tp_plan_shard_ranks(dev(w), "rowwise", 8, 6, 3, fused_splits=[32, 32], device=DEV)
    assert e.value.name == "TP_ERR_INVALID_ARG"


def test_extract_pageable_host_refused():
    w = tp.bf16_from_bits(tp_inputs.random_bits(101, 0, (16, 16)))   # ordinary (pageable) CPU tensor
    with pytest.raises(tp.TPError) as e:
        tp.tp_plan_shard(w, "colwise", 2, 0, device=DEV)
    assert e.value.name == "TP_ERR_NOT_PINNED"


@pytest.mark.parametrize("which", ["attn_qkv", "attn_out", "mlp_gate_up", "mlp_down"])
@pytest.mark.parametrize("source", ["device", "pinned_host"])
def test_extract_full_size_bit_exact(which, source):
    if which == "attn_qkv":
        shape, style, splits, h, d = (9216, 3072), "colwise", [3072] * 3, 24, 128
    elif which == "attn_out":
        shape, style, splits, h, d = (3072, 3072), "rowwise", None, 24, 128
    elif which == "mlp_gate_up":
        shape, style, splits, h, d = (36864, 6144), "colwise", [18432, 18432], 48, 0
    else:
        shape, style, splits, h, d = (6144, 18432), "rowwise", None, 48, 0
    w = tp_inputs.random_bits(102, len(which), shape)
    src = dev(w) if source == "device" else pinned(w)
    for r in range(4):
        out = tp.tp_plan_shard(src, style, 4, r, splits, h, d, device=DEV)
        assert np.array_equal(host_bits(out), O.shard(w, style, 4, r, splits, num_heads=h, head_dim=d)), r


# ----------------------------------------------------------------------------- combine

def test_gather_bit_exact():
    for p, T, n in ((4, 37, 24), (3, 5, 3), (2, 300, 512)):
        parts = [tp_inputs.random_bits(103, 10 * p + r, (T, n)) for r in range(p)]
        got = host_bits(tp.tp_combine("gather", [dev(b) for b in parts]))
        assert np.array_equal(got, O.combine_gather(parts))


def test_reduce_integer_exact_and_normal_within_tolerance():
    p, T, n = 4, 129, 200
    rng = np.random.default_rng(104)
    ints = [rng.integers(-300, 300, size=(T, n)).astype(np.float32) for _ in range(p)]
    got = host_bits(tp.tp_combine("reduce", [torch.from_numpy(a).to(DEV) for a in ints]))
    assert np.array_equal(got, O.f64_to_bf16(O.combine_reduce(ints)))
    normals = [rng.standard_normal((T, n)).astype(np.float32) for _ in range(p)]
    out = tp.tp_combine("reduce", [torch.from_numpy(a).to(DEV) for a in normals])
    assert_close(f64(out), O.combine_reduce(normals), "reduce")
    # Unaligned length: scalar tail path.
    odd = [rng.integers(-5, 5, size=(3, 7)).astype(np.float32) for _ in range(3)]
    got = host_bits(tp.tp_combine("reduce", [torch.from_numpy(a).to(DEV) for a in odd]))
    assert np.array_equal(got, O.f64_to_bf16(O.combine_reduce(odd)))


# ----------------------------------------------------------------------------- colwise GEMM

COLWISE_SHAPES = [
    # (T, K, N_r, p): several tiles with ragged tails in M, N and K.
    (300, 200, 520, 2),
    (64, 256, 512, 2),
    (129, 64, 264, 3),
    (1, 8, 8, 1),
    (517, 1032, 1040, 4),
]


@pytest.mark.parametrize("shape", COLWISE_SHAPES, ids=str)
def test_colwise_integer_bit_exact(shape):
    T, K, N_r, p = shape
    x = tp_inputs.int_bf16(110, 0, (T, K))
    w = tp_inputs.int_bf16(110, 1, (N_r * p, K))
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "none")
    ref = O.colwise_forward(x, shards, "none")
    for r in range(p):
        assert np.array_equal(host_bits(ys[r]), O.f64_to_bf16(ref[r])), r


@pytest.mark.parametrize("act", ["none", "gelu_tanh", "swiglu"])
@pytest.mark.parametrize("shape", COLWISE_SHAPES[:3] + [(1000, 512, 1024, 4)], ids=str)
def test_colwise_normal_within_tolerance(shape, act):
    T, K, N_r, p = shape
    if act == "swiglu":
        N_r = ((N_r + 15) // 16) * 16   # gate and up halves of whole 8-column groups
    x = tp_inputs.activation_bf16(111, 0, (T, K))
    w = tp_inputs.weight_bf16(111, 1, (N_r * p, K))
    splits = [N_r * p // 2] * 2 if act == "swiglu" else None
    shards = [O.shard(w, "colwise", p, r, splits) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], act)
    ref = O.colwise_forward(x, shards, act)
    for r in range(p):
        assert_close(f64(ys[r]), ref[r], f"{act} rank {r}")


def test_colwise_bias_and_gathered_output():
    T, K, N_r, p = 200, 128, 136, 3
    x = tp_inputs.activation_bf16(112, 0, (T, K))
    w = tp_inputs.weight_bf16(112, 1, (N_r * p, K))
    b = tp_inputs.weight_bf16(112, 2, (N_r * p,))
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    bsh = [np.ascontiguousarray(b[r * N_r:(r + 1) * N_r]) for r in range(p)]
    # Write every rank's slice straight into the joined [T, p*N_r] output (the AllGather fused away).
    y = torch.empty((T, p * N_r), dtype=torch.bfloat16, device=DEV)
    tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "gelu_tanh", bias_shards=[dev(v) for v in bsh],
                         y_shards=[y[:, r * N_r:] for r in range(p)], ldy=p * N_r)
    ref = O.combine_gather(O.colwise_forward(x, shards, "gelu_tanh", bsh))
    assert_close(f64(y), ref, "colwise bias gathered")
    # And the unsharded layer equals it (tp_degree=1 is the plain layer).
    y1 = tp.tp_linear_colwise(dev(x), [dev(w)], "gelu_tanh", bias_shards=[dev(b)])[0]
    assert_close(f64(y1), ref, "tp=1 plain layer")


def test_colwise_swiglu_bias():
    T, K, F, p = 130, 64, 96, 2
    x = tp_inputs.activation_bf16(113, 0, (T, K))
    w = tp_inputs.weight_bf16(113, 1, (2 * F, K))
    b = tp_inputs.weight_bf16(113, 2, (2 * F,))
    shards = [O.shard(w, "colwise", p, r, [F, F]) for r in range(p)]
    bsh = [O.shard(b[:, None], "colwise", p, r, [F, F])[:, 0].copy() for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "swiglu", bias_shards=[dev(v) for v in bsh])
    ref = O.colwise_forward(x, shards, "swiglu", bsh)
    for r in range(p):
        assert_close(f64(ys[r]), ref[r], f"swiglu bias rank {r}")


# Shapes whose wave-count heuristic picks each accumulator width (160, 192, 224, 256 columns) on
# 76 resident CTA pairs; K is small to keep them quick, values integer so the check is exact.
WIDTH_SHAPES = [(257, 64, 1600, 3), (257, 64, 1472, 4), (257, 64, 2368, 3), (257, 64, 2048, 4)]


@pytest.mark.parametrize("shape", WIDTH_SHAPES, ids=str)
def test_tile_widths_integer_bit_exact(shape):
    T, K, N, p = shape
    x = tp_inputs.int_bf16(114, 0, (T, K * p))
    w = tp_inputs.int_bf16(114, 1, (N * p, K))
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    xk = x[:, :K]
    ys = tp.tp_linear_colwise(dev(xk), [dev(s) for s in shards], "none")
    ref = O.colwise_forward(xk, shards, "none")
    for r in range(p):
        assert np.array_equal(host_bits(ys[r]), O.f64_to_bf16(ref[r])), ("colwise", r)
    # The same widths through the rowwise workspace and unfused modes (one output group per rank).
    wr = tp_inputs.int_bf16(114, 2, (N, K * p))
    xs = [O.shard(x, "rowwise", p, r) for r in range(p)]
    wsh = [O.shard(wr, "rowwise", p, r) for r in range(p)]
    exp = O.f64_to_bf16(O.rowwise_forward(xs, wsh))
    for mode in ("workspace", "none"):
        assert np.array_equal(host_bits(_rowwise_gpu(xs, wsh, mode)), exp), mode


# ----------------------------------------------------------------------------- rowwise GEMM

ROWWISE_SHAPES = [
    # (T, K_r, N, p)
    (300, 200, 520, 2),
    (64, 512, 256, 2),
    (129, 72, 264, 3),
    (517, 1032, 1040, 4),
    (33, 16, 8, 8),
]
MODES = ["accum", "workspace", "none"]


def _rowwise_gpu(xs, ws, mode, bias=None):
    out = tp.tp_linear_rowwise([dev(a) for a in xs], [dev(a) for a in ws], bias=None if bias is None else dev(bias),
                               mode=mode)
    if mode == "none":
        return tp.tp_combine("reduce", list(out))
    return out


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", ROWWISE_SHAPES, ids=str)
def test_rowwise_integer_bit_exact(shape, mode):
    T, K_r, N, p = shape
    x = tp_inputs.int_bf16(120, 0, (T, K_r * p))
    w = tp_inputs.int_bf16(120, 1, (N, K_r * p))
    xs = [O.shard(x, "rowwise", p, r) for r in range(p)]
    ws = [O.shard(w, "rowwise", p, r) for r in range(p)]
    z = _rowwise_gpu(xs, ws, mode)
    assert np.array_equal(host_bits(z), O.f64_to_bf16(O.rowwise_forward(xs, ws)))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", ROWWISE_SHAPES[:4], ids=str)
def test_rowwise_normal_within_tolerance(shape, mode):
    T, K_r, N, p = shape
    x = tp_inputs.activation_bf16(121, 0, (T, K_r * p))
    w = tp_inputs.weight_bf16(121, 1, (N, K_r * p))
    b = tp_inputs.weight_bf16(121, 2, (N,))
    xs = [O.shard(x, "rowwise", p, r) for r in range(p)]
    ws = [O.shard(w, "rowwise", p, r) for r in range(p)]
    z = _rowwise_gpu(xs, ws, mode, bias=b)
    assert_close(f64(z), O.rowwise_forward(xs, ws, b), mode)


def test_rowwise_workspace_reused_across_calls():
    # The tile counters reset themselves; a second call on the same workspace gives the same answer.
    T, K_r, N, p = 260, 64, 264, 4
    x = tp_inputs.int_bf16(122, 0, (T, K_r * p))
    w = tp_inputs.int_bf16(122, 1, (N, K_r * p))
    xs = [dev(O.shard(x, "rowwise", p, r)) for r in range(p)]
    ws = [dev(O.shard(w, "rowwise", p, r)) for r in range(p)]
    space = torch.empty(tp.tp_rowwise_workspace_bytes(p, T, N), dtype=torch.uint8, device=DEV)
    exp = O.f64_to_bf16(O.rowwise_forward([O.shard(x, "rowwise", p, r) for r in range(p)],
                                          [O.shard(w, "rowwise", p, r) for r in range(p)]))
    for _ in range(3):
        z = tp.tp_linear_rowwise(xs, ws, mode="workspace", workspace=space)
        assert np.array_equal(host_bits(z), exp)


# ----------------------------------------------------------------------------- rowwise_split_input

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(300, 1600, 520, 4), (2, 3072, 18432, 4), (129, 96, 264, 3)], ids=str)
def test_rowwise_split_input_integer_bit_exact(shape, mode):
    # (2, 3072, 18432): an AdaLN-modulation-like projection -- two timestep-embedding rows,
    # six hidden-size modulation vectors out.
    T, K, N, p = shape
    x = tp_inputs.int_bf16(160, 0, (T, K))
    w = tp_inputs.int_bf16(160, 1, (N, K))
    ws = [O.shard(w, "rowwise", p, r) for r in range(p)]
    z = tp.tp_linear_rowwise_split_input(dev(x), [dev(a) for a in ws], mode=mode)
    if mode == "none":
        z = tp.tp_combine("reduce", list(z))
    assert np.array_equal(host_bits(z), O.f64_to_bf16(O.rowwise_split_input_forward(x, ws)))


def test_rowwise_split_input_normal_with_bias_and_strided_input():
    T, K, N, p = 517, 1024, 1040, 4
    wide = tp_inputs.activation_bf16(161, 0, (T, K + 64))
    x = np.ascontiguousarray(wide[:, :K])
    w = tp_inputs.weight_bf16(161, 1, (N, K))
    b = tp_inputs.weight_bf16(161, 2, (N,))
    ws = [O.shard(w, "rowwise", p, r) for r in range(p)]
    xd = dev(wide)[:, :K]       # row stride K + 64: each rank's slice is read in place
    z = tp.tp_linear_rowwise_split_input(xd, [dev(a) for a in ws], bias=dev(b))
    assert_close(f64(z), O.rowwise_split_input_forward(x, ws, b), "split input")


def test_rowwise_split_input_rejects_indivisible_input():
    with pytest.raises(tp.TPError) as e:
        tp.tp_linear_rowwise_split_input(dev(tp_inputs.int_bf16(162, 0, (8, 100))),
                                         [dev(tp_inputs.int_bf16(162, 1, (16, 33)))] * 3)
    assert e.value.name == "TP_ERR_SPLIT_NOT_DIVISIBLE"


# ----------------------------------------------------------------------------- workloads

def _shard_all(w, style, p, splits=None, h=0, d=0):
    return [O.shard(w, style, p, r, splits, num_heads=h, head_dim=d) for r in range(p)]


def _plan_all(w_dev, rows, cols, style, p, splits=None, h=0, d=0):
    return [tp.tp_plan_shard(w_dev, style, p, r, splits, h, d, device=DEV) for r in range(p)]


def test_tiny_mlp_block():
    """Tiny MLP, tp_degree 2: colwise up-projection + GELU(tanh), rowwise down-projection, summed."""
    cfg = tp_inputs.WORKLOADS["tiny_mlp_tp2"]
    p, H, F = cfg["tp"], cfg["hidden"], cfg["ffn"]
    w_up, w_down, x = tp_inputs.tiny_mlp_inputs()
    up = _plan_all(dev(w_up), F, H, "colwise", p, h=cfg["heads"])
    down = _plan_all(dev(w_down), H, F, "rowwise", p, h=cfg["heads"])
    for r in range(p):   # extraction is bit-exact
        assert np.array_equal(host_bits(up[r]), O.shard(w_up, "colwise", p, r))
        assert np.array_equal(host_bits(down[r]), O.shard(w_down, "rowwise", p, r))
    h_ref, z_ref = O.mlp_forward(x, _shard_all(w_up, "colwise", p), _shard_all(w_down, "rowwise", p), "gelu_tanh")
    for mode in MODES:
        hs = tp.tp_linear_colwise(dev(x), up, "gelu_tanh")
        z = tp.tp_linear_rowwise(hs, down, mode=mode)
        if mode == "none":
            z = tp.tp_combine("reduce", list(z))
        assert_close(f64(z), z_ref, f"tiny mlp {mode}")
        for r in range(p):
            assert_close(f64(hs[r]), O.bf16_to_f64(h_ref[r]), "hidden")


@pytest.mark.slow
def test_attention_projections_full_size():
    """Fused QKV colwise (6 whole heads per rank) + out-projection rowwise, tp 4, at full size, sampled rows."""
    cfg = tp_inputs.WORKLOADS["attn_proj_tp4"]
    p, T, H, h, d = cfg["tp"], cfg["tokens"], cfg["hidden"], cfg["heads"], cfg["head_dim"]
    w_qkv, w_out, x, a = tp_inputs.attn_proj_inputs()
    qkv = _plan_all(dev(w_qkv), 3 * H, H, "colwise", p, [H] * 3, h, d)
    wo = _plan_all(dev(w_out), H, H, "rowwise", p, None, h, d)
    a_sh = [dev(O.shard(a, "rowwise", p, r)) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), qkv, "none")
    rows = tp_inputs.sample_rows(cfg["seed"], T, 256)
    qkv_ref = O.colwise_forward(x[rows], _shard_all(w_qkv, "colwise", p, [H] * 3, h, d), "none")
    for r in range(p):
        assert_close(f64(ys[r])[rows], qkv_ref[r], f"qkv rank {r}")
    z_ref = O.rowwise_forward([O.shard(a[rows], "rowwise", p, r) for r in range(p)], _shard_all(w_out, "rowwise", p))
    for mode in MODES:
        z = tp.tp_linear_rowwise(a_sh, wo, mode=mode)
        if mode == "none":
            z = tp.tp_combine("reduce", list(z))
        assert_close(f64(z)[rows], z_ref, f"out-proj {mode}")


@pytest.mark.slow
def test_swiglu_mlp_full_size():
    """Fused gate/up colwise with SwiGLU + down rowwise, tp 4, full size, sampled rows."""
    cfg = tp_inputs.WORKLOADS["swiglu_mlp_tp4"]
    p, T, H, F = cfg["tp"], cfg["tokens"], cfg["hidden"], cfg["ffn"]
    w_gu, w_down, x = tp_inputs.swiglu_mlp_inputs()
    gu = _plan_all(dev(w_gu), 2 * F, H, "colwise", p, [F, F], cfg["heads"], 0)
    dn = _plan_all(dev(w_down), H, F, "rowwise", p, None, cfg["heads"], 0)
    hs = tp.tp_linear_colwise(dev(x), gu, "swiglu")
    z = tp.tp_linear_rowwise(hs, dn, mode="accum")
    rows = tp_inputs.sample_rows(cfg["seed"], T, 128)
    h_ref, z_ref = O.mlp_forward(x[rows], _shard_all(w_gu, "colwise", p, [F, F]), _shard_all(w_down, "rowwise", p),
                                 "swiglu")
    for r in range(p):
        assert_close(f64(hs[r])[rows], O.bf16_to_f64(h_ref[r]), f"h rank {r}")
    assert_close(f64(z)[rows], z_ref, "swiglu mlp out")


def test_plan_shard_many_equals_the_single_calls():
    # The attention projections' two weights and a page-locked SwiGLU weight in one call: the
    # device sources share one launch, the host source gets its own; every shard is bit-exact.
    H, heads, d, F, p = 768, 6, 128, 1152, 3
    w_qkv = tp_inputs.random_bits(90, 0, (3 * H, H))
    w_out = tp_inputs.random_bits(90, 1, (H, H))
    w_gu = tp_inputs.random_bits(90, 2, (2 * F, H))
    gu_pin = torch.empty(w_gu.shape, dtype=torch.bfloat16, pin_memory=True)
    gu_pin.copy_(tp.bf16_from_bits(w_gu))
    got = tp.tp_plan_shard_many([
        dict(weight=tp.bf16_from_bits(w_qkv, DEV), style="colwise", tp_degree=p, fused_splits=[H] * 3,
             num_heads=heads, head_dim=d),
        dict(weight=tp.bf16_from_bits(w_out, DEV), style="rowwise", tp_degree=p, num_heads=heads, head_dim=d),
        dict(weight=gu_pin, style="colwise", tp_degree=p, rank_begin=1, rank_count=2, fused_splits=[F, F]),
    ], device=DEV)
    torch.cuda.synchronize()
    for r in range(p):
        assert np.array_equal(tp.bits_from_bf16(got[0][r]), O.shard(w_qkv, "colwise", p, r, [H] * 3))
        assert np.array_equal(tp.bits_from_bf16(got[1][r]), O.shard(w_out, "rowwise", p, r))
    for i, r in enumerate((1, 2)):
        assert np.array_equal(tp.bits_from_bf16(got[2][i]), O.shard(w_gu, "colwise", p, r, [F, F]))


def test_plan_shard_many_refusal_touches_nothing():
    H, p = 256, 2
    w = tp.bf16_from_bits(tp_inputs.random_bits(91, 0, (H, H)), DEV)
    outs = [torch.full((H // p, H), 7, dtype=torch.int16, device=DEV).view(torch.bfloat16) for _ in range(p)]
    with pytest.raises(tp.TPError) as e:
        tp.tp_plan_shard_many([dict(weight=w, style="colwise", tp_degree=p, outs=outs),
                               dict(weight=w, style="rowwise", tp_degree=3, outs=outs[:1])])
    assert e.value.name == "TP_ERR_SPLIT_NOT_DIVISIBLE"
    torch.cuda.synchronize()
    for t in outs:
        assert torch.all(t.view(torch.int16) == 7)


# CTA-pair launches run as 4-CTA clusters whose two pairs share one operand by multicast:
# n-adjacent tiles (shared A) when the n-tile count is even, m-adjacent tiles (shared B) when
# only the m-tile count (256-row tiles) is even.  Shapes that take each form, several k-blocks,
# every rank; integer inputs, so the results must equal the oracle's bit for bit.
MULTICAST_COLWISE = [
    (1024, 320, 2304, 2),   # 4 m-tiles, 9 n-tiles of 256: B shared
    (1000, 192, 512, 3),    # 4 m-tiles, 2 n-tiles: A shared
    (1536, 128, 768, 4),    # 6 m-tiles, 3 n-tiles: B shared
]


@pytest.mark.parametrize("shape", MULTICAST_COLWISE, ids=str)
def test_multicast_clusters_colwise_bit_exact(shape):
    T, K, N_r, p = shape
    x = tp_inputs.int_bf16(131, 0, (T, K), lim=3)
    w = tp_inputs.int_bf16(131, 1, (N_r * p, K), lim=3)
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "none")
    ref = O.colwise_forward(x, shards, "none")
    for r in range(p):
        assert np.array_equal(host_bits(ys[r]), O.f64_to_bf16(ref[r])), (shape, r)


@pytest.mark.parametrize("T, F_r", [(768, 256), (1024, 384)], ids=str)
def test_multicast_clusters_swiglu(T, F_r):
    # (768, 256): 3 m-tiles, 2 n-tiles of 128 gate columns: A shared; (1024, 384): 4 m-tiles,
    # 3 n-tiles: B shared (each pair's gate and up rows split between the two pairs).
    p, K = 2, 256
    x = tp_inputs.activation_bf16(132, 0, (T, K))
    w = tp_inputs.weight_bf16(132, 1, (2 * F_r * p, K))
    shards = [O.shard(w, "colwise", p, r, [F_r * p, F_r * p]) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "swiglu")
    ref = O.colwise_forward(x, shards, "swiglu")
    for r in range(p):
        assert_close(f64(ys[r]), ref[r], f"swiglu T={T} F_r={F_r} rank {r}")


@pytest.mark.parametrize("T, N", [(1024, 1536), (1024, 1280), (2048, 768)], ids=str)
def test_multicast_clusters_rowwise_bit_exact(T, N):
    # 6 n-tiles: A (every rank's slice in turn) shared; 5 n-tiles, 4 m-tiles: B shared; 8 m-tiles,
    # 3 n-tiles: B shared.  Three ranks, so the shared operand changes at each rank boundary.
    p, K_r = 3, 320
    x = tp_inputs.int_bf16(133, 0, (T, K_r * p), lim=3)
    w = tp_inputs.int_bf16(133, 1, (N, K_r * p), lim=3)
    x_sh = [O.shard(x, "rowwise", p, r) for r in range(p)]
    w_sh = [O.shard(w, "rowwise", p, r) for r in range(p)]
    z = tp.tp_linear_rowwise([dev(a) for a in x_sh], [dev(b) for b in w_sh], mode="accum")
    assert np.array_equal(host_bits(z), O.f64_to_bf16(O.rowwise_forward(x_sh, w_sh))), (T, N)
