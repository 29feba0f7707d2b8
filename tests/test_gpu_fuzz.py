"""Seeded random shapes through every entry point, against the oracle.

Each case draws a plan and a shape (ragged token counts, widths that are not
multiples of the tile sizes, packed blocks, every join mode, plain and chunked
accumulation) from a seeded generator.  Inputs are small integers, so every product sum is exact in fp32
and the bf16 results must equal the oracle's bit for bit, whatever the
kernels' summation order.  Attention cases use normal inputs and the
tolerance of tests/tolerance.py.
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
N_CASES = 64


def dev(bits):
    return tp.bf16_from_bits(bits, DEV)


def bits(t):
    torch.cuda.synchronize()
    return tp.bits_from_bf16(t)


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    tp.tp_device_status()


def _packed(rng, p, n_blocks, unit):
    """n_blocks positive block sizes, each a multiple of p * unit."""
    return [int(rng.integers(1, 5)) * p * unit for _ in range(n_blocks)]


@pytest.mark.parametrize("case", range(N_CASES))
def test_fuzz_colwise_projection(case):
    rng = np.random.default_rng([7001, case])
    p = int(rng.integers(1, 9))
    T = int(rng.integers(1, 700))
    K = 8 * int(rng.integers(1, 80))
    act = ["none", "swiglu", "none"][case % 3]
    chunked = case % 3 == 2          # chunked fp32 accumulation (TP_ACCUM_CHUNKED)
    if chunked:
        K = 8 * int(rng.integers(1, 400))   # up to 50 k-blocks: several chunks of 16 and a tail
    if act == "swiglu":
        F = 8 * p * int(rng.integers(1, 40))
        splits = [F, F]
    else:
        splits = _packed(rng, p, int(rng.integers(1, 4)), 8)
    rows = sum(splits)
    w = tp_inputs.int_bf16(7001, case * 10 + 1, (rows, K), lim=3)
    x = tp_inputs.int_bf16(7001, case * 10 + 2, (T, K), lim=3)
    shards = tp.tp_plan_shard_ranks(dev(w), "colwise", p, 0, p, splits, device=DEV)
    for r in range(p):
        assert np.array_equal(bits(shards[r]), O.shard(w, "colwise", p, r, splits)), ("extract", case, r)
    bias_sh = None
    if case % 3 == 0:   # a bias, sharded like the weight's rows (integer values: sums stay exact)
        b = tp_inputs.int_bf16(7001, case * 10 + 3, (rows, 1), lim=3)
        bias_sh = [np.ascontiguousarray(O.shard(b, "colwise", p, r, splits).reshape(-1)) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), shards, act, bias_shards=None if bias_sh is None else [dev(v) for v in bias_sh],
                              chunked=chunked)
    want = O.colwise_forward(x, [O.shard(w, "colwise", p, r, splits) for r in range(p)], act, bias_sh)
    for r in range(p):
        if act == "swiglu":
            # SiLU is not exact: within the bar.
            assert_close(O.bf16_to_f64(bits(ys[r])), want[r], f"case {case} rank {r}")
        else:
            assert np.array_equal(bits(ys[r]), O.f64_to_bf16(want[r])), ("colwise", case, r)


@pytest.mark.parametrize("case", range(N_CASES))
def test_fuzz_rowwise_projection(case):
    rng = np.random.default_rng([7002, case])
    p = int(rng.integers(1, 9))
    T = int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 90))
    splits = _packed(rng, p, int(rng.integers(1, 3)), 8)
    K = sum(splits)
    mode = ["accum", "workspace", "none"][case % 3]
    w = tp_inputs.int_bf16(7002, case * 10 + 1, (N, K), lim=3)
    x = tp_inputs.int_bf16(7002, case * 10 + 2, (T, K), lim=3)
    w_sh = tp.tp_plan_shard_ranks(dev(w), "rowwise", p, 0, p, splits, device=DEV)
    x_sh = [O.shard(x, "rowwise", p, r, splits) for r in range(p)]
    for r in range(p):
        assert np.array_equal(bits(w_sh[r]), O.shard(w, "rowwise", p, r, splits)), ("extract", case, r)
    b = tp_inputs.int_bf16(7002, case * 10 + 3, (N,), lim=3) if case % 4 == 0 else None  # added once
    z = tp.tp_linear_rowwise([dev(a) for a in x_sh], w_sh, bias=None if b is None else dev(b), mode=mode)
    if mode == "none":
        z = tp.tp_combine("reduce", list(z))
    want = O.rowwise_forward(x_sh, [O.shard(w, "rowwise", p, r, splits) for r in range(p)], b)
    assert np.array_equal(bits(z), O.f64_to_bf16(want)), (case, p, T, K, N, mode)


@pytest.mark.parametrize("case", range(24))
def test_fuzz_attention(case):
    rng = np.random.default_rng([7003, case])
    n = int(rng.integers(1, 5))
    T = 8 * int(rng.integers(1, 90))
    heads = int(rng.integers(1, 4))
    d = [64, 128][case % 2]
    H = heads * d
    qkvs = [tp_inputs.activation_bf16(7003, case * 10 + r, (T, 3 * H)) for r in range(n)]
    outs = tp.tp_attention_heads_ranks([dev(q) for q in qkvs], heads, d)
    for r, qkv in enumerate(qkvs):
        qf = O.bf16_to_f64(qkv)
        ref = O.attention_core(qf[:, :H], qf[:, H:2 * H], qf[:, 2 * H:], heads, d)
        assert_close(O.bf16_to_f64(bits(outs[r])), ref, f"case {case} rank {r} T={T} heads={heads} d={d}")
