"""The single-stream block through the library, against the oracle.

"Tensor parallelism" page, §Fused projections: one Linear packs Q, K, V, gate
and up as [1, 1, 1, 3, 3] (mlp_ratio 3) and is sharded block by block; the
single-stream to_out stores its input blocks [inner_dim, mlp_hidden_dim] and is
sharded block by block along its input.  Each rank's fused shard is
[Q_r; K_r; V_r; gate_r; up_r]: its Q/K/V rows go through a plain colwise GEMM
into the attention core, its gate/up rows through the SwiGLU colwise GEMM, and
both results land side by side in one [T, H/p + F/p] buffer -- attention in the
first columns, the MLP state after it -- which is exactly the input of the
rank's packed to_out shard.
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


def f64(t):
    torch.cuda.synchronize()
    return O.bf16_to_f64(tp.bits_from_bf16(t))


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    tp.tp_device_status()


def gpu_single_stream(x_bits, w_in, w_out, p, heads, d, F, mode="accum"):
    H = heads * d
    w, f = H // p, F // p
    x = dev(x_bits)
    T = x.shape[0]
    in_sh = tp.tp_plan_shard_ranks(dev(w_in), "colwise", p, 0, p, [H, H, H, F, F], heads, 0, device=DEV)
    out_sh = tp.tp_plan_shard_ranks(dev(w_out), "rowwise", p, 0, p, [H, F], heads, 0, device=DEV)
    cat = [torch.full((T, w + f), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(p)]
    qkv = tp.tp_linear_colwise(x, [s[:3 * w] for s in in_sh], "none", chunked=True)
    tp.tp_linear_colwise(x, [s[3 * w:] for s in in_sh], "swiglu", y_shards=[c[:, w:] for c in cat], ldy=w + f)
    tp.tp_attention_heads_ranks(qkv, heads // p, d, outs=[c[:, :w] for c in cat])
    z = tp.tp_linear_rowwise(cat, out_sh, mode=mode)
    if mode == "none":
        z = tp.tp_combine("reduce", list(z))
    return dict(cat=cat, z=z, w=w)


def oracle_single_stream(x_bits, w_in, w_out, p, heads, d, F, q_rows=None):
    H = heads * d
    return O.single_stream_block_forward(
        x_bits, [O.shard(w_in, "colwise", p, r, [H, H, H, F, F], num_heads=heads) for r in range(p)],
        [O.shard(w_out, "rowwise", p, r, [H, F], num_heads=heads) for r in range(p)],
        n_local_heads=heads // p, head_dim=d, q_rows=q_rows)


def check_against_oracle(got, ref, rows, what):
    # Each stored result against the oracle's value before its own bf16 storage, all at the
    # one bar.  Every check runs before the first failure is raised.
    w = got["w"]
    failures = []

    def check(fn, *a):
        try:
            fn(*a)
        except AssertionError as e:
            failures.append(e.args[0])

    for r, c in enumerate(got["cat"]):
        cr = f64(c)[rows]
        check(assert_close, cr[:, :w], ref["o"][r], f"rank {r} attention, {what}")
        check(assert_close, cr[:, w:], ref["h"][r], f"rank {r} SwiGLU, {what}")
    check(assert_close, f64(got["z"])[rows], ref["z"], f"out-projection, {what}")
    assert not failures, failures


SMALL = dict(T=328, heads=6, d=128, ratio=3)   # fused attention (head_dim 128), ragged token tail


@pytest.mark.parametrize("p", [1, 2, 3, 6])
def test_single_stream_small_matches_oracle(p):
    T, heads, d, ratio = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["ratio"]
    H, F = heads * d, ratio * heads * d
    w_in, w_out, x = tp_inputs.single_stream_inputs(5, tokens=T, hidden=H, mlp_ratio=ratio)
    got = gpu_single_stream(x, w_in, w_out, p, heads, d, F)
    ref = oracle_single_stream(x, w_in, w_out, p, heads, d, F)
    check_against_oracle(got, ref, np.arange(T), f"tp={p}")


@pytest.mark.parametrize("mode", ["workspace", "none"])
def test_single_stream_small_other_join_modes(mode):
    T, heads, d, ratio = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["ratio"]
    H, F = heads * d, ratio * heads * d
    w_in, w_out, x = tp_inputs.single_stream_inputs(5, tokens=T, hidden=H, mlp_ratio=ratio)
    got = gpu_single_stream(x, w_in, w_out, 3, heads, d, F, mode=mode)
    ref = oracle_single_stream(x, w_in, w_out, 3, heads, d, F)
    check_against_oracle(got, ref, np.arange(T), mode)


def test_single_stream_integer_projections_bit_exact():
    # Integer-valued weights and input: the fused in-projection's Q/K/V rows and the packed
    # out-projection of a given [attention, mlp] input are exact, so both match bit for bit.
    T, heads, d, ratio, p = 136, 4, 64, 3, 2
    H, F = heads * d, ratio * heads * d
    w, f = H // p, F // p
    w_in, w_out, x = tp_inputs.single_stream_inputs(6, tokens=T, hidden=H, mlp_ratio=ratio, kind="int")
    in_o = [O.shard(w_in, "colwise", p, r, [H, H, H, F, F]) for r in range(p)]
    out_o = [O.shard(w_out, "rowwise", p, r, [H, F]) for r in range(p)]
    in_sh = tp.tp_plan_shard_ranks(dev(w_in), "colwise", p, 0, p, [H, H, H, F, F], heads, 0, device=DEV)
    out_sh = tp.tp_plan_shard_ranks(dev(w_out), "rowwise", p, 0, p, [H, F], heads, 0, device=DEV)
    for r in range(p):
        assert np.array_equal(tp.bits_from_bf16(in_sh[r]), in_o[r])
        assert np.array_equal(tp.bits_from_bf16(out_sh[r]), out_o[r])
    qkv = tp.tp_linear_colwise(dev(x), [s[:3 * w] for s in in_sh], "none")
    for r in range(p):
        want = O.f64_to_bf16(O.colwise_forward(x, [in_o[r][:3 * w]])[0])
        assert np.array_equal(tp.bits_from_bf16(qkv[r]), want)
    cat = [tp_inputs.int_bf16(6, 10 + r, (T, w + f)) for r in range(p)]
    z = tp.tp_linear_rowwise([dev(c) for c in cat], out_sh, mode="accum")
    assert np.array_equal(tp.bits_from_bf16(z), O.f64_to_bf16(O.rowwise_forward(cat, out_o)))


def test_single_stream_rejects_blocks_not_divisible():
    # 6 heads at tp_degree 4 is refused before any weight is touched, and so is a packed
    # to_out whose blocks [24, 24] tp_degree 16 does not divide although it divides their sum.
    heads, d = 6, 128
    H, F = heads * d, 3 * heads * d
    with pytest.raises(tp.TPError) as e:
        tp.tp_validate(3 * H + 2 * F, H, "colwise", 4, heads, 0, [H, H, H, F, F])
    assert e.value.name == "TP_ERR_HEADS_NOT_DIVISIBLE"
    with pytest.raises(tp.TPError) as e:
        tp.tp_validate(H, 3 * 8 + 2 * 12, "rowwise", 16, 0, 0, [24, 24])
    assert e.value.name == "TP_ERR_SPLIT_NOT_DIVISIBLE"


@pytest.mark.slow
def test_single_stream_full_size():
    """hidden 6144, 48 heads x 128, mlp_ratio 3, 4608 tokens, tp_degree 4: sampled rows against the oracle."""
    cfg = tp_inputs.WORKLOADS["single_stream_tp4"]
    T, H, heads, d, p = cfg["tokens"], cfg["hidden"], cfg["heads"], cfg["head_dim"], cfg["tp"]
    F = cfg["mlp_ratio"] * H
    w_in, w_out, x = tp_inputs.single_stream_inputs(cfg["seed"], T, H, cfg["mlp_ratio"])
    rows = tp_inputs.sample_rows(cfg["seed"], T, 48)
    got = gpu_single_stream(x, w_in, w_out, p, heads, d, F)
    ref = oracle_single_stream(x, w_in, w_out, p, heads, d, F, q_rows=rows)
    check_against_oracle(got, ref, rows, "full size")
