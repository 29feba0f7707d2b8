"""Attention over a rank's local heads, and the full attention + SwiGLU MLP block, against the oracle.

The block is: x -> fused QKV (colwise, whole heads per rank) -> attention over
each rank's heads -> out-projection (rowwise, partials summed) -> fused
gate/up (colwise, SwiGLU) -> down-projection (rowwise, summed).  tp_degree is
swept over the divisors of the head count the workload names; 5 and 7 must be
refused before any weight is touched.
"""
import math

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


# ----------------------------------------------------------------------------- attention core

@pytest.mark.parametrize("T,heads,d", [(304, 3, 64), (520, 5, 128), (256, 18, 32), (8, 1, 8), (8, 2, 128),
                                       (136, 3, 128), (1160, 1, 128), (8, 2, 64), (1160, 2, 64), (296, 3, 96)])
def test_attention_heads_within_tolerance(T, heads, d):
    qkv = tp_inputs.activation_bf16(150, heads * 1000 + T, (T, 3 * heads * d))
    out = tp.tp_attention_heads(dev(qkv), heads, d)
    qf = O.bf16_to_f64(qkv)
    H = heads * d
    ref = O.attention_core(qf[:, :H], qf[:, H:2 * H], qf[:, 2 * H:], heads, d)
    assert_close(f64(out), ref, f"attention T={T} heads={heads} d={d}")


@pytest.mark.parametrize("T,heads,d,n", [(520, 2, 128, 3), (136, 4, 128, 2), (200, 2, 64, 3), (392, 3, 64, 4),
                                         (200, 2, 32, 3)])
def test_attention_of_several_ranks_in_one_call(T, heads, d, n):
    # Every rank's heads in one call (one launch at head_dim 128): each rank's output equals
    # the single-rank call bit for bit and the oracle within tolerance.
    H = heads * d
    qkvs = [tp_inputs.activation_bf16(160 + r, T, (T, 3 * H)) for r in range(n)]
    outs = tp.tp_attention_heads_ranks([dev(q) for q in qkvs], heads, d)
    for r, qkv in enumerate(qkvs):
        single = tp.tp_attention_heads(dev(qkv), heads, d)
        assert torch.equal(outs[r].view(torch.int16), single.view(torch.int16)), r
        qf = O.bf16_to_f64(qkv)
        ref = O.attention_core(qf[:, :H], qf[:, H:2 * H], qf[:, 2 * H:], heads, d)
        assert_close(f64(outs[r]), ref, f"rank {r} of {n}, T={T}")


def test_attention_ranks_workspace_and_limits():
    # head_dim 64 and 128 read Q, K and V in place: no workspace; other sizes share one across ranks.
    for d in (64, 128):
        assert tp.tp_attention_ranks_workspace_bytes(4, 4608, 12, d) == 0
        assert tp.tp_attention_workspace_bytes(4608, 12, d) == 0
    assert tp.tp_attention_ranks_workspace_bytes(4, 300, 2, 32) == tp.tp_attention_workspace_bytes(300, 2, 32) > 0
    q = torch.zeros((16, 3 * 128), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tp.TPError) as e:
        tp.tp_attention_heads_ranks([q] * 17, 1, 128)
    assert e.value.name == "TP_ERR_UNSUPPORTED"
    q32 = torch.zeros((16, 3 * 32), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tp.TPError) as e:
        tp.tp_attention_heads_ranks([q32, q32], 1, 32, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert e.value.name == "TP_ERR_WORKSPACE"
    out = tp.tp_attention_heads_ranks([q, q], 1, 128)   # no workspace at all
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(o).item() == 0 for o in out)  # zero Q, K, V -> zero output


def test_attention_one_dominant_key_returns_its_value():
    # Query t is 400*e_t and key u is e_u (head_dim 64): its own key scores 400/8 = 50
    # above the others, so the softmax puts all but e^-50 of its weight there and O ~= V.
    T, d = 64, 64
    q = np.zeros((T, d))
    k = np.zeros((T, d))
    for t in range(T):
        q[t, t] = 400.0
        k[t, t] = 1.0
    v = O.bf16_to_f64(tp_inputs.activation_bf16(151, 0, (T, d)))
    qkv = O.f64_to_bf16(np.concatenate([q, k, v], axis=1))
    out = f64(tp.tp_attention_heads(dev(qkv), 1, d))
    ref = O.attention_core(q, k, v, 1, d)
    assert np.max(np.abs(ref - v)) < 1e-12
    assert_close(out, ref, "one-hot attention")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T", [512, 1000])
def test_attention_running_max_raised_in_some_rows(T, d):
    # Key tiles of growing magnitude (x1, x3, x9, ...): a query's scores jump between tiles
    # when it aligns with the keys (its running max is raised and its output rescaled) and
    # not when it does not -- rows of the same warp take different paths.
    heads = 2
    rng = np.random.default_rng(153)
    q = rng.standard_normal((T, heads * d))
    k = rng.standard_normal((T, heads * d)) * (3.0 ** (np.arange(T) // 128))[:, None] * 0.5
    v = rng.standard_normal((T, heads * d))
    qkv = O.f64_to_bf16(np.concatenate([q, k, v], axis=1))
    out = f64(tp.tp_attention_heads(dev(qkv), heads, d))
    qf = O.bf16_to_f64(qkv)
    H = heads * d
    ref = O.attention_core(qf[:, :H], qf[:, H:2 * H], qf[:, 2 * H:], heads, d)
    assert_close(out, ref, f"growing keys T={T}")


@pytest.mark.parametrize("d", [32, 64])
def test_attention_writes_into_strided_output(d):
    # The rank's attention output can land in a wider buffer (row stride ldo): the unfused path
    # (head_dim 32) and the fused one (64).
    T, heads = 136, 2
    qkv = tp_inputs.activation_bf16(152, 0, (T, 3 * heads * d))
    wide = torch.zeros((T, 3 * heads * d), dtype=torch.bfloat16, device=DEV)
    tp.tp_attention_heads(dev(qkv), heads, d, out=wide[:, :heads * d])
    qf = O.bf16_to_f64(qkv)
    H = heads * d
    ref = O.attention_core(qf[:, :H], qf[:, H:2 * H], qf[:, 2 * H:], heads, d)
    got = f64(wide)
    assert_close(got[:, :H], ref, "strided attention output")
    assert np.all(got[:, H:] == 0)


# ----------------------------------------------------------------------------- full block

def gpu_block(x_bits, wqkv, wout, wgu, wdown, p, heads, d, F, mode="accum"):
    """The block through the library: every rank's shards extracted from device copies of the weights."""
    H = heads * d
    x = dev(x_bits)
    qkv_sh = tp.tp_plan_shard_ranks(dev(wqkv), "colwise", p, 0, p, [H] * 3, heads, d, device=DEV)
    out_sh = tp.tp_plan_shard_ranks(dev(wout), "rowwise", p, 0, p, None, heads, d, device=DEV)
    gu_sh = tp.tp_plan_shard_ranks(dev(wgu), "colwise", p, 0, p, [F, F], heads, 0, device=DEV)
    dn_sh = tp.tp_plan_shard_ranks(dev(wdown), "rowwise", p, 0, p, None, heads, 0, device=DEV)
    # Q, K and V feed the softmax, which amplifies one-ulp rounding differences: chunked accumulation.
    ys = tp.tp_linear_colwise(x, qkv_sh, "none", chunked=True)
    hl = heads // p
    os_ = tp.tp_attention_heads_ranks(ys, hl, d)
    z1 = tp.tp_linear_rowwise(os_, out_sh, mode=mode)
    if mode == "none":
        z1 = tp.tp_combine("reduce", list(z1))
    hs = tp.tp_linear_colwise(z1, gu_sh, "swiglu")
    z2 = tp.tp_linear_rowwise(hs, dn_sh, mode=mode)
    if mode == "none":
        z2 = tp.tp_combine("reduce", list(z2))
    return dict(qkv=ys, o=os_, z1=z1, h=hs, z=z2)


def oracle_block(x_bits, wqkv, wout, wgu, wdown, p, heads, d, F, q_rows=None):
    H = heads * d
    return O.transformer_block_forward(
        x_bits,
        [O.shard(wqkv, "colwise", p, r, [H] * 3, num_heads=heads, head_dim=d) for r in range(p)],
        [O.shard(wout, "rowwise", p, r, num_heads=heads, head_dim=d) for r in range(p)],
        [O.shard(wgu, "colwise", p, r, [F, F]) for r in range(p)],
        [O.shard(wdown, "rowwise", p, r) for r in range(p)],
        n_local_heads=heads // p, head_dim=d, q_rows=q_rows)


SMALL = dict(T=256, heads=48, d=16, F=1536)   # the sweep's 48 heads, at a size the oracle runs in full


def gpu_mlp(z1_bits, wgu, wdown, p, F, heads, mode="accum"):
    """The MLP block alone through the library, from a given input."""
    gu_sh = tp.tp_plan_shard_ranks(dev(wgu), "colwise", p, 0, p, [F, F], heads, 0, device=DEV)
    dn_sh = tp.tp_plan_shard_ranks(dev(wdown), "rowwise", p, 0, p, None, heads, 0, device=DEV)
    hs = tp.tp_linear_colwise(dev(z1_bits), gu_sh, "swiglu")
    z = tp.tp_linear_rowwise(hs, dn_sh, mode=mode)
    return tp.tp_combine("reduce", list(z)) if mode == "none" else z


def oracle_from_stored_qkv(qkv_bits, wout, wgu, wdown, p, heads, d, F, rows):
    """The oracle's block from the rank's stored QKV on: attention, out-projection, SwiGLU MLP.

    qkv_bits: every rank's QKV output as the path stored it; only the query rows `rows`
    are computed (K and V use every token), which is exact for those rows.
    """
    H = heads * d
    w = H // p
    o = []
    for y in qkv_bits:
        qb, kb, vb = O.split_qkv(y, w)
        o.append(O.f64_to_bf16(O.attention_core(O.bf16_to_f64(qb[rows]), O.bf16_to_f64(kb), O.bf16_to_f64(vb),
                                                heads // p, d)))
    z1 = O.rowwise_forward(o, [O.shard(wout, "rowwise", p, r, num_heads=heads, head_dim=d) for r in range(p)])
    _, z = O.mlp_forward(O.f64_to_bf16(z1), [O.shard(wgu, "colwise", p, r, [F, F]) for r in range(p)],
                         [O.shard(wdown, "rowwise", p, r) for r in range(p)], "swiglu")
    return z


def check_block_against_oracle(got, ref, x_rows, wout, wgu, wdown, p, F, heads, d, what, mode="accum"):
    """Every check at the one bar, against the oracle's exact-softmax block; all run before a failure is raised."""
    failures = []

    def check(*a):
        try:
            st = assert_close(*a)
            print(a[2], {k: round(v, 5) for k, v in st.items()})
        except AssertionError as e:
            failures.append(e.args[0])

    # The attention half (QKV -> attention -> out-projection) from the input x.
    check(f64(got["z1"])[x_rows], ref["z1"], f"attention half, {what}")
    # The MLP half (gate/up + SwiGLU -> down) from the oracle's own stored attention-half output.
    check(f64(gpu_mlp(ref["z1_bits"], wgu, wdown, p, F, heads, mode)), ref["z"], f"MLP half, {what}")
    # The whole attention + MLP block from x.
    z = f64(got["z"])[x_rows]
    check(z, ref["z"], f"attention + MLP block from x, {what}")
    # The whole block again, the oracle starting from the QKV the path stored (the block's first
    # stored tensor): attention, out-projection and the MLP against the oracle's own arithmetic.
    qkv_bits = [tp.bits_from_bf16(y) for y in got["qkv"]]
    check(z, oracle_from_stored_qkv(qkv_bits, wout, wgu, wdown, p, heads, d, F, x_rows),
          f"attention + MLP block from the stored QKV, {what}")
    assert not failures, failures


@pytest.mark.parametrize("p", [1, 2, 3, 4, 6, 8])
def test_block_small_matches_oracle(p):
    T, heads, d, F = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["F"]
    H = heads * d
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(3, tokens=T, hidden=H, ffn=F)
    got = gpu_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)
    ref = oracle_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)
    check_block_against_oracle(got, ref, np.arange(T), wout, wgu, wdown, p, F, heads, d, f"tp={p}")


def test_block_small_every_tp_degree_is_bit_identical_to_tp1():
    # With the on-chip rank-ordered sum and K slices on 64-element boundaries, every output
    # element is accumulated over the same products in the same order for every tp_degree:
    # the sharded block reproduces the plain one exactly.
    T, heads, d, F = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["F"]
    H = heads * d
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(3, tokens=T, hidden=H, ffn=F)
    base = tp.bits_from_bf16(gpu_block(x, wqkv, wout, wgu, wdown, 1, heads, d, F)["z"])
    for p in (2, 3, 4, 6, 8):
        got = tp.bits_from_bf16(gpu_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)["z"])
        assert np.array_equal(got, base), p


MID = dict(T=392, heads=24, d=128, F=3072)   # head_dim 128 (the fused attention), a ragged token tail


@pytest.mark.parametrize("p", [1, 3, 8])
def test_block_head_dim_128_matches_oracle(p):
    T, heads, d, F = MID["T"], MID["heads"], MID["d"], MID["F"]
    H = heads * d
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(3, tokens=T, hidden=H, ffn=F)
    got = gpu_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)
    ref = oracle_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)
    check_block_against_oracle(got, ref, np.arange(T), wout, wgu, wdown, p, F, heads, d, f"tp={p}")


@pytest.mark.parametrize("p", [5, 7])
def test_block_rejects_tp_not_dividing_heads(p):
    T, heads, d, F = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["F"]
    H = heads * d
    wqkv = tp_inputs.weight_bf16(3, 0, (3 * H, H))
    for style, rows, cols, splits, hd in (("colwise", 3 * H, H, [H] * 3, d), ("rowwise", H, H, None, d)):
        with pytest.raises(tp.TPError) as e:
            tp.tp_validate(rows, cols, style, p, heads, hd, splits)
        assert e.value.name == "TP_ERR_HEADS_NOT_DIVISIBLE"
    with pytest.raises(tp.TPError) as e:
        tp.tp_plan_shard_ranks(dev(wqkv), "colwise", p, 0, p, [H] * 3, heads, d, device=DEV)
    assert e.value.name == "TP_ERR_HEADS_NOT_DIVISIBLE"


@pytest.mark.parametrize("mode", ["workspace", "none"])
def test_block_small_other_join_modes(mode):
    T, heads, d, F = SMALL["T"], SMALL["heads"], SMALL["d"], SMALL["F"]
    H = heads * d
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(3, tokens=T, hidden=H, ffn=F)
    got = gpu_block(x, wqkv, wout, wgu, wdown, 4, heads, d, F, mode=mode)
    ref = oracle_block(x, wqkv, wout, wgu, wdown, 4, heads, d, F)
    check_block_against_oracle(got, ref, np.arange(T), wout, wgu, wdown, 4, F, heads, d, mode, mode=mode)


@pytest.mark.slow
def test_block_sweep_full_size():
    """hidden 6144, 48 heads x 128, ffn 18432, tokens 4608: every tp_degree against tp_degree 1 and the oracle."""
    cfg = tp_inputs.WORKLOADS["block_sweep"]
    T, H, F, heads, d = cfg["tokens"], cfg["hidden"], cfg["ffn"], cfg["heads"], cfg["head_dim"]
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(cfg["seed"], tokens=T, hidden=H, ffn=F)
    rows = tp_inputs.sample_rows(cfg["seed"], T, 48)
    ref = oracle_block(x, wqkv, wout, wgu, wdown, 1, heads, d, F, q_rows=rows)
    base = None
    for p in cfg["tp_list"]:
        got = gpu_block(x, wqkv, wout, wgu, wdown, p, heads, d, F)
        z = tp.bits_from_bf16(got["z"])
        if base is None:
            base = z
            check_block_against_oracle(got, ref, rows, wout, wgu, wdown, p, F, heads, d, "tp=1 full size")
        else:
            # The sum / concatenation invariant against tp_degree 1, bit for bit.
            assert np.array_equal(z, base), f"tp={p} differs from tp=1"
        del got
        torch.cuda.empty_cache()
