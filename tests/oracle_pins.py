"""Pins of the CPU oracle: checks of its functions against facts fixed outside it.

Each ``pin_*`` function raises AssertionError when the oracle (the module
``oracle.tp_oracle``, looked up at call time) disagrees with a closed form, a
brute-force loop, a library routine on a special case, or a hand-derived
fixture from ``tests/golden``.  ``test_oracle_pins.py`` runs them against the
real oracle; ``test_oracle_mutations.py`` plants plausible mistakes in the
oracle and checks that at least one pin fails for each.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import tp_inputs
from oracle import tp_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- fixtures --

def read_index_fixture(name):
    """Parse a tests/golden/*.txt index fixture -> dict."""
    out = {"ranks": {}}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "rank":
                r, _, idx = rest.partition(":")
                out["ranks"][int(r)] = [int(v) for v in idx.split()]
            elif key in ("blocks", "sizes"):
                out[key] = [int(v) for v in rest.split()]
            elif key in ("dim", "tp"):
                out[key] = int(rest)
            else:
                out[key] = rest.strip()
    return out


def read_plan_fixture(name="plan_rejections.txt"):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            style, r, c, tp, h, d, sizes, expected = line.split()
            sizes = None if sizes == "-" else [int(v) for v in sizes.split(",")]
            rows.append((style, int(r), int(c), int(tp), int(h), int(d), sizes, expected))
    return rows


def _bits_from_f32(x):
    """bf16 bits of float32 values via torch's own conversion (a library routine)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------ bf16 --

def pin_bf16_rounding():
    # Hand-worked encodings: 1.0 = 0x3F80; 1 + 2^-8 is a tie between 0x3F80 and
    # 0x3F81 and goes to the even one; 1 + 3*2^-8 ties up to 0x3F82; just above
    # a tie rounds up; -2.5 = 0xC020; max bf16 0x7F7F; its next tie overflows.
    cases = [
        (1.0, 0x3F80), (1.0 + 2.0 ** -8, 0x3F80), (1.0 + 3 * 2.0 ** -8, 0x3F82),
        (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81), (-2.5, 0xC020), (0.0, 0x0000), (-0.0, 0x8000),
        (3.3895313892515355e38, 0x7F7F), (2.0 ** 128 - 2.0 ** 119, 0x7F80), (float("inf"), 0x7F80),
        (-float("inf"), 0xFF80), (2.0 ** -133, 0x0001), (2.0 ** -134, 0x0000), (3 * 2.0 ** -134, 0x0002),
        (2.0 ** -126, 0x0080), (-1e-45, 0x8000),
    ]
    xs = np.array([c[0] for c in cases], dtype=np.float64)
    got = O.f64_to_bf16(xs)
    exp = np.array([c[1] for c in cases], dtype=np.uint16)
    assert np.array_equal(got, exp), (got, exp)
    assert O.f64_to_bf16(np.array([np.nan]))[0] == 0x7FC0
    # Against torch's float32 -> bf16 conversion on values exact in float32.
    rng = np.random.default_rng(7)
    x32 = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),   # subnormal range
        np.clip(rng.standard_normal(2000) * 1e38, -3.3e38, 3.3e38).astype(np.float32),
    ])
    # Construct exact ties: bf16 value + half an ulp.
    base = rng.standard_normal(2000).astype(np.float32)
    bb = base.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (bb | np.uint32(0x8000)).view(np.float32)
    x32 = np.concatenate([x32, ties])
    assert np.array_equal(O.f64_to_bf16(x32.astype(np.float64)), _bits_from_f32(x32))
    # Widening is exact and inverse on every non-NaN pattern.
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wide = O.bf16_to_f64(allbits)
    ok = ~np.isnan(wide)
    assert np.array_equal(O.f64_to_bf16(wide[ok]), allbits[ok])
    assert np.array_equal(wide[ok].astype(np.float32), (allbits[ok].astype(np.uint32) << 16).view(np.float32))


# ------------------------------------------------------------------ plan --

def pin_plan_rejections():
    for style, r, c, tp, h, d, sizes, expected in read_plan_fixture():
        try:
            O.check_plan(r, c, style, tp, num_heads=h, head_dim=d, splits=sizes)
            got = "OK"
        except O.PlanRejected as e:
            got = e.reason
        assert got == expected, (style, r, c, tp, h, d, sizes, got, expected)
    # Argument errors.
    for kw in (dict(tp_degree=0), dict(tp_degree=-1), dict(tp_degree=2, rank=2), dict(tp_degree=2, rank=-1)):
        tp = kw.pop("tp_degree")
        try:
            O.check_plan(8, 8, O.COLWISE, tp, **kw)
            raise AssertionError(f"accepted {tp} {kw}")
        except O.PlanRejected as e:
            assert e.reason == O.INVALID_ARG
    # Heads rule against a brute-force divisor list: 48 heads pass exactly at its divisors.
    divisors = [p for p in range(1, 49) if 48 % p == 0]
    passed = []
    for p in range(1, 49):
        try:
            O.check_plan(48 * 128, 64, O.COLWISE, p, num_heads=48, head_dim=128)
            passed.append(p)
        except O.PlanRejected:
            pass
    assert passed == divisors == [1, 2, 3, 4, 6, 8, 12, 16, 24, 48]


def pin_packed_blocks():
    # The pages' proportional forms against hand arithmetic.
    assert O.packed_block_sizes(36864, [1, 1]) == [18432, 18432]
    assert O.packed_block_sizes(18, [1, 1, 1, 3, 3]) == [2, 2, 2, 6, 6]
    assert O.packed_block_sizes(3072 * 9, [1, 1, 1, 3, 3]) == [3072, 3072, 3072, 9216, 9216]
    try:
        O.packed_block_sizes(10, [1, 1, 1])
        raise AssertionError("sum 3 does not divide 10")
    except O.PlanRejected as e:
        assert e.reason == O.SPLIT_SUM


def _index_weight(rows, cols):
    """W[i, j] = i * cols + j as int64 so every element names its own position."""
    return np.arange(rows * cols, dtype=np.int64).reshape(rows, cols)


def pin_shard_golden():
    for name in ("packed_colwise_qkv_gate_up.txt", "packed_colwise_swiglu.txt", "plain_colwise_tp4.txt",
                 "packed_rowwise_to_out.txt"):
        fx = read_index_fixture(name)
        dim, tp = fx["dim"], fx["tp"]
        sizes = fx.get("sizes") or O.packed_block_sizes(dim, fx["blocks"])
        style = fx["style"]
        other = 3
        if style == O.COLWISE:
            w = _index_weight(dim, other)
        else:
            w = _index_weight(other, dim)
        for r, idx in fx["ranks"].items():
            s = O.shard(w, style, tp, r, sizes)
            if style == O.COLWISE:
                assert np.array_equal(s, w[idx, :]), (name, r)
            else:
                assert np.array_equal(s, w[:, idx]), (name, r)
            assert s.shape == O.shard_shape(w.shape[0], w.shape[1], style, tp, sizes)


def pin_shard_reassembly():
    rng = np.random.default_rng(11)
    for style in (O.COLWISE, O.ROWWISE):
        for tp, sizes in ((1, None), (2, None), (3, [6, 12, 6]), (4, [8, 8]), (6, [12, 12, 12]), (2, [2, 2, 2, 6, 6])):
            dim = sum(sizes) if sizes else 24
            shape = (dim, 40) if style == O.COLWISE else (40, dim)
            w = rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)   # any bit pattern survives
            blocks = sizes or [dim]
            shards = [O.shard(w, style, tp, r, sizes) for r in range(tp)]
            # Independent reassembly: block b of W is the concatenation over ranks of part b.
            pieces = []
            for b, s in enumerate(blocks):
                part = s // tp
                off = sum(blocks[:b]) // tp
                for r in range(tp):
                    sl = shards[r][off:off + part, :] if style == O.COLWISE else shards[r][:, off:off + part]
                    pieces.append(sl)
            re = np.concatenate(pieces, axis=0 if style == O.COLWISE else 1)
            assert re.dtype == np.uint16 and np.array_equal(re, w), (style, tp, sizes)
            if tp == 1:
                assert np.array_equal(shards[0], w)


def pin_whole_heads():
    # Tag every row of a fused QKV weight with (which, head): rank r must hold
    # exactly heads [r*h/p, (r+1)*h/p) of each of Q, K and V.
    h, d = 12, 4
    H = h * d
    tags = np.zeros((3 * H, 2), dtype=np.int64)
    for which in range(3):
        for row in range(H):
            tags[which * H + row] = (which, row // d)
    for p in (1, 2, 3, 4, 6, 12):
        for r in range(p):
            s = O.shard(tags, O.COLWISE, p, r, [H, H, H], num_heads=h, head_dim=d)
            hp = h // p
            expect = [(which, head) for which in range(3) for head in range(r * hp, (r + 1) * hp) for _ in range(d)]
            assert [tuple(t) for t in s] == expect, (p, r)


# ----------------------------------------------------------- arithmetic --

def _brute_linear(x, w):
    T, K = x.shape
    N = w.shape[0]
    y = [[0.0] * N for _ in range(T)]
    for t in range(T):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(x[t, k]) * float(w[n, k])
            y[t][n] = acc
    return np.array(y)


def pin_linear_bruteforce():
    for (T, K, N) in ((1, 1, 1), (3, 5, 2), (4, 7, 6), (2, 8, 3)):
        xb = tp_inputs.int_bf16(5, T * 100 + K, (T, K), lim=4)
        wb = tp_inputs.int_bf16(6, N * 100 + K, (N, K), lim=4)
        xf, wf = O.bf16_to_f64(xb), O.bf16_to_f64(wb)
        assert np.array_equal(O.linear(xb, wb), _brute_linear(xf, wf)), (T, K, N)
    # Identity input returns W transposed; a one-hot row picks one column of W^T.
    w = tp_inputs.weight_bf16(9, 0, (6, 5))
    eye = O.f64_to_bf16(np.eye(5))
    assert np.array_equal(O.linear(eye, w), O.bf16_to_f64(w).T)


def pin_activations():
    x = np.linspace(-9, 9, 4001)
    g = O.gelu_tanh(x)
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.allclose(g - O.gelu_tanh(-x), x, rtol=0, atol=1e-12)          # tanh is odd
    assert np.allclose(O.gelu_tanh(np.array([30.0, -30.0])), [30.0, 0.0], atol=1e-12)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(g, ref, rtol=1e-14, atol=1e-14)
    s = O.silu(x)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(s - O.silu(-x), x, rtol=0, atol=1e-12)               # sigmoid(x)+sigmoid(-x)=1
    assert np.allclose(s, torch.nn.functional.silu(torch.from_numpy(x)).numpy(), rtol=1e-14, atol=1e-14)
    assert math.isclose(O.silu(np.array([1.0]))[0], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    gate = np.array([[0.0, 1.0, -2.0]])
    up = np.array([[5.0, 3.0, 0.5]])
    assert np.allclose(O.swiglu(gate, up), [[0.0, 3.0 / (1 + math.exp(-1.0)), 0.5 * -2.0 / (1 + math.exp(2.0))]],
                       rtol=1e-15)


def pin_colwise_concat():
    # Concatenating colwise outputs gives the unsharded output (plain split), and
    # tp_degree=1 is the plain layer.
    T, K, N = 9, 24, 36
    x = tp_inputs.activation_bf16(21, 0, (T, K))
    w = tp_inputs.weight_bf16(21, 1, (N, K))
    full = O.bf16_to_f64(x) @ O.bf16_to_f64(w).T
    for p in (1, 2, 3, 4, 6):
        ys = O.colwise_forward(x, [O.shard(w, O.COLWISE, p, r) for r in range(p)], "none")
        assert np.allclose(np.concatenate(ys, axis=1), full, rtol=1e-13, atol=1e-15), p
    xi = tp_inputs.int_bf16(22, 0, (T, K))
    wi = tp_inputs.int_bf16(22, 1, (N, K))
    fi = O.bf16_to_f64(xi) @ O.bf16_to_f64(wi).T
    for p in (1, 2, 3):
        ys = O.colwise_forward(xi, [O.shard(wi, O.COLWISE, p, r) for r in range(p)], "none")
        assert np.array_equal(np.concatenate(ys, axis=1), fi)
    # GELU is applied after the projection, per element.
    ys = O.colwise_forward(x, [O.shard(w, O.COLWISE, 2, r) for r in range(2)], "gelu_tanh")
    gref = torch.nn.functional.gelu(torch.from_numpy(full), approximate="tanh").numpy()
    assert np.allclose(np.concatenate(ys, axis=1), gref, rtol=1e-12, atol=1e-14)


def pin_swiglu_packed():
    # Packed [gate; up] sharded block by block + SwiGLU per rank, concatenated,
    # equals the unsharded silu(X Wg^T) * (X Wu^T) written here from torch ops.
    T, K, F = 7, 16, 24
    x = tp_inputs.activation_bf16(31, 0, (T, K))
    wg = tp_inputs.weight_bf16(31, 1, (F, K))
    wu = tp_inputs.weight_bf16(31, 2, (F, K))
    wgu = np.concatenate([wg, wu], axis=0)
    xt = torch.from_numpy(O.bf16_to_f64(x))
    ref = (torch.nn.functional.silu(xt @ torch.from_numpy(O.bf16_to_f64(wg)).T)
           * (xt @ torch.from_numpy(O.bf16_to_f64(wu)).T)).numpy()
    for p in (1, 2, 3, 4):
        shards = [O.shard(wgu, O.COLWISE, p, r, [F, F]) for r in range(p)]
        hs = O.colwise_forward(x, shards, "swiglu")
        assert all(h.shape == (T, F // p) for h in hs)
        assert np.allclose(np.concatenate(hs, axis=1), ref, rtol=1e-12, atol=1e-15), p


def pin_rowwise_sum():
    T, K, N = 5, 48, 10
    x = tp_inputs.activation_bf16(41, 0, (T, K))
    w = tp_inputs.weight_bf16(41, 1, (N, K))
    full = O.bf16_to_f64(x) @ O.bf16_to_f64(w).T
    for p in (1, 2, 3, 4, 6, 8):
        xs = [O.shard(x, O.ROWWISE, p, r) for r in range(p)]     # activations split like the weight's columns
        ws = [O.shard(w, O.ROWWISE, p, r) for r in range(p)]
        z = O.rowwise_forward(xs, ws)
        assert np.allclose(z, full, rtol=1e-13, atol=1e-15), p
        parts = O.rowwise_partials(xs, ws)
        # Each partial is the product over the rank's columns only (brute force on the slice).
        bk = _brute_linear(O.bf16_to_f64(xs[-1]), O.bf16_to_f64(ws[-1]))
        assert np.allclose(parts[-1], bk, rtol=1e-13, atol=1e-15)
    # Integer-valued inputs: exact.
    xi = tp_inputs.int_bf16(42, 0, (T, K))
    wi = tp_inputs.int_bf16(42, 1, (N, K))
    zi = O.rowwise_forward([O.shard(xi, O.ROWWISE, 4, r) for r in range(4)],
                           [O.shard(wi, O.ROWWISE, 4, r) for r in range(4)])
    assert np.array_equal(zi, _brute_linear(O.bf16_to_f64(xi), O.bf16_to_f64(wi)))
    # The bias is added once, not once per rank.
    b = tp_inputs.weight_bf16(43, 0, (N,))
    zb = O.rowwise_forward([O.shard(x, O.ROWWISE, 4, r) for r in range(4)],
                           [O.shard(w, O.ROWWISE, 4, r) for r in range(4)], b)
    assert np.allclose(zb, full + O.bf16_to_f64(b)[None, :], rtol=1e-13, atol=1e-15)


def pin_rowwise_split_input():
    # Each rank slicing the replicated input and the sum over ranks is the plain layer,
    # checked against a brute-force loop and the slice arithmetic by hand on a tiny case.
    T, K, N = 3, 12, 5
    x = tp_inputs.int_bf16(44, 0, (T, K))
    w = tp_inputs.int_bf16(44, 1, (N, K))
    brute = _brute_linear(O.bf16_to_f64(x), O.bf16_to_f64(w))
    for p in (1, 2, 3, 4, 6):
        z = O.rowwise_split_input_forward(x, [O.shard(w, O.ROWWISE, p, r) for r in range(p)])
        assert np.array_equal(z, brute), p
    # With tp_degree 3 rank 1 sees input columns 4..7 only: zeroing them changes only its partial.
    x2 = O.bf16_to_f64(x).copy()
    x2[:, 4:8] = 0
    z2 = O.rowwise_split_input_forward(O.f64_to_bf16(x2), [O.shard(w, O.ROWWISE, 3, r) for r in range(3)])
    part1 = O.bf16_to_f64(x)[:, 4:8] @ O.bf16_to_f64(w)[:, 4:8].T
    assert np.array_equal(brute - z2, part1)


def pin_combine():
    parts = [np.full((3, 2), r, dtype=np.uint16) for r in range(4)]
    g = O.combine_gather(parts)
    assert g.shape == (3, 8) and g.dtype == np.uint16
    assert np.array_equal(g[1], [0, 0, 1, 1, 2, 2, 3, 3])
    red = O.combine_reduce([np.full((2, 2), float(r + 1), dtype=np.float32) for r in range(4)])
    assert np.array_equal(red, np.full((2, 2), 10.0))


def _brute_attention(q, k, v, n_heads, d):
    T, Tk = q.shape[0], k.shape[0]
    out = np.zeros((T, n_heads * d))
    for h in range(n_heads):
        c0 = h * d
        for t in range(T):
            s = [sum(q[t, c0 + i] * k[u, c0 + i] for i in range(d)) / math.sqrt(d) for u in range(Tk)]
            m = max(s)
            e = [math.exp(v_ - m) for v_ in s]
            z = sum(e)
            for i in range(d):
                out[t, c0 + i] = sum(e[u] / z * v[u, c0 + i] for u in range(Tk))
    return out


def pin_attention():
    rng = np.random.default_rng(51)
    T, h, d = 4, 2, 3
    q, k, v = (rng.standard_normal((T, h * d)) for _ in range(3))
    o = O.attention_core(q, k, v, h, d)
    assert np.allclose(o, _brute_attention(q, k, v, h, d), rtol=1e-13, atol=1e-14)
    # Q = 0: every key gets the same weight, so O is the column mean of V.
    o0 = O.attention_core(np.zeros_like(q), k, v, h, d)
    assert np.allclose(o0, np.tile(v.mean(axis=0), (T, 1)), rtol=1e-13, atol=1e-14)
    # One dominant key per query: key u is the unit vector e_u and query t is
    # 200*e_t, so query t's softmax puts all its weight on key t and O = V.
    d2 = 4
    kk = np.zeros((T, d2))
    qq = np.zeros((T, d2))
    for t in range(T):
        kk[t, t] = 1.0
        qq[t, t] = 200.0
    vv = rng.standard_normal((T, d2))
    oo = O.attention_core(qq, kk, vv, 1, d2)
    assert np.allclose(oo, vv, rtol=0, atol=1e-12)
    # Against torch's scaled-dot-product attention in float64 (a library routine).
    T2, h2, d3 = 17, 3, 8
    q2, k2, v2 = (rng.standard_normal((T2, h2 * d3)) for _ in range(3))

    def heads(a):
        return torch.from_numpy(a).reshape(T2, h2, d3).permute(1, 0, 2)

    ref = torch.nn.functional.scaled_dot_product_attention(heads(q2), heads(k2), heads(v2))
    ref = ref.permute(1, 0, 2).reshape(T2, h2 * d3).numpy()
    assert np.allclose(O.attention_core(q2, k2, v2, h2, d3), ref, rtol=1e-12, atol=1e-13)


def pin_block_tp_invariance():
    # The sharded block at tp_degree p equals the block at tp_degree 1 (the plain
    # layer) up to float64 reassociation and the bf16 storage between steps.
    T, h, d, F = 12, 6, 8, 72
    H = h * d
    wqkv, wout, wgu, wdown, x = tp_inputs.block_inputs(61, tokens=T, hidden=H, ffn=F)
    ref = None
    for p in (1, 2, 3, 6):
        sh = dict(
            wqkv_shards=[O.shard(wqkv, O.COLWISE, p, r, [H, H, H], num_heads=h, head_dim=d) for r in range(p)],
            wout_shards=[O.shard(wout, O.ROWWISE, p, r, num_heads=h, head_dim=d) for r in range(p)],
            wgu_shards=[O.shard(wgu, O.COLWISE, p, r, [F, F]) for r in range(p)],
            wdown_shards=[O.shard(wdown, O.ROWWISE, p, r) for r in range(p)],
        )
        res = O.transformer_block_forward(x, n_local_heads=h // p, head_dim=d, **sh)
        if ref is None:
            ref = res
            # tp=1: independent plain computation from torch ops in float64.
            xf = torch.from_numpy(O.bf16_to_f64(x))
            wq = torch.from_numpy(O.bf16_to_f64(wqkv))
            qkv = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16((xf @ wq.T).numpy())))
            qh = qkv[:, :H].reshape(T, h, d).permute(1, 0, 2)
            kh = qkv[:, H:2 * H].reshape(T, h, d).permute(1, 0, 2)
            vh = qkv[:, 2 * H:].reshape(T, h, d).permute(1, 0, 2)
            att = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh).permute(1, 0, 2).reshape(T, H)
            att = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(att.numpy())))
            z1 = att @ torch.from_numpy(O.bf16_to_f64(wout)).T
            z1 = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(z1.numpy())))
            gu = z1 @ torch.from_numpy(O.bf16_to_f64(wgu)).T
            hh = torch.nn.functional.silu(gu[:, :F]) * gu[:, F:]
            hh = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(hh.numpy())))
            z2 = (hh @ torch.from_numpy(O.bf16_to_f64(wdown)).T).numpy()
            rms = math.sqrt(float(np.mean(z2 ** 2)))
            assert np.max(np.abs(res["z"] - z2)) <= 1e-2 * rms
        else:
            rms = math.sqrt(float(np.mean(ref["z"] ** 2)))
            assert np.max(np.abs(res["z"] - ref["z"])) <= 1e-2 * rms, p
            # Every rank's QKV slice equals the matching columns of the tp=1 output.
            Hp = H // p
            for r in range(p):
                full = ref["qkv"][0]
                cols = np.concatenate([np.arange(j * H + r * Hp, j * H + (r + 1) * Hp) for j in range(3)])
                assert np.array_equal(res["qkv"][r], full[:, cols]), (p, r)


def pin_single_stream_block():
    # The fused [1,1,1,3,3] in-projection and the packed [inner, mlp] out-projection:
    # every tp_degree gives the unsharded block (tp_degree 1), and tp_degree 1 equals an
    # independent torch float64 computation from the packed weights.
    T, h, d, ratio = 10, 6, 8, 3
    H, F = h * d, ratio * h * d
    w_in, w_out, x = tp_inputs.single_stream_inputs(63, tokens=T, hidden=H, mlp_ratio=ratio)
    assert O.packed_block_sizes(3 * H + 2 * F, [1, 1, 1, 3, 3]) == [H, H, H, F, F]
    res = {}
    for p in (1, 2, 3, 6):
        win = [O.shard(w_in, O.COLWISE, p, r, [H, H, H, F, F], num_heads=h, head_dim=0) for r in range(p)]
        wout = [O.shard(w_out, O.ROWWISE, p, r, [H, F]) for r in range(p)]
        res[p] = O.single_stream_block_forward(x, win, wout, h // p, d)["z"]
    xt = torch.from_numpy(O.bf16_to_f64(x))
    y = xt @ torch.from_numpy(O.bf16_to_f64(w_in)).T
    qkv = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(y[:, :3 * H].numpy())))
    heads = lambda a: a.reshape(T, h, d).permute(1, 0, 2)  # noqa: E731
    att = torch.nn.functional.scaled_dot_product_attention(heads(qkv[:, :H]), heads(qkv[:, H:2 * H]),
                                                           heads(qkv[:, 2 * H:]))
    att = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(att.permute(1, 0, 2).reshape(T, H).numpy())))
    mlp = torch.nn.functional.silu(y[:, 3 * H:3 * H + F]) * y[:, 3 * H + F:]
    mlp = torch.from_numpy(O.bf16_to_f64(O.f64_to_bf16(mlp.numpy())))
    z = (torch.cat([att, mlp], dim=1) @ torch.from_numpy(O.bf16_to_f64(w_out)).T).numpy()
    rms = math.sqrt(float(np.mean(z ** 2)))
    for p, zp in res.items():
        assert np.max(np.abs(zp - z)) <= 1e-2 * rms, p
    # Asking for a subset of token rows (queries) gives those rows of the full result.
    rows = np.array([1, 4, 9])
    win = [O.shard(w_in, O.COLWISE, 2, r, [H, H, H, F, F]) for r in range(2)]
    wout = [O.shard(w_out, O.ROWWISE, 2, r, [H, F]) for r in range(2)]
    full = O.single_stream_block_forward(x, win, wout, h // 2, d)
    part = O.single_stream_block_forward(x, win, wout, h // 2, d, q_rows=rows)
    assert np.array_equal(part["z"], full["z"][rows])
    for k in ("o", "o_bits", "h", "h_bits"):
        for a, b in zip(part[k], full[k]):
            assert np.array_equal(a, b[rows]), k


def pin_safetensors_reader():
    # A file assembled byte by byte from the published layout: header length (little-endian
    # u64), the JSON header, then data whose offsets count from the first byte after it.
    import os
    import struct
    import tempfile
    from oracle import st_oracle
    hdr = (b'{"__metadata__":{"format":"pt"},'
           b'"w":{"dtype":"BF16","shape":[2,3],"data_offsets":[8,20]},'
           b'"b":{"dtype":"F32","shape":[2],"data_offsets":[0,8]},'
           b'"s":{"dtype":"I8","shape":[],"data_offsets":[20,21]}}')
    data = struct.pack("<2f", 1.5, -2.0) + struct.pack("<6H", 0x3F80, 0xC000, 0x0001, 0x7FC1, 0xFF80, 0x8000) + b"\xfe"
    blob = struct.pack("<Q", len(hdr)) + hdr + data
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "hand.safetensors")
        with open(path, "wb") as f:
            f.write(blob)
        ts, meta = st_oracle.read_safetensors(path)
    assert meta == {"format": "pt"}
    assert sorted(ts) == ["b", "s", "w"]
    assert ts["w"].dtype == np.uint16 and ts["w"].shape == (2, 3)
    assert ts["w"].tolist() == [[0x3F80, 0xC000, 0x0001], [0x7FC1, 0xFF80, 0x8000]]
    assert O.bf16_to_f64(ts["w"][0, :2]).tolist() == [1.0, -2.0]
    assert ts["b"].tolist() == [1.5, -2.0]
    assert ts["s"].shape == () and int(ts["s"]) == -2


ALL_PINS = [pin_bf16_rounding, pin_plan_rejections, pin_packed_blocks, pin_shard_golden, pin_shard_reassembly,
            pin_whole_heads, pin_linear_bruteforce, pin_activations, pin_colwise_concat, pin_swiglu_packed,
            pin_rowwise_sum, pin_rowwise_split_input, pin_combine, pin_attention, pin_block_tp_invariance,
            pin_single_stream_block, pin_safetensors_reader]
