"""CPU oracle for the tensor-parallel sharded transformer projection.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  The
product path (the CUDA library under ``tensor_sharded_linear_tp_gb300`` and
its binding) never imports it, and this module imports nothing from there.

What it computes, and where the definition comes from (diffusers
documentation, "Tensor parallelism" page, English edition, unless noted):

* Plan checks -- §Load a sharded model (tp_degree must divide the number of
  attention heads) and §Constraints and verification (every packed block must
  be divisible by tp_degree on its own, checked before any weight is touched).
* Shard extraction -- §Colwise and rowwise table ("colwise" shards weight
  dim 0, "rowwise" shards weight dim 1) and §Fused projections (a packed
  Linear is sharded block by block, so each rank keeps the same slice of
  every logical sub-projection).
* Colwise projection -- each rank computes a slice of the output
  (§Colwise and rowwise); slices are joined by concatenation (AllGather,
  opening paragraph of the page).
* Rowwise projection -- each rank computes a partial sum from its slice of
  the input features; partials are joined by summation (AllReduce, opening
  paragraph and §Colwise and rowwise: one AllReduce per colwise/rowwise pair).
* Attention heads -- the colwise Q, K and V projections give each rank a
  subset of heads (§Colwise and rowwise), so attention runs per rank over its
  local heads.

The pages give no arithmetic precision and no activation; the readings taken
here (bf16 storage with round-to-nearest-even, fp64 accumulation, GELU with
the tanh form, SwiGLU with the gate block first, no mask/norm/residual) are
the plainest ones the rest of the text supports, and each function says so.

Everything is plain numpy in float64.  A float64 matrix product (BLAS) is the
only library primitive used as a step.  No blocking, fusion or reordering is
done beyond what the definitions state.

Parity status: every function below is pinned by ``tests/test_oracle_*.py``
against closed forms, brute force on tiny inputs, library routines for the
special cases (torch's bf16 conversion, GELU, SiLU and scaled-dot-product
attention in float64) and hand-derived fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np

COLWISE = "colwise"
ROWWISE = "rowwise"

# Reasons a plan is rejected, named like the library's status codes.
INVALID_ARG = "INVALID_ARG"
HEADS_NOT_DIVISIBLE = "HEADS_NOT_DIVISIBLE"
SPLIT_NOT_DIVISIBLE = "SPLIT_NOT_DIVISIBLE"
SPLIT_SUM = "SPLIT_SUM"
NOT_WHOLE_HEADS = "NOT_WHOLE_HEADS"


class PlanRejected(ValueError):
    """A sharding plan that the pages say must raise before any weight is loaded."""

    def __init__(self, reason: str, message: str):
        super().__init__(f"{reason}: {message}")
        self.reason = reason


# ---------------------------------------------------------------------------
# Plan: packed blocks and the divisibility rules
# ---------------------------------------------------------------------------

def packed_block_sizes(dim: int, blocks: Sequence[int]) -> list[int]:
    """Absolute sizes of the packed blocks of a fused dimension.

    "Tensor parallelism" page, §Fused projections: ``blocks`` is a list of
    proportional integers whose sum divides the packed dimension (e.g. [1, 1]
    for SwiGLU gate and up, [1, 1, 1, 3, 3] for Q, K, V, gate, up at
    mlp_ratio 3).  Reading: one unit is ``dim / sum(blocks)`` rows and block i
    spans ``blocks[i]`` units.
    """
    blocks = [int(b) for b in blocks]
    if not blocks or any(b <= 0 for b in blocks):
        raise PlanRejected(INVALID_ARG, f"blocks must be positive integers, got {blocks}")
    total = sum(blocks)
    if dim % total != 0:
        raise PlanRejected(SPLIT_SUM, f"sum(blocks)={total} does not divide the packed dim {dim}")
    unit = dim // total
    return [unit * b for b in blocks]


def check_plan(rows: int, cols: int, style: str, tp_degree: int, *, rank: int | None = None,
               num_heads: int = 0, head_dim: int = 0, splits: Sequence[int] | None = None) -> list[int]:
    """Validate one weight's sharding plan; return the absolute block sizes.

    Rules, in the order they are checked:

    1. Arguments: ``tp_degree >= 1``, ``0 <= rank < tp_degree``, non-negative
       shape, style "colwise" or "rowwise", positive split sizes.
    2. "Tensor parallelism" page, §Load a sharded model and §Constraints and
       verification: tp_degree must divide the attention-head count
       (``num_heads`` > 0 turns this on; it is a model-wide rule).
    3. §Fused projections: the packed blocks must cover the sharded dimension
       (their sum equals it).
    4. §Constraints and verification: every packed block must be divisible by
       tp_degree on its own, not only their sum.
    5. §Colwise and rowwise (Q, K, V give each rank a subset of heads): when
       the sharded dimension is made of heads (``head_dim`` > 0), each rank's
       part of every block holds whole heads.
    """
    if style not in (COLWISE, ROWWISE):
        raise PlanRejected(INVALID_ARG, f"unknown style {style!r}")
    if tp_degree < 1:
        raise PlanRejected(INVALID_ARG, f"tp_degree must be >= 1, got {tp_degree}")
    if rank is not None and not (0 <= rank < tp_degree):
        raise PlanRejected(INVALID_ARG, f"rank {rank} outside [0, {tp_degree})")
    if rows < 0 or cols < 0 or num_heads < 0 or head_dim < 0:
        raise PlanRejected(INVALID_ARG, "sizes must be non-negative")
    dim = rows if style == COLWISE else cols
    if splits is None or len(splits) == 0:
        sizes = [dim]
    else:
        sizes = [int(s) for s in splits]
        if any(s <= 0 for s in sizes):
            raise PlanRejected(INVALID_ARG, f"split sizes must be positive, got {sizes}")
    if num_heads > 0 and num_heads % tp_degree != 0:
        raise PlanRejected(HEADS_NOT_DIVISIBLE,
                           f"tp_degree={tp_degree} does not divide num_heads={num_heads}")
    if sum(sizes) != dim:
        raise PlanRejected(SPLIT_SUM, f"blocks sum to {sum(sizes)}, sharded dim is {dim}")
    for s in sizes:
        if s % tp_degree != 0:
            raise PlanRejected(SPLIT_NOT_DIVISIBLE, f"block of {s} not divisible by tp_degree={tp_degree}")
    if head_dim > 0:
        for s in sizes:
            if (s // tp_degree) % head_dim != 0:
                raise PlanRejected(NOT_WHOLE_HEADS,
                                   f"block of {s} split {tp_degree} ways is not whole heads of {head_dim}")
    return sizes


def shard_shape(rows: int, cols: int, style: str, tp_degree: int, splits=None) -> tuple[int, int]:
    """Shape of every rank's dense shard: the sharded dimension divided by tp_degree."""
    check_plan(rows, cols, style, tp_degree, splits=splits)
    if style == COLWISE:
        return rows // tp_degree, cols
    return rows, cols // tp_degree


# ---------------------------------------------------------------------------
# Shard extraction (a pure copy: works on any dtype, bf16 bit patterns included)
# ---------------------------------------------------------------------------

def shard(w: np.ndarray, style: str, tp_degree: int, rank: int, splits=None, *,
          num_heads: int = 0, head_dim: int = 0) -> np.ndarray:
    """Rank ``rank``'s slice of weight ``w`` ([out_features, in_features]).

    "Tensor parallelism" page, §Colwise and rowwise: "colwise" shards
    dimension 0 (output features), "rowwise" shards dimension 1 (input
    features).  §Fused projections: a packed dimension is sharded block by
    block -- block b (offset o_b, size s_b) contributes its part
    ``[o_b + rank*s_b/p, o_b + (rank+1)*s_b/p)`` and the parts are
    concatenated in block order, so the rank holds the same slice of every
    logical sub-projection.  With one block this is the plain even split.
    The plan is validated first (see ``check_plan``).
    """
    rows, cols = w.shape
    sizes = check_plan(rows, cols, style, tp_degree, rank=rank, num_heads=num_heads,
                       head_dim=head_dim, splits=splits)
    parts = []
    offset = 0
    for s in sizes:
        part = s // tp_degree
        lo = offset + rank * part
        if style == COLWISE:
            parts.append(w[lo:lo + part, :])
        else:
            parts.append(w[:, lo:lo + part])
        offset += s
    axis = 0 if style == COLWISE else 1
    return np.ascontiguousarray(np.concatenate(parts, axis=axis))


# ---------------------------------------------------------------------------
# bf16 storage.  The pages run the model in bf16 (dtype=torch.bfloat16 in the
# loading example); the reading taken is: values are stored in bf16 wherever
# a tensor is materialised, rounded to nearest with ties to even.
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact: bf16 is the top half of binary32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (round to nearest, ties to even); return the bits.

    bf16 keeps 8 significant bits and binary32's exponent range: a value with
    leading bit 2^e is rounded to a multiple of 2^(e-7) for e >= -126, and to a
    multiple of 2^-133 (the subnormal spacing) below that.  The rounding is done
    once, directly from float64 (no double rounding through binary32).
    Overflow goes to infinity; NaN becomes the quiet NaN 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    nan = np.isnan(x)
    xs = np.where(nan, 0.0, x)
    _, e = np.frexp(np.abs(xs))            # |x| in [2^(e-1), 2^e)
    quantum_exp = np.maximum((e - 1) - 7, -133)
    q = np.ldexp(np.rint(np.ldexp(xs, -quantum_exp)), quantum_exp)   # np.rint: ties to even
    with np.errstate(over="ignore"):
        f = q.astype(np.float32)           # exact, or +-inf past the bf16 range
    out[...] = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out[nan] = 0x7FC0
    return out


# ---------------------------------------------------------------------------
# Activations (fused after the colwise projection)
# ---------------------------------------------------------------------------

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)


def gelu_tanh(x: np.ndarray) -> np.ndarray:
    """GELU, tanh form: 0.5*x*(1 + tanh(sqrt(2/pi)*(x + 0.044715*x^3))).

    The pages name no activation; the tiny MLP workload uses GELU(tanh).
    """
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + 0.044715 * x * x * x)))


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU: x * sigmoid(x) = x / (1 + exp(-x))."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SwiGLU: silu(gate) * up.

    "Tensor parallelism" page, §Fused projections: [1, 1] packs "a SwiGLU gate
    and up projection of equal halves".  Reading: the gate block comes first
    in the packed weight and the up block second.
    """
    return silu(gate) * np.asarray(up, dtype=np.float64)


# ---------------------------------------------------------------------------
# Projections
# ---------------------------------------------------------------------------

def linear(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """Plain nn.Linear without bias in float64: Y = X @ W^T, W is [out, in]."""
    return bf16_to_f64(x_bits) @ bf16_to_f64(w_bits).T


def apply_act(acc: np.ndarray, act: str) -> np.ndarray:
    """Activation applied to the unrounded accumulator (the fused-epilogue reading).

    ``act`` is "none", "gelu_tanh" or "swiglu".  For "swiglu" the accumulator's
    first half of columns is the gate and the second half the up projection of
    the same rank (the rank's shard is [gate_r; up_r], see ``shard``).
    """
    if act == "none":
        return acc
    if act == "gelu_tanh":
        return gelu_tanh(acc)
    if act == "swiglu":
        n = acc.shape[1]
        assert n % 2 == 0, "swiglu needs an even number of accumulator columns"
        return swiglu(acc[:, : n // 2], acc[:, n // 2:])
    raise ValueError(f"unknown activation {act!r}")


def colwise_forward(x_bits: np.ndarray, w_shards: Sequence[np.ndarray], act: str = "none",
                    bias_shards: Sequence[np.ndarray] | None = None) -> list[np.ndarray]:
    """Colwise-sharded projection: rank r computes Y_r = act(X @ W_r^T + b_r) (float64).

    "Tensor parallelism" page, §Colwise and rowwise: the input X is replicated,
    each rank holds a slice of the output features and computes that slice of
    the output.  The bias (none in the workloads) is sharded like the weight's
    rows.  The returned values are unrounded; ``f64_to_bf16`` gives what a rank
    stores.
    """
    out = []
    for r, w in enumerate(w_shards):
        acc = linear(x_bits, w)
        if bias_shards is not None and bias_shards[r] is not None:
            acc = acc + bf16_to_f64(bias_shards[r])[None, :]
        out.append(apply_act(acc, act))
    return out


def rowwise_partials(x_shards: Sequence[np.ndarray], w_shards: Sequence[np.ndarray]) -> list[np.ndarray]:
    """Rowwise-sharded projection: rank r computes the partial P_r = X_r @ W_r^T (float64).

    "Tensor parallelism" page, §Colwise and rowwise: "rowwise" shards the input
    features and each rank computes a partial sum from its slice.
    """
    return [linear(x, w) for x, w in zip(x_shards, w_shards)]


def rowwise_forward(x_shards, w_shards, bias_bits: np.ndarray | None = None) -> np.ndarray:
    """Rowwise projection joined by summation: Z = sum_r P_r (+ bias once), float64.

    The partials are added in rank order.  The bias is added once, after the
    sum (adding it on every rank would count it tp_degree times); the pages do
    not discuss bias, this is the plainest reading.
    """
    parts = rowwise_partials(x_shards, w_shards)
    z = np.zeros_like(parts[0])
    for p in parts:
        z = z + p
    if bias_bits is not None:
        z = z + bf16_to_f64(bias_bits)[None, :]
    return z


def rowwise_split_input_forward(x_bits: np.ndarray, w_shards, bias_bits: np.ndarray | None = None) -> np.ndarray:
    """"rowwise_split_input": the input X is replicated and each rank takes its own slice of it.

    "Tensor parallelism" page, §Colwise and rowwise table: the style shards the
    weight's input features like "rowwise", but the rank computes its partial
    from its slice of the replicated input (e.g. an AdaLN modulation projection
    reading the timestep embedding), and the AllReduce sum gives every rank all
    output features.  Rank r's slice is columns [r*K/p, (r+1)*K/p) of X.
    """
    p = len(w_shards)
    x_shards = [shard(x_bits, ROWWISE, p, r) for r in range(p)]
    return rowwise_forward(x_shards, w_shards, bias_bits)


def combine_gather(parts: Sequence[np.ndarray]) -> np.ndarray:
    """AllGather of colwise outputs: concatenate rank slices along the feature axis."""
    return np.ascontiguousarray(np.concatenate(list(parts), axis=1))


def combine_reduce(parts: Sequence[np.ndarray]) -> np.ndarray:
    """AllReduce of rowwise partials: their sum in rank order, float64."""
    z = np.zeros(np.shape(parts[0]), dtype=np.float64)
    for p in parts:
        z = z + np.asarray(p, dtype=np.float64)
    return z


# ---------------------------------------------------------------------------
# Attention over a rank's local heads
# ---------------------------------------------------------------------------

def attention_core(q: np.ndarray, k: np.ndarray, v: np.ndarray, n_heads: int, head_dim: int) -> np.ndarray:
    """softmax(Q_h K_h^T / sqrt(d)) V_h for each of the rank's local heads, float64.

    "Tensor parallelism" page, §Colwise and rowwise: colwise Q, K and V give
    each rank a subset of heads, so attention needs no communication.  The
    pages define no attention variant; reading: no mask, no positional
    embedding, no QK-norm (norms are replicated and left out of the plan,
    §What to leave out), scale 1/sqrt(head_dim), max-subtracted softmax, head j
    occupying columns [j*d, (j+1)*d) of each of Q, K, V.  ``q`` may hold only
    some query rows; ``k`` and ``v`` hold every token.  The probabilities are
    never rounded: the pages fix no storage for them, so this is the plain
    definition, exact in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    scale = 1.0 / math.sqrt(head_dim)
    out = np.empty((q.shape[0], n_heads * head_dim), dtype=np.float64)
    for j in range(n_heads):
        cols = slice(j * head_dim, (j + 1) * head_dim)
        s = (q[:, cols] @ k[:, cols].T) * scale
        s = s - s.max(axis=1, keepdims=True)
        e = np.exp(s)
        pr = e / e.sum(axis=1, keepdims=True)
        out[:, cols] = pr @ v[:, cols]
    return out


def split_qkv(y: np.ndarray, local_width: int):
    """Q, K, V of one rank from its colwise QKV output [T, 3*local_width]."""
    return y[:, :local_width], y[:, local_width:2 * local_width], y[:, 2 * local_width:]


# ---------------------------------------------------------------------------
# Whole workloads.  Every tensor a rank would store is rounded to bf16 between
# steps; the final value is returned unrounded (the tolerance reference).
# ---------------------------------------------------------------------------

def mlp_forward(x_bits, w_in_shards, w_out_shards, act: str):
    """Colwise in-projection + activation, then rowwise out-projection joined by a sum.

    "Tensor parallelism" page, §Colwise and rowwise: pair "colwise" then
    "rowwise"; the colwise output stays sharded and feeds the rowwise
    projection directly, and one AllReduce at the block boundary rebuilds the
    result.  Returns (h_bits per rank, Z float64).
    """
    h = [f64_to_bf16(y) for y in colwise_forward(x_bits, w_in_shards, act)]
    z = rowwise_forward(h, w_out_shards)
    return h, z


def attention_block_forward(x_bits, wqkv_shards, wout_shards, n_local_heads: int, head_dim: int,
                            q_rows: np.ndarray | None = None):
    """QKV colwise -> per-rank attention -> out-projection rowwise + sum.

    Returns (qkv_bits per rank, o_bits per rank, Z float64).  With ``q_rows``
    only those token rows are computed for the query side (K and V always use
    every token), which is exact for those rows.  Q, K, V and the attention
    output are stored in bf16 like every tensor the path stores; the
    probabilities are exact (``attention_core``).
    """
    width = n_local_heads * head_dim
    qkv = [f64_to_bf16(y) for y in colwise_forward(x_bits, wqkv_shards, "none")]
    o = []
    for y in qkv:
        qb, kb, vb = split_qkv(y, width)
        if q_rows is not None:
            qb = qb[q_rows]
        o.append(f64_to_bf16(attention_core(bf16_to_f64(qb), bf16_to_f64(kb), bf16_to_f64(vb),
                                            n_local_heads, head_dim)))
    z = rowwise_forward(o, wout_shards)
    return qkv, o, z


def transformer_block_forward(x_bits, wqkv_shards, wout_shards, wgu_shards, wdown_shards,
                              n_local_heads: int, head_dim: int, q_rows: np.ndarray | None = None):
    """Attention + SwiGLU MLP block, both halves sharded colwise -> rowwise.

    x -> QKV (colwise) -> attention over local heads -> out-projection
    (rowwise, summed) -> gate/up (colwise, SwiGLU) -> down (rowwise, summed).
    No norms and no residual: they are replicated modules outside the plan
    ("Tensor parallelism" page, §What to leave out).  Returns a dict of the
    intermediates and the unrounded final output ``z``.
    """
    qkv, o, z1 = attention_block_forward(x_bits, wqkv_shards, wout_shards, n_local_heads, head_dim,
                                         q_rows=q_rows)
    z1_bits = f64_to_bf16(z1)
    h, z2 = mlp_forward(z1_bits, wgu_shards, wdown_shards, "swiglu")
    return dict(qkv=qkv, o=o, z1=z1, z1_bits=z1_bits, h=h, z=z2)


def single_stream_block_forward(x_bits, w_in_shards, w_out_shards, n_local_heads: int, head_dim: int,
                                q_rows: np.ndarray | None = None):
    """Single-stream block: one fused colwise in-projection and one packed rowwise out-projection.

    "Tensor parallelism" page, §Fused projections: [1, 1, 1, 3, 3] packs Q, K,
    V, gate and up (mlp_ratio 3) into one Linear, sharded block by block
    (PackedColwiseParallel), and the single-stream to_out stores its input's
    absolute blocks [inner_dim, mlp_hidden_dim] and is sharded block by block
    along its input (PackedRowwiseParallel).  Rank r's fused output is
    [Q_r, K_r, V_r, gate_r, up_r]; attention runs over its local heads, SwiGLU
    joins gate_r and up_r, and [attention_r, mlp_r] -- exactly the columns of
    its packed to_out shard -- feeds the rowwise projection; the partials are
    summed.  Returns a dict: per-rank attention output "o" (float64, before its
    bf16 storage) and "o_bits" (stored), per-rank SwiGLU output "h" and
    "h_bits" likewise, and the final "z" (float64).
    """
    width = n_local_heads * head_dim
    rows = x_bits if q_rows is None else x_bits[q_rows]
    res = dict(o=[], o_bits=[], h=[], h_bits=[])
    cs = []
    for w in w_in_shards:
        # The rank's five outputs for the token rows asked for, and K, V for every token.
        y = colwise_forward(rows, [w], "none")[0]
        kv = y[:, width:3 * width] if q_rows is None else colwise_forward(x_bits, [w[width:3 * width]], "none")[0]
        qb = f64_to_bf16(y[:, :width])
        kb, vb = f64_to_bf16(kv[:, :width]), f64_to_bf16(kv[:, width:])
        o = attention_core(bf16_to_f64(qb), bf16_to_f64(kb), bf16_to_f64(vb), n_local_heads, head_dim)
        h = apply_act(y[:, 3 * width:], "swiglu")
        ob, hb = f64_to_bf16(o), f64_to_bf16(h)
        for k, v in (("o", o), ("o_bits", ob), ("h", h), ("h_bits", hb)):
            res[k].append(v)
        cs.append(np.concatenate([ob, hb], axis=1))
    res["z"] = rowwise_forward(cs, w_out_shards)
    return res
