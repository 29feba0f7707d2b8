"""Seeded synthetic inputs for the tensor-parallel sharded projection.

This module only draws random numbers and stores them as bf16 bit patterns.
It holds none of the method's arithmetic (no sharding, no products, no
activations), so the CPU oracle and the CUDA path can both consume its
tensors without sharing any of the computation they are checked on.

Recipe (one generator per tensor, so tensors never depend on each other):

* ``np.random.default_rng([seed, tensor_index])`` (PCG64) for tensor number
  ``tensor_index`` of a workload; tensors are numbered weights first, in the
  order they are used inside a block, then activations.
* Normal tensors: ``standard_normal(float32) * sigma`` rounded to bf16 with
  round-to-nearest-even; sigma = 0.02 for weights and 1.0 for activations.
* Integer tensors (exactness cases): uniform integers in ``[-lim, lim]``,
  which are exact in bf16 for ``lim <= 256``.
* Bit tensors (copy cases): uniform 16-bit patterns, NaN and Inf encodings
  included.

Everything returned is a C-contiguous ``numpy.uint16`` array of bf16 bits.
"""
from __future__ import annotations

import numpy as np

WEIGHT_SIGMA = 0.02
ACT_SIGMA = 1.0


def _rng(seed: int, index: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(index)])


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Store finite float32 values as bf16 bits, rounding to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(seed: int, index: int, shape, sigma: float) -> np.ndarray:
    """N(0, sigma^2) samples stored as bf16 bits."""
    x = _rng(seed, index).standard_normal(size=tuple(shape), dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return _f32_to_bf16_bits(x)


def weight_bf16(seed: int, index: int, shape) -> np.ndarray:
    return normal_bf16(seed, index, shape, WEIGHT_SIGMA)


def activation_bf16(seed: int, index: int, shape) -> np.ndarray:
    return normal_bf16(seed, index, shape, ACT_SIGMA)


def int_bf16(seed: int, index: int, shape, lim: int = 4) -> np.ndarray:
    """Uniform integers in [-lim, lim] stored as bf16 bits (exact for lim <= 256)."""
    assert 0 <= lim <= 256
    v = _rng(seed, index).integers(-lim, lim + 1, size=tuple(shape), dtype=np.int32)
    return _f32_to_bf16_bits(v.astype(np.float32))


def random_bits(seed: int, index: int, shape) -> np.ndarray:
    """Uniform 16-bit patterns (any bf16 encoding, NaN/Inf/subnormal included)."""
    return _rng(seed, index).integers(0, 1 << 16, size=tuple(shape), dtype=np.uint16)


def sample_rows(seed: int, n_rows: int, n_sample: int) -> np.ndarray:
    """A sorted seeded sample of row indices, for checks that cannot afford every row."""
    n_sample = min(int(n_sample), int(n_rows))
    idx = np.random.default_rng([int(seed), 1_000_003]).choice(n_rows, size=n_sample, replace=False)
    return np.sort(idx)


# ---------------------------------------------------------------------------
# Workloads (tensor shapes and seeds).  Weights are nn.Linear layout
# [out_features, in_features]; activations are [tokens, features].
# ---------------------------------------------------------------------------

WORKLOADS = {
    # Tiny MLP block: up-projection (colwise) -> GELU(tanh) -> down-projection (rowwise).
    "tiny_mlp_tp2": dict(seed=0, tp=2, tokens=64, hidden=256, ffn=1024, heads=4, head_dim=64,
                         act="gelu_tanh"),
    # Attention projections: fused QKV (colwise, whole heads) and out-projection (rowwise).
    "attn_proj_tp4": dict(seed=1, tp=4, tokens=4096, hidden=3072, heads=24, head_dim=128),
    # Large DiT MLP with fused SwiGLU: gate/up (colwise, halves paired) and down (rowwise).
    "swiglu_mlp_tp4": dict(seed=2, tp=4, tokens=4608, hidden=6144, ffn=18432, heads=48, head_dim=128,
                           act="swiglu"),
    # Full attention + MLP block, tp_degree swept (5 and 7 must be rejected: 48 heads).
    "block_sweep": dict(seed=3, tp_list=(1, 2, 3, 4, 6, 8), tp_rejected=(5, 7), tokens=4608,
                        hidden=6144, ffn=18432, heads=48, head_dim=128, act="swiglu"),
    # Single-stream block at the block sweep's sizes: one fused in-projection packed
    # [1,1,1,3,3] (Q, K, V, gate, up at mlp_ratio 3) and a packed rowwise out-projection over
    # [attention, MLP] inputs ([inner_dim, mlp_hidden_dim] = [6144, 18432]).
    "single_stream_tp4": dict(seed=5, tp=4, tokens=4608, hidden=6144, heads=48, head_dim=128, mlp_ratio=3),
    # Eight SwiGLU MLP blocks loaded shard-on-read from pinned host memory.
    "stack8_swiglu_tp4": dict(seed=4, tp=4, blocks=8, tokens=4608, hidden=6144, ffn=18432, heads=48,
                              head_dim=128, act="swiglu"),
}


def tiny_mlp_inputs(seed=0, tokens=64, hidden=256, ffn=1024, kind="normal"):
    """Tensors of the tiny MLP block: (W_up [ffn,hidden], W_down [hidden,ffn], X [tokens,hidden])."""
    if kind == "int":
        return (int_bf16(seed, 0, (ffn, hidden)), int_bf16(seed, 1, (hidden, ffn)),
                int_bf16(seed, 2, (tokens, hidden)))
    return (weight_bf16(seed, 0, (ffn, hidden)), weight_bf16(seed, 1, (hidden, ffn)),
            activation_bf16(seed, 2, (tokens, hidden)))


def attn_proj_inputs(seed=1, tokens=4096, hidden=3072, kind="normal"):
    """Tensors of the attention-projection workload.

    Returns (W_qkv [3*hidden, hidden], W_out [hidden, hidden], X [tokens, hidden],
    A [tokens, hidden]); A stands for the attention output the out-projection reads.
    """
    if kind == "int":
        return (int_bf16(seed, 0, (3 * hidden, hidden)), int_bf16(seed, 1, (hidden, hidden)),
                int_bf16(seed, 2, (tokens, hidden)), int_bf16(seed, 3, (tokens, hidden)))
    return (weight_bf16(seed, 0, (3 * hidden, hidden)), weight_bf16(seed, 1, (hidden, hidden)),
            activation_bf16(seed, 2, (tokens, hidden)), activation_bf16(seed, 3, (tokens, hidden)))


def swiglu_mlp_inputs(seed=2, tokens=4608, hidden=6144, ffn=18432, kind="normal", index_base=0):
    """Tensors of one SwiGLU MLP block: (W_gate_up [2*ffn, hidden], W_down [hidden, ffn], X [tokens, hidden])."""
    b = index_base
    if kind == "int":
        return (int_bf16(seed, b + 0, (2 * ffn, hidden)), int_bf16(seed, b + 1, (hidden, ffn)),
                int_bf16(seed, b + 2, (tokens, hidden)))
    return (weight_bf16(seed, b + 0, (2 * ffn, hidden)), weight_bf16(seed, b + 1, (hidden, ffn)),
            activation_bf16(seed, b + 2, (tokens, hidden)))


def block_inputs(seed=3, tokens=4608, hidden=6144, ffn=18432, kind="normal"):
    """Tensors of one attention + SwiGLU MLP block.

    Returns (W_qkv [3*hidden, hidden], W_out [hidden, hidden], W_gate_up [2*ffn, hidden],
    W_down [hidden, ffn], X [tokens, hidden]).
    """
    shapes = [(3 * hidden, hidden), (hidden, hidden), (2 * ffn, hidden), (hidden, ffn)]
    if kind == "int":
        ws = [int_bf16(seed, i, s) for i, s in enumerate(shapes)]
        return (*ws, int_bf16(seed, 4, (tokens, hidden)))
    ws = [weight_bf16(seed, i, s) for i, s in enumerate(shapes)]
    return (*ws, activation_bf16(seed, 4, (tokens, hidden)))


def stack_weight(seed: int, block: int, which: str, hidden=6144, ffn=18432) -> np.ndarray:
    """One weight of the stacked SwiGLU workload: which in {"gate_up", "down"}; block-major numbering."""
    if which == "gate_up":
        return weight_bf16(seed, 2 * block, (2 * ffn, hidden))
    if which == "down":
        return weight_bf16(seed, 2 * block + 1, (hidden, ffn))
    raise ValueError(which)


def stack_input(seed: int, blocks: int, tokens=4608, hidden=6144) -> np.ndarray:
    return activation_bf16(seed, 2 * blocks, (tokens, hidden))


def single_stream_inputs(seed=5, tokens=4608, hidden=6144, mlp_ratio=3, kind="normal"):
    """Tensors of one single-stream block.

    Returns (W_in [3*hidden + 2*ffn, hidden] packed as Q, K, V, gate, up;
    W_out [hidden, hidden + ffn] whose input packs the attention output then the
    MLP hidden state; X [tokens, hidden]), with ffn = mlp_ratio * hidden.
    """
    ffn = mlp_ratio * hidden
    shapes = [(3 * hidden + 2 * ffn, hidden), (hidden, hidden + ffn)]
    if kind == "int":
        return (*[int_bf16(seed, i, s) for i, s in enumerate(shapes)], int_bf16(seed, 2, (tokens, hidden)))
    return (*[weight_bf16(seed, i, s) for i, s in enumerate(shapes)], activation_bf16(seed, 2, (tokens, hidden)))


def write_safetensors(path, tensors, metadata=None, ensure_ascii=True) -> None:
    """Write ``tensors`` (a list of (name, dtype, array)) as a safetensors file.

    The published layout: an 8-byte little-endian header length N, N bytes of
    JSON (each tensor's dtype, shape and [begin, end) data offsets counted from
    the first data byte; an optional "__metadata__" of strings), padded with
    spaces to a multiple of 8, then the tensors' bytes in list order.  Each
    array's raw bytes are written as they are (bf16 as its uint16 bit
    patterns), C order.
    """
    import json
    header = {}
    if metadata is not None:
        header["__metadata__"] = dict(metadata)
    offset = 0
    blobs = []
    for name, dtype, arr in tensors:
        raw = np.ascontiguousarray(arr).tobytes()
        header[name] = {"dtype": dtype, "shape": [int(d) for d in np.shape(arr)],
                        "data_offsets": [offset, offset + len(raw)]}
        blobs.append(raw)
        offset += len(raw)
    text = json.dumps(header, ensure_ascii=ensure_ascii, separators=(",", ":")).encode("utf-8")
    text += b" " * ((-len(text)) % 8)
    with open(path, "wb") as f:
        f.write(len(text).to_bytes(8, "little"))
        f.write(text)
        for raw in blobs:
            f.write(raw)
