"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

A pin set that still passes with a dropped term, a wrong sign or index, or a
transposed operand would not be pinning the oracle to anything.
"""
import numpy as np
import pytest

import oracle_pins
from oracle import st_oracle
from oracle import tp_oracle as O

_orig = {name: getattr(O, name) for name in dir(O) if callable(getattr(O, name))}
_orig_st = {"read_safetensors": st_oracle.read_safetensors}


def _shard_plain_split(w, style, tp_degree, rank, splits=None, **kw):
    # Ignores the packed blocks: slices straight across the concatenation.
    return _orig["shard"](w, style, tp_degree, rank, None)


def _shard_wrong_rank(w, style, tp_degree, rank, splits=None, **kw):
    return _orig["shard"](w, style, tp_degree, (rank + 1) % tp_degree, splits, **kw)


def _check_plan_sum_only(rows, cols, style, tp_degree, *, rank=None, num_heads=0, head_dim=0, splits=None):
    dim = rows if style == O.COLWISE else cols
    if num_heads > 0 and num_heads % tp_degree:
        raise O.PlanRejected(O.HEADS_NOT_DIVISIBLE, "")
    if dim % tp_degree:
        raise O.PlanRejected(O.SPLIT_NOT_DIVISIBLE, "")
    return list(splits) if splits else [dim]


def _check_plan_heads_reversed(rows, cols, style, tp_degree, *, rank=None, num_heads=0, head_dim=0, splits=None):
    if num_heads > 0 and tp_degree % num_heads:
        raise O.PlanRejected(O.HEADS_NOT_DIVISIBLE, "")
    return _orig["check_plan"](rows, cols, style, tp_degree, rank=rank, num_heads=0, head_dim=head_dim,
                               splits=splits)


def _bf16_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    return (x.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _gelu_no_cubic(x):
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * x))


def _silu_sign(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(x))


def _swiglu_swapped(gate, up):
    return _orig["silu"](up) * np.asarray(gate, dtype=np.float64)


def _linear_drop_last_k(x_bits, w_bits):
    return O.bf16_to_f64(x_bits)[:, :-1] @ O.bf16_to_f64(w_bits)[:, :-1].T


def _linear_transposed(x_bits, w_bits):
    w = O.bf16_to_f64(w_bits)
    x = O.bf16_to_f64(x_bits)
    if w.shape[0] == w.shape[1]:
        return x @ w
    return x @ w.T[:, ::-1]


def _rowwise_bias_per_rank(x_shards, w_shards, bias_bits=None):
    z = 0
    for x, w in zip(x_shards, w_shards):
        z = z + O.linear(x, w)
        if bias_bits is not None:
            z = z + O.bf16_to_f64(bias_bits)[None, :]
    return z


def _rowwise_drop_rank0(x_shards, w_shards, bias_bits=None):
    parts = O.rowwise_partials(x_shards, w_shards)
    z = np.zeros_like(parts[0])
    for p in parts[1:]:
        z = z + p
    return z


def _attention_no_scale(q, k, v, n_heads, head_dim):
    return _orig["attention_core"](np.asarray(q) * np.sqrt(head_dim), k, v, n_heads, head_dim)


def _attention_wrong_axis(q, k, v, n_heads, head_dim):
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    out = np.empty((q.shape[0], n_heads * head_dim))
    for j in range(n_heads):
        c = slice(j * head_dim, (j + 1) * head_dim)
        s = q[:, c] @ k[:, c].T / np.sqrt(head_dim)
        e = np.exp(s - s.max(axis=0, keepdims=True))
        out[:, c] = (e / e.sum(axis=0, keepdims=True)) @ v[:, c]
    return out


def _attention_p_rounded_bf16(q, k, v, n_heads, head_dim):
    # Rounds the probabilities to bf16 before the product with V.
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    out = np.empty((q.shape[0], n_heads * head_dim))
    for j in range(n_heads):
        c = slice(j * head_dim, (j + 1) * head_dim)
        s = q[:, c] @ k[:, c].T / np.sqrt(head_dim)
        e = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, c] = O.bf16_to_f64(O.f64_to_bf16(e / e.sum(axis=1, keepdims=True))) @ v[:, c]
    return out


def _gather_wrong_axis(parts):
    return np.concatenate(list(parts), axis=0)


def _single_stream_concat_swapped(x_bits, w_in_shards, w_out_shards, n_local_heads, head_dim, q_rows=None):
    # Feeds [mlp, attention] to the packed out-projection instead of [attention, mlp].
    res = _orig["single_stream_block_forward"](x_bits, w_in_shards, w_out_shards, n_local_heads, head_dim,
                                               q_rows=q_rows)
    res["z"] = O.rowwise_forward([np.concatenate([h, o], axis=1) for o, h in zip(res["o_bits"], res["h_bits"])],
                                 w_out_shards)
    return res


def _read_offsets_from_file_start(path):
    # Counts data_offsets from the start of the file instead of the end of the header.
    import json
    with open(path, "rb") as f:
        raw = f.read()
    n = int.from_bytes(raw[:8], "little")
    header = json.loads(raw[8:8 + n])
    meta = header.pop("__metadata__", None)
    out = {}
    for name, e in header.items():
        dt = np.dtype(st_oracle.DTYPES[e["dtype"]])
        b, _ = e["data_offsets"]
        cnt = int(np.prod(e["shape"], dtype=np.int64)) if e["shape"] else 1
        out[name] = np.frombuffer(raw, dtype=dt, count=cnt, offset=b).reshape(e["shape"])
    return out, meta


def _read_big_endian(path):
    ts, meta = _orig_st["read_safetensors"](path)
    return {k: v.byteswap() for k, v in ts.items()}, meta


MUTATIONS = {
    "shard_ignores_packed_blocks": ("shard", _shard_plain_split),
    "shard_wrong_rank_offset": ("shard", _shard_wrong_rank),
    "plan_checks_only_the_sum": ("check_plan", _check_plan_sum_only),
    "plan_heads_rule_reversed": ("check_plan", _check_plan_heads_reversed),
    "bf16_truncates": ("f64_to_bf16", _bf16_truncate),
    "gelu_drops_cubic_term": ("gelu_tanh", _gelu_no_cubic),
    "silu_wrong_sign": ("silu", _silu_sign),
    "swiglu_gate_up_swapped": ("swiglu", _swiglu_swapped),
    "linear_drops_last_k": ("linear", _linear_drop_last_k),
    "linear_transposed_operand": ("linear", _linear_transposed),
    "rowwise_bias_per_rank": ("rowwise_forward", _rowwise_bias_per_rank),
    "rowwise_drops_a_partial": ("rowwise_forward", _rowwise_drop_rank0),
    "attention_no_scale": ("attention_core", _attention_no_scale),
    "attention_softmax_wrong_axis": ("attention_core", _attention_wrong_axis),
    "attention_p_rounded_bf16": ("attention_core", _attention_p_rounded_bf16),
    "gather_wrong_axis": ("combine_gather", _gather_wrong_axis),
    "single_stream_concat_swapped": ("single_stream_block_forward", _single_stream_concat_swapped),
}

ST_MUTATIONS = {
    "safetensors_offsets_from_file_start": ("read_safetensors", _read_offsets_from_file_start),
    "safetensors_big_endian": ("read_safetensors", _read_big_endian),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, bad = MUTATIONS[name]
    monkeypatch.setattr(O, attr, bad)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin()
        except Exception as e:  # AssertionError or a shape error: the pin noticed
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(ST_MUTATIONS))
def test_pins_catch_planted_reader_mistake(name, monkeypatch):
    attr, bad = ST_MUTATIONS[name]
    monkeypatch.setattr(st_oracle, attr, bad)
    with pytest.raises(Exception):
        oracle_pins.pin_safetensors_reader()
