"""The safetensors reader of libtp on the host: header parsing, checks and plan refusals (no GPU).

Opening a file and inspecting its tensors allocates nothing on a GPU, and a
load whose plan is refused fails before any byte is read or any CUDA call is
made, so all of this runs on the CPU.  Expected values come from the oracle's
reader (oracle/st_oracle.py) on files written by tp_inputs.write_safetensors.
"""
import json
import os
import struct

import numpy as np
import pytest

import tp_inputs
from oracle import st_oracle

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")

FAKE = 1 << 40  # a pointer value no call may dereference: refusals happen first


def _status(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except tp.TPError as e:
        return e.name
    return "TP_OK"


def _sample_tensors(seed=0):
    rng = np.random.default_rng(seed)
    return [
        ("blocks.0.attn.to_qkv_mlp.weight", "BF16", tp_inputs.random_bits(seed, 0, (40, 16))),
        ("blocks.0.attn.to_out.weight", "BF16", tp_inputs.random_bits(seed, 1, (16, 24))),
        ("blocks.0.norm.weight", "F32", rng.standard_normal(16).astype(np.float32)),
        ("blocks.0.adaln.linear.weight", "F16", rng.standard_normal((12, 8)).astype(np.float16)),
        ("quant.scales", "I8", rng.integers(-128, 128, (6, 10), dtype=np.int8)),
        ("conv.weight", "F64", rng.standard_normal((4, 2, 3, 3))),
        ("step", "I64", np.array(7, dtype=np.int64)),
        ("empty", "U8", np.zeros((0, 5), dtype=np.uint8)),
    ]


def _write(tmp_path, tensors, name="m.safetensors", **kw):
    path = str(tmp_path / name)
    tp_inputs.write_safetensors(path, tensors, **kw)
    return path


def _table(path):
    with tp.SafetensorsFile(path) as f:
        return {t["name"]: t for t in f.tensors()}


def test_parse_agrees_with_oracle_reader(tmp_path):
    tensors = _sample_tensors()
    path = _write(tmp_path, tensors, metadata={"format": "pt", "note": "a \"quoted\" value"})
    want, meta = st_oracle.read_safetensors(path)
    assert meta["format"] == "pt"
    got = _table(path)
    assert sorted(got) == sorted(want)
    raw = open(path, "rb").read()
    for name, dtype, arr in tensors:
        g = got[name]
        assert g["dtype"] == dtype
        assert g["shape"] == tuple(np.shape(arr))
        assert g["nbytes"] == want[name].nbytes
        # The reported offset addresses the tensor's bytes in the file.
        assert raw[g["offset"]:g["offset"] + g["nbytes"]] == np.ascontiguousarray(want[name]).tobytes()
    offsets = [t["offset"] for t in _table(path).values()]
    assert offsets == sorted(offsets)


@pytest.mark.parametrize("ensure_ascii", [True, False])
def test_names_with_escapes_and_unicode(tmp_path, ensure_ascii):
    names = ["plain", "with \"quotes\" and \\backslash\\", "tab\there/slash", "café.weight",
             "模型.weight", "emoji\U0001F600.bias"]
    tensors = [(n, "U8", np.full((2,), i, dtype=np.uint8)) for i, n in enumerate(names)]
    path = _write(tmp_path, tensors, ensure_ascii=ensure_ascii)
    got = _table(path)
    assert sorted(got) == sorted(names)
    h = tp.tp_st_open(path)
    try:
        for n in names:
            assert tp.tp_st_find(h, n) >= 0
        assert tp.tp_st_find(h, "missing") == -1
    finally:
        tp.tp_st_close(h)


def test_hand_made_header_with_whitespace_and_extra_keys(tmp_path):
    hdr = (b'{ "__metadata__" : { "k" : "v" } ,\n'
           b'  "b" : { "data_offsets" : [ 0 , 8 ] , "shape" : [ 2 ] , "dtype" : "F32" , "extra" : [1, {"x": null}] },\n'
           b'  "a" : { "dtype" : "BF16" , "shape" : [ 1 , 2 ] , "data_offsets" : [ 8 , 12 ] } }   ')
    data = struct.pack("<2f", 1.0, 2.0) + struct.pack("<2H", 1, 2)
    path = tmp_path / "hand.safetensors"
    path.write_bytes(struct.pack("<Q", len(hdr)) + hdr + data)
    got = _table(str(path))
    assert got["b"]["shape"] == (2,) and got["b"]["dtype"] == "F32" and got["b"]["offset"] == 8 + len(hdr)
    assert got["a"]["shape"] == (1, 2) and got["a"]["offset"] == 8 + len(hdr) + 8


def _raw_file(tmp_path, header_obj_or_bytes, data=b"", name="bad.safetensors", length=None):
    hdr = header_obj_or_bytes if isinstance(header_obj_or_bytes, bytes) else json.dumps(header_obj_or_bytes).encode()
    n = len(hdr) if length is None else length
    path = tmp_path / name
    path.write_bytes(struct.pack("<Q", n) + hdr + data)
    return str(path)


def _ok_entry(b=0, e=4, shape=(2,), dtype="BF16"):
    return {"dtype": dtype, "shape": list(shape), "data_offsets": [b, e]}


@pytest.mark.parametrize("case", [
    "short_file", "header_past_end", "header_too_large", "not_json", "not_object", "trailing_text",
    "unknown_dtype", "missing_field", "negative_dim", "fraction_offset", "reversed_offsets",
    "offsets_past_end", "size_mismatch", "overlap", "duplicate_name", "too_many_dims", "bad_escape",
    "lone_surrogate", "deep_nesting",
])
def test_malformed_files_are_refused(tmp_path, case):
    data = bytes(16)
    if case == "short_file":
        path = tmp_path / "short.safetensors"
        path.write_bytes(b"\x01\x02\x03")
        path = str(path)
    elif case == "header_past_end":
        path = _raw_file(tmp_path, {"a": _ok_entry()}, data, length=10 ** 6)
    elif case == "header_too_large":
        path = _raw_file(tmp_path, {"a": _ok_entry()}, data, length=200_000_000)
    elif case == "not_json":
        path = _raw_file(tmp_path, b'{"a": {"dtype": "BF16", "shape": [2], "data_offsets": [0, 4]', data)
    elif case == "not_object":
        path = _raw_file(tmp_path, b'[1, 2, 3]', data)
    elif case == "trailing_text":
        path = _raw_file(tmp_path, json.dumps({"a": _ok_entry()}).encode() + b" x", data)
    elif case == "unknown_dtype":
        path = _raw_file(tmp_path, {"a": _ok_entry(dtype="BF17")}, data)
    elif case == "missing_field":
        path = _raw_file(tmp_path, {"a": {"dtype": "BF16", "shape": [2]}}, data)
    elif case == "negative_dim":
        path = _raw_file(tmp_path, {"a": {"dtype": "BF16", "shape": [-2], "data_offsets": [0, 4]}}, data)
    elif case == "fraction_offset":
        path = _raw_file(tmp_path, b'{"a": {"dtype": "BF16", "shape": [2], "data_offsets": [0, 4.0]}}', data)
    elif case == "reversed_offsets":
        path = _raw_file(tmp_path, {"a": _ok_entry(4, 0)}, data)
    elif case == "offsets_past_end":
        path = _raw_file(tmp_path, {"a": _ok_entry(14, 18)}, data)
    elif case == "size_mismatch":
        path = _raw_file(tmp_path, {"a": _ok_entry(0, 6)}, data)
    elif case == "overlap":
        path = _raw_file(tmp_path, {"a": _ok_entry(0, 4), "b": _ok_entry(2, 6)}, data)
    elif case == "duplicate_name":
        path = _raw_file(tmp_path, b'{"a": {"dtype": "U8", "shape": [1], "data_offsets": [0, 1]}, '
                                   b'"a": {"dtype": "U8", "shape": [1], "data_offsets": [1, 2]}}', data)
    elif case == "too_many_dims":
        path = _raw_file(tmp_path, {"a": {"dtype": "U8", "shape": [1] * 9, "data_offsets": [0, 1]}}, data)
    elif case == "bad_escape":
        path = _raw_file(tmp_path, b'{"a\\q": {"dtype": "U8", "shape": [1], "data_offsets": [0, 1]}}', data)
    elif case == "lone_surrogate":
        path = _raw_file(tmp_path, b'{"a\\ud800": {"dtype": "U8", "shape": [1], "data_offsets": [0, 1]}}', data)
    elif case == "deep_nesting":
        deep = b'[' * 100 + b']' * 100
        path = _raw_file(tmp_path, b'{"__metadata__": ' + deep + b'}', data)
    assert _status(tp.tp_st_open, path) == "TP_ERR_FORMAT", tp.tp_last_error()


def test_missing_file_is_an_io_error(tmp_path):
    assert _status(tp.tp_st_open, str(tmp_path / "nope.safetensors")) == "TP_ERR_IO"
    assert "nope.safetensors" in tp.tp_last_error()


def test_empty_header_is_a_file_without_tensors(tmp_path):
    path = _raw_file(tmp_path, b"{}", b"")
    with tp.SafetensorsFile(path) as f:
        assert f.tensors() == []


def test_plan_refusals_come_before_any_read(tmp_path):
    H, F, heads = 48, 144, 6
    tensors = [("in", "BF16", tp_inputs.random_bits(1, 0, (3 * H + 2 * F, H))),
               ("out", "BF16", tp_inputs.random_bits(1, 1, (H, H + F))),
               ("bias", "BF16", tp_inputs.random_bits(1, 2, (3 * H + 2 * F,))),
               ("conv", "F32", np.zeros((8, 2, 3), dtype=np.float32)),
               ("bytes", "U8", np.zeros((4, 6), dtype=np.uint8))]
    path = _write(tmp_path, tensors)
    h = tp.tp_st_open(path)
    try:
        def load(name, style, p, rank_begin=0, rank_count=1, splits=None, heads_=0, hd=0):
            arr = (tp._i64 * len(splits))(*splits) if splits else None
            n_outs = min(max(1, rank_count), 16)   # a refused call reads none of them
            outs = (tp._vp * n_outs)(*([FAKE] * n_outs))
            st = tp.lib.tp_st_plan_shard_ranks(h, name.encode(), tp.STYLES[style], p, rank_begin, rank_count, arr,
                                               len(splits) if splits else 0, heads_, hd, outs, None)
            return tp.STATUS_NAMES[st]
        assert load("missing", "colwise", 2) == "TP_ERR_NOT_FOUND"
        assert load("in", "colwise", 4, heads_=heads, splits=[H, H, H, F, F]) == "TP_ERR_HEADS_NOT_DIVISIBLE"
        assert load("in", "colwise", 2, splits=[H, H, H, F, F - 1]) == "TP_ERR_SPLIT_SUM"
        assert load("out", "rowwise", 32, splits=[H, F]) == "TP_ERR_SPLIT_NOT_DIVISIBLE"
        assert load("in", "colwise", 3, splits=[H, H, H, F, F], heads_=heads, hd=32) == "TP_ERR_NOT_WHOLE_HEADS"
        assert load("bias", "rowwise", 2) == "TP_ERR_INVALID_ARG"
        assert load("conv", "rowwise", 2) == "TP_ERR_UNSUPPORTED"
        assert load("bytes", "rowwise", 6) == "TP_ERR_UNSUPPORTED"        # 1-byte slices of odd width
        assert load("in", "colwise", 2, rank_begin=1, rank_count=2) == "TP_ERR_INVALID_ARG"
        assert load("in", "colwise", 2, rank_count=-1) == "TP_ERR_INVALID_ARG"
        # A rank count whose sum with rank_begin would overflow an int is still refused.
        assert load("in", "colwise", 2, rank_begin=1, rank_count=2 ** 31 - 1) == "TP_ERR_INVALID_ARG"
        # rank_count 0 validates and reads nothing: the binding's pre-allocation check.
        assert load("in", "colwise", 2, rank_count=0, splits=[H, H, H, F, F]) == "TP_OK"
    finally:
        tp.tp_st_close(h)


def test_rowwise_row_must_fit_the_staging_buffer(tmp_path):
    path = _write(tmp_path, [("w", "BF16", tp_inputs.random_bits(2, 0, (2, 4096)))])
    h = tp.tp_st_open(path, 4096)   # one row is 8192 bytes
    try:
        outs = (tp._vp * 1)(FAKE)
        st = tp.lib.tp_st_plan_shard_ranks(h, b"w", 1, 2, 0, 1, None, 0, 0, 0, outs, None)
        assert tp.STATUS_NAMES[st] == "TP_ERR_UNSUPPORTED"
        assert "staging" in tp.tp_last_error()
    finally:
        tp.tp_st_close(h)


def test_close_of_null_and_count_of_null():
    assert tp.lib.tp_st_close(None) == 0
    assert tp.lib.tp_st_count(None) == -1
    assert tp.lib.tp_st_find(None, b"x") == -1


def test_dtype_sizes():
    sizes = {"BOOL": 1, "U8": 1, "I8": 1, "F8_E4M3": 1, "F8_E5M2": 1, "I16": 2, "U16": 2, "F16": 2, "BF16": 2,
             "I32": 4, "U32": 4, "F32": 4, "I64": 8, "U64": 8, "F64": 8}
    for name, size in sizes.items():
        assert tp.tp_st_dtype_size(name) == size
        assert np.dtype(st_oracle.DTYPES[name]).itemsize == size


def test_read_mode_choice_needs_no_gpu(tmp_path):
    path = _write(tmp_path, [("w", "BF16", tp_inputs.random_bits(3, 0, (4, 8)))])
    h = tp.tp_st_open(path)
    try:
        tp.tp_st_set_read_mode(h, "staged")
        assert tp.tp_st_read_mode_on_device(h) == "staged"   # staged is never resolved against a device
        for bad in (-1, 3, 1000):
            assert tp.STATUS_NAMES[tp.lib.tp_st_set_read_mode(h, bad)] == "TP_ERR_INVALID_ARG"
        assert tp.tp_st_read_mode_on_device(h) == "staged"   # a refused value changes nothing
        assert tp.STATUS_NAMES[tp.lib.tp_st_set_read_mode(None, 0)] == "TP_ERR_INVALID_ARG"
        assert tp.STATUS_NAMES[tp.lib.tp_st_read_mode_on_device(h, None)] == "TP_ERR_INVALID_ARG"
    finally:
        tp.tp_st_close(h)
    with pytest.raises(ValueError):
        tp.SafetensorsFile(path, read_mode="mmap")
