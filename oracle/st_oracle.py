"""CPU oracle (test infrastructure): reading a safetensors checkpoint, for the shard-on-read tests.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
module; the product path never does.

"Tensor parallelism" page, §Load a sharded model and §Limitations: the
tensor-parallel loading path reads safetensors files (non-safetensors weights
raise).  The pages do not define the file format; this reader follows the
published safetensors layout, read plainly: the first 8 bytes are the header
length N as a little-endian unsigned integer, the next N bytes a JSON object
mapping each tensor name to its dtype, shape and [begin, end) data offsets,
counted from the first byte after the header (the key "__metadata__", if
present, holds string metadata and is not a tensor); a tensor's bytes are its
elements in row-major order.  The whole file is read into memory (this is a
checker, not a loader), and each tensor comes back as a numpy array of its
dtype -- bf16 as uint16 bit patterns, the 8-bit float types as uint8 bytes.

Parity: pinned by a hand-assembled file whose every byte follows from the
layout above (tests/oracle_pins.py, pin_safetensors_reader).
"""
from __future__ import annotations

import json

import numpy as np

DTYPES = {
    "BOOL": np.bool_, "U8": np.uint8, "I8": np.int8, "F8_E4M3": np.uint8, "F8_E5M2": np.uint8,
    "I16": np.int16, "U16": np.uint16, "F16": np.float16, "BF16": np.uint16, "I32": np.int32,
    "U32": np.uint32, "F32": np.float32, "I64": np.int64, "U64": np.uint64, "F64": np.float64,
}


def read_safetensors(path: str):
    """Return ({name: array}, metadata dict or None) for a safetensors file."""
    with open(path, "rb") as f:
        raw = f.read()
    n = int.from_bytes(raw[:8], "little")
    header = json.loads(raw[8:8 + n].decode("utf-8"))
    data = raw[8 + n:]
    metadata = header.pop("__metadata__", None)
    out = {}
    for name, entry in header.items():
        dt = np.dtype(DTYPES[entry["dtype"]]).newbyteorder("<")
        begin, end = entry["data_offsets"]
        shape = tuple(entry["shape"])
        count = int(np.prod(shape, dtype=np.int64)) if shape else 1
        if end - begin != count * dt.itemsize or end > len(data):
            raise ValueError(f"tensor {name!r}: offsets [{begin}, {end}) disagree with shape {shape}")
        out[name] = np.frombuffer(data, dtype=dt, count=count, offset=begin).reshape(shape).astype(dt.newbyteorder("="))
    return out, metadata
