"""GB300-native tensor-parallel sharded projections: a thin binding over libtp.so.

Every function here has the name of the C entry point it calls (see
``include/tp.h``) and does argument marshalling only: it checks dtypes,
allocates outputs with PyTorch when the caller passes none, and hands raw
pointers and the current CUDA stream to the library.  All computation runs in
the library's CUDA kernels; there is no other path.  If ``libtp.so`` has not
been built, importing this package raises ImportError.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtp.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python tensor_sharded_linear_tp_gb300/build.py` "
        "(the CUDA library is the only implementation)")

lib = ctypes.CDLL(LIB_PATH)

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_status = ctypes.c_int

# Status codes and enums, mirrored from include/tp.h.
TP_OK = 0
STATUS_NAMES = ["TP_OK", "TP_ERR_INVALID_ARG", "TP_ERR_HEADS_NOT_DIVISIBLE", "TP_ERR_SPLIT_NOT_DIVISIBLE",
                "TP_ERR_SPLIT_SUM", "TP_ERR_NOT_WHOLE_HEADS", "TP_ERR_ALIGNMENT", "TP_ERR_NOT_PINNED",
                "TP_ERR_WORKSPACE", "TP_ERR_CUDA", "TP_ERR_TIMEOUT", "TP_ERR_UNSUPPORTED", "TP_ERR_IO",
                "TP_ERR_FORMAT", "TP_ERR_NOT_FOUND"]
STYLES = {"colwise": 0, "rowwise": 1}
ACTS = {"none": 0, "gelu_tanh": 1, "swiglu": 2}
ACCUM_CHUNKED = 0x100   # TP_ACCUM_CHUNKED (include/tp.h): OR'd into the colwise act argument
REDUCE_MODES = {"none": 0, "workspace": 1, "accum": 2}
COMBINE_MODES = {"gather": 0, "reduce": 1}
MAX_DEGREE = 16
MAX_SPLITS = 16

_SIGS = {
    "tp_validate": (_status, [_i64, _i64, ctypes.c_int, ctypes.c_int, _i64, _i64, ctypes.POINTER(_i64), ctypes.c_int]),
    "tp_shard_shape": (_status, [_i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_i64), ctypes.c_int,
                                 ctypes.POINTER(_i64), ctypes.POINTER(_i64)]),
    "tp_plan_shard": (_status, [_vp, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_i64),
                                ctypes.c_int, _i64, _i64, _vp, _vp]),
    "tp_plan_shard_ranks": (_status, [_vp, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(_i64), ctypes.c_int, _i64, _i64, ctypes.POINTER(_vp), _vp]),
    "tp_linear_colwise": (_status, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_int, _i64,
                                    _i64, _i64, ctypes.POINTER(_vp), _i64, _vp]),
    "tp_linear_rowwise": (_status, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, ctypes.c_int, _i64, _i64, _i64,
                                    ctypes.c_int, _vp, ctypes.c_size_t, _vp, _vp]),
    "tp_linear_rowwise_split_input": (_status, [_vp, _i64, ctypes.POINTER(_vp), _vp, ctypes.c_int, _i64, _i64, _i64,
                                                ctypes.c_int, _vp, ctypes.c_size_t, _vp, _vp]),
    "tp_linear_rowwise_noalloc": (_status, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp, ctypes.c_int, _i64, _i64,
                                            _i64, _vp, _vp]),
    "tp_rowwise_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, _i64, _i64, ctypes.c_int]),
    "tp_attention_heads": (_status, [_vp, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_size_t, _vp, _i64,
                                     _vp]),
    "tp_attention_workspace_bytes": (ctypes.c_size_t, [_i64, ctypes.c_int, ctypes.c_int]),
    "tp_attention_heads_ranks": (_status, [ctypes.c_int, ctypes.POINTER(_vp), _i64, _i64, ctypes.c_int, ctypes.c_int,
                                           _vp, ctypes.c_size_t, ctypes.POINTER(_vp), _i64, _vp]),
    "tp_attention_ranks_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, _i64, ctypes.c_int, ctypes.c_int]),
    "tp_combine": (_status, [ctypes.c_int, ctypes.POINTER(_vp), ctypes.c_int, _i64, _i64, _vp, _vp]),
    "tp_last_error": (ctypes.c_char_p, []),
    "tp_status_name": (ctypes.c_char_p, [ctypes.c_int]),
    "tp_device_status": (_status, [_vp]),
    "tp_abi_version": (ctypes.c_int, []),
    "tp_set_tile_wait_limit_ns": (None, [ctypes.c_uint64]),
    "tp_tile_wait_limit_ns": (ctypes.c_uint64, []),
    # include/tp_safetensors.h
    "tp_st_dtype_size": (ctypes.c_size_t, [ctypes.c_int]),
    "tp_st_open": (_status, [ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(_vp)]),
    "tp_st_close": (_status, [_vp]),
    "tp_st_set_read_mode": (_status, [_vp, ctypes.c_int]),
    "tp_st_read_mode_on_device": (_status, [_vp, ctypes.POINTER(ctypes.c_int)]),
    "tp_st_count": (_i64, [_vp]),
    "tp_st_info": (_status, [_vp, _i64, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_int),
                             ctypes.POINTER(ctypes.c_int), ctypes.POINTER(_i64), ctypes.POINTER(ctypes.c_uint64),
                             ctypes.POINTER(ctypes.c_uint64)]),
    "tp_st_find": (_i64, [_vp, ctypes.c_char_p]),
    "tp_st_plan_shard_ranks": (_status, [_vp, ctypes.c_char_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(_i64), ctypes.c_int, _i64, _i64, ctypes.POINTER(_vp), _vp]),
}
class ShardRequest(ctypes.Structure):
    """Mirror of tp_shard_request (include/tp.h)."""
    _fields_ = [("weight", _vp), ("rows", _i64), ("cols", _i64), ("style", ctypes.c_int), ("tp_degree", ctypes.c_int),
                ("rank_begin", ctypes.c_int), ("rank_count", ctypes.c_int), ("fused_splits", ctypes.POINTER(_i64)),
                ("n_splits", ctypes.c_int), ("num_heads", _i64), ("head_dim", _i64),
                ("dev_outs", ctypes.POINTER(_vp))]


_SIGS["tp_plan_shard_many"] = (_status, [ctypes.POINTER(ShardRequest), ctypes.c_int, _vp])

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


class TPError(RuntimeError):
    """A libtp call returned a status other than TP_OK."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else f"status {status}"
        super().__init__(message or self.name)


def _check(status: int) -> None:
    if status != TP_OK:
        raise TPError(status, lib.tp_last_error().decode())


def _splits(fused_splits):
    if not fused_splits:
        return None, 0
    arr = (_i64 * len(fused_splits))(*[int(s) for s in fused_splits])
    return arr, len(fused_splits)


def _ptrs(tensors):
    return (_vp * len(tensors))(*[_ptr(t) for t in tensors])


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need_bf16(name, t):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_bf16_rows(name, t):
    """bf16 2-D with contiguous rows (any row stride): the library takes the stride."""
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 2 or t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name} must be 2-D with contiguous rows")


# ---------------------------------------------------------------------------
# Plan
# ---------------------------------------------------------------------------

def tp_validate(rows: int, cols: int, style: str, tp_degree: int, num_heads: int = 0, head_dim: int = 0,
                fused_splits: Sequence[int] | None = None) -> None:
    """Raise TPError unless the plan is valid (tp_degree divides the heads, blocks divide, whole heads)."""
    arr, n = _splits(fused_splits)
    _check(lib.tp_validate(rows, cols, STYLES[style], tp_degree, num_heads, head_dim, arr, n))


def tp_shard_shape(rows: int, cols: int, style: str, tp_degree: int,
                   fused_splits: Sequence[int] | None = None) -> tuple[int, int]:
    arr, n = _splits(fused_splits)
    r, c = _i64(), _i64()
    _check(lib.tp_shard_shape(rows, cols, STYLES[style], tp_degree, arr, n, ctypes.byref(r), ctypes.byref(c)))
    return r.value, c.value


# ---------------------------------------------------------------------------
# Shard extraction
# ---------------------------------------------------------------------------

def tp_plan_shard(weight: torch.Tensor, style: str, tp_degree: int, rank: int,
                  fused_splits: Sequence[int] | None = None, num_heads: int = 0, head_dim: int = 0,
                  out: torch.Tensor | None = None, device=None, stream=None) -> torch.Tensor:
    """Rank ``rank``'s dense shard of a bf16 weight, on the GPU.

    ``weight`` is a bf16 [rows, cols] tensor in page-locked host memory
    (shard-on-read: only the slice crosses to the device) or on the GPU.
    """
    _need_bf16("weight", weight)
    rows, cols = weight.shape
    arr, n = _splits(fused_splits)
    if out is None:
        tp_validate(rows, cols, style, tp_degree, num_heads, head_dim, fused_splits)  # before allocating
        shape = tp_shard_shape(rows, cols, style, tp_degree, fused_splits)
        dev = device if device is not None else (weight.device if weight.is_cuda else torch.device("cuda"))
        out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    _check(lib.tp_plan_shard(_ptr(weight), rows, cols, STYLES[style], tp_degree, rank, arr, n, num_heads, head_dim,
                             _ptr(out), _stream(stream)))
    return out


def tp_plan_shard_ranks(weight: torch.Tensor, style: str, tp_degree: int, rank_begin: int = 0,
                        rank_count: int | None = None, fused_splits: Sequence[int] | None = None, num_heads: int = 0,
                        head_dim: int = 0, outs: Sequence[torch.Tensor] | None = None, device=None,
                        stream=None) -> list[torch.Tensor]:
    """Shards of ranks [rank_begin, rank_begin + rank_count) in one launch (default: every rank)."""
    _need_bf16("weight", weight)
    rows, cols = weight.shape
    if rank_count is None:
        rank_count = tp_degree - rank_begin
    arr, n = _splits(fused_splits)
    if outs is None:
        tp_validate(rows, cols, style, tp_degree, num_heads, head_dim, fused_splits)  # before allocating
        shape = tp_shard_shape(rows, cols, style, tp_degree, fused_splits)
        dev = device if device is not None else (weight.device if weight.is_cuda else torch.device("cuda"))
        outs = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(rank_count)]
    _check(lib.tp_plan_shard_ranks(_ptr(weight), rows, cols, STYLES[style], tp_degree, rank_begin, rank_count, arr, n,
                                   num_heads, head_dim, _ptrs(outs) if outs else None, _stream(stream)))
    return list(outs)


# ---------------------------------------------------------------------------
# Projections
# ---------------------------------------------------------------------------

def tp_plan_shard_many(requests: Sequence[dict], device=None, stream=None) -> list[list[torch.Tensor]]:
    """Several tp_plan_shard_ranks extractions in as few launches as possible.

    Each request is a dict with keys weight, style, tp_degree and optionally rank_begin,
    rank_count, fused_splits, num_heads, head_dim, outs (as for tp_plan_shard_ranks).
    Every request is checked before anything is copied.  Returns each request's outputs.
    """
    keep = []
    arr = (ShardRequest * max(1, len(requests)))()
    all_outs = []
    for i, rq in enumerate(requests):
        w = rq["weight"]
        _need_bf16("weight", w)
        rows, cols = w.shape
        style, p = rq["style"], rq["tp_degree"]
        rb = rq.get("rank_begin", 0)
        rc = rq.get("rank_count")
        rc = p - rb if rc is None else rc
        splits = rq.get("fused_splits")
        heads, hd = rq.get("num_heads", 0), rq.get("head_dim", 0)
        outs = rq.get("outs")
        if outs is None:
            tp_validate(rows, cols, style, p, heads, hd, splits)  # before allocating
            shape = tp_shard_shape(rows, cols, style, p, splits)
            dev = device if device is not None else (w.device if w.is_cuda else torch.device("cuda"))
            outs = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(rc)]
        sp, n = _splits(splits)
        ptrs = _ptrs(outs) if outs else None
        keep += [sp, ptrs]
        arr[i] = ShardRequest(_ptr(w), rows, cols, STYLES[style], p, rb, rc, sp, n, heads, hd, ptrs)
        all_outs.append(list(outs))
    _check(lib.tp_plan_shard_many(arr, len(requests), _stream(stream)))
    return all_outs


def tp_linear_colwise(x: torch.Tensor, w_shards: Sequence[torch.Tensor], act: str = "none",
                      bias_shards: Sequence[torch.Tensor | None] | None = None,
                      y_shards: Sequence[torch.Tensor] | None = None, ldy: int = 0, stream=None,
                      chunked: bool = False):
    """Y_r = act(X W_r^T + b_r) for every rank r, one launch.  Returns the list of Y_r.

    chunked=True (act "none" only): the K sum is formed in chunks of 1024 on the tensor core and
    the chunks are added with round-to-nearest (TP_ACCUM_CHUNKED), for outputs that feed
    attention."""
    _need_bf16("x", x)
    p = len(w_shards)
    T, K = x.shape
    N_r = w_shards[0].shape[0]
    for w in w_shards:
        _need_bf16("w_shards[i]", w)
    n_out = N_r // 2 if act == "swiglu" else N_r
    if y_shards is None:
        y_shards = [torch.empty((T, n_out), dtype=torch.bfloat16, device=x.device) for _ in range(p)]
    bias_arr = _ptrs(bias_shards) if bias_shards is not None else None
    code = ACTS[act] | (ACCUM_CHUNKED if chunked else 0)
    _check(lib.tp_linear_colwise(_ptr(x), _ptrs(w_shards), bias_arr, code, p, T, K, N_r, _ptrs(y_shards), ldy,
                                 _stream(stream)))
    return y_shards


def tp_rowwise_workspace_bytes(tp_degree: int, T: int, N: int, mode: str = "workspace") -> int:
    return int(lib.tp_rowwise_workspace_bytes(tp_degree, T, N, REDUCE_MODES[mode]))


def tp_linear_rowwise(x_shards: Sequence[torch.Tensor], w_shards: Sequence[torch.Tensor],
                      bias: torch.Tensor | None = None, mode: str = "accum", workspace: torch.Tensor | None = None,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Z = sum_r X_r W_r^T (+ bias once), one launch.

    mode "accum" / "workspace" return bf16 [T, N]; "none" returns the fp32
    partials [tp_degree, T, N] (join them with ``tp_combine("reduce", ...)``).
    """
    p = len(w_shards)
    T, K_r = x_shards[0].shape
    N = w_shards[0].shape[0]
    for t in list(x_shards) + list(w_shards):
        _need_bf16("shard", t)
    dev = x_shards[0].device
    if out is None:
        if mode == "none":
            out = torch.empty((p, T, N), dtype=torch.float32, device=dev)
        else:
            out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    need = tp_rowwise_workspace_bytes(p, T, N, mode)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.tp_linear_rowwise(_ptrs(x_shards), _ptrs(w_shards), _ptr(bias), p, T, K_r, N, REDUCE_MODES[mode],
                                 _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)))
    return out


def tp_linear_rowwise_split_input(x: torch.Tensor, w_shards: Sequence[torch.Tensor], bias: torch.Tensor | None = None,
                                  mode: str = "accum", workspace: torch.Tensor | None = None,
                                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Z = sum_r X[:, r*K/p:(r+1)*K/p] W_r^T (+ bias once): each rank slices the replicated input itself."""
    _need_bf16_rows("x", x)
    p = len(w_shards)
    T, K = x.shape
    N = w_shards[0].shape[0]
    if out is None:
        shape = (p, T, N) if mode == "none" else (T, N)
        out = torch.empty(shape, dtype=torch.float32 if mode == "none" else torch.bfloat16, device=x.device)
    need = tp_rowwise_workspace_bytes(p, T, N, mode)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.tp_linear_rowwise_split_input(_ptr(x), x.stride(0), _ptrs(w_shards), _ptr(bias), p, T, K, N,
                                             REDUCE_MODES[mode], _ptr(workspace), ws_bytes, _ptr(out),
                                             _stream(stream)))
    return out


NOALLOC_SCRATCH_BYTES = 64 << 20


def tp_linear_rowwise_noalloc(x_shards: Sequence[torch.Tensor], w_shards: Sequence[torch.Tensor],
                              bias: torch.Tensor | None = None, out: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """Rowwise projection with the summed partials, using the library's built-in scratch.

    For callers that may not allocate device memory: the fp32 partials live in
    a fixed 64 MiB array inside libtp.so instead of a caller workspace.  Only
    ``out`` (bf16 [T, N]) is allocated here, and only when none is passed.
    Calls that overlap on the GPU share that array and must be serialised.
    """
    p = len(w_shards)
    T, K_r = x_shards[0].shape
    N = w_shards[0].shape[0]
    for t in list(x_shards) + list(w_shards):
        _need_bf16("shard", t)
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=x_shards[0].device)
    _check(lib.tp_linear_rowwise_noalloc(_ptrs(x_shards), _ptrs(w_shards), _ptr(bias), p, T, K_r, N, _ptr(out),
                                         _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# Attention over a rank's local heads
# ---------------------------------------------------------------------------

def tp_attention_workspace_bytes(T: int, n_heads: int, head_dim: int) -> int:
    return int(lib.tp_attention_workspace_bytes(T, n_heads, head_dim))


def tp_attention_heads(qkv: torch.Tensor, n_heads: int, head_dim: int, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """softmax(Q_h K_h^T / sqrt(d)) V_h for each local head of a rank's QKV output [T, 3*n_heads*d]."""
    _need_bf16_rows("qkv", qkv)
    T = qkv.shape[0]
    width = n_heads * head_dim
    if out is None:
        out = torch.empty((T, width), dtype=torch.bfloat16, device=qkv.device)
    need = tp_attention_workspace_bytes(T, n_heads, head_dim)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.tp_attention_heads(_ptr(qkv), qkv.stride(0), T, n_heads, head_dim, _ptr(workspace), ws_bytes,
                                  _ptr(out), out.stride(0), _stream(stream)))
    return out


def tp_attention_ranks_workspace_bytes(n_ranks: int, T: int, n_heads: int, head_dim: int) -> int:
    return int(lib.tp_attention_ranks_workspace_bytes(n_ranks, T, n_heads, head_dim))


def tp_attention_heads_ranks(qkv: Sequence[torch.Tensor], n_heads: int, head_dim: int,
                             outs: Sequence[torch.Tensor] | None = None, workspace: torch.Tensor | None = None,
                             stream=None) -> list[torch.Tensor]:
    """tp_attention_heads for every rank's QKV output in one call (one launch at head_dim 64 or 128)."""
    n = len(qkv)
    for t in qkv:
        _need_bf16_rows("qkv[r]", t)
    if len({t.stride(0) for t in qkv}) != 1:
        raise ValueError("every rank's qkv must have the same row stride")
    T = qkv[0].shape[0]
    width = n_heads * head_dim
    if outs is None:
        outs = [torch.empty((T, width), dtype=torch.bfloat16, device=qkv[0].device) for _ in range(n)]
    if len({t.stride(0) for t in outs}) != 1:
        raise ValueError("every rank's output must have the same row stride")
    need = tp_attention_ranks_workspace_bytes(n, T, n_heads, head_dim)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=qkv[0].device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.tp_attention_heads_ranks(n, _ptrs(qkv), qkv[0].stride(0), T, n_heads, head_dim, _ptr(workspace),
                                        ws_bytes, _ptrs(outs), outs[0].stride(0), _stream(stream)))
    return list(outs)


# ---------------------------------------------------------------------------
# Join
# ---------------------------------------------------------------------------

def tp_combine(mode: str, partials: Sequence[torch.Tensor], out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """Gather bf16 [T, N_each] slices into [T, p*N_each], or reduce fp32 partials into bf16 [T, N_each]."""
    p = len(partials)
    T, N_each = partials[0].shape
    if out is None:
        cols = N_each * p if mode == "gather" else N_each
        out = torch.empty((T, cols), dtype=torch.bfloat16, device=partials[0].device)
    _check(lib.tp_combine(COMBINE_MODES[mode], _ptrs(partials), p, T, N_each, _ptr(out), _stream(stream)))
    return out


# ---------------------------------------------------------------------------
# Diagnostics
# ---------------------------------------------------------------------------

def tp_last_error() -> str:
    return lib.tp_last_error().decode()


def tp_status_name(status: int) -> str:
    return lib.tp_status_name(status).decode()


def tp_device_status(stream=None) -> None:
    """Synchronise the stream; raise TPError if a kernel gave up on a bounded wait."""
    _check(lib.tp_device_status(_stream(stream)))


def tp_abi_version() -> int:
    return int(lib.tp_abi_version())


def tp_set_tile_wait_limit_ns(ns: int) -> None:
    """Bound, in ns, on a workspace-mode CTA's wait for the other ranks' partials (0: the default 2 s)."""
    lib.tp_set_tile_wait_limit_ns(int(ns))


def tp_tile_wait_limit_ns() -> int:
    return int(lib.tp_tile_wait_limit_ns())


def bf16_from_bits(bits, device=None) -> torch.Tensor:
    """A bf16 tensor holding the given uint16 bit patterns (numpy array), optionally moved to `device`."""
    import numpy as np
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def bits_from_bf16(t: torch.Tensor):
    """uint16 numpy bit patterns of a bf16 tensor (copied to the host)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# Shard-on-read from a safetensors file (include/tp_safetensors.h)
# ---------------------------------------------------------------------------

ST_DTYPES = ["BOOL", "U8", "I8", "F8_E4M3", "F8_E5M2", "I16", "U16", "F16", "BF16", "I32", "U32", "F32", "I64",
             "U64", "F64"]
ST_MAX_DIMS = 8
_ST_TORCH = {"BOOL": "bool", "U8": "uint8", "I8": "int8", "F8_E4M3": "float8_e4m3fn", "F8_E5M2": "float8_e5m2",
             "I16": "int16", "U16": "uint16", "F16": "float16", "BF16": "bfloat16", "I32": "int32", "U32": "uint32",
             "F32": "float32", "I64": "int64", "U64": "uint64", "F64": "float64"}


def st_torch_dtype(dtype: str) -> torch.dtype:
    """The torch dtype holding a safetensors dtype's elements."""
    return getattr(torch, _ST_TORCH[dtype])


def tp_st_dtype_size(dtype: str) -> int:
    return int(lib.tp_st_dtype_size(ST_DTYPES.index(dtype)))


def tp_st_open(path: str, staging_bytes: int = 0) -> int:
    """Open a safetensors file and check its header; returns the handle (close it with tp_st_close)."""
    h = _vp()
    _check(lib.tp_st_open(os.fsencode(path), staging_bytes, ctypes.byref(h)))
    return h.value


def tp_st_close(handle: int) -> None:
    _check(lib.tp_st_close(handle))


ST_READ_MODES = ["auto", "staged", "mapped"]   # tp_st_read_mode order


def tp_st_set_read_mode(handle: int, mode: str) -> None:
    """How the following loads read the file: "auto", "staged" or "mapped"."""
    _check(lib.tp_st_set_read_mode(handle, ST_READ_MODES.index(mode)))


def tp_st_read_mode_on_device(handle: int) -> str:
    """The mode a load on the current device uses ("staged" or "mapped")."""
    m = ctypes.c_int(-1)
    _check(lib.tp_st_read_mode_on_device(handle, ctypes.byref(m)))
    return ST_READ_MODES[m.value]


def tp_st_count(handle: int) -> int:
    return int(lib.tp_st_count(handle))


def tp_st_info(handle: int, index: int) -> dict:
    name = ctypes.c_char_p()
    dtype, ndim = ctypes.c_int(), ctypes.c_int()
    shape = (_i64 * ST_MAX_DIMS)()
    off, nbytes = ctypes.c_uint64(), ctypes.c_uint64()
    _check(lib.tp_st_info(handle, index, ctypes.byref(name), ctypes.byref(dtype), ctypes.byref(ndim), shape,
                          ctypes.byref(off), ctypes.byref(nbytes)))
    return {"name": name.value.decode("utf-8"), "dtype": ST_DTYPES[dtype.value],
            "shape": tuple(shape[i] for i in range(ndim.value)), "offset": off.value, "nbytes": nbytes.value}


def tp_st_find(handle: int, name: str) -> int:
    return int(lib.tp_st_find(handle, name.encode("utf-8")))


def _st_shard_shape(info: dict, style: str, tp_degree: int) -> tuple:
    shape = info["shape"]
    if style == "colwise":
        if not shape:
            return ()
        return (shape[0] // tp_degree, *shape[1:])
    return (shape[0], shape[1] // tp_degree) if len(shape) == 2 else shape


def tp_st_plan_shard_ranks(handle: int, name: str, style: str, tp_degree: int, rank_begin: int = 0,
                           rank_count: int | None = None, fused_splits: Sequence[int] | None = None,
                           num_heads: int = 0, head_dim: int = 0, outs: Sequence[torch.Tensor] | None = None,
                           device=None, stream=None) -> list[torch.Tensor]:
    """Ranks [rank_begin, rank_begin + rank_count)'s shards of tensor ``name``, read from the file to the GPU."""
    if rank_count is None:
        rank_count = tp_degree - rank_begin
    arr, n = _splits(fused_splits)
    if outs is None:
        idx = tp_st_find(handle, name)
        if idx < 0:
            raise TPError(STATUS_NAMES.index("TP_ERR_NOT_FOUND"), f"TP_ERR_NOT_FOUND: no tensor {name!r}")
        info = tp_st_info(handle, idx)
        # Validate before allocating: a refused plan allocates nothing.
        _check(lib.tp_st_plan_shard_ranks(handle, name.encode("utf-8"), STYLES[style], tp_degree, rank_begin, 0, arr,
                                          n, num_heads, head_dim, None, None))
        dev = device if device is not None else torch.device("cuda")
        outs = [torch.empty(_st_shard_shape(info, style, tp_degree), dtype=st_torch_dtype(info["dtype"]), device=dev)
                for _ in range(rank_count)]
    _check(lib.tp_st_plan_shard_ranks(handle, name.encode("utf-8"), STYLES[style], tp_degree, rank_begin, rank_count,
                                      arr, n, num_heads, head_dim, _ptrs(outs) if outs else None, _stream(stream)))
    return list(outs)


class SafetensorsFile:
    """A safetensors file opened for shard-on-read (closes on exit of a ``with`` block)."""

    def __init__(self, path: str, staging_bytes: int = 0, read_mode: str = "auto"):
        self.handle = tp_st_open(path, staging_bytes)
        if read_mode != "auto":
            try:
                tp_st_set_read_mode(self.handle, read_mode)
            except BaseException:
                self.close()
                raise

    def read_mode_on_device(self) -> str:
        return tp_st_read_mode_on_device(self.handle)

    def tensors(self) -> list[dict]:
        return [tp_st_info(self.handle, i) for i in range(tp_st_count(self.handle))]

    def shard_ranks(self, name: str, style: str, tp_degree: int, **kw) -> list[torch.Tensor]:
        return tp_st_plan_shard_ranks(self.handle, name, style, tp_degree, **kw)

    def close(self) -> None:
        if self.handle:
            h, self.handle = self.handle, None
            tp_st_close(h)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
