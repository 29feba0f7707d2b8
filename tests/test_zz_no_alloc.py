"""The allocation-free rowwise entry point, tp_linear_rowwise_noalloc.

Some callers may not allocate device memory (a plug-in inside a framework
that owns every byte of the GPU, or a process whose memory a pool claimed up
front).  For them the library keeps its rowwise scratch in a fixed array of
its own.  This test calls that entry point through the C ABI and checks it
against the ordinary workspace entry point on two calls in a row, so that a
second call on a scratch array that still holds the first call's partials
and counters gives the right answer too.  The file sorts last, so a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import tp_inputs
from oracle import tp_oracle as O
from tolerance import assert_close

pytestmark = pytest.mark.gpu

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")


def _noalloc_raw(xs, ws, bias, out):
    """Call the C entry point directly with raw device pointers."""
    p = len(ws)
    T, K_r = xs[0].shape
    N = ws[0].shape[0]
    xp = (ctypes.c_void_p * p)(*[t.data_ptr() for t in xs])
    wp = (ctypes.c_void_p * p)(*[t.data_ptr() for t in ws])
    st = tp.lib.tp_linear_rowwise_noalloc(xp, wp, None if bias is None else bias.data_ptr(), p, T, K_r, N,
                                          out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return tp.STATUS_NAMES[st]


def _case(seed, T, K_r, N, p):
    x = tp_inputs.activation_bf16(seed, 0, (T, K_r * p))
    w = tp_inputs.weight_bf16(seed, 1, (N, K_r * p))
    b = tp_inputs.weight_bf16(seed, 2, (N,))
    xs = [tp.bf16_from_bits(O.shard(x, "rowwise", p, r), "cuda") for r in range(p)]
    ws = [tp.bf16_from_bits(O.shard(w, "rowwise", p, r), "cuda") for r in range(p)]
    return xs, ws, tp.bf16_from_bits(b, "cuda")


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # Two different problems back to back through the same built-in scratch array.
    for seed, (T, K_r, N, p) in ((140, (300, 200, 520, 4)), (141, (1000, 512, 1040, 3))):
        xs, ws, b = _case(seed, T, K_r, N, p)
        ref = tp.tp_linear_rowwise(xs, ws, bias=b, mode="workspace")
        out = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc_raw(xs, ws, b, out) == "TP_OK", tp.tp_last_error()
        tp.tp_device_status()
        got = O.bf16_to_f64(tp.bits_from_bf16(out))
        want = O.bf16_to_f64(tp.bits_from_bf16(ref))
        assert_close(got, want, f"noalloc call seed {seed}")


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # p*T*N*4 bytes of partials above 64 MiB: refused on the host before any device work.
    p, T, K_r, N = 4, 4096, 64, 1536
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "workspace") > tp.NOALLOC_SCRATCH_BYTES
    fake = (ctypes.c_void_p * p)(*([0x10000] * p))
    st = tp.lib.tp_linear_rowwise_noalloc(fake, fake, None, p, T, K_r, N, 0x10000, None)
    assert tp.STATUS_NAMES[st] == "TP_ERR_WORKSPACE"
    assert "TP_NOALLOC_SCRATCH_BYTES" in tp.tp_last_error()
