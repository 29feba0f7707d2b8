"""The allocation-free rowwise entry point, tp_linear_rowwise_noalloc.

Some callers may not allocate device memory (a plug-in inside a framework
that owns every byte of the GPU, or a process whose memory a pool claimed up
front).  For them the library keeps its rowwise scratch in a fixed array of
its own.  This test calls that entry point through the C ABI and checks it
against the ordinary workspace entry point -- the same kernel on the same
inputs, so bit for bit -- and against the oracle within the bar, on calls in a
row, so that a call on a scratch array that still holds the previous call's
partials and counters gives the right answer too; it also checks that a call
claims no device memory.  The file sorts last, so a run that stops at the
first failure has already run every other test.
"""
import ctypes
import gc

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
    xs_bits = [O.shard(x, "rowwise", p, r) for r in range(p)]
    ws_bits = [O.shard(w, "rowwise", p, r) for r in range(p)]
    ref = O.rowwise_forward(xs_bits, ws_bits, bias_bits=b)
    xs = [tp.bf16_from_bits(a, "cuda") for a in xs_bits]
    ws = [tp.bf16_from_bits(a, "cuda") for a in ws_bits]
    return xs, ws, tp.bf16_from_bits(b, "cuda"), ref


def _device_free_bytes():
    free, _ = torch.cuda.mem_get_info()
    return free


def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row():
    # Problems back to back through the same built-in scratch array: CTA pairs (T > 128),
    # then single CTAs (T <= 128) through the Python wrapper, then the first problem again.
    cases = [(140, (300, 200, 520, 4)), (141, (1000, 512, 1040, 3)), (142, (96, 64, 264, 2)),
             (140, (300, 200, 520, 4))]
    for k, (seed, (T, K_r, N, p)) in enumerate(cases):
        xs, ws, b, ref_o = _case(seed, T, K_r, N, p)
        ref = tp.tp_linear_rowwise(xs, ws, bias=b, mode="workspace")
        out = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        # Python's collector must not free other tests' tensors inside the measured call:
        # that would change torch's count of allocated bytes without this call doing anything.
        gc.collect()
        gc.disable()
        try:
            free0, alloc0 = _device_free_bytes(), torch.cuda.memory_allocated()
            if T <= 128:
                tp.tp_linear_rowwise_noalloc(xs, ws, bias=b, out=out)
            else:
                assert _noalloc_raw(xs, ws, b, out) == "TP_OK", tp.tp_last_error()
            tp.tp_device_status()
            free1, alloc1 = _device_free_bytes(), torch.cuda.memory_allocated()
        finally:
            gc.enable()
        if k > 0:
            # After the first call on the device (which may load the module that holds the
            # array), a call claims no device memory at all.
            assert free1 == free0
            assert alloc1 == alloc0
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"case {k}: differs from the workspace call"
        assert_close(O.bf16_to_f64(tp.bits_from_bf16(out)), ref_o, f"noalloc call {k} (seed {seed})")


def test_noalloc_at_exactly_its_scratch_size_and_one_tile_above():
    # p 2, T 1030, N 8144: partials and tile counters fill the 64 MiB array exactly -- accepted;
    # 128 more rows (one more row of tiles) -- refused on the host before any device work.
    p, T, K_r, N = 2, 1030, 64, 8144
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "workspace") == tp.NOALLOC_SCRATCH_BYTES
    xs, ws, b, ref_o = _case(143, T, K_r, N, p)
    out = torch.full((T, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _noalloc_raw(xs, ws, b, out) == "TP_OK", tp.tp_last_error()
    tp.tp_device_status()
    ref = tp.tp_linear_rowwise(xs, ws, bias=b, mode="workspace")
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert_close(O.bf16_to_f64(tp.bits_from_bf16(out)), ref_o, "noalloc at the scratch size")
    T2 = T + 128
    assert tp.tp_rowwise_workspace_bytes(p, T2, N, "workspace") > tp.NOALLOC_SCRATCH_BYTES
    fake = (ctypes.c_void_p * p)(*([0x10000] * p))
    st = tp.lib.tp_linear_rowwise_noalloc(fake, fake, None, p, T2, K_r, N, 0x10000, None)
    assert tp.STATUS_NAMES[st] == "TP_ERR_WORKSPACE"
    assert "TP_NOALLOC_SCRATCH_BYTES" in tp.tp_last_error()


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # p*T*N*4 bytes of partials above 64 MiB: refused on the host before any device work.
    p, T, K_r, N = 4, 4096, 64, 1536
    assert tp.tp_rowwise_workspace_bytes(p, T, N, "workspace") > tp.NOALLOC_SCRATCH_BYTES
    fake = (ctypes.c_void_p * p)(*([0x10000] * p))
    st = tp.lib.tp_linear_rowwise_noalloc(fake, fake, None, p, T, K_r, N, 0x10000, None)
    assert tp.STATUS_NAMES[st] == "TP_ERR_WORKSPACE"
    assert "TP_NOALLOC_SCRATCH_BYTES" in tp.tp_last_error()
