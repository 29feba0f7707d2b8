"""The give-up path of the library's one cross-CTA wait, made to run out without a fault.

In TP_REDUCE_WORKSPACE every rank's CTA of an output tile publishes its fp32
partial, counts it on the tile's counter and waits (bounded) until all ranks'
partials are in.  With the bound set far below the time the ranks take to
arrive (tp_set_tile_wait_limit_ns), the waiting CTAs give up: the call still
returns, the kernel drains and exits, tp_device_status reports
TP_ERR_TIMEOUT, and the next call with the default bound is exact again.
Nothing here faults, traps or hangs the GPU: the wait that runs out is a
counter that the other ranks do set, only later than the bound allows.
"""
import numpy as np
import pytest

import tp_inputs
from oracle import tp_oracle as O

pytestmark = pytest.mark.gpu

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")


def _integer_case(p=4, T=128, K_r=4096, N=4096):
    # Integer-valued inputs: every product sum is exact in fp32 (|sum| <= 16 * 4 * 4096 < 2^24),
    # so a valid result equals the oracle's bit for bit.  T <= 128 runs single CTAs (no CTA
    # pairs).  The K slices are long (64 k-blocks per rank), so the ranks' CTAs of a tile
    # publish their partials microseconds apart, more than the device timer's tick: the first
    # to arrive then always waits long enough for a bound of 1 ns to run out.
    x = tp_inputs.int_bf16(170, 0, (T, K_r * p))
    w = tp_inputs.int_bf16(170, 1, (N, K_r * p))
    xs = [O.shard(x, "rowwise", p, r) for r in range(p)]
    ws = [O.shard(w, "rowwise", p, r) for r in range(p)]
    want = O.f64_to_bf16(O.rowwise_forward(xs, ws))
    return ([tp.bf16_from_bits(a, "cuda") for a in xs], [tp.bf16_from_bits(a, "cuda") for a in ws], want)


def test_tile_wait_runs_out_and_is_reported_then_recovers():
    xs, ws, want = _integer_case()
    tp.tp_device_status()                        # start from a clean status record
    assert tp.tp_tile_wait_limit_ns() == 2_000_000_000
    try:
        tp.tp_set_tile_wait_limit_ns(1)
        assert tp.tp_tile_wait_limit_ns() == 1
        # A CTA gives up unless every other rank's partial of its tile is already in when it
        # first looks; the ranks' CTAs run side by side, so some CTA nearly always looks too
        # early.  Several tries make the outcome certain.
        reported = []
        for _ in range(10):
            out = tp.tp_linear_rowwise(xs, ws, mode="workspace")   # returns: the kernel gives up, drains, exits
            assert out.shape == (128, 4096)
            try:
                tp.tp_device_status()
            except tp.TPError as e:
                reported.append(e.name)
                break
        assert reported == ["TP_ERR_TIMEOUT"], reported
    finally:
        tp.tp_set_tile_wait_limit_ns(0)
    assert tp.tp_tile_wait_limit_ns() == 2_000_000_000
    tp.tp_device_status()                        # the record was cleared by the report above
    for _ in range(2):                           # the context is healthy: exact results again
        got = tp.bits_from_bf16(tp.tp_linear_rowwise(xs, ws, mode="workspace"))
        tp.tp_device_status()
        assert np.array_equal(got, want)
    got = tp.bits_from_bf16(tp.tp_linear_rowwise(xs, ws, mode="accum"))
    assert np.array_equal(got, want)
