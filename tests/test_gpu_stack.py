"""Eight SwiGLU MLP blocks loaded shard-on-read from page-locked host memory, then run.

"Tensor parallelism" page, §Load a sharded model: each rank reads only its
slice of each weight and places it directly on its device, so no full-size
weight is ever held there.  Here every rank's slices of the 16 weights
(hidden 6144, ffn 18432, tp_degree 4: 5.44 GB of bf16) are extracted from a
page-locked host state dict straight into device shards; the device never
holds more than the shards.  Then the 8 blocks run on 4608 tokens.
"""
import numpy as np
import pytest
import torch

import tp_inputs
from oracle import tp_oracle as O
from tolerance import assert_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")

DEV = "cuda"


def f64(t):
    torch.cuda.synchronize()
    return O.bf16_to_f64(tp.bits_from_bf16(t))


def pinned(bits):
    t = torch.empty(bits.shape, dtype=torch.bfloat16, pin_memory=True)
    t.copy_(tp.bf16_from_bits(bits))
    return t


def test_stack_of_eight_blocks_shard_on_read():
    cfg = tp_inputs.WORKLOADS["stack8_swiglu_tp4"]
    seed, p, nb, T, H, F = cfg["seed"], cfg["tp"], cfg["blocks"], cfg["tokens"], cfg["hidden"], cfg["ffn"]
    heads = cfg["heads"]
    host = []   # (gate_up bits, down bits) per block, and their page-locked copies
    for b in range(nb):
        gu = tp_inputs.stack_weight(seed, b, "gate_up", H, F)
        dn = tp_inputs.stack_weight(seed, b, "down", H, F)
        host.append((gu, dn, pinned(gu), pinned(dn)))
    x = tp_inputs.stack_input(seed, nb, T, H)

    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    shards = []
    for gu, dn, gu_pin, dn_pin in host:
        gu_sh = tp.tp_plan_shard_ranks(gu_pin, "colwise", p, 0, p, [F, F], heads, 0, device=DEV)
        dn_sh = tp.tp_plan_shard_ranks(dn_pin, "rowwise", p, 0, p, None, heads, 0, device=DEV)
        shards.append((gu_sh, dn_sh))
    torch.cuda.synchronize()
    shard_bytes = sum(t.numel() * 2 for gu_sh, dn_sh in shards for t in gu_sh + dn_sh)
    assert shard_bytes == nb * (2 * F * H + H * F) * 2
    # Nothing but the shards reached the device: no full-size weight was staged.
    assert torch.cuda.max_memory_allocated() - base <= shard_bytes + (1 << 20)

    # Every shard is bit-exact (checked on a sample of its rows).
    rng = np.random.default_rng(7)
    for (gu, dn, _, _), (gu_sh, dn_sh) in zip(host, shards):
        for r in range(p):
            want_gu = O.shard(gu, "colwise", p, r, [F, F])
            want_dn = O.shard(dn, "rowwise", p, r)
            for want, got in ((want_gu, gu_sh[r]), (want_dn, dn_sh[r])):
                idx = np.sort(rng.choice(want.shape[0], size=32, replace=False))
                sel = got[torch.from_numpy(idx).to(DEV)]
                assert np.array_equal(tp.bits_from_bf16(sel), want[idx])
    host = [(gu, dn) for gu, dn, _, _ in host]  # drop the page-locked copies

    # The forward pass through all 8 blocks, with the calls the benchmark times (each block:
    # tp_linear_colwise with SwiGLU, then tp_linear_rowwise with the on-chip sum), keeping
    # every block's stored output.
    zs = [tp.bf16_from_bits(x, DEV)]
    for gu_sh, dn_sh in shards:
        h = tp.tp_linear_colwise(zs[-1], gu_sh, "swiglu")
        zs.append(tp.tp_linear_rowwise(h, dn_sh, mode="accum"))
    tp.tp_device_status()

    # Each block of that forward against the oracle, from the block's own stored input (the
    # previous block's output as the path stored it) on sampled token rows, at the one bar.
    # Without the replicated norms between blocks (left out of the plan) the activations
    # grow roughly quadratically per block (SwiGLU is quadratic in its input): blocks 0-4
    # stay finite, block 5's SwiGLU output passes the bf16 range and its output is no longer
    # finite -- in the oracle too.  Every block with a finite input and a finite oracle
    # output is checked; the first block whose oracle output is not finite must be
    # non-finite on the GPU as well; past it there is nothing finite to compare.
    rows = tp_inputs.sample_rows(seed, T, 32)
    checked = []
    for b in range(nb):
        xin = tp.bits_from_bf16(zs[b][torch.from_numpy(rows).to(DEV)])
        if not np.all(np.isfinite(O.bf16_to_f64(xin))):
            break
        gu, dn = host[b]
        with np.errstate(all="ignore"):
            _, zo = O.mlp_forward(xin, [O.shard(gu, "colwise", p, r, [F, F]) for r in range(p)],
                                  [O.shard(dn, "rowwise", p, r) for r in range(p)], "swiglu")
        got = f64(zs[b + 1])[rows]
        if np.all(np.isfinite(O.bf16_to_f64(O.f64_to_bf16(zo)))):
            assert_close(got, zo, f"block {b} of the forward, from its stored input")
            checked.append(b)
        else:
            assert not np.all(np.isfinite(got)), f"block {b}: the oracle overflows, the path does not"
            break
    assert checked == [0, 1, 2, 3, 4], checked

    # Every block also from a bounded seeded input of its own (N(0,1) rows).
    for b in range(nb):
        gu, dn = host[b]
        gu_o = [O.shard(gu, "colwise", p, r, [F, F]) for r in range(p)]
        dn_o = [O.shard(dn, "rowwise", p, r) for r in range(p)]
        xb = tp_inputs.activation_bf16(seed, 100 + b, (32, H))
        _, zo = O.mlp_forward(xb, gu_o, dn_o, "swiglu")
        gu_sh, dn_sh = shards[b]
        hb = tp.tp_linear_colwise(tp.bf16_from_bits(xb, DEV), gu_sh, "swiglu")
        zb = tp.tp_linear_rowwise(hb, dn_sh, mode="accum")
        assert_close(f64(zb), zo, f"block {b} from a fresh input")
