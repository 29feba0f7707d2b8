"""The colwise projection with chunked fp32 accumulation (TP_ACCUM_CHUNKED).

The tensor core adds every step of 16 products into its fp32 accumulator
without rounding to nearest, so over a long K the sum drifts and a bf16
output lands on the other neighbour of the exact value more often than a
round-to-nearest fp32 sum would.  With TP_ACCUM_CHUNKED the K sum is formed
on the tensor core in chunks of 1024, each from zero, and the chunks are added
in fp32 with round-to-nearest by the epilogue.  Integer-valued inputs are
exact either way, so those cases are compared bit for bit across chunk tails,
tile widths, single CTAs, CTA pairs and clusters, bias and a gathered output;
on N(0, sigma) inputs at K = 6144 the share of outputs that differ from the
correctly rounded exact value is measured.
"""
import numpy as np
import pytest
import torch

import tp_inputs
from oracle import tp_oracle as O
from tolerance import assert_close

pytestmark = pytest.mark.gpu

tp = pytest.importorskip("tensor_sharded_linear_tp_gb300")

DEV = "cuda"


def dev(bits):
    return tp.bf16_from_bits(bits, DEV)


def host_bits(t):
    torch.cuda.synchronize()
    return tp.bits_from_bf16(t)


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    tp.tp_device_status()


CHUNKED_SHAPES = [
    # (T, K, N_r, p)
    (100, 2112, 520, 2),     # single CTAs (T <= 128); 33 k-blocks: chunks of 16, 16, 1
    (300, 2112, 520, 2),     # CTA pairs, ragged rows and columns
    (517, 1032, 1040, 4),    # one chunk, with a K tail inside the last k-block
    (300, 3080, 264, 3),     # a chunk tail with a K tail (49 k-blocks, the last one partial)
    (257, 320, 1472, 4),     # tile widths other than 256
    (257, 320, 2368, 3),
    (1536, 320, 768, 4),     # clusters of two pairs sharing B
    (768, 320, 1024, 2),     # clusters of two pairs sharing A
    (1, 8, 8, 1),
]


@pytest.mark.parametrize("shape", CHUNKED_SHAPES, ids=str)
def test_chunked_colwise_integer_bit_exact(shape):
    T, K, N_r, p = shape
    x = tp_inputs.int_bf16(180, 0, (T, K), lim=3)
    w = tp_inputs.int_bf16(180, 1, (N_r * p, K), lim=3)
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    ys = tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "none", chunked=True)
    ref = O.colwise_forward(x, shards, "none")
    for r in range(p):
        assert np.array_equal(host_bits(ys[r]), O.f64_to_bf16(ref[r])), (shape, r)


def test_chunked_colwise_bias_and_gathered_output():
    T, K, N_r, p = 300, 576, 136, 3
    x = tp_inputs.int_bf16(181, 0, (T, K), lim=3)
    w = tp_inputs.int_bf16(181, 1, (N_r * p, K), lim=3)
    b = tp_inputs.int_bf16(181, 2, (N_r * p,), lim=3)
    shards = [O.shard(w, "colwise", p, r) for r in range(p)]
    bsh = [np.ascontiguousarray(b[r * N_r:(r + 1) * N_r]) for r in range(p)]
    y = torch.empty((T, p * N_r), dtype=torch.bfloat16, device=DEV)
    tp.tp_linear_colwise(dev(x), [dev(s) for s in shards], "none", bias_shards=[dev(v) for v in bsh],
                         y_shards=[y[:, r * N_r:] for r in range(p)], ldy=p * N_r, chunked=True)
    ref = O.combine_gather(O.colwise_forward(x, shards, "none", bsh))
    assert np.array_equal(host_bits(y), O.f64_to_bf16(ref))


def test_chunked_accumulation_rounds_like_a_round_to_nearest_sum():
    # K = 6144 (the block's hidden size), N(0,1) activations and N(0,0.02) weights: the share of
    # bf16 outputs that differ from the correctly rounded exact value.  A round-to-nearest fp32
    # sum differs on about 0.02 %, chunks of K = 1024 on about 0.07 %; the tensor core's own
    # accumulation over the whole K on about 0.35 %.
    T, K, N = 512, 6144, 2048
    x = tp_inputs.activation_bf16(182, 0, (T, K))
    w = tp_inputs.weight_bf16(182, 1, (N, K))
    exact = O.linear(x, w)
    want = O.f64_to_bf16(exact)
    y_chunked = host_bits(tp.tp_linear_colwise(dev(x), [dev(w)], "none", chunked=True)[0])
    y_plain = host_bits(tp.tp_linear_colwise(dev(x), [dev(w)], "none")[0])
    flips_chunked = float(np.mean(y_chunked != want))
    flips_plain = float(np.mean(y_plain != want))
    print(f"bf16 outputs off the correctly rounded value: chunked {flips_chunked:.5f}, plain {flips_plain:.5f}")
    assert flips_chunked <= 1.2e-3, flips_chunked
    assert_close(O.bf16_to_f64(y_chunked), exact, "chunked accumulation")
