"""The numeric acceptance bar for floating-point outputs of the CUDA path.

bf16 inputs, fp32 accumulation, bf16 outputs, compared with the oracle's
unrounded float64 value ``ref``:

* max |gpu - ref| <= 2e-2 * RMS(ref), RMS = sqrt(mean(ref^2));
* sum |gpu - ref| / sum |ref| <= 5e-3 (the mean relative error, weighted by
  |ref| so that entries near zero do not dominate).

Rounding the output to bf16 alone costs at most 2^-9 relative per element
(about 1e-3 on average), so the bar leaves room for fp32 reassociation and for
bf16 storage between steps, and no more.  Integer, byte and index results
(shard extraction, gather, integer-valued products) are compared bit for bit
instead.
"""
import numpy as np

MAX_ABS_OVER_RMS = 2e-2
MEAN_REL = 5e-3


def error_stats(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite values in the GPU output"
    err = np.abs(gpu - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    return dict(max_abs=float(err.max()) if err.size else 0.0, rms=rms,
                max_over_rms=float(err.max() / rms) if rms > 0 else 0.0,
                mean_rel=float(err.sum() / np.abs(ref).sum()) if np.abs(ref).sum() > 0 else 0.0)


def assert_close(gpu, ref, what=""):
    s = error_stats(gpu, ref)
    assert s["max_over_rms"] <= MAX_ABS_OVER_RMS, (what, s)
    assert s["mean_rel"] <= MEAN_REL, (what, s)
    return s
