"""Comparison of the CUDA path with the FP64 oracle.

Tolerances: max-abs 1e-2 for FP16 and 2e-2 for BF16 outputs, mean-abs 2e-3,
no NaN or Inf anywhere in the output.
"""
import numpy as np
import torch

MAX_ABS = {torch.float16: 1e-2, torch.bfloat16: 2e-2}
MEAN_ABS = 2e-3


def check(got: torch.Tensor, want: np.ndarray, dtype: torch.dtype, what: str = ""):
    g = got.detach().to("cpu", torch.float64).numpy().reshape(want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    if want.size == 0:
        return 0.0, 0.0
    err = np.abs(g - want)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS[dtype], f"{what}: max-abs {mx:.3g} > {MAX_ABS[dtype]} (mean {mean:.3g})"
    assert mean <= MEAN_ABS, f"{what}: mean-abs {mean:.3g} > {MEAN_ABS}"
    return mx, mean
