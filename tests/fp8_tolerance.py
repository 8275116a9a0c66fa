"""Error model of the forward on E4M3 inputs, for its parity tests.

The inputs are exact (the oracle decodes the same bytes), products are exact and
accumulate in FP32, so the one coarse rounding is that of the probabilities: the
kernel rounds each p_j (taken against its row's running reference maximum, so at
most 2^8) to E4M3, to nearest, before the value product, while the row sum l adds
the unrounded values. E4M3 keeps 3 mantissa bits, so |p_hat - p| <= 2^-4 p in its
normal range (p >= 2^-6) and <= 2^-10 (half the subnormal spacing 2^-9) below it.
Divided by l >= l_true = sum_j exp(s_j - max_j s_j), key j moves output element
(i, d) by at most b_j |V_jd| with

    b_j = max(2^-4 w_j, 2^-10 / l_true)        (w: the exact attention weights).

Hard bound H = sum_j b_j |V_jd|. Taking the roundings as independent and uniform,
the error's standard deviation is at most sigma = sqrt(sum_j b_j^2 V_jd^2 / 3).
An element may miss by min(H, 6 sigma), plus half an ulp of the output cast
(2^-8 relative for BF16, 2^-11 for FP16) and 2^-12 sum_j w_j |V_jd| for the FP32
accumulation; the mean error may not exceed the mean of sigma plus half of the
cast term.
"""
from __future__ import annotations

import numpy as np
import torch

CAST = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def _visible(M, N, causal, window):
    i = np.arange(M)[:, None] + (N - M)
    j = np.arange(N)[None, :]
    keep = np.ones((M, N), dtype=bool)
    if causal:
        keep &= j <= i
    if window > 0:
        keep &= j > i - window
    return keep


def bounds(qf, kf, vf, causal, window, scale):
    """Per-element (H, sigma, sum_j w_j |V_jd|) for dequantized FP64 inputs
    q [B,Hq,M,D], k and v [B,Hkv,N,D]."""
    B, Hq, M, D = qf.shape
    Hkv, N = kf.shape[1], kf.shape[2]
    G = Hq // Hkv
    kk = np.repeat(kf, G, axis=1)
    vv = np.repeat(vf, G, axis=1)
    keep = _visible(M, N, causal, window)
    s = np.einsum("bhmd,bhnd->bhmn", qf, kk) * scale
    s = np.where(keep, s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    mx = np.where(np.isfinite(mx), mx, 0.0)
    e = np.where(keep, np.exp(s - mx), 0.0)
    l_true = e.sum(axis=-1, keepdims=True)
    safe = np.where(l_true > 0, l_true, 1.0)
    w = e / safe
    b = np.where(keep, np.maximum(2.0 ** -4 * w, 2.0 ** -10 / safe), 0.0)
    H = np.einsum("bhmn,bhnd->bhmd", b, np.abs(vv))
    sigma = np.sqrt(np.einsum("bhmn,bhnd->bhmd", b * b, vv * vv) / 3.0)
    wabs = np.einsum("bhmn,bhnd->bhmd", w, np.abs(vv))
    return H, sigma, wabs


def row_bounds(qf, kf, vf, rows, causal, window, scale):
    """The same for selected rows of the flattened [B*Hq*M] row axis; arrays [len(rows), D]."""
    B, Hq, M, D = qf.shape
    Hkv, N = kf.shape[1], kf.shape[2]
    G = Hq // Hkv
    out = [np.zeros((len(rows), D)) for _ in range(3)]
    for r_i, r in enumerate(rows):
        b_, rem = divmod(r, Hq * M)
        h, i = divmod(rem, M)
        keep = _visible(M, N, causal, window)[i]
        kv = b_, h // G
        s = np.where(keep, kf[kv] @ qf[b_, h, i] * scale, -np.inf)
        if not keep.any():
            continue
        e = np.where(keep, np.exp(s - s[keep].max()), 0.0)
        l_true = e.sum()
        w = e / l_true
        b = np.where(keep, np.maximum(2.0 ** -4 * w, 2.0 ** -10 / l_true), 0.0)
        v = vf[kv]
        out[0][r_i] = b @ np.abs(v)
        out[1][r_i] = np.sqrt((b * b) @ (v * v) / 3.0)
        out[2][r_i] = w @ np.abs(v)
    return out


def check_fp8(got: torch.Tensor, want: np.ndarray, H, sigma, wabs, out_dtype, what: str = ""):
    g = got.detach().to("cpu", torch.float64).numpy().reshape(want.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    if want.size == 0:
        return
    err = np.abs(g - want)
    allow = np.minimum(H, 6.0 * sigma)
    cast = CAST[out_dtype] * (np.abs(want) + allow)
    tol = allow + cast + 2.0 ** -12 * wabs + 1e-6
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), (f"{what}: err {err[worst]:.3g} > tol {tol[worst]:.3g} at {worst} "
                                f"(want {want[worst]:.3g}, sigma {sigma[worst]:.3g})")
    mean_allow = sigma.mean() + 0.5 * CAST[out_dtype] * np.abs(want).mean() + 2.0 ** -12 * wabs.mean() + 1e-6
    assert err.mean() <= mean_allow, f"{what}: mean err {err.mean():.3g} > {mean_allow:.3g}"
