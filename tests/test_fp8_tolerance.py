"""The E4M3 error model on the CPU: a float64 simulation of the kernel's one
coarse rounding (probabilities rounded to E4M3 against a stale reference
maximum up to 8 base-2 units below the true one) stays inside the tolerance,
and outputs with a planted mistake do not."""
import numpy as np
import pytest
import torch

import oracle
from fp8_tolerance import _visible, bounds, check_fp8
from streaming_attention_gb300.inputs import make_qkv_fp8

SHAPE = (1, 2, 2, 64, 200, 128)


def simulate(qf, kf, vf, causal, window, scale, seed, drop_last=False):
    rng = np.random.default_rng(seed)
    B, Hq, M, D = qf.shape
    Hkv, N = kf.shape[1], kf.shape[2]
    G = Hq // Hkv
    keep = _visible(M, N, causal, window)
    out = np.zeros_like(qf)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for i in range(M):
                vis = np.flatnonzero(keep[i])
                if drop_last and vis.size > 1:
                    vis = vis[:-1]
                if vis.size == 0:
                    continue
                t = (kf[b, g][vis] @ qf[b, h, i]) * scale * np.log2(np.e)
                m_ref = t.max() - rng.uniform(0, 8)
                p = np.exp2(t - m_ref)
                p_hat = torch.from_numpy(p).to(torch.float8_e4m3fn).to(torch.float64).numpy()
                out[b, h, i] = (p_hat @ vf[b, g][vis]) / p.sum()
    return torch.from_numpy(out).to(torch.bfloat16)


def inputs(shape=SHAPE):
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 31, 1.0, 1.0, 1.0)
    return oracle.decode_e4m3(q) * 2.0, oracle.decode_e4m3(k), oracle.decode_e4m3(v)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 40)])
def test_simulated_rounding_is_inside_the_tolerance(causal, window):
    qf, kf, vf = inputs()
    scale = 1.0 / np.sqrt(qf.shape[-1])
    want = oracle.attention(qf, kf, vf, causal=causal, window=window)
    H, sigma, wabs = bounds(qf, kf, vf, causal, window, scale)
    for seed in range(3):
        check_fp8(simulate(qf, kf, vf, causal, window, scale, seed), want, H, sigma, wabs, torch.bfloat16)


def test_planted_mistake_is_outside_the_tolerance():
    qf, kf, vf = inputs()
    scale = 1.0 / np.sqrt(qf.shape[-1])
    want = oracle.attention(qf, kf, vf, causal=True)
    H, sigma, wabs = bounds(qf, kf, vf, True, 0, scale)
    with pytest.raises(AssertionError):
        check_fp8(simulate(qf, kf, vf, True, 0, scale, 0, drop_last=True), want, H, sigma, wabs, torch.bfloat16)
    with pytest.raises(AssertionError):  # V dequantization factor applied twice
        check_fp8(simulate(qf, kf, 2 * vf, True, 0, scale, 0), want, H, sigma, wabs, torch.bfloat16)


@pytest.mark.parametrize("shape,causal,window", [
    ((1, 4, 2, 48, 160, 128), True, 50),   # GQA (two query heads per KV head) with a window
    ((1, 2, 1, 90, 40, 64), True, 0),      # M > N: the first rows see no key and must be exactly 0
])
def test_simulated_rounding_gqa_window_and_empty_rows(shape, causal, window):
    qf, kf, vf = inputs(shape)
    scale = 1.0 / np.sqrt(qf.shape[-1])
    want = oracle.attention(qf, kf, vf, causal=causal, window=window)
    H, sigma, wabs = bounds(qf, kf, vf, causal, window, scale)
    got = simulate(qf, kf, vf, causal, window, scale, 5)
    check_fp8(got, want, H, sigma, wabs, torch.bfloat16)
    if shape[3] > shape[4]:  # rows before the first key: zero output, zero allowance
        n_empty = shape[3] - shape[4]
        assert torch.all(got[:, :, :n_empty] == 0) and np.all(H[:, :, :n_empty] == 0)
