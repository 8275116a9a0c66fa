"""Log-sum-exp output of the forward and the backward pass (attn_fwd_lse,
attn_bwd) against the FP64 oracle, through the C ABI.

Gradient tolerance: every gradient element is a sum over up to M (or N) products
of 16-bit-rounded operands (P, dS, dO, Q, K), so its error grows with its size:
|got - want| <= atol + rtol * |want| elementwise with atol = rtol = 2e-2 (BF16)
or 1e-2 (FP16), and the mean error at most 2e-3 * max(1, mean |want|)."""

import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300.inputs import PREFILL_D128, make_qkv, workload_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = {torch.bfloat16: 2e-2, torch.float16: 1e-2}


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


def grad_check(got, want, dtype, what):
    g = got.detach().to("cpu", torch.float64).numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite gradient"
    if want.size == 0:
        return
    err = np.abs(g - want)
    tol = TOL[dtype] * (1.0 + np.abs(want))
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), f"{what}: err {err[worst]:.3g} at {worst} (want {want[worst]:.3g})"
    assert err.mean() <= 2e-3 * max(1.0, float(np.abs(want).mean())), f"{what}: mean err {err.mean():.3g}"


def lse_check(got, want, what):
    g = got.detach().cpu().double().numpy()
    assert np.array_equal(np.isneginf(g), np.isneginf(want)), f"{what}: -inf pattern differs"
    fin = np.isfinite(want)
    assert np.isfinite(g[fin]).all()
    if fin.any():
        err = np.abs(g[fin] - want[fin]).max()
        assert err <= 2e-3, f"{what}: lse max err {err:.3g}"


@pytest.mark.parametrize("path", [sa.PATH_SIMT, sa.PATH_PREFILL, sa.PATH_DECODE, sa.PATH_AUTO])
@pytest.mark.parametrize("shape,causal,window", [
    ((2, 4, 2, 200, 333, 128), True, 0),
    ((1, 2, 2, 130, 130, 64), False, 0),
    ((2, 8, 2, 1, 1500, 128), True, 700),     # decode: 6 splits per group, merged in a cluster
    ((1, 4, 1, 1, 5000, 128), False, 0),      # decode: 40 splits, merged by the merge kernel
    ((1, 2, 1, 300, 100, 64), True, 0),   # rows past the keys see nothing: lse = -inf
])
def test_forward_lse(path, shape, causal, window):
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 5)
    o, lse = sa.attention_lse(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, path=path)
    torch.cuda.synchronize()
    want_o, want_lse = oracle.attention_lse(q, k, v, causal=causal, window=window)
    check(o, want_o, torch.bfloat16, f"o path={path}")
    lse_check(lse, want_lse, f"path={path}")


def run_bwd(q, k, v, d_o, causal, window):
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), d_o.to(DEV)
    o, lse = sa.attention_lse(qd, kd, vd, causal=causal, window=window)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    sa.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, causal=causal, window=window)
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shape,causal,window", [
    ((1, 2, 2, 256, 256, 128), True, 0),
    ((1, 2, 2, 256, 256, 128), False, 0),
    ((2, 4, 2, 200, 333, 128), True, 0),      # GQA, ragged, M < N
    ((1, 4, 1, 384, 384, 64), True, 150),     # window, D = 64, four heads share one KV head
    ((1, 2, 2, 333, 200, 64), False, 0),      # M > N, noncausal
    ((1, 2, 2, 300, 100, 128), True, 0),      # rows with no visible key
    ((1, 1, 1, 1, 517, 128), True, 64),       # one query row (decode shape)
])
def test_backward_against_oracle(dtype, shape, causal, window):
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, dtype, 9)
    d_o = torch.randn(B, Hq, M, D, generator=torch.Generator().manual_seed(10)).to(dtype)
    dq, dk, dv = run_bwd(q, k, v, d_o, causal, window)
    wq, wk, wv = oracle.attention_backward(q, k, v, d_o, causal=causal, window=window)
    grad_check(dq, wq, dtype, "dq")
    grad_check(dk, wk, dtype, "dk")
    grad_check(dv, wv, dtype, "dv")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shape,causal,window", [
    ((1, 2, 2, 77, 77, 16), True, 0),
    ((2, 4, 2, 100, 150, 32), False, 0),      # GQA, M < N
    ((1, 4, 1, 130, 130, 32), True, 40),      # window, four heads share one KV head
    ((1, 2, 2, 90, 40, 16), True, 0),         # rows with no visible key
    ((1, 3, 3, 1, 200, 32), True, 17),        # one query row
])
def test_backward_small_head_dims(dtype, shape, causal, window):
    """D = 16 and 32 (the pages' own head dimensions) on the CUDA-core backward."""
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, dtype, 13)
    d_o = torch.randn(B, Hq, M, D, generator=torch.Generator().manual_seed(14)).to(dtype)
    dq, dk, dv = run_bwd(q, k, v, d_o, causal, window)
    wq, wk, wv = oracle.attention_backward(q, k, v, d_o, causal=causal, window=window)
    grad_check(dq, wq, dtype, "dq")
    grad_check(dk, wk, dtype, "dk")
    grad_check(dv, wv, dtype, "dv")


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("scale", [0.2, -0.1])
def test_backward_explicit_scales(D, scale):
    """A caller-given logit scale (including a negative one) through the forward
    log-sum-exp and the backward."""
    B, Hq, Hkv, M, N = 1, 4, 2, 150, 200
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 15)
    d_o = torch.randn(B, Hq, M, D, generator=torch.Generator().manual_seed(16)).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(DEV), k.to(DEV), v.to(DEV), d_o.to(DEV)
    o, lse = sa.attention_lse(qd, kd, vd, causal=True, scale=scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    sa.attn_bwd(qd, kd, vd, o, dod, lse, dq, dk, dv, causal=True, scale=scale)
    torch.cuda.synchronize()
    wq, wk, wv = oracle.attention_backward(q, k, v, d_o, causal=True, scale=scale)
    grad_check(dq, wq, torch.bfloat16, "dq")
    grad_check(dk, wk, torch.bfloat16, "dk")
    grad_check(dv, wv, torch.bfloat16, "dv")


def test_backward_empty_dims():
    q, k, v = make_qkv(1, 2, 2, 0, 64, 128, torch.bfloat16, 0)
    d_o = torch.zeros_like(q)
    dq, dk, dv = run_bwd(q, k, v, d_o, True, 0)
    assert dq.shape == (1, 2, 0, 128) and torch.all(dk == 0) and torch.all(dv == 0)
    q, k, v = make_qkv(1, 2, 2, 64, 0, 128, torch.bfloat16, 0)
    d_o = torch.randn_like(q.float()).to(torch.bfloat16)
    dq, dk, dv = run_bwd(q, k, v, d_o, False, 0)
    assert torch.all(dq == 0) and dk.shape == (1, 2, 0, 128)


def test_backward_full_size_sampled_heads():
    """The causal D=128 prefill workload (B=2, H=32, M=N=4096) at full size; the
    oracle takes two whole heads in FP64 (dk, dv of a head need all its rows)."""
    w = PREFILL_D128
    q, k, v = workload_inputs(w)
    d_o = torch.randn(q.shape, generator=torch.Generator().manual_seed(12)).to(w.dtype)
    dq, dk, dv = run_bwd(q, k, v, d_o, True, 0)
    for b, h in ((0, 0), (1, 31)):
        wq, wk, wv = oracle.attention_backward(q, k, v, d_o, causal=True, heads=[(b, h)])
        grad_check(dq[b, h], wq[b, h], w.dtype, f"dq head {b},{h}")
        grad_check(dk[b, h], wk[b, h], w.dtype, f"dk head {b},{h}")
        grad_check(dv[b, h], wv[b, h], w.dtype, f"dv head {b},{h}")
