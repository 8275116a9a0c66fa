"""Wide-row split softmax (attn_split_softmax) against the FP64 oracle.

Tolerance (derived, not from the pages): outputs are probabilities in [0, 1]
with one final cast, so |got - want| <= rtol * want + 1e-6 with rtol = 1e-4
(FP32), 2e-3 (FP16), 1e-2 (BF16)."""
import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
RTOL = {torch.float32: 1e-4, torch.float16: 2e-3, torch.bfloat16: 1e-2}


def check(y, want, dtype, what):
    g = y.detach().cpu().double().numpy()
    assert np.isfinite(g).all(), what
    err = np.abs(g - want)
    tol = RTOL[dtype] * want + 1e-6
    assert (err <= tol).all(), f"{what}: worst {err.max():.3g}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16], ids=["fp32", "fp16", "bf16"])
@pytest.mark.parametrize("chunk", [256, 1024, 4096, 0], ids=["c256", "c1024", "c4096", "resident"])
@pytest.mark.parametrize("M,N", [(4, 32769), (3, 1), (5, 1000), (2, 131072), (7, 4097), (3, 32768), (2, 98303)])
def test_split_softmax(dtype, chunk, M, N):
    g = torch.Generator().manual_seed(M * 7 + N)
    x = (torch.randn(M, N, generator=g) * 4).to(dtype)
    y = sa.split_softmax(x.to(DEV), chunk)
    torch.cuda.synchronize()
    check(y, oracle.softmax_rows(x), dtype, f"M={M} N={N} chunk={chunk}")


@pytest.mark.parametrize("chunk", [1024, 0], ids=["c1024", "resident"])
def test_split_softmax_peaked_and_empty(chunk):
    x = torch.zeros(3, 20000)
    x[0, 12345] = 50.0       # one dominant column
    x[1] = torch.linspace(-60, 60, 20000)  # maximum in the last chunk
    y = sa.split_softmax(x.to(DEV), chunk)
    torch.cuda.synchronize()
    check(y, oracle.softmax_rows(x), torch.float32, "peaked")
    y0 = sa.split_softmax(torch.zeros(0, 100, device=DEV), 256)
    assert y0.shape == (0, 100)


def test_resident_and_three_kernel_forms_agree_at_full_width():
    """The row-resident form and the three-kernel form on the bench's 1024 x 131072
    BF16 matrix: both within the tolerance of the oracle on sampled rows."""
    M, N = 1024, 131072
    x = (torch.randn(M, N, generator=torch.Generator().manual_seed(7)) * 4).to(torch.bfloat16)
    xd = x.to(DEV)
    y0 = sa.split_softmax(xd, 0)
    y1 = sa.split_softmax(xd, 4096)
    torch.cuda.synchronize()
    rows = [0, 1, 511, 1023]
    want = oracle.softmax_rows(x[rows])
    check(y0[rows], want, torch.bfloat16, "resident")
    check(y1[rows], want, torch.bfloat16, "three kernels")
