"""The pair-MMA prefill path (ATTN_PATH_PREFILL_PAIR: tcgen05 cta_group::2, two
CTAs per 512-row work tile, each loading half of every K/V tile) against the
FP64 oracle, element by element, and bit for bit against the one-CTA prefill
kernel, which does the same arithmetic per row in the same order."""
import math

import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300.inputs import PREFILL_D128, make_qkv, sample_rows, workload_inputs
from test_parity_gpu import whole_heads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAIR, ONE = sa.PATH_PREFILL_PAIR, sa.PATH_PREFILL


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


def both(q, k, v, causal, window=0, scale=0.0):
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o2 = sa.attention(q, k, v, causal=causal, window=window, scale=scale, path=PAIR)
    o1 = sa.attention(q, k, v, causal=causal, window=window, scale=scale, path=ONE)
    torch.cuda.synchronize()
    return o2, o1


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shape", [(1, 2, 2, 64, 64), (1, 2, 2, 37, 37), (1, 2, 2, 300, 300), (2, 4, 2, 129, 385),
                                   (1, 2, 1, 385, 129), (1, 1, 1, 1, 257), (1, 3, 3, 600, 600)], ids=str)
@pytest.mark.parametrize("mask", [(False, 0), (True, 0), (True, 100), (False, 70)], ids=str)
def test_pair_mid_sizes(shape, mask, dtype):
    """Ragged tails, M != N both ways, GQA, every mask: rows past M in one CTA
    of a pair, pairs whose second CTA holds no row below M."""
    B, Hq, Hkv, M, N = shape
    causal, window = mask
    q, k, v = make_qkv(B, Hq, Hkv, M, N, 128, dtype, seed=M * 7 + N)
    o2, o1 = both(q, k, v, causal, window)
    check(o2, oracle.attention(q, k, v, causal=causal, window=window), dtype, f"pair {shape} {mask}")
    assert torch.equal(o2, o1)


@pytest.mark.parametrize("case", [(40, 8, 4, 600, 200, True, 0), (24, 16, 16, 384, 384, True, 0),
                                  (20, 12, 3, 1024, 700, False, 0), (30, 8, 8, 300, 900, True, 257)], ids=str)
def test_pair_many_work_tiles(case):
    """More work tiles than pairs: the ring, barrier phases and relays carry
    across tiles; (first case) some work tiles see no key (M > N causal)."""
    B, Hq, Hkv, M, N, causal, window = case
    q, k, v = make_qkv(B, Hq, Hkv, M, N, 128, torch.bfloat16, seed=B + M + N)
    o2, o1 = both(q, k, v, causal, window)
    rows = sample_rows(B, Hq, M, 400, seed=M)
    want = oracle.attention_rows(q, k, v, rows, causal=causal, window=window)
    assert torch.isfinite(o2).all()
    check(o2.reshape(-1, 128)[torch.tensor(rows, device=o2.device)], want, torch.bfloat16, f"pair {case}")
    assert torch.equal(o2, o1)


@pytest.mark.parametrize("causal", [True, False])
def test_pair_full_size_whole_heads(causal):
    w = PREFILL_D128
    q, k, v = workload_inputs(w)
    o2, o1 = both(q, k, v, causal)
    rows = sorted(set(sample_rows(w.B, w.Hq, w.M, 192, seed=w.seed)) | set(whole_heads(w.B, w.Hq, w.M)))
    want = oracle.attention_rows(q, k, v, rows, causal=causal)
    check(o2.reshape(-1, w.D)[torch.tensor(rows, device=o2.device)], want, w.dtype, f"pair full causal={causal}")
    assert torch.equal(o2, o1)


def test_pair_log_sum_exp():
    q, k, v = make_qkv(2, 4, 2, 700, 900, 128, torch.bfloat16, seed=31)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o2, l2 = sa.attention_lse(q, k, v, causal=True, path=PAIR)
    o1, l1 = sa.attention_lse(q, k, v, causal=True, path=ONE)
    torch.cuda.synchronize()
    assert torch.equal(o2, o1) and torch.equal(l2, l1)
    want = oracle.attention_lse(q.cpu(), k.cpu(), v.cpu(), causal=True)[1]
    assert np.abs(l2.double().cpu().numpy() - want).max() <= 2e-3


def test_pair_a3_worked_example_across_tiles():
    """The answer key's A3 example (6, not the 7 of an unrescaled accumulator)
    at D = 128 with the ln 2 key in the second key tile."""
    D, N = 128, 129
    q = torch.zeros(1, 1, 1, D)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, N, D)
    k[0, 0, :, 0] = -80.0
    k[0, 0, 0, 0] = 0.0
    k[0, 0, 1, 0] = 0.0
    k[0, 0, 128, 0] = math.log(2.0)
    v = torch.zeros(1, 1, N, D)
    v[0, 0, 0, 0], v[0, 0, 1, 0], v[0, 0, 128, 0] = 1.0, 3.0, 10.0
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        o2, _ = both(q, k, v, causal, scale=1.0)
        x = float(o2[0, 0, 0, 0])
        assert abs(x - 6.0) <= 2e-2 and abs(x - 7.0) > 0.5, x


def test_pair_empty_dims_and_head_dim():
    q, k, v = make_qkv(1, 2, 2, 0, 16, 128, torch.bfloat16, 0)
    assert sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, path=PAIR).shape == (1, 2, 0, 128)
    q, k, v = make_qkv(1, 2, 2, 16, 0, 128, torch.bfloat16, 0)
    o = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), path=PAIR)
    torch.cuda.synchronize()
    assert torch.all(o == 0)
    q, k, v = make_qkv(1, 2, 2, 64, 64, 64, torch.bfloat16, 0)
    with pytest.raises(sa.AttnError) as e:
        sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), path=PAIR)
    assert e.value.status == -4
