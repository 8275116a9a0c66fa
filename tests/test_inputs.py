"""The seeded generator is deterministic and follows the stated recipe."""
import torch

from streaming_attention_gb300.inputs import LONG_CAUSAL, TINY, make_qkv, sample_rows, workload_inputs


def test_deterministic_and_rounded():
    a = workload_inputs(TINY)
    b = workload_inputs(TINY)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16 and torch.equal(x, y)
    g = torch.Generator().manual_seed(0)
    q32 = torch.randn((1, 2, 64, 64), generator=g)
    assert torch.equal(a[0], q32.to(torch.bfloat16))


def test_ramp_bias_construction():
    q, k, v = make_qkv(1, 2, 2, 8, 33, 16, torch.float16, 4, ramp_bias=True)
    assert torch.all(q[..., -1] == 8)
    ramp = k[0, 0, :, -1].float()
    assert ramp[0] == -42 and ramp[-1] == 42 and torch.all(ramp[1:] > ramp[:-1])
    assert LONG_CAUSAL.ramp_bias and LONG_CAUSAL.dtype == torch.float16


def test_sample_rows_in_range():
    rows = sample_rows(2, 3, 300, 50)
    assert len(rows) >= 20 and all(0 <= r < 2 * 3 * 300 for r in rows)
    assert 299 in rows and 2 * 3 * 300 - 1 in rows


def test_fp8_inputs_follow_the_recipe():
    from streaming_attention_gb300.inputs import make_qkv_fp8

    q, k, v = make_qkv_fp8(1, 2, 1, 16, 32, 128, 7, q_descale=0.5, k_descale=2.0, v_descale=1.0)
    assert q.dtype == torch.float8_e4m3fn and k.shape == (1, 1, 32, 128)
    g = torch.Generator().manual_seed(7)  # the same draws as make_qkv, divided by each factor, then rounded
    q32 = torch.randn((1, 2, 16, 128), generator=g) / 0.5
    k32 = torch.randn((1, 1, 32, 128), generator=g) / 2.0
    assert torch.equal(q.view(torch.uint8), q32.to(torch.float8_e4m3fn).view(torch.uint8))
    assert torch.equal(k.view(torch.uint8), k32.to(torch.float8_e4m3fn).view(torch.uint8))
    # dequantized values are about N(0, 1)
    deq = q.float() * 0.5
    assert abs(deq.mean().item()) < 0.1 and 0.9 < deq.std().item() < 1.1
