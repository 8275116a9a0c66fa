"""Failure detection without a GPU fault: a wait that nothing completes gives up
after its limit and reports through the device status word; the context stays
usable and the next call reports OK."""
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300.inputs import TINY, workload_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert sa.last_device_status() == 0
    sa.selftest_bounded_wait(20000)  # 20 ms
    assert sa.last_device_status() == -10  # ATTN_ERR_TIMEOUT, read and cleared
    assert sa.last_device_status() == 0
    q, k, v = workload_inputs(TINY)
    o = sa.attention(q.to("cuda"), k.to("cuda"), v.to("cuda"), causal=True)
    torch.cuda.synchronize()
    check(o, oracle.attention(q, k, v, causal=True), TINY.dtype, "after the timeout")
    assert sa.last_device_status() == 0


def test_prefill_abort_path_reports_timeout_and_context_survives():
    """The real prefill kernel with one P-ready arrival withheld: its issuing
    thread gives up after the wait limit, every CTA drains, frees TMEM and exits,
    the status word reads ATTN_ERR_TIMEOUT, and the next calls run normally."""
    import torch
    from streaming_attention_gb300.inputs import make_qkv

    assert sa.last_device_status() == 0
    q, k, v = (t.to("cuda") for t in make_qkv(2, 8, 8, 512, 1024, 128, torch.bfloat16, 61))
    o = torch.empty_like(q)
    sa.selftest_prefill_abort(q, k, v, o, withhold_at=3)
    assert sa.last_device_status() == -10  # ATTN_ERR_TIMEOUT, read and cleared
    assert sa.last_device_status() == 0
    for _ in range(2):  # TMEM was freed: the same kernel allocates and runs again
        qq, kk, vv = workload_inputs(TINY)
        got = sa.attention(qq.to("cuda"), kk.to("cuda"), vv.to("cuda"), causal=True)
        torch.cuda.synchronize()
        check(got, oracle.attention(qq, kk, vv, causal=True), TINY.dtype, "after the prefill abort")
        got = sa.attention(q, k, v)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
    assert sa.last_device_status() == 0
