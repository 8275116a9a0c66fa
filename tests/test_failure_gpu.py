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
