"""attn_fwd_decode_noalloc: the split-KV decode for callers that cannot
allocate device memory (allocator hooks, pools that must not re-enter
cudaMalloc, allocation-free hot loops). It keeps its split summaries in the
library's fixed device array instead of a workspace.

Checked through the C ABI against attn_fwd (the existing entry point, which
allocates its workspace stream-ordered) on two different calls in a row, so
the second call runs over the array the first one left behind. This file is
collected last on purpose."""
import ctypes

import pytest
import torch

import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300 import build as sab
from streaming_attention_gb300.inputs import DECODE_GQA, make_qkv, workload_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DT = {torch.bfloat16: sa.ATTN_BF16, torch.float16: sa.ATTN_FP16}


def noalloc(q, k, v, causal, window):
    o = torch.empty_like(q)
    B, Hq, M, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    st = sa.lib().attn_fwd_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), B, Hq, Hkv, M, N, D, int(causal), int(window), 0.0, DT[q.dtype],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, sa.strerror(st)
    return o


def existing(q, k, v, causal, window):
    o = torch.empty_like(q)
    sa.attn_fwd(q, k, v, o, causal=causal, window=window)
    return o


def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row():
    sab.build()
    cases = [
        (workload_inputs(DECODE_GQA), True, DECODE_GQA.window, DECODE_GQA.dtype),
        (make_qkv(2, 16, 4, 2, 3000, 128, torch.float16, seed=77), True, 1000, torch.float16),
    ]
    for (q, k, v), causal, window, dtype in cases:
        q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
        got = noalloc(q, k, v, causal, window)
        want = existing(q, k, v, causal, window)
        torch.cuda.synchronize()
        check(got, want.double().cpu().numpy(), dtype, "noalloc vs attn_fwd")
    assert sa.last_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_array():
    """A decode whose split summaries exceed the fixed array is refused with
    ATTN_ERR_WORKSPACE. The tensors are real device buffers of the full shape,
    so nothing could touch invalid memory even if the call were accepted."""
    B, Hq, Hkv, M, N, D = 8, 32, 8, 4, 8192, 64
    need = sa.attn_workspace_bytes(B, Hq, Hkv, M, N, D, True, 0, sa.PATH_DECODE)
    assert need > 8 << 20, need  # precondition: the problem does not fit the array
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=5)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    o = torch.empty_like(q)
    st = sa.lib().attn_fwd_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), B, Hq, Hkv, M, N, D, 1, 0, 0.0, sa.ATTN_BF16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == -8, sa.strerror(st)
