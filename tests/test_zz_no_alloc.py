"""attn_fwd_decode_noalloc: the split-KV decode for callers that cannot
allocate device memory (allocator hooks, pools that must not re-enter
cudaMalloc, allocation-free hot loops). It keeps its split summaries in the
library's fixed device array instead of a workspace.

Checked through the C ABI against attn_fwd (the existing entry point, which
allocates its workspace stream-ordered) and against the FP64 oracle, on calls
in a row whose summaries all go through the array: a larger problem first,
then smaller ones, so each later call runs over what the earlier ones left
behind. This file is collected last on purpose."""
import ctypes

import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300 import build as sab
from streaming_attention_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
DT = {torch.bfloat16: sa.ATTN_BF16, torch.float16: sa.ATTN_FP16}
ARRAY_BYTES = 8 << 20  # ATTN_NOALLOC_SCRATCH_BYTES


def noalloc(q, k, v, causal, window):
    o = torch.full_like(q, float("nan"))
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


# (B, Hq, Hkv, M, N, D, dtype, causal, window, seed). Every case plans more
# splits per KV head than one thread-block cluster merges, so its summaries go
# through the fixed array.
THROUGH_ARRAY = [
    (1, 32, 4, 1, 32768, 128, torch.bfloat16, True, 0, 71),    # 64 splits per KV head, 1.1 MB of summaries
    (2, 16, 4, 2, 3000, 128, torch.float16, True, 1000, 77),  # 9 splits, 64 rows
    (2, 8, 2, 1, 5000, 64, torch.bfloat16, False, 0, 78),      # D = 64: 40 splits per KV head
    (1, 20, 1, 1, 3000, 128, torch.bfloat16, True, 0, 80),     # 20 grouped rows: two CTAs of 16 rows, 24 splits
]


def test_noalloc_matches_attn_fwd_and_oracle_on_calls_in_a_row():
    sab.build()
    for B, Hq, Hkv, M, N, D, dtype, causal, window, seed in THROUGH_ARRAY:
        need = sa.attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, causal, window, sa.PATH_DECODE)
        assert 0 < need <= ARRAY_BYTES
        q, k, v = make_qkv(B, Hq, Hkv, M, N, D, dtype, seed=seed)
        want = oracle.attention(q, k, v, causal=causal, window=window)
        q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
        got = noalloc(q, k, v, causal, window)
        ref = existing(q, k, v, causal, window)
        torch.cuda.synchronize()
        what = f"{(B, Hq, Hkv, M, N, D)}"
        check(got, ref.double().cpu().numpy(), dtype, "noalloc vs attn_fwd " + what)
        check(got, want, dtype, "noalloc vs oracle " + what)
    assert sa.last_device_status() == 0


def test_noalloc_cluster_merge_is_not_limited_by_the_array():
    """128 sequences of 16 grouped query heads: one split per KV head, merged
    inside the split kernel. Stored summaries would need more than the array
    holds, but none is stored, so the call is accepted and matches."""
    B, Hq, Hkv, M, N, D = 128, 128, 8, 1, 640, 128
    assert sa.attn_workspace_bytes_ex(B, Hq, Hkv, M, N, D, True, 0, sa.PATH_DECODE) > ARRAY_BYTES
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=79)
    rows = [0, 17, 4095, 9000, B * Hq * M - 1]
    want = oracle.attention_rows(q, k, v, rows, causal=True)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    got = noalloc(q, k, v, True, 0)
    ref = existing(q, k, v, True, 0)
    torch.cuda.synchronize()
    check(got, ref.double().cpu().numpy(), torch.bfloat16, "cluster-merged noalloc vs attn_fwd")
    picked = got.reshape(-1, D)[torch.tensor(rows, device=DEV)]
    check(picked, want, torch.bfloat16, "cluster-merged noalloc vs oracle")
    assert sa.last_device_status() == 0


def test_noalloc_large_d64_decode_merges_in_cluster():
    """A D = 64 decode whose stored summaries would exceed the fixed array
    (B=8, Hq=32, Hkv=8, M=4, N=8192): the tcgen05 split kernel plans at most 8
    splits per KV head and merges them in its cluster, so the call is accepted
    and matches attn_fwd and the oracle on sampled rows."""
    B, Hq, Hkv, M, N, D = 8, 32, 8, 4, 8192, 64
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=5)
    rows = [0, 5, 130, 517, 1023]
    want = oracle.attention_rows(q, k, v, rows, causal=True)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    got = noalloc(q, k, v, True, 0)
    ref = existing(q, k, v, True, 0)
    torch.cuda.synchronize()
    check(got, ref.double().cpu().numpy(), torch.bfloat16, "D = 64 noalloc vs attn_fwd")
    picked = got.reshape(-1, D)[torch.tensor(rows, device=DEV)]
    check(picked, want, torch.bfloat16, "D = 64 noalloc vs oracle")
    assert sa.last_device_status() == 0
