"""Every entry point is asynchronous on its stream and never synchronizes, so it
can be captured in a CUDA graph, including the calls that allocate their
workspace stream-ordered (cudaMallocAsync / cudaFreeAsync become graph memory
nodes). Each case captures one call, replays it on fresh inputs copied into the
captured buffers, and compares with an eager call: the same kernels run, so the
outputs are identical."""
import pytest
import torch

import streaming_attention_gb300 as sa
from streaming_attention_gb300.inputs import make_qkv, make_qkv_fp8

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


def capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm-up outside the graph (tensor maps, attributes, first-use setup)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("shape,causal,window", [
    ((2, 8, 8, 384, 384, 128), True, 0),       # prefill path
    ((4, 32, 8, 1, 4096, 128), True, 2048),    # decode path, workspace allocated inside the call
    ((1, 8, 1, 1, 9000, 128), False, 0),       # decode with more than 8 splits: separate merge kernel
])
def test_attn_fwd_in_a_graph(shape, causal, window):
    B, Hq, Hkv, M, N, D = shape
    q, k, v = (t.to(DEV) for t in make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 41))
    o = torch.empty_like(q)
    g = capture(lambda: sa.attn_fwd(q, k, v, o, causal, window))
    for seed in (42, 43):
        q2, k2, v2 = (t.to(DEV) for t in make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed))
        q.copy_(q2), k.copy_(k2), v.copy_(v2)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, sa.attention(q2, k2, v2, causal=causal, window=window))


@pytest.mark.parametrize("path", [sa.PATH_PREFILL, sa.PATH_DECODE], ids=["prefill", "decode"])
def test_attn_fwd_fp8_in_a_graph(path):
    B, Hq, Hkv, M, N, D = (2, 16, 4, 1, 3000, 128) if path == sa.PATH_DECODE else (1, 4, 4, 300, 500, 128)
    q, k, v = (t.to(DEV) for t in make_qkv_fp8(B, Hq, Hkv, M, N, D, 44))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    g = capture(lambda: sa.attn_fwd_fp8(q, k, v, o, lse, True, 0, 0.0, 0.5, 1.0, 2.0, path))
    q2, k2, v2 = (t.to(DEV) for t in make_qkv_fp8(B, Hq, Hkv, M, N, D, 45))
    q.copy_(q2), k.copy_(k2), v.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    want_o, want_lse = sa.attention_fp8(q2, k2, v2, causal=True, q_descale=0.5, v_descale=2.0, with_lse=True,
                                        path=path)
    assert torch.equal(o, want_o) and torch.equal(lse, want_lse)


@pytest.mark.parametrize("D", [32, 64, 128])  # 32: the grouped CUDA-core kernel; 64, 128: tcgen05
def test_paged_decode_in_a_graph(D):
    B, Hq, Hkv, M, page, npg = 3, 8, 2, 1, 64, 12
    g0 = torch.Generator().manual_seed(46)
    q = torch.randn(B, Hq, M, D, generator=g0).to(torch.bfloat16).to(DEV)
    kp = torch.randn(B * npg, Hkv, page, D, generator=g0).to(torch.bfloat16).to(DEV)
    vp = torch.randn(B * npg, Hkv, page, D, generator=g0).to(torch.bfloat16).to(DEV)
    table = torch.randperm(B * npg, generator=g0).reshape(B, npg).to(torch.int32).to(DEV)
    lens = torch.tensor([700, 5, 768], dtype=torch.int32, device=DEV)
    o = torch.empty_like(q)
    g = capture(lambda: sa.attn_decode_paged(q, kp, vp, table, lens, o, npg * page))
    lens.copy_(torch.tensor([768, 300, 1], dtype=torch.int32))  # lengths are read on the device
    g.replay()
    torch.cuda.synchronize()
    want = torch.empty_like(q)
    sa.attn_decode_paged(q, kp, vp, table, lens, want, npg * page)
    torch.cuda.synchronize()
    assert torch.equal(o, want)


@pytest.mark.parametrize("D", [32, 128])  # 32: the CUDA-core backward; 128: tcgen05
def test_backward_in_a_graph(D):
    B, Hq, Hkv, M, N = 1, 4, 2, 256, 384
    q, k, v = (t.to(DEV) for t in make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 47))
    d_o = torch.randn(q.shape, generator=torch.Generator().manual_seed(48)).to(torch.bfloat16).to(DEV)
    o, lse = sa.attention_lse(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    g = capture(lambda: sa.attn_bwd(q, k, v, o, d_o, lse, dq, dk, dv, causal=True))
    d_o.mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    wq, wk, wv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sa.attn_bwd(q, k, v, o, d_o, lse, wq, wk, wv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dq, wq) and torch.equal(dk, wk) and torch.equal(dv, wv)
