"""Calls that overlap on the GPU or come from several host threads: every
entry point keeps its state in the caller's buffers (or, for the host-buffer
entry, serializes its internal streams), so results match the same calls made
one at a time."""
import threading

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


def test_prefill_and_decode_on_two_streams():
    """A prefill and two decode calls (cluster-merged and merge-kernel forms) run
    concurrently on separate streams, each with its own workspace."""
    pq, pk, pv = (t.to(DEV) for t in make_qkv(2, 8, 8, 512, 512, 128, torch.bfloat16, 51))
    dq, dk, dv = (t.to(DEV) for t in make_qkv(8, 32, 8, 1, 4096, 128, torch.bfloat16, 52))
    eq, ek, ev = (t.to(DEV) for t in make_qkv(1, 8, 1, 1, 9000, 128, torch.bfloat16, 53))
    want = [sa.attention(pq, pk, pv, causal=True), sa.attention(dq, dk, dv, causal=True, window=1024),
            sa.attention(eq, ek, ev, causal=True)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(3)]
    outs = [torch.empty_like(pq), torch.empty_like(dq), torch.empty_like(eq)]
    for _ in range(5):
        for st, (q, k, v, o, cw) in zip(streams, [(pq, pk, pv, outs[0], (True, 0)), (dq, dk, dv, outs[1], (True, 1024)),
                                                   (eq, ek, ev, outs[2], (True, 0))]):
            with torch.cuda.stream(st):
                sa.attn_fwd(q, k, v, o, cw[0], cw[1], stream=st)
    torch.cuda.synchronize()
    for got, ref in zip(outs, want):
        assert torch.equal(got, ref)


def test_fp8_decode_and_split_softmax_on_two_streams():
    q, k, v = (t.to(DEV) for t in make_qkv_fp8(8, 32, 8, 1, 4096, 128, 54))
    x = (torch.randn(256, 65536, generator=torch.Generator().manual_seed(55)) * 3).to(torch.bfloat16).to(DEV)
    want_o = sa.attention_fp8(q, k, v, causal=True)
    want_y = sa.split_softmax(x, 0)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o = torch.empty_like(want_o)
    y = torch.empty_like(want_y)
    for _ in range(5):
        with torch.cuda.stream(s1):
            sa.attn_fwd_fp8(q, k, v, o, None, True, stream=s1)
        with torch.cuda.stream(s2):
            sa.split_softmax(x, 0, y=y, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(o, want_o) and torch.equal(y, want_y)


def test_host_entry_from_two_threads():
    """Two host threads call the host-buffer entry point at once on their own
    buffers; the library serializes its internal copy streams."""
    cases = []
    for seed in (56, 57):
        q, k, v = make_qkv(2, 8, 4, 256, 384, 128, torch.bfloat16, seed)
        qh, kh, vh = (t.pin_memory() for t in (q, k, v))
        oh = torch.empty_like(qh).pin_memory()
        dev_bufs = [torch.empty_like(t, device=DEV) for t in (q, k, v, q)]
        cases.append((qh, kh, vh, oh, dev_bufs, sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True).cpu()))
    errors = []

    def work(c):
        try:
            qh, kh, vh, oh, (qd, kd, vd, od), _ = c
            st = torch.cuda.Stream()
            for _ in range(3):
                sa.attn_fwd_host(qh, kh, vh, oh, qd, kd, vd, od, causal=True, stream=st)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for c in cases:
        assert torch.equal(c[3], c[5])
