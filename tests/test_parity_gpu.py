"""CUDA path against the FP64 oracle, element by element on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from parity import check
from streaming_attention_gb300.inputs import (DECODE_GQA, LONG_CAUSAL, PREFILL_D64, PREFILL_D128, TINY,
                                              TINY_RAGGED, make_qkv, sample_rows, workload_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
ALL_PATHS = [sa.PATH_AUTO, sa.PATH_SIMT, sa.PATH_PREFILL, sa.PATH_DECODE]
PATH_NAMES = {0: "auto", 1: "simt", 2: "prefill", 3: "decode"}


def run(q, k, v, causal, window=0, path=sa.PATH_AUTO, scale=0.0):
    o = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, path=path, scale=scale)
    torch.cuda.synchronize()
    return o


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_NAMES.get)
@pytest.mark.parametrize("w", [TINY, TINY_RAGGED], ids=lambda w: w.name)
@pytest.mark.parametrize("causal", [False, True])
def test_tiny(w, causal, path):
    q, k, v = workload_inputs(w)
    want = oracle.attention(q, k, v, causal=causal)
    check(run(q, k, v, causal, path=path), want, w.dtype, f"{w.name} causal={causal} path={path}")


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_NAMES.get)
def test_empty_dims(path):
    q, k, v = make_qkv(1, 2, 2, 0, 16, 64, torch.bfloat16, 0)
    o = run(q, k, v, True, path=path)
    assert o.shape == (1, 2, 0, 64)
    q, k, v = make_qkv(1, 2, 2, 16, 0, 64, torch.bfloat16, 0)
    o = run(q, k, v, False, path=path)
    assert o.shape == (1, 2, 16, 64) and torch.all(o == 0)
    q, k, v = make_qkv(0, 2, 2, 16, 16, 64, torch.bfloat16, 0)
    assert run(q, k, v, False, path=path).shape == (0, 2, 16, 64)


@pytest.mark.parametrize("path", [sa.PATH_SIMT, sa.PATH_PREFILL, sa.PATH_DECODE], ids=PATH_NAMES.get)
def test_a3_worked_example_across_tiles(path):
    """The answer key's A3 example (logits 0, 0, ln 2 over values 1, 3, 10 give
    6; leaving the accumulator unrescaled gives 7) at D=64, with the ln 2 key in the second
    128-key tile so that the running maximum rises in a later tile. Filler keys
    score -80 and carry value 0."""
    D, N = 64, 129
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
        o = run(q, k, v, causal, path=path, scale=1.0)
        x = float(o[0, 0, 0, 0])
        assert abs(x - 6.0) <= 2e-2 and abs(x - 7.0) > 0.5, x
        check(o, oracle.attention(q, k, v, causal=causal, scale=1.0), torch.bfloat16, "a3")


@pytest.mark.parametrize("path", [sa.PATH_SIMT, sa.PATH_PREFILL], ids=PATH_NAMES.get)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape", [(1, 2, 2, 300, 300), (2, 4, 2, 129, 385), (1, 2, 1, 385, 129),
                                   (1, 1, 1, 1, 257), (1, 3, 3, 256, 256)], ids=str)
@pytest.mark.parametrize("mask", [(False, 0), (True, 0), (True, 100), (False, 70)], ids=str)
def test_mid_sizes_full_compare(shape, mask, D, dtype, path):
    """Several tiles with ragged tails, M != N (both ways), GQA, all masks."""
    B, Hq, Hkv, M, N = shape
    causal, window = mask
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, dtype, seed=M * 7 + N)
    want = oracle.attention(q, k, v, causal=causal, window=window)
    check(run(q, k, v, causal, window, path), want, dtype, f"{shape} {mask} D={D} path={path}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("case", [(40, 8, 4, 600, 200, True, 0), (24, 16, 16, 384, 384, True, 0),
                                  (20, 12, 3, 512, 700, False, 0), (30, 8, 8, 300, 900, True, 257)], ids=str)
def test_prefill_many_work_tiles(case, D):
    """More work tiles than SMs, so each persistent CTA walks several of them:
    the K/V ring and barrier phases carry across tiles, and (first case) some
    work tiles see no key at all (M > N causal) and are written as zeros."""
    B, Hq, Hkv, M, N, causal, window = case
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=B + M + N)
    o = run(q, k, v, causal, window, sa.PATH_PREFILL)
    rows = sample_rows(B, Hq, M, 400, seed=M)
    want = oracle.attention_rows(q, k, v, rows, causal=causal, window=window)
    assert torch.isfinite(o).all()
    check(o.reshape(-1, D)[torch.tensor(rows, device=o.device)], want, torch.bfloat16, f"{case} D={D}")


def test_prefill_noncausal_head_groups():
    """Noncausal work tiles of equal length over at least four waves: the
    persistent CTAs walk the heads in groups of about one wave's worth (here
    160 query heads x 4 query blocks = 640 work tiles, groups of 38 heads, the
    last one of 8), GQA groups of 5. Whole first, middle and last heads and
    sampled rows against the oracle."""
    B, Hq, Hkv, M, N, D = 2, 80, 16, 1024, 1024, 64
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=31)
    o = run(q, k, v, False, 0, sa.PATH_PREFILL)
    rows = sorted(set(sample_rows(B, Hq, M, 300, seed=31)) | set(whole_heads(B, Hq, M)))
    want = oracle.attention_rows(q, k, v, rows, causal=False)
    assert torch.isfinite(o).all()
    check(o.reshape(-1, D)[torch.tensor(rows, device=o.device)], want, torch.bfloat16, "head groups")


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_NAMES.get)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape,causal,window", [
    ((1, 2, 2, 1, 1), False, 0),        # one query, one key
    ((1, 2, 2, 1, 1), True, 0),
    ((1, 2, 2, 5, 1), True, 0),         # one key: only the last row sees it (causal), the rest output 0
    ((1, 2, 2, 129, 1), False, 0),      # one key for a tile and a ragged row
    ((2, 4, 2, 1, 3), True, 1),         # window 1: each row sees only its own position
    ((1, 2, 2, 200, 200), True, 1),     # window 1 over several tiles: the diagonal alone
    ((1, 2, 1, 1, 129), False, 0),      # one row over a tile and one key
], ids=str)
def test_extreme_small_shapes(shape, causal, window, D, path):
    """Single keys, single rows and a one-key window on every forward path."""
    B, Hq, Hkv, M, N = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=M + N + D)
    want = oracle.attention(q, k, v, causal=causal, window=window)
    o = run(q, k, v, causal, window, path)
    check(o, want, torch.bfloat16, f"{shape} causal={causal} window={window} D={D} path={path}")


@pytest.mark.parametrize("path", ALL_PATHS, ids=PATH_NAMES.get)
@pytest.mark.parametrize("scale", [0.05, 0.3, -0.08])
@pytest.mark.parametrize("shape,causal,window", [
    ((1, 4, 2, 300, 300, 128), True, 0),
    ((2, 4, 1, 1, 1500, 64), True, 600),    # decode shape
    ((1, 2, 2, 200, 333, 64), False, 0),
], ids=str)
def test_explicit_scales(shape, causal, window, scale, path):
    """A caller-given logit scale, including a negative one (masked keys must
    still get probability 0 whatever the sign of the scaled scores)."""
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=M + N)
    want = oracle.attention(q, k, v, causal=causal, window=window, scale=scale)
    check(run(q, k, v, causal, window, path, scale=scale), want, torch.bfloat16,
          f"{shape} scale={scale} path={path}")


@pytest.mark.parametrize("D", [16, 32])
@pytest.mark.parametrize("mask", [(False, 0), (True, 0), (True, 9)], ids=str)
def test_small_head_dims_simt(D, mask):
    q, k, v = make_qkv(2, 4, 2, 77, 45, D, torch.float16, seed=D)
    want = oracle.attention(q, k, v, causal=mask[0], window=mask[1])
    check(run(q, k, v, mask[0], mask[1], sa.PATH_AUTO), want, torch.float16, f"D={D}")


@pytest.mark.parametrize("path", [sa.PATH_SIMT, sa.PATH_PREFILL], ids=PATH_NAMES.get)
def test_fully_masked_rows_are_zero(path):
    """Causal with M > N: the first M-N rows see no key and must be 0, not NaN."""
    q, k, v = make_qkv(1, 2, 2, 200, 50, 64, torch.bfloat16, seed=5)
    o = run(q, k, v, True, path=path)
    assert torch.isfinite(o).all() and torch.all(o[:, :, :150] == 0)
    check(o, oracle.attention(q, k, v, causal=True), torch.bfloat16, "M>N causal")


@pytest.mark.parametrize("shape", [(2, 8, 2, 1, 1000), (1, 16, 4, 3, 2500), (3, 4, 4, 2, 700), (1, 32, 2, 1, 600),
                                   (32, 8, 8, 1, 1000), (16, 16, 4, 2, 1500), (40, 4, 4, 1, 2100),
                                   (1, 32, 1, 1, 1000), (2, 8, 2, 5, 900), (4, 64, 2, 3, 1300)],
                         ids=str)
@pytest.mark.parametrize("mask", [(True, 0), (True, 333), (False, 0)], ids=str)
@pytest.mark.parametrize("D", [64, 128])
def test_decode_split_paths(shape, mask, D):
    """D = 64 runs the same tcgen05 kernel with the upper 64 columns of every
    tile read as zeros. Few groups give many splits of one tile; many groups (shapes 5-7) give
    few splits of several tiles each, which runs the K/V ring around several
    times; the last three have 32, 20 and 96 grouped rows per KV head, which the
    decode path takes in CTAs of 16 rows (the last one partly empty, rows of one
    query head split across two CTAs)."""
    B, Hq, Hkv, M, N = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, seed=N)
    want = oracle.attention(q, k, v, causal=mask[0], window=mask[1])
    for path in (sa.PATH_DECODE, sa.PATH_AUTO, sa.PATH_SIMT):
        check(run(q, k, v, mask[0], mask[1], path), want, torch.bfloat16, f"{shape} {mask} D={D} path={path}")


def whole_heads(B, H, M):
    """Every row of the first, the middle and the last (batch, head): the
    persistent prefill kernel deals each CTA work tiles from many heads, so
    whole heads cover every work tile of those heads, the last ones scheduled
    included."""
    heads = sorted({0, (B * H) // 2, B * H - 1})
    return [bh * M + i for bh in heads for i in range(M)]


def sampled(w, causal, window, path, dtype=None, count=192, heads=False):
    dtype = dtype or w.dtype
    q, k, v = workload_inputs(w, dtype)
    o = run(q, k, v, causal, window, path)
    rows = sample_rows(w.B, w.Hq, w.M, count, seed=w.seed)
    if heads:
        rows = sorted(set(rows) | set(whole_heads(w.B, w.Hq, w.M)))
    want = oracle.attention_rows(q, k, v, rows, causal=causal, window=window)
    got = o.reshape(-1, w.D)[torch.tensor(rows, device=o.device)]
    assert torch.isfinite(o).all()
    return check(got, want, dtype, f"{w.name} causal={causal} path={path}")


@pytest.mark.parametrize("path", [sa.PATH_AUTO, sa.PATH_SIMT], ids=PATH_NAMES.get)
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_d64_full_size(causal, path):
    sampled(PREFILL_D64, causal, 0, path)


@pytest.mark.parametrize("variant", ["bf16_causal", "bf16_noncausal", "fp16_causal"])
def test_prefill_d128_full_size(variant):
    dtype = torch.float16 if variant.startswith("fp16") else torch.bfloat16
    sampled(PREFILL_D128, "noncausal" not in variant, 0, sa.PATH_AUTO, dtype, heads=True)


@pytest.mark.parametrize("path", [sa.PATH_AUTO, sa.PATH_DECODE, sa.PATH_SIMT], ids=PATH_NAMES.get)
def test_decode_gqa_full_size(path):
    w = DECODE_GQA
    q, k, v = workload_inputs(w)
    o = run(q, k, v, True, w.window, path)
    want = oracle.attention(q, k, v, causal=True, window=w.window)  # 256 rows: the full output
    check(o, want, w.dtype, f"decode path={path}")


def test_long_causal_stress_full_size():
    sampled(LONG_CAUSAL, True, 0, sa.PATH_AUTO, count=160, heads=True)


def test_merge_kernel_worked_example():
    """The answer key's A1 worked answer through the GPU merge kernel."""
    m = torch.tensor([[2.0, 4.0], [-math.inf, -math.inf], [-math.inf, 1.5]], device=DEV)
    l = torch.tensor([[2.0, 1.0], [0.0, 0.0], [0.0, 2.5]], device=DEV)
    acc = torch.tensor([[[3.0], [5.0]], [[0.0], [0.0]], [[0.0], [4.0]]], device=DEV)
    o, mo, lo = sa.attn_merge(m, l, acc, torch.float32, with_stats=True)
    torch.cuda.synchronize()
    assert float(mo[0]) == 4.0 and abs(float(lo[0]) - (1 + 2 * math.exp(-2))) < 1e-6
    assert abs(float(o[0, 0]) - (5 + 3 * math.exp(-2)) / (1 + 2 * math.exp(-2))) < 1e-6
    assert float(mo[1]) == -math.inf and float(lo[1]) == 0.0 and float(o[1, 0]) == 0.0
    assert float(mo[2]) == 1.5 and abs(float(lo[2]) - 2.5) < 1e-6 and abs(float(o[2, 0]) - 1.6) < 1e-6


def test_merge_kernel_random_against_oracle():
    g = torch.Generator().manual_seed(3)
    rows, S, D = 37, 19, 128
    m = torch.randn(rows, S, generator=g) * 4
    m[::5, ::3] = -math.inf
    l = torch.rand(rows, S, generator=g) * 3
    l[m == -math.inf] = 0
    acc = torch.randn(rows, S, D, generator=g)
    acc[m == -math.inf] = 0
    o = sa.attn_merge(m.to(DEV), l.to(DEV), acc.to(DEV), torch.float32).cpu().double().numpy()
    for r in range(rows):
        mm, ll, aa = oracle.merge(m[r].double().numpy(), l[r].double().numpy(), acc[r].double().numpy())
        want = aa / ll if ll > 0 else np.zeros(D)
        assert np.allclose(o[r], want, rtol=1e-5, atol=1e-5)


def test_host_end_to_end_matches_device_call():
    w = TINY_RAGGED
    q, k, v = workload_inputs(w)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.empty_like(qh).pin_memory()
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    od = torch.empty_like(qd)
    sa.attn_fwd_host(qh, kh, vh, oh, qd, kd, vd, od, causal=True)
    ref = run(q, k, v, True)
    assert torch.equal(oh, ref.cpu())


@pytest.mark.parametrize("shape,causal,window", [
    ((1, 3, 3, 300, 300, 128), True, 0),        # three chunks of one KV head
    ((1, 20, 20, 130, 257, 64), False, 0),      # seven chunks of three heads, the last of two
    ((3, 10, 5, 130, 257, 64), False, 0),       # two chunks per batch (3 + 2 heads)
    ((17, 2, 1, 70, 90, 64), True, 33),         # chunks of whole batches (3, 3, ..., 2)
    ((2, 16, 4, 256, 512, 128), True, 0),       # GQA groups kept whole within a chunk
    ((1, 2, 2, 40, 40, 32), False, 0),          # SIMT path (D = 32)
])
def test_host_pipelined_chunks_match_device_call(shape, causal, window):
    """The host-buffer entry point cuts the problem into chunks of (batch, KV
    head) groups; every row is computed by the same kernel as in one device
    call, so the outputs are identical, and they match the oracle."""
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 17)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh = torch.full_like(qh, float("nan")).pin_memory()
    qd, kd, vd = (torch.empty_like(t, device=DEV) for t in (q, k, v))
    od = torch.empty_like(qd)
    sa.attn_fwd_host(qh, kh, vh, oh, qd, kd, vd, od, causal=causal, window=window)
    ref = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window)
    torch.cuda.synchronize()
    assert torch.equal(oh, ref.cpu())
    assert torch.equal(od, ref)
    check(oh, oracle.attention(q, k, v, causal=causal, window=window), torch.bfloat16, f"host {shape}")


@pytest.mark.parametrize("case", ["decode", "prefill"])
def test_fwd_ws_boundary_against_oracle(case):
    """The workspace boundary calls through ctypes: attn_workspace_bytes sizes the
    caller's workspace for attn_fwd_ws (per-call scratch, as the course's
    wide-row split softmax keeps it), which takes the path attn_fwd takes."""
    import ctypes

    if case == "decode":
        w = DECODE_GQA
        q, k, v = workload_inputs(w)
        causal, window = True, w.window
    else:
        q, k, v = make_qkv(1, 4, 2, 300, 700, 128, torch.bfloat16, seed=21)
        causal, window = True, 0
    B, Hq, M, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    L = sa.lib()
    n = L.attn_workspace_bytes(B, Hq, Hkv, M, N, D, window)
    assert (n > 0) == (case == "decode")
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device=DEV)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o = torch.full_like(qd, float("nan"))
    st = L.attn_fwd_ws(ctypes.c_void_p(qd.data_ptr()), ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(vd.data_ptr()),
                       ctypes.c_void_p(o.data_ptr()), B, Hq, Hkv, M, N, D, int(causal), window, 0.0, sa.ATTN_BF16,
                       ctypes.c_void_p(ws.data_ptr()) if n else None, n,
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, sa.strerror(st)
    torch.cuda.synchronize()
    check(o, oracle.attention(q, k, v, causal=causal, window=window), torch.bfloat16, f"attn_fwd_ws {case}")
