"""Forward pass on E4M3 inputs (attn_fwd_fp8) against the FP64 oracle of the
dequantized tensors, through the C ABI. Tolerances: the rounding model of the
probabilities in ``fp8_tolerance``; exact-mean cases (all-zero queries, where
every probability is exactly 1) at the output cast's precision."""
import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from fp8_tolerance import CAST, bounds, check_fp8, row_bounds
from streaming_attention_gb300.inputs import PREFILL_D128, make_qkv_fp8, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


def deq(t, d):
    return float(d) * oracle.decode_e4m3(t)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16], ids=["bf16", "fp16"])
@pytest.mark.parametrize("shape,causal,window,descale", [
    ((1, 2, 2, 256, 256, 128), False, 0, (1.0, 1.0, 1.0)),
    ((1, 2, 2, 256, 256, 128), True, 0, (1.0, 1.0, 1.0)),
    ((2, 4, 2, 200, 333, 128), True, 0, (0.5, 0.25, 2.0)),     # GQA, ragged, M < N, descales
    ((1, 4, 1, 384, 384, 128), True, 150, (1.0, 1.0, 1.0)),    # window, four heads share one KV head
    ((1, 2, 2, 333, 200, 128), False, 0, (0.125, 1.0, 0.5)),   # M > N
    ((1, 2, 2, 300, 100, 128), True, 0, (1.0, 1.0, 1.0)),      # rows with no visible key
    ((1, 3, 1, 1, 777, 128), True, 64, (1.0, 1.0, 1.0)),       # one query row
])
@pytest.mark.parametrize("D", [64, 128])
def test_fp8_forward_against_oracle(out_dtype, shape, causal, window, descale, D):
    """D = 64 runs the 128-column prefill with the upper half of every tile
    read as zeros (AUTO never takes the 8-bit split decode at D = 64)."""
    B, Hq, Hkv, M, N, _ = shape
    qd, kd, vd = descale
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 21, qd, kd, vd)
    scale = 1.0 / np.sqrt(D)
    o, lse = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, q_descale=qd,
                              k_descale=kd, v_descale=vd, out_dtype=out_dtype, with_lse=True)
    torch.cuda.synchronize()
    want, want_lse = oracle.attention_fp8(q, k, v, qd, kd, vd, causal=causal, window=window, with_lse=True)
    H, sigma, wabs = bounds(deq(q, qd), deq(k, kd), deq(v, vd), causal, window, scale)
    check_fp8(o, want, H, sigma, wabs, out_dtype, f"{shape} causal={causal} window={window}")
    g = lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(g), np.isneginf(want_lse))
    fin = np.isfinite(want_lse)
    if fin.any():
        assert np.abs(g[fin] - want_lse[fin]).max() <= 2e-3


@pytest.mark.parametrize("path", [sa.PATH_AUTO, sa.PATH_PREFILL, sa.PATH_DECODE], ids=["auto", "prefill", "decode"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("shape,causal,window", [
    ((1, 2, 2, 1, 1), False, 0),      # one query, one key
    ((1, 2, 2, 5, 1), True, 0),       # one key: rows before it output 0
    ((2, 4, 2, 1, 3), True, 1),       # window 1: each row sees only its own position
    ((1, 2, 2, 200, 200), True, 1),   # window 1 over several tiles
])
def test_fp8_extreme_small_shapes(shape, causal, window, D, path):
    B, Hq, Hkv, M, N = shape
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 30, 1.0, 1.0, 1.0)
    if path == sa.PATH_DECODE and D == 64:  # the 8-bit split decode takes D = 128 only
        with pytest.raises(sa.AttnError) as e:
            sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, path=path)
        assert e.value.status == -11
        return
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, path=path)
    torch.cuda.synchronize()
    want = oracle.attention_fp8(q, k, v, causal=causal, window=window)
    H, sigma, wabs = bounds(deq(q, 1.0), deq(k, 1.0), deq(v, 1.0), causal, window, 1.0 / np.sqrt(D))
    check_fp8(o, want, H, sigma, wabs, torch.bfloat16, f"{shape} causal={causal} window={window} D={D}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_zero_queries_give_exact_means(causal):
    """All-zero queries: every visible key scores 0, every probability is exactly
    1 in E4M3, and each output row is the mean of its visible V rows."""
    B, Hq, Hkv, M, N, D = 1, 2, 1, 256, 300, 128
    _, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 22, 1.0, 1.0, 0.5)
    q = torch.zeros(B, Hq, M, D).to(torch.float8_e4m3fn)
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, v_descale=0.5)
    torch.cuda.synchronize()
    want = oracle.attention_fp8(q, k, v, 1.0, 1.0, 0.5, causal=causal)
    err = np.abs(o.cpu().double().numpy() - want)
    assert (err <= CAST[torch.bfloat16] * np.abs(want) + 1e-5).all(), err.max()


def test_fp8_empty_dims():
    q, k, v = make_qkv_fp8(1, 2, 2, 0, 64, 128, 0)
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    assert o.shape == (1, 2, 0, 128)
    q, k, v = make_qkv_fp8(1, 2, 2, 64, 0, 128, 0)
    o, lse = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), with_lse=True)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_fp8_d64_many_work_tiles_and_no_decode_path():
    """E4M3 at D = 64 over more work tiles than SMs (each persistent CTA walks
    several), every row; the explicit split-decode path refuses D = 64."""
    B, Hq, Hkv, M, N, D = 2, 16, 4, 1100, 1300, 64
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 29, 1.0, 0.5, 1.0)
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, k_descale=0.5)
    torch.cuda.synchronize()
    want = oracle.attention_fp8(q, k, v, 1.0, 0.5, 1.0, causal=True)
    H, sigma, wabs = bounds(deq(q, 1.0), deq(k, 0.5), deq(v, 1.0), True, 0, 1.0 / np.sqrt(D))
    check_fp8(o, want, H, sigma, wabs, torch.bfloat16, "E4M3 D=64 many work tiles")
    o2 = torch.empty(q.shape, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(sa.AttnError) as e:
        sa.attn_fwd_fp8(q.to(DEV), k.to(DEV), v.to(DEV), o2, None, True, 0, path=sa.PATH_DECODE)
    assert e.value.status == -11


def test_fp8_full_size_sampled_rows():
    """The causal prefill shape (B=2, H=32, M=N=4096, D=128) in E4M3, checked on
    sampled rows: first and last rows of query tiles, the tail, random rows."""
    w = PREFILL_D128
    q, k, v = make_qkv_fp8(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, 23)
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.Hq, w.M, 96)
    qf, kf, vf = deq(q, 1.0), deq(k, 1.0), deq(v, 1.0)
    want = oracle.attention_rows(qf, kf, vf, rows, causal=True)
    got = o.reshape(-1, w.D)[torch.tensor(rows)].cpu()
    H, sigma, wabs = row_bounds(qf, kf, vf, rows, True, 0, 1.0 / np.sqrt(w.D))
    check_fp8(got, want, H, sigma, wabs, torch.bfloat16, "full size")


# --------------------------------------------------------------------------
# Split-KV decode on E4M3 inputs (contiguous and paged caches)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("shape,causal,window,descale", [
    ((2, 8, 2, 1, 1500, 128), True, 700, (1.0, 1.0, 1.0)),
    ((1, 32, 8, 1, 8192, 128), True, 0, (0.5, 0.25, 2.0)),
    ((1, 4, 1, 3, 777, 128), True, 0, (1.0, 1.0, 1.0)),      # speculative rows: G * M = 12
    ((3, 16, 1, 1, 2049, 128), False, 0, (1.0, 0.5, 1.0)),   # G = 16, ragged N
    ((2, 32, 1, 1, 1500, 128), True, 300, (1.0, 1.0, 1.0)),  # 32 grouped rows: two CTAs of 16 on the decode path
    ((1, 8, 2, 5, 900, 128), True, 0, (0.5, 1.0, 1.0)),      # 20 grouped rows, the second CTA partly empty
])
@pytest.mark.parametrize("path", [sa.PATH_AUTO, sa.PATH_DECODE, sa.PATH_PREFILL],
                         ids=["auto", "decode", "prefill"])
def test_fp8_decode_shapes(shape, causal, window, descale, path):
    B, Hq, Hkv, M, N, D = shape
    qd, kd, vd = descale
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 24, qd, kd, vd)
    o, lse = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, q_descale=qd,
                              k_descale=kd, v_descale=vd, with_lse=True, path=path)
    torch.cuda.synchronize()
    want, want_lse = oracle.attention_fp8(q, k, v, qd, kd, vd, causal=causal, window=window, with_lse=True)
    H, sigma, wabs = bounds(deq(q, qd), deq(k, kd), deq(v, vd), causal, window, 1.0 / np.sqrt(D))
    check_fp8(o, want, H, sigma, wabs, torch.bfloat16, f"{shape} path={path}")
    assert np.abs(lse.cpu().double().numpy() - want_lse).max() <= 2e-3


@pytest.mark.parametrize("N,causal,window", [(256, True, 0), (384, True, 0), (512, False, 0), (640, True, 0),
                                             (1100, True, 300), (1100, False, 0)])
def test_fp8_decode_round_counts(N, causal, window):
    """304 KV groups (B = 76, Hkv = 4) take one split each, so a CTA streams all
    ceil(N / 128) key tiles: the 8-bit decode's rounds of two tiles with an even
    and an odd tile count, several rounds, and a window that starts inside a round."""
    B, Hq, Hkv, M, D = 76, 8, 4, 1, 128
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 31, 1.0, 1.0, 1.0)
    o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, path=sa.PATH_DECODE)
    torch.cuda.synchronize()
    want = oracle.attention_fp8(q, k, v, causal=causal, window=window)
    H, sigma, wabs = bounds(deq(q, 1.0), deq(k, 1.0), deq(v, 1.0), causal, window, 1.0 / np.sqrt(D))
    check_fp8(o, want, H, sigma, wabs, torch.bfloat16, f"rounds N={N} causal={causal} window={window}")


def test_fp8_decode_workload_full_size():
    """The GQA decode shape (B=8, Hq=32, Hkv=8, M=1, N=8192, window 4096) in E4M3,
    every row, with a caller workspace."""
    from streaming_attention_gb300.inputs import DECODE_GQA as w
    q, k, v = make_qkv_fp8(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, 25)
    nb = sa.attn_fwd_fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, True, w.window, sa.PATH_DECODE)
    assert nb > 0 and sa.attn_fwd_fp8_workspace_bytes(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, True, w.window,
                                                       sa.PATH_PREFILL) == 0
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=DEV)
    sa.attn_fwd_fp8(q.to(DEV), k.to(DEV), v.to(DEV), o, None, True, w.window, path=sa.PATH_DECODE, workspace=ws)
    torch.cuda.synchronize()
    want = oracle.attention_fp8(q, k, v, causal=True, window=w.window)
    H, sigma, wabs = bounds(deq(q, 1.0), deq(k, 1.0), deq(v, 1.0), True, w.window, 1.0 / np.sqrt(w.D))
    check_fp8(o, want, H, sigma, wabs, torch.bfloat16, "decode workload")


@pytest.mark.parametrize("page_size", [16, 64, 128, 256])
def test_fp8_paged_ragged_lengths(page_size):
    from oracle_pins import to_pages
    B, Hq, Hkv, M, Ncap, D = 4, 8, 2, 2, 1024, 128
    qd, kd, vd = 0.5, 1.0, 2.0
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, Ncap, D, 26, qd, kd, vd)
    rng = np.random.default_rng(5)
    kp, table = to_pages(k.float().numpy(), page_size, rng)
    rng = np.random.default_rng(5)
    vp, _ = to_pages(v.float().numpy(), page_size, rng)
    f8 = torch.float8_e4m3fn
    kp, vp = torch.from_numpy(kp).to(f8), torch.from_numpy(vp).to(f8)  # exact: the values came from E4M3
    table = torch.from_numpy(table.astype(np.int32))
    lens = [1000, 1, 1024, 517]
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    use_ws = page_size in (16, 128)  # the others let the library allocate it
    nb = sa.attn_decode_paged_fp8_workspace_bytes(B, Hq, Hkv, M, D, page_size, table.shape[1], Ncap, True, 0)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV) if use_ws else None
    sa.attn_decode_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV),
                             torch.tensor(lens, dtype=torch.int32, device=DEV), o, Ncap, causal=True,
                             q_descale=qd, k_descale=kd, v_descale=vd, workspace=ws)
    torch.cuda.synchronize()
    want = oracle.attention_paged(deq(q, qd), deq(kp, kd), deq(vp, vd), table, lens, Ncap, True, 0)
    qf, kf, vf = deq(q, qd), deq(k, kd), deq(v, vd)
    for b, L in enumerate(lens):
        H, sigma, wabs = bounds(qf[b:b + 1], kf[b:b + 1, :, :L], vf[b:b + 1, :, :L], True, 0, 1.0 / np.sqrt(D))
        check_fp8(o[b:b + 1], want[b:b + 1], H, sigma, wabs, torch.bfloat16, f"page {page_size} seq {b}")


@pytest.mark.parametrize("D,G,M,page_size", [(64, 4, 1, 16), (32, 2, 2, 64), (128, 8, 4, 32), (128, 32, 1, 128)])
def test_fp8_paged_group_shapes(D, G, M, page_size):
    """E4M3 paged decode on the grouped CUDA-core kernel: D < 128, or more than
    16 grouped rows per KV head at D = 128; FP16 output for one case."""
    from oracle_pins import to_pages
    B, Hkv, Ncap = 3, 2, 1024
    Hq = G * Hkv
    qd, kd, vd = 0.5, 1.0, 2.0
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, Ncap, D, 28, qd, kd, vd)
    rng = np.random.default_rng(6)
    kp, table = to_pages(k.float().numpy(), page_size, rng)
    rng = np.random.default_rng(6)
    vp, _ = to_pages(v.float().numpy(), page_size, rng)
    f8 = torch.float8_e4m3fn
    kp, vp = torch.from_numpy(kp).to(f8), torch.from_numpy(vp).to(f8)  # exact: the values came from E4M3
    table = torch.from_numpy(table.astype(np.int32))
    lens = [1000, 2, 517]
    out_dtype = torch.float16 if D == 32 else torch.bfloat16
    for window in (0, 300):
        o = torch.full(q.shape, float("nan"), dtype=out_dtype, device=DEV)
        sa.attn_decode_paged_fp8(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV),
                                 torch.tensor(lens, dtype=torch.int32, device=DEV), o, Ncap, causal=True,
                                 window=window, q_descale=qd, k_descale=kd, v_descale=vd)
        torch.cuda.synchronize()
        want = oracle.attention_paged(deq(q, qd), deq(kp, kd), deq(vp, vd), table, lens, Ncap, True, window)
        qf, kf, vf = deq(q, qd), deq(k, kd), deq(v, vd)
        for b, L in enumerate(lens):
            H, sigma, wabs = bounds(qf[b:b + 1], kf[b:b + 1, :, :L], vf[b:b + 1, :, :L], True, window,
                                    1.0 / np.sqrt(D))
            check_fp8(o[b:b + 1], want[b:b + 1], H, sigma, wabs, out_dtype,
                      f"D={D} G={G} M={M} window={window} seq {b}")


def test_fp8_rising_maximum_stress():
    """The long causal stress construction in E4M3 (Q[..., D-1] = 8, K[..., j, D-1]
    rising from -42 to 42, each rounded to E4M3): the logit row maximum rises by
    about 60 base-2 units along the keys, so the lazy rescale fires again and
    again, while P stays within E4M3's range. Sampled rows, causal and noncausal."""
    from streaming_attention_gb300.inputs import _ramp_bias
    B, H, M, N, D = 1, 4, 4096, 4096, 128
    g = torch.Generator().manual_seed(27)
    q = torch.randn(B, H, M, D, generator=g)
    k = torch.randn(B, H, N, D, generator=g)
    v = torch.randn(B, H, N, D, generator=g)
    _ramp_bias(q, k)
    q, k, v = (t.to(torch.float8_e4m3fn) for t in (q, k, v))
    qf, kf, vf = deq(q, 1.0), deq(k, 1.0), deq(v, 1.0)
    rows = sample_rows(B, H, M, 64, seed=28)
    for causal in (True, False):
        o = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal)
        torch.cuda.synchronize()
        want = oracle.attention_rows(qf, kf, vf, rows, causal=causal)
        got = o.reshape(-1, D)[torch.tensor(rows)].cpu()
        H_, sigma, wabs = row_bounds(qf, kf, vf, rows, causal, 0, 1.0 / np.sqrt(D))
        check_fp8(got, want, H_, sigma, wabs, torch.bfloat16, f"stress causal={causal}")


@pytest.mark.parametrize("shape,causal,window,out_dtype", [
    ((40, 16, 1, 1, 1000, 128), True, 0, torch.float16),     # 16 grouped rows (the widest softmax form), cluster merge
    ((2, 8, 2, 4, 2500, 128), True, 600, torch.float16),     # speculative rows with a window
    ((1, 8, 1, 2, 20000, 128), False, 0, torch.bfloat16),    # more than 8 splits: the merge kernel path
])
def test_fp8_decode_output_types_and_split_forms(shape, causal, window, out_dtype):
    B, Hq, Hkv, M, N, D = shape
    q, k, v = make_qkv_fp8(B, Hq, Hkv, M, N, D, 29, 1.0, 0.5, 1.5)
    o, lse = sa.attention_fp8(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, k_descale=0.5,
                              v_descale=1.5, out_dtype=out_dtype, with_lse=True, path=sa.PATH_DECODE)
    torch.cuda.synchronize()
    want, want_lse = oracle.attention_fp8(q, k, v, 1.0, 0.5, 1.5, causal=causal, window=window, with_lse=True)
    H, sigma, wabs = bounds(deq(q, 1.0), deq(k, 0.5), deq(v, 1.5), causal, window, 1.0 / np.sqrt(D))
    check_fp8(o, want, H, sigma, wabs, out_dtype, f"{shape} {out_dtype}")
    g = lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(g), np.isneginf(want_lse))
    fin = np.isfinite(want_lse)
    assert np.abs(g[fin] - want_lse[fin]).max() <= 2e-3
