"""Decode over a paged KV cache (attn_decode_paged) against the FP64 oracle's
paged definition, on the same seeded inputs, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import streaming_attention_gb300 as sa
from oracle_pins import to_pages
from parity import check
from streaming_attention_gb300.inputs import DECODE_GQA, make_qkv, workload_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(autouse=True)
def no_device_timeouts():
    yield
    assert sa.last_device_status() == 0, "a kernel gave up on a bounded wait"


def paged_case(B, Hq, Hkv, M, Ncap, page_size, dtype, seed, shuffle=True, D=128):
    """Seeded q and a contiguous cache cut into pages (shuffled in the pool)."""
    q, k, v = make_qkv(B, Hq, Hkv, M, Ncap, D, dtype, seed)
    r = np.random.default_rng(seed) if shuffle else None
    kp, table = to_pages(k.float().numpy(), page_size, r)
    r = np.random.default_rng(seed) if shuffle else None
    vp, _ = to_pages(v.float().numpy(), page_size, r)
    kp, vp = torch.from_numpy(kp).to(dtype), torch.from_numpy(vp).to(dtype)
    return q, kp, vp, torch.from_numpy(table.astype(np.int32))


def run_paged(q, kp, vp, table, lens, max_seq_len, causal, window, workspace=True):
    qd, kd, vd = q.to(DEV), kp.to(DEV), vp.to(DEV)
    td, ld = table.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV)
    o = torch.full_like(qd, float("nan"))
    ws = None
    if workspace:
        B, Hq, M, D = q.shape
        nb = sa.attn_decode_paged_workspace_bytes(B, Hq, kp.shape[1], M, D, kp.shape[2], table.shape[1],
                                                  max_seq_len, causal, window)
        ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    sa.attn_decode_paged(qd, kd, vd, td, ld, o, max_seq_len, causal, window, workspace=ws)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("causal,window", [(True, 0), (True, 300), (False, 0), (False, 200)])
def test_paged_ragged_lengths(page_size, causal, window):
    B, Hq, Hkv, M, Ncap = 5, 8, 2, 1, 1024
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, page_size, torch.bfloat16, 7)
    lens = [1000, 1, 0, 1024, 517]
    o = run_paged(q, kp, vp, table, lens, Ncap, causal, window)
    want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, causal, window)
    check(o, want, torch.bfloat16, f"page {page_size} causal={causal} window={window}")
    assert torch.all(o[2] == 0)  # the empty sequence


@pytest.mark.parametrize("G,M", [(4, 4), (2, 8), (16, 1), (1, 3)])
def test_paged_grouped_and_speculative_rows(G, M):
    """Speculative decode: M > 1 query rows per sequence, G * M <= 16 grouped rows."""
    B, Hkv, Ncap, ps = 3, 2, 768, 64
    q, kp, vp, table = paged_case(B, G * Hkv, Hkv, M, Ncap, ps, torch.float16, 11)
    lens = [768, 301, 2]
    for causal, window in ((True, 0), (True, 129)):
        o = run_paged(q, kp, vp, table, lens, Ncap, causal, window)
        want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, causal, window)
        check(o, want, torch.float16, f"G={G} M={M} causal={causal} window={window}")


def test_paged_contiguous_cache_is_one_page_per_sequence():
    """A contiguous [B, Hkv, N, D] cache is the pool with page_size N and the
    block table [[0], [1], ...]: equal to attn_fwd's decode on the same cache."""
    B, Hq, Hkv, M, N = 4, 16, 4, 1, 1280
    q, k, v = make_qkv(B, Hq, Hkv, M, N, 128, torch.bfloat16, 13)
    table = torch.arange(B, dtype=torch.int32).reshape(B, 1)
    o = run_paged(q, k, v, table, [N] * B, N, True, 1000)
    ref = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=1000, path=sa.PATH_DECODE)
    torch.cuda.synchronize()
    assert torch.allclose(o.float(), ref.float(), atol=2e-2, rtol=0)
    check(o, oracle.attention(q, k, v, causal=True, window=1000), torch.bfloat16, "contiguous as one page")


def test_paged_max_seq_len_cuts_lengths_and_library_workspace():
    B, Hq, Hkv, M, Ncap, ps = 2, 4, 1, 2, 640, 32
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, ps, torch.bfloat16, 17)
    lens = [640, 640]
    o = run_paged(q, kp, vp, table, lens, 333, True, 0, workspace=False)
    want = oracle.attention_paged(q, kp, vp, table, lens, 333, True, 0)
    check(o, want, torch.bfloat16, "max_seq_len 333, library-allocated workspace")


def test_paged_empty_problems():
    q, kp, vp, table = paged_case(2, 4, 2, 1, 256, 16, torch.bfloat16, 19)
    o = run_paged(q, kp, vp, table, [0, 0], 256, True, 0)
    assert torch.all(o == 0)
    o = run_paged(q, kp, vp, table, [256, 100], 0, True, 0)  # max_seq_len 0
    assert torch.all(o == 0)
    q0 = q[:0].contiguous()
    o = run_paged(q0, kp, vp, table[:0].contiguous(), [], 256, True, 0)
    assert o.shape == (0, 4, 1, 128)


def test_paged_decode_workload_full_size():
    """The GQA decode workload (B=8, Hq=32, Hkv=8, N=8192, window 4096) with its
    cache cut into 16-key pages in shuffled order, against the oracle on every
    row and against the contiguous decode path."""
    w = DECODE_GQA
    q, k, v = workload_inputs(w)
    r = np.random.default_rng(3)
    kp, table = to_pages(k.float().numpy(), 16, r)
    r = np.random.default_rng(3)
    vp, _ = to_pages(v.float().numpy(), 16, r)
    kp, vp = torch.from_numpy(kp).to(w.dtype), torch.from_numpy(vp).to(w.dtype)
    table = torch.from_numpy(table.astype(np.int32))
    o = run_paged(q, kp, vp, table, [w.N] * w.B, w.N, w.causal, w.window)
    want = oracle.attention_paged(q, kp, vp, table, [w.N] * w.B, w.N, w.causal, w.window)
    check(o, want, w.dtype, "paged decode workload")
    ref = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, window=w.window, path=sa.PATH_DECODE)
    torch.cuda.synchronize()
    assert torch.allclose(o.float(), ref.float(), atol=2e-2, rtol=0)


# ---------------------------------------------------------------------------
# Head dimensions 16 and 32 (the grouped CUDA-core kernel) and 64 (the tcgen05
# kernel, the upper 64 columns of each tile read as zeros); more than 16
# grouped query rows per KV head
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D", [16, 32, 64])
@pytest.mark.parametrize("page_size", [16, 64, 128])
@pytest.mark.parametrize("causal,window", [(True, 0), (True, 300), (False, 0), (False, 200)])
def test_paged_group_head_dims(D, page_size, causal, window):
    B, Hq, Hkv, M, Ncap = 5, 8, 2, 1, 1024
    dtype = torch.bfloat16 if page_size != 64 else torch.float16
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, page_size, dtype, 31, D=D)
    lens = [1000, 1, 0, 1024, 517]
    o = run_paged(q, kp, vp, table, lens, Ncap, causal, window)
    want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, causal, window)
    check(o, want, dtype, f"D={D} page {page_size} causal={causal} window={window}")
    assert torch.all(o[2] == 0)  # the empty sequence


@pytest.mark.parametrize("D,G,M", [(128, 8, 4), (128, 32, 1), (128, 4, 5), (128, 16, 9), (64, 4, 5), (64, 16, 1),
                                   (32, 2, 11)])
def test_paged_group_many_grouped_rows(D, G, M):
    """More than 16 grouped rows per KV head at D = 128 and 64 (the tcgen05
    kernel in CTAs of 16 rows, the last one partly empty) and D = 32 (the
    grouped CUDA-core kernel in blocks of eight rows), with sequences shorter
    than M (rows with no visible key under causal)."""
    B, Hkv, Ncap, ps = 3, 2, 768, 32
    q, kp, vp, table = paged_case(B, G * Hkv, Hkv, M, Ncap, ps, torch.float16, 37, D=D)
    lens = [768, 301, 3]
    for causal, window in ((True, 0), (True, 129), (False, 0)):
        o = run_paged(q, kp, vp, table, lens, Ncap, causal, window)
        want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, causal, window)
        check(o, want, torch.float16, f"D={D} G={G} M={M} causal={causal} window={window}")


def test_paged_group_one_split_writes_output():
    """Enough (sequence, KV head) pairs that the grouped CUDA-core kernel (D = 32)
    plans one split: no workspace (its size is 0), the kernel writes o itself."""
    B, Hq, Hkv, M, Ncap, ps, D = 96, 8, 8, 1, 256, 16, 32
    nb = sa.attn_decode_paged_workspace_bytes(B, Hq, Hkv, M, D, ps, Ncap // ps, Ncap, True, 0)
    assert nb == 0
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, ps, torch.bfloat16, 41, D=D)
    lens = [int(x) for x in np.random.default_rng(41).integers(0, Ncap + 1, size=B)]
    for workspace in (True, False):
        o = run_paged(q, kp, vp, table, lens, Ncap, True, 0, workspace=workspace)
        want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, True, 0)
        check(o, want, torch.bfloat16, f"one split, workspace={workspace}")


def test_paged_decode_workload_d64():
    """The GQA decode workload's shape at D = 64 (B=8, Hq=32, Hkv=8, N=8192,
    window 4096), its cache cut into 16-key pages in shuffled order, against the
    oracle on every row and against the contiguous decode path."""
    B, Hq, Hkv, M, N, W, D = 8, 32, 8, 1, 8192, 4096, 64
    q, k, v = make_qkv(B, Hq, Hkv, M, N, D, torch.bfloat16, 43)
    r = np.random.default_rng(43)
    kp, table = to_pages(k.float().numpy(), 16, r)
    r = np.random.default_rng(43)
    vp, _ = to_pages(v.float().numpy(), 16, r)
    kp, vp = torch.from_numpy(kp).to(torch.bfloat16), torch.from_numpy(vp).to(torch.bfloat16)
    table = torch.from_numpy(table.astype(np.int32))
    o = run_paged(q, kp, vp, table, [N] * B, N, True, W)
    want = oracle.attention_paged(q, kp, vp, table, [N] * B, N, True, W)
    check(o, want, torch.bfloat16, "paged decode D=64")
    ref = sa.attention(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, window=W, path=sa.PATH_DECODE)
    torch.cuda.synchronize()
    assert torch.allclose(o.float(), ref.float(), atol=2e-2, rtol=0)


@pytest.mark.parametrize("D", [32, 128])
def test_paged_table_entries_outside_the_pool_read_zeros(D):
    """Block-table entries outside [0, num_pages) (negative or past the pool)
    read a page of zeros on both kernels (the tcgen05 kernel through a TMA
    coordinate past the pool, the grouped kernel through a bounds check): the
    result equals the oracle on the pool extended by one zero page that those
    entries point to."""
    B, Hq, Hkv, M, Ncap, ps = 3, 8, 2, 1, 512, 32
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, ps, torch.bfloat16, 47, D=D)
    num_pages = kp.shape[0]
    bad = table.clone()
    bad[0, 3] = -1
    bad[1, 0] = num_pages
    bad[2, 7] = num_pages + 1000
    lens = [500, 512, 300]
    o = run_paged(q, kp, vp, bad, lens, Ncap, True, 0)
    zero = torch.zeros((1,) + tuple(kp.shape[1:]), dtype=kp.dtype)
    kz, vz = torch.cat([kp, zero]), torch.cat([vp, zero])
    fixed = torch.where((bad < 0) | (bad >= num_pages), torch.full_like(bad, num_pages), bad)
    want = oracle.attention_paged(q, kz, vz, fixed, lens, Ncap, True, 0)
    check(o, want, torch.bfloat16, f"out-of-pool table entries D={D}")


@pytest.mark.parametrize("D", [32, 128])
@pytest.mark.parametrize("scale", [0.3, -0.1])
def test_paged_explicit_scales(D, scale):
    """A caller-given logit scale, including a negative one, on both paged kernels."""
    B, Hq, Hkv, M, Ncap, ps = 3, 8, 2, 2, 512, 32
    q, kp, vp, table = paged_case(B, Hq, Hkv, M, Ncap, ps, torch.bfloat16, 53, D=D)
    lens = [500, 7, 512]
    qd, kd, vd = q.to(DEV), kp.to(DEV), vp.to(DEV)
    td, ld = table.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV)
    o = torch.full_like(qd, float("nan"))
    sa.attn_decode_paged(qd, kd, vd, td, ld, o, Ncap, True, 100, scale)
    torch.cuda.synchronize()
    want = oracle.attention_paged(q, kp, vp, table, lens, Ncap, True, 100, scale)
    check(o, want, torch.bfloat16, f"paged D={D} scale={scale}")
