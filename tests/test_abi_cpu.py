"""The C-ABI library loads and exports every symbol declared in include/attn.h,
and metadata validation answers with status codes. No compute call is made:
everything here runs without a GPU."""
import ctypes
import os
import re

import pytest

import streaming_attention_gb300 as sa
from streaming_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    B.build()
    return sa.lib()


def declared_symbols():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert "attn_fwd" in names and len(names) >= 8, names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_version_and_strerror(L):
    assert L.attn_version() >= 100
    for st in range(0, -12, -1):
        assert sa.strerror(st) and sa.strerror(st) != "unknown status", st
    assert sa.strerror(-99) == "unknown status"


A16 = ctypes.c_void_p(0x10000)   # 16-byte aligned placeholder (never dereferenced)
A8 = ctypes.c_void_p(0x10008)


def fwd(L, q=A16, k=A16, v=A16, o=A16, B_=1, Hq=2, Hkv=2, M=8, N=8, D=64, causal=0, window=0, dtype=0):
    return L.attn_fwd(q, k, v, o, B_, Hq, Hkv, M, N, D, causal, window, 0.0, dtype, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=7), -3),
    (dict(B_=-1), -2),
    (dict(M=-1), -2),
    (dict(N=-5), -2),
    (dict(D=0), -2),
    (dict(Hkv=0), -2),
    (dict(Hq=6, Hkv=4), -5),
    (dict(D=48), -4),
    (dict(D=256), -4),
    (dict(B_=64, Hq=64, M=4096, D=128), -6),
    (dict(q=None), -1),
    (dict(o=None), -1),
    (dict(k=None), -1),
    (dict(q=A8), -7),
    (dict(v=A8), -7),
])
def test_validation_status(L, kw, status):
    assert fwd(L, **kw) == status


def test_forced_path_checks(L):
    # an out-of-range path value is rejected before any launch
    st = L.attn_fwd_ex(A16, A16, A16, A16, 1, 2, 2, 8, 8, 64, 0, 0, 0.0, 0, 9, None, 0, None)
    assert st == -11
    # decode and prefill need D in {64, 128}; the pair-MMA prefill D = 128
    for path in (sa.PATH_DECODE, sa.PATH_PREFILL, sa.PATH_PREFILL_PAIR):
        st = L.attn_fwd_ex(A16, A16, A16, A16, 1, 2, 2, 8, 8, 32, 0, 0, 0.0, 0, path, None, 0, None)
        assert st == -4, path
    assert L.attn_fwd_ex(A16, A16, A16, A16, 1, 2, 2, 8, 8, 64, 0, 0, 0.0, 0, sa.PATH_PREFILL_PAIR, None, 0,
                         None) == -4
    assert L.attn_fwd_ex(A16, A16, A16, A16, 1, 2, 2, 8, 8, 128, 0, 0, 0.0, 0, 5, None, 0, None) == -11
    # the E4M3 entry point offers neither the CUDA-core nor the pair path
    assert L.attn_fwd_fp8(A16, A16, A16, A16, None, 1, 2, 2, 8, 8, 128, 0, 0, 0.0, 1.0, 1.0, 1.0, 0,
                          sa.PATH_PREFILL_PAIR, None, 0, None) == -11


def test_simt_grid_limit(L):
    # the CUDA-core kernel takes at most 65535 (batch, query head) pairs; the
    # check comes before any launch
    for D in (16, 32):  # AUTO has no other kernel for these head dimensions
        assert fwd(L, B_=1, Hq=65536, Hkv=65536, M=1, N=8, D=D) == -11, D
    args = (A16, A16, A16, A16, 1, 65536, 65536, 1, 256, 64, 0, 0, 0.0, 0)
    assert L.attn_fwd_ex(*args, sa.PATH_SIMT, None, 0, None) == -11
    # B*Hkv > 65535 is past the tcgen05 decode's grid too, so its D = 64 splits run on the CUDA-core kernel
    assert L.attn_fwd_ex(*args, sa.PATH_DECODE, None, 0, None) == -11
    assert L.attn_fwd_decode_noalloc(*args, None) == -11
    # the tcgen05 decode (D = 64 and 128) only needs B*Hkv <= 65535: B*Hq may exceed it
    assert sa.attn_workspace_bytes_ex(1, 4096, 4096, 1, 512, 64, 0, 0, sa.PATH_AUTO) > 0
    assert sa.attn_workspace_bytes_ex(1, 65536, 4096, 1, 512, 64, 0, 0, sa.PATH_AUTO) > 0
    # AUTO leaves decode to the prefill kernel when no split kernel fits (D = 64, B*Hkv > 65535)
    assert sa.attn_workspace_bytes_ex(1, 65536, 65536, 1, 512, 64, 0, 0, sa.PATH_AUTO) == 0


def test_workspace_bytes(L):
    # prefill and SIMT need none; decode needs room for its split summaries
    assert sa.attn_workspace_bytes_ex(2, 32, 32, 4096, 4096, 128, True, 0, sa.PATH_SIMT) == 0
    n = sa.attn_workspace_bytes_ex(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_DECODE)
    rows = 8 * 32
    assert n >= rows * 4 * (128 + 2)
    assert sa.attn_workspace_bytes_ex(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_AUTO) == n
    assert sa.attn_workspace_bytes_ex(-1, 32, 8, 1, 8192, 128, True, 4096, 0) == 0


def test_boundary_workspace_query_and_fwd_ws(L):
    """The workspace boundary calls: attn_workspace_bytes(B, Hq, Hkv, M, N, D, window)
    sizes the workspace of attn_fwd_ws (the path attn_fwd takes) for either
    causal value, and attn_fwd_ws refuses a missing or short workspace before
    launching anything."""
    dec = (8, 32, 8, 1, 8192, 128)
    n = sa.attn_workspace_bytes(*dec, 4096)
    assert n > 0
    assert n == max(sa.attn_workspace_bytes_ex(*dec, c, 4096, sa.PATH_AUTO) for c in (0, 1))
    assert sa.attn_workspace_bytes(2, 32, 32, 4096, 4096, 128, 0) == 0  # prefill needs none
    assert sa.attn_workspace_bytes(-1, 32, 8, 1, 8192, 128, 0) == 0
    assert sa.attn_workspace_bytes(8, 32, 8, 0, 8192, 128, 0) == 0  # empty output
    args = (A16, A16, A16, A16, *dec, 1, 4096, 0.0, 0)
    assert L.attn_fwd_ws(*args, None, 0, None) == -8
    assert L.attn_fwd_ws(*args, A16, n - 1, None) == -8
    assert L.attn_fwd_ws(*args, A8, n, None) == -7
    # metadata validation comes first, as for attn_fwd
    assert L.attn_fwd_ws(A16, A16, A16, A16, 1, 6, 4, 8, 8, 64, 0, 0, 0.0, 0, None, 0, None) == -5
    assert L.attn_fwd_ws(A16, A16, A16, A16, 1, 2, 2, 8, 8, 64, 0, 0, 0.0, 9, None, 0, None) == -3


def test_merge_validation(L):
    assert L.attn_merge(A16, A16, A16, A16, None, None, 4, 0, 64, 2, None) == -2
    assert L.attn_merge(A16, A16, A16, A16, None, None, 4, 2, 64, 5, None) == -3
    assert L.attn_merge(None, A16, A16, A16, None, None, 4, 2, 64, 2, None) == -1
    assert L.attn_merge(A16, A16, A16, A16, None, None, 0, 2, 64, 2, None) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from streaming_attention_gb300 import binding

    monkeypatch.setattr(binding, "_LIB_FILE", str(tmp_path / "absent.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(FileNotFoundError):
        binding.lib()


A4 = ctypes.c_void_p(0x10004)


def paged(L, q=A16, kp=A16, vp=A16, table=A16, lens=A16, o=A16, B_=2, Hq=8, Hkv=2, M=1, D=128, num_pages=4,
          page_size=16, max_pages=2, max_seq_len=32, dtype=0):
    return L.attn_decode_paged(q, kp, vp, table, lens, o, B_, Hq, Hkv, M, D, num_pages, page_size, max_pages,
                               max_seq_len, 1, 0, 0.0, dtype, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), -3),
    (dict(B_=-1), -2),
    (dict(num_pages=-1), -2),
    (dict(max_pages=-3), -2),
    (dict(max_seq_len=-1), -2),
    (dict(page_size=48), -2),
    (dict(page_size=8), -2),
    (dict(page_size=0), -2),
    (dict(Hkv=0), -2),
    (dict(Hq=6, Hkv=4), -5),
    (dict(D=48), -4),
    (dict(D=256), -4),
    (dict(Hq=2, Hkv=2, M=1100000), -6),        # D = 128 (and 64): more than 16 x 65535 grouped rows
    (dict(Hq=2, Hkv=2, M=600000, D=32), -6),   # D = 32: more than 8 x 65535 grouped rows
    (dict(num_pages=1 << 20, page_size=128), -6),
    (dict(B_=70000, Hkv=1, Hq=1), -6),
    (dict(q=None), -1),
    (dict(kp=None), -1),
    (dict(table=None), -1),
    (dict(lens=None), -1),
    (dict(o=A8), -7),
    (dict(vp=A8), -7),
    (dict(table=ctypes.c_void_p(0x10002)), -7),
])
def test_paged_validation_status(L, kw, status):
    assert paged(L, **kw) == status


def test_paged_workspace_bytes(L):
    # the decode workload as pages of 16 keys: rows x splits x (2 + D) floats, 256-byte aligned parts
    nb = sa.attn_decode_paged_workspace_bytes(8, 32, 8, 1, 128, 16, 512, 8192, True, 4096)
    rows = 8 * 32
    assert nb > 0 and nb % 256 == 0
    S = nb // (rows * 4 * 130)
    assert 1 <= S <= 64
    assert sa.attn_decode_paged_workspace_bytes(8, 32, 8, 1, 48, 16, 512, 8192, True, 0) == 0   # D = 48
    # D = 64 (the grouped CUDA-core kernel) and 32 grouped rows per KV head at D = 128 (two CTAs of 16)
    assert sa.attn_decode_paged_workspace_bytes(8, 32, 8, 1, 64, 16, 512, 8192, True, 0) % 256 == 0
    assert sa.attn_decode_paged_workspace_bytes(2, 32, 1, 1, 128, 16, 512, 8192, True, 0) > 0
    assert sa.attn_decode_paged_workspace_bytes(8, 32, 8, 1, 128, 16, 512, 0, True, 0) == 0     # no keys
    assert sa.attn_decode_paged_workspace_bytes(0, 32, 8, 1, 128, 16, 512, 8192, True, 0) == 0  # no rows
    # a 4-byte aligned table and length array are accepted (validation passes, nothing launched: B = 0)
    assert paged(L, table=A4, lens=A4, B_=0) == 0


def test_split_softmax_resident_needs_no_scratch(L):
    assert sa.attn_split_softmax_workspace_bytes(1024, 131072, 0) == 0
    assert sa.attn_split_softmax_workspace_bytes(1024, 131072, 4096) == 8 * 1024 * 33


def test_split_softmax_scratch_matches_the_a2_worked_answer(L):
    import json
    fx = json.load(open(os.path.join(ROOT, "tests", "golden", "a2_split_softmax_example.json")))
    assert -(-fx["N"] // fx["chunk"]) == fx["chunks"]
    assert sa.attn_split_softmax_workspace_bytes(fx["M"], fx["N"], fx["chunk"]) == fx["scratch_bytes"]


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=9), -3),
    (dict(M=-1), -2),
    (dict(N=0), -2),
    (dict(N=131073), -2),
    (dict(chunk=512), -2),
    (dict(M=20000, N=131072), -6),
    (dict(M=70000, N=16), -2),       # more rows than one grid dimension holds
    (dict(x=None), -1),
    (dict(y=A8), -7),
])
def test_split_softmax_validation(L, kw, status):
    a = dict(x=A16, y=A16, M=4, N=100, chunk=1024, dtype=0)
    a.update(kw)
    assert L.attn_split_softmax(a["x"], a["y"], a["M"], a["N"], a["chunk"], a["dtype"], None, 0, None) == status


def test_selftest_rejects_bad_limits(L):
    assert L.attn_selftest_bounded_wait(0, None) == -2
    assert L.attn_selftest_bounded_wait(3000000, None) == -2


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=7), -3),
    (dict(dtype=2), -3),                 # FP32 output is not offered
    (dict(D=32), -4),
    (dict(D=48), -4),
    (dict(path=3, D=64), -11),           # the 8-bit split decode is D = 128 only; D = 64 runs the prefill
    (dict(Hq=6, Hkv=4), -5),
    (dict(k=None), -1),
    (dict(q=A8), -7),
    (dict(lse=ctypes.c_void_p(0x10002)), -7),
    (dict(M=0), 0),                      # empty output: nothing to do, no launch
    (dict(path=1), -11),                 # no SIMT form for 8-bit inputs
    (dict(path=7), -11),
    (dict(path=3, Hq=1, Hkv=1, M=1100000), -11),  # more than 16 x 65535 grouped rows for the decode grid
])
def test_fp8_validation_status(L, kw, status):
    a = dict(q=A16, k=A16, v=A16, o=A16, lse=None, B_=1, Hq=2, Hkv=2, M=8, N=8, D=128, dtype=0, path=0)
    a.update(kw)
    st = L.attn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B_"], a["Hq"], a["Hkv"], a["M"], a["N"],
                        a["D"], 1, 0, 0.0, 1.0, 1.0, 1.0, a["dtype"], a["path"], None, 0, None)
    assert st == status


def test_fp8_workspace_bytes(L):
    # the 8-bit decode plan has its own query (today the same split plan as the 16-bit one)
    n8 = sa.attn_fwd_fp8_workspace_bytes(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_DECODE)
    n16 = sa.attn_workspace_bytes_ex(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_DECODE)
    assert n8 == n16 > 0
    assert sa.attn_fwd_fp8_workspace_bytes(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_AUTO) == n8
    assert sa.attn_fwd_fp8_workspace_bytes(8, 32, 8, 1, 8192, 128, True, 4096, sa.PATH_PREFILL) == 0
    assert sa.attn_fwd_fp8_workspace_bytes(8, 32, 8, 1, 8192, 64, True, 4096, sa.PATH_DECODE) == 0
    assert sa.attn_fwd_fp8_workspace_bytes(2, 32, 32, 4096, 4096, 128, True, 0, sa.PATH_AUTO) == 0
    p8 = sa.attn_decode_paged_fp8_workspace_bytes(8, 32, 8, 1, 128, 16, 512, 8192, True, 4096)
    assert p8 >= sa.attn_decode_paged_workspace_bytes(8, 32, 8, 1, 128, 16, 512, 8192, True, 4096) > 0


def paged_fp8(L, q=A16, kp=A16, vp=A16, table=A16, lens=A16, o=A16, B_=2, Hq=8, Hkv=2, M=1, D=128, num_pages=4,
              page_size=16, max_pages=2, max_seq_len=32, dtype=0):
    return L.attn_decode_paged_fp8(q, kp, vp, table, lens, o, B_, Hq, Hkv, M, D, num_pages, page_size, max_pages,
                                   max_seq_len, 1, 0, 0.0, 1.0, 1.0, 1.0, dtype, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=2), -3),               # the output is BF16 or FP16
    (dict(page_size=48), -2),
    (dict(Hq=6, Hkv=4), -5),
    (dict(D=48), -4),
    (dict(kp=None), -1),
    (dict(o=A8), -7),
    (dict(B_=0), 0),                   # no rows: nothing to do, no launch
])
def test_paged_fp8_validation_status(L, kw, status):
    assert paged_fp8(L, **kw) == status


def test_fp8_workspace_queries_reject_bad_shapes(L):
    assert sa.attn_fwd_fp8_workspace_bytes(-1, 32, 8, 1, 8192, 128, True, 0, sa.PATH_DECODE) == 0
    assert sa.attn_fwd_fp8_workspace_bytes(8, 32, 8, 1, 8192, 128, True, 0, sa.PATH_SIMT) == 0
    # 64 grouped rows: four CTAs of 16 rows per KV head on the decode path; AUTO takes the prefill
    assert sa.attn_fwd_fp8_workspace_bytes(1, 64, 1, 1, 8192, 128, True, 0, sa.PATH_DECODE) > 0
    assert sa.attn_fwd_fp8_workspace_bytes(1, 64, 1, 1, 8192, 128, True, 0, sa.PATH_AUTO) == 0
    assert sa.attn_decode_paged_fp8_workspace_bytes(8, 32, 8, 1, 48, 16, 512, 8192, True, 0) == 0  # D = 48
    assert sa.attn_decode_paged_fp8_workspace_bytes(8, 32, 8, 1, 128, 48, 512, 8192, True, 0) == 0  # page 48


def test_prefill_abort_selftest_validation(L):
    # validation answers before any launch
    st = L.attn_selftest_prefill_abort(A16, A16, A16, A16, 1, 2, 2, 64, 64, 64, 0, 1, None)
    assert st == -4  # D must be 128
    st = L.attn_selftest_prefill_abort(A16, A16, A16, A16, 1, 2, 2, 64, 64, 128, 0, -1, None)
    assert st == -2
    st = L.attn_selftest_prefill_abort(A16, A16, A16, A16, 1, 2, 2, 0, 64, 128, 0, 1, None)
    assert st == -2


def test_host_entry_validation(L):
    # device buffers validated as attn_fwd does, then the host pointers; no copy is started
    args = [A16, A16, A16, A16, A16, A16, A16, A16, 1, 2, 2, 8, 8, 64, 0, 0, 0.0, 0, None, 0, None]
    bad_host = list(args)
    bad_host[0] = None  # q_h
    assert L.attn_fwd_host(*bad_host) == -1
    bad_dev = list(args)
    bad_dev[4] = ctypes.c_void_p(0x10008)  # q_d misaligned
    assert L.attn_fwd_host(*bad_dev) == -7
    bad_shape = list(args)
    bad_shape[9], bad_shape[10] = 6, 4  # Hq % Hkv != 0
    assert L.attn_fwd_host(*bad_shape) == -5


@pytest.mark.parametrize("kw,status", [
    (dict(D=48), -4),
    (dict(D=256), -4),
    (dict(Hq=6, Hkv=4), -5),
    (dict(dq=None), -1),
    (dict(lse=ctypes.c_void_p(0x10002)), -7),
    (dict(B_=0, D=16), 0),   # no rows and no keys: nothing to write, no launch
    (dict(B_=0, D=32), 0),
    (dict(B_=1, Hq=65536, Hkv=65536, D=16), -11),   # past the CUDA-core kernels' grid
])
def test_bwd_validation_status(L, kw, status):
    """attn_bwd takes D in {16, 32, 64, 128}; validation answers before any launch."""
    a = dict(q=A16, k=A16, v=A16, o=A16, d_o=A16, lse=A16, dq=A16, dk=A16, dv=A16, B_=1, Hq=2, Hkv=2, M=8,
             N=8, D=128)
    a.update(kw)
    st = L.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["d_o"], a["lse"], a["dq"], a["dk"], a["dv"], a["B_"],
                    a["Hq"], a["Hkv"], a["M"], a["N"], a["D"], 1, 0, 0.0, 0, None, 0, None)
    assert st == status
