"""FP64 attention oracle (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package. The CUDA library never calls it, and it
shares no code with the CUDA library: the two meet only in the seeded input
generator, which holds none of the method's arithmetic.

The C source (``attn_oracle.c``) computes the plain definition: per query
row, materialize the FP64 score row over the allowed keys, take its maximum,
exponentiate, sum, divide ("Compare reasoning after your own attempt",
"Reference tradeoffs to challenge": the FP64 materializing oracle). The
summary merge follows the same page's A1 row and worked answer.
``decode_e4m3`` writes out the E4M3 code table of the OCP 8-bit
floating-point format, and ``attention_fp8`` is the plain attention of the
decoded tensors times their dequantization factors.

Parity pins: every exported function is pinned in ``tests/test_oracle_pins.py``
against worked answers from the pages, closed forms, invariants and an
independent library formula; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LOCK = threading.Lock()
_LIBS: dict = {}

# Planted-mistake switch of the Python functions below, the counterpart of the
# C source's ORACLE_MUTANT: 0 is the real oracle; the pin tests set another
# value for the length of one test to show that each planted mistake fails a pin.
PY_MUTANT = 0

# -ffp-contract=off keeps the FP64 results identical on x86_64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math"]


def lib_path(mutant: int = 0, out_dir: Optional[str] = None) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(out_dir or _HERE, name)


def build(mutant: int = 0, out_dir: Optional[str] = None, force: bool = False) -> str:
    """Compile the oracle with gcc; returns the shared-library path."""
    path = lib_path(mutant, out_dir)
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def _load(mutant: int = 0, out_dir: Optional[str] = None) -> ctypes.CDLL:
    key = (mutant, out_dir)
    with _LOCK:
        if key not in _LIBS:
            lib = ctypes.CDLL(build(mutant, out_dir))
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci, cd = ctypes.c_int, ctypes.c_double
            shape = [ci] * 6 + [ci, ci, cd]
            lib.oracle_attn_f64.argtypes = [dp, dp, dp, dp, *shape, ci]
            lib.oracle_attn_f64.restype = ci
            lib.oracle_attn_lse_f64.argtypes = [dp, dp, dp, dp, dp, *shape, ci]
            lib.oracle_attn_lse_f64.restype = ci
            lib.oracle_attn_rows_f64.argtypes = [dp, dp, dp, dp, *shape, i64p, ctypes.c_int64, ci]
            lib.oracle_attn_rows_f64.restype = ci
            lib.oracle_attn_weights_f64.argtypes = [dp, dp, *shape, ctypes.c_int64, dp]
            lib.oracle_attn_weights_f64.restype = ci
            lib.oracle_partial_f64.argtypes = [dp, dp, dp, *shape, ctypes.c_int64, ci, ci, dp, dp, dp]
            lib.oracle_partial_f64.restype = ci
            lib.oracle_merge_f64.argtypes = [ci, ci, dp, dp, dp, dp, dp, dp]
            lib.oracle_merge_f64.restype = None
            lib.oracle_mutant_id.restype = ci
            _LIBS[key] = lib
        return _LIBS[key]


def _f64(a) -> np.ndarray:
    """Exact widening to a contiguous float64 array (accepts numpy or torch CPU tensors)."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch

        a = a.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class Oracle:
    """Handle on one build of the oracle (mutant 0 is the real one)."""

    def __init__(self, mutant: int = 0, out_dir: Optional[str] = None):
        self.lib = _load(mutant, out_dir)

    @staticmethod
    def _dims(q, k, v):
        B, Hq, M, D = q.shape
        Bk, Hkv, N, Dk = k.shape
        if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
            raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
        return B, Hq, Hkv, M, N, D

    def attention(self, q, k, v, causal=False, window=0, scale=None, nthreads=0) -> np.ndarray:
        """Full FP64 output [B, Hq, M, D]."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, M, N, D = self._dims(q, k, v)
        scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
        o = np.zeros((B, Hq, M, D), dtype=np.float64)
        rc = self.lib.oracle_attn_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D,
                                      int(causal), int(window), scale, int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_f64 rejected the shape (rc={rc})")
        return o

    def attention_lse(self, q, k, v, causal=False, window=0, scale=None, nthreads=0):
        """Full FP64 output [B, Hq, M, D] and each row's log-sum-exp [B, Hq, M]
        (natural log of the sum of exp of its allowed logits; -inf when none)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, M, N, D = self._dims(q, k, v)
        scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
        o = np.zeros((B, Hq, M, D), dtype=np.float64)
        lse = np.full((B, Hq, M), -np.inf, dtype=np.float64)
        rc = self.lib.oracle_attn_lse_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, M, N, D,
                                          int(causal), int(window), scale, int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_lse_f64 rejected the shape (rc={rc})")
        return o, lse

    def attention_rows(self, q, k, v, rows: Sequence[int], causal=False, window=0, scale=None,
                       nthreads=0) -> np.ndarray:
        """FP64 output of selected rows only; rows index the flattened [B*Hq*M] row axis."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, M, N, D = self._dims(q, k, v)
        scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.zeros((len(r), D), dtype=np.float64)
        rc = self.lib.oracle_attn_rows_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, M, N, D,
                                           int(causal), int(window), scale,
                                           r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                           len(r), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_rows_f64 rejected the call (rc={rc})")
        return o

    def weights(self, q, k, row: int, causal=False, window=0, scale=None) -> np.ndarray:
        """Normalized attention weights of one row over the N keys."""
        q, k = _f64(q), _f64(k)
        B, Hq, Hkv, M, N, D = self._dims(q, k, k)
        scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
        w = np.zeros(max(N, 1), dtype=np.float64)
        rc = self.lib.oracle_attn_weights_f64(_ptr(q), _ptr(k), B, Hq, Hkv, M, N, D, int(causal),
                                              int(window), scale, int(row), _ptr(w))
        if rc != 0:
            raise ValueError(f"oracle_attn_weights_f64 rejected the call (rc={rc})")
        return w[:N]

    def partial(self, q, k, v, row: int, j0: int, j1: int, causal=False, window=0, scale=None):
        """Unnormalized summary (m, l, acc[D]) of one row over allowed keys in [j0, j1)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, M, N, D = self._dims(q, k, v)
        scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
        m = np.zeros(1)
        l = np.zeros(1)
        acc = np.zeros(D)
        rc = self.lib.oracle_partial_f64(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, M, N, D, int(causal),
                                         int(window), scale, int(row), int(j0), int(j1), _ptr(m),
                                         _ptr(l), _ptr(acc))
        if rc != 0:
            raise ValueError(f"oracle_partial_f64 rejected the call (rc={rc})")
        return float(m[0]), float(l[0]), acc

    def attention_paged(self, q, k_pages, v_pages, block_table, seq_lens, max_seq_len, causal=True, window=0,
                        scale=None, nthreads=0) -> np.ndarray:
        """Decode over a paged KV cache, by its definition: gather each
        sequence's first L_b keys out of the pages into a contiguous cache,
        then take the plain attention of that sequence's rows over them.
        q [B, Hq, M, D]; pools [num_pages, Hkv, page_size, D]; block_table
        [B, max_pages]; L_b = clamp(seq_lens[b], 0, min(max_seq_len,
        max_pages * page_size)). Returns [B, Hq, M, D] in FP64."""
        q, kp, vp = _f64(q), _f64(k_pages), _f64(v_pages)
        table = np.asarray(block_table, dtype=np.int64)
        lens = np.asarray(seq_lens, dtype=np.int64).reshape(-1)
        B, Hq, M, D = q.shape
        num_pages, Hkv, page_size, _ = kp.shape
        # 19 plants lengths that ignore max_seq_len
        cap = table.shape[1] * page_size if PY_MUTANT == 19 else min(int(max_seq_len), table.shape[1] * page_size)
        o = np.zeros((B, Hq, M, D), dtype=np.float64)
        for b in range(B):
            L = int(min(max(lens[b], 0), cap))
            j = np.arange(L)
            pages, rows = table[b, j // page_size], j % page_size
            if PY_MUTANT == 20:  # planted: pages taken in pool order, not through the table
                pages = b * table.shape[1] + j // page_size
            kb = np.ascontiguousarray(kp[pages, :, rows, :].transpose(1, 0, 2))[None]  # [1, Hkv, L, D]
            vb = np.ascontiguousarray(vp[pages, :, rows, :].transpose(1, 0, 2))[None]
            o[b] = self.attention(q[b:b + 1], kb, vb, causal, window, scale, nthreads)[0]
        return o

    def merge(self, m, l, acc):
        """Merge S summaries: m[S], l[S], acc[S, D] -> (m, l, acc[D])."""
        m = np.ascontiguousarray(np.asarray(m, dtype=np.float64).reshape(-1))
        l = np.ascontiguousarray(np.asarray(l, dtype=np.float64).reshape(-1))
        S = m.shape[0]
        acc = np.ascontiguousarray(np.asarray(acc, dtype=np.float64).reshape(S, -1))
        D = acc.shape[1]
        mo, lo, ao = np.zeros(1), np.zeros(1), np.zeros(max(D, 1))
        self.lib.oracle_merge_f64(S, D, _ptr(m), _ptr(l), _ptr(acc), _ptr(mo), _ptr(lo), _ptr(ao))
        return float(mo[0]), float(lo[0]), ao[:D]


_DEFAULT: Optional[Oracle] = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(0)
    return _DEFAULT


def attention(q, k, v, causal=False, window=0, scale=None, nthreads=0):
    return default().attention(q, k, v, causal, window, scale, nthreads)


def attention_lse(q, k, v, causal=False, window=0, scale=None, nthreads=0):
    return default().attention_lse(q, k, v, causal, window, scale, nthreads)


def attention_rows(q, k, v, rows, causal=False, window=0, scale=None, nthreads=0):
    return default().attention_rows(q, k, v, rows, causal, window, scale, nthreads)


def merge(m, l, acc):
    return default().merge(m, l, acc)


def attention_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, causal=True, window=0, scale=None,
                    nthreads=0):
    return default().attention_paged(q, k_pages, v_pages, block_table, seq_lens, max_seq_len, causal, window,
                                     scale, nthreads)


def cpu_threads() -> int:
    return os.cpu_count() or 1


# --------------------------------------------------------------------------
# Backward pass, FP64, by its definition
# --------------------------------------------------------------------------
def visible_mask(M, N, causal, window):
    """[M, N] boolean: key j visible to query row i (position i + N - M)."""
    pos = np.arange(M)[:, None] + (0 if PY_MUTANT == 14 else N - M)  # 14 plants top-left alignment
    j = np.arange(N)[None, :]
    keep = np.ones((M, N), dtype=bool)
    if causal:
        keep &= j <= pos
    if window > 0:
        keep &= j > pos - window
    return keep


def attention_backward(q, k, v, do, causal=False, window=0, scale=None, heads=None):
    """Gradients (dq, dk, dv) of L = sum(do * o) for o = attention(q, k, v), in FP64.

    For each (b, h): the weights P = softmax(scale * q k^T over the visible
    keys) are materialized; dv = P^T do; dP = do v^T; each row of dS is the
    softmax vector-Jacobian product of that row, dS = P * (dP - sum_j P dP)
    ("Intermediate and advanced kernel workshops", workshop I2, softmax
    backward: one reduction of y*g, then y * (g - that sum)); dq = scale dS k;
    dk = scale dS^T q. With GQA, dk and dv of a KV head sum over its query
    heads. Rows with no visible key contribute nothing. `heads`, if given, is a
    list of (b, h) pairs to evaluate (dk, dv then hold only their share)."""
    q, k, v, do = (_f64(x) for x in (q, k, v, do))
    B, Hq, M, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    G = Hq // Hkv if Hkv else 1
    scale = 1.0 / np.sqrt(D) if scale is None else float(scale)
    keep = visible_mask(M, N, causal, window)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(Hq)]
    for b, h in pairs:
        g = h // G
        s = np.where(keep, scale * (q[b, h] @ k[b, g].T), -np.inf)
        mu = s.max(axis=1, keepdims=True)
        any_key = np.isfinite(mu)
        e = np.where(keep, np.exp(s - np.where(any_key, mu, 0.0)), 0.0)
        z = e.sum(axis=1, keepdims=True)
        p = np.divide(e, z, out=np.zeros_like(e), where=z > 0)
        if PY_MUTANT == 12:  # planted: a KV head keeps only its last query head's share
            dv[b, g] = p.T @ do[b, h]
        else:
            dv[b, g] += p.T @ do[b, h]
        dp = do[b, h] @ v[b, g].T
        if PY_MUTANT == 11:  # planted: the row-sum term of the softmax VJP dropped
            ds = p * dp
        else:
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
        dq[b, h] = (1.0 if PY_MUTANT == 13 else scale) * (ds @ k[b, g])  # 13 plants a dropped scale
        dk[b, g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


# --------------------------------------------------------------------------
# Row softmax, FP64, by its definition
# --------------------------------------------------------------------------
def softmax_rows(x):
    """softmax of each row of a 2-D array in FP64: exp(x - max) / sum. The
    wide-row split method ("Intermediate and advanced kernel workshops", A2)
    reaches this exactly up to rounding; the oracle is the definition."""
    x = _f64(x)
    if x.shape[0] == 0:
        return x.copy()
    e = np.exp(x - x.max(axis=1, keepdims=True))
    if PY_MUTANT == 15:  # planted: normalized over columns instead of rows
        return e / e.sum(axis=0, keepdims=True)
    return e / e.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# 8-bit E4M3 inputs, by definition


def decode_e4m3(codes) -> np.ndarray:
    """Exact FP64 values of E4M3 codes (the OCP 8-bit floating-point format's
    E4M3 encoding): bit 7 sign, bits 6-3 exponent field e (bias 7), bits 2-0
    mantissa m; e = 0 is subnormal, m/8 * 2^-6; otherwise (1 + m/8) * 2^(e-7);
    e = 15 with m = 7 is NaN (no infinities). Accepts a uint8 array or an
    E4M3 / uint8 torch tensor."""
    if hasattr(codes, "detach"):
        import torch

        t = codes.detach().to("cpu")
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        codes = t.numpy()
    b = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    bias = 8 if PY_MUTANT == 16 else 7  # 16 plants a wrong exponent bias
    lead = 1.0 if PY_MUTANT == 17 else 0.0  # 17 plants an implicit one on subnormals
    mag = np.where(e == 0, (lead + m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - bias).astype(np.float64)))
    mag = np.where((e == 15) & (b & 0x7 == 7), np.nan, mag)
    return sign * mag


def attention_fp8(q, k, v, q_descale=1.0, k_descale=1.0, v_descale=1.0, causal=False, window=0, scale=None,
                  nthreads=0, with_lse=False):
    """Attention of dequantized E4M3 inputs: Q = q_descale * q, K = k_descale * k,
    V = v_descale * v (each product exact in FP64), then the plain FP64
    attention (and log-sum-exp) of those tensors."""
    qd = float(q_descale) * decode_e4m3(q)
    kd = float(k_descale) * decode_e4m3(k)
    vd = (1.0 if PY_MUTANT == 18 else float(v_descale)) * decode_e4m3(v)  # 18 plants a dropped V factor
    if with_lse:
        return attention_lse(qd, kd, vd, causal, window, scale, nthreads)
    return attention(qd, kd, vd, causal, window, scale, nthreads)
