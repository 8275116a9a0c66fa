"""Pins for the FP64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with an outside fact: a worked answer printed on the pages
(fixtures under ``tests/golden/``), a closed form, an invariant, or an
independent library formula on tiny inputs. ``test_oracle_pins.py`` runs them
on the real oracle, and on deliberately broken builds to show that each
planted mistake is caught by at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float64).numpy()


# --------------------------------------------------------------------------
# Worked answers printed on the pages
# --------------------------------------------------------------------------
def a3_inputs():
    """D=1 encoding of the A3 example: q = 1, k_j = logit_j, scale = 1."""
    fx = _golden("a3_worked_example.json")
    logits = [math.log(2.0) if x == "ln2" else float(x) for x in fx["logits"]]
    q = np.ones((1, 1, 1, 1))
    k = np.array(logits, dtype=np.float64).reshape(1, 1, 3, 1)
    v = np.array(fx["values"], dtype=np.float64).reshape(1, 1, 3, 1)
    return fx, q, k, v


def pin_a3_worked_example(orc):
    fx, q, k, v = a3_inputs()
    for causal in (False, True):  # M=1 sits at position N-1, so causal sees every key
        o = orc.attention(q, k, v, causal=causal, scale=1.0)[0, 0, 0, 0]
        assert abs(o - fx["expected"]) <= fx["tol"], (causal, o)
        assert abs(o - fx["missing_alpha_bug"]) > 0.5, o


def pin_a1_merge_example(orc):
    fx = _golden("a1_merge_example.json")
    (m1, l1), (m2, l2) = fx["a"], fx["b"]
    want_l = 1.0 + 2.0 * math.exp(-2.0)
    for order in ((0, 1), (1, 0)):
        ms = np.array([m1, m2])[list(order)]
        ls = np.array([l1, l2])[list(order)]
        acc = np.array([[3.0], [5.0]])[list(order)]
        m, l, a = orc.merge(ms, ls, acc)
        assert abs(m - fx["expected_m"]) <= fx["tol"], m
        assert abs(l - want_l) <= fx["tol"], l
        # the numerator follows the same weights: 3 e^{2-4} + 5 e^{4-4}
        want_a = (3.0 * math.exp(-2.0) + 5.0) if order == (0, 1) else (5.0 + 3.0 * math.exp(-2.0))
        assert abs(a[0] - want_a) <= 1e-12, a


def pin_merge_empty(orc):
    m, l, a = orc.merge([-np.inf, -np.inf], [0.0, 0.0], [[0.0, 0.0], [0.0, 0.0]])
    assert m == -np.inf and l == 0.0 and np.all(a == 0.0), (m, l, a)
    assert not np.isnan(l) and not np.any(np.isnan(a))
    # the empty summary is an identity on either side
    for order in ((0, 1), (1, 0)):
        ms = np.array([-np.inf, 1.5])[list(order)]
        ls = np.array([0.0, 2.5])[list(order)]
        acc = np.array([[0.0, 0.0], [4.0, -1.0]])[list(order)]
        m, l, a = orc.merge(ms, ls, acc)
        assert m == 1.5 and abs(l - 2.5) < 1e-15 and np.allclose(a, [4.0, -1.0], atol=0, rtol=1e-15)


def pin_merge_algebra(orc):
    rng = np.random.default_rng(7)
    for _ in range(20):
        ms = rng.normal(0, 3, 3)
        ls = rng.uniform(0.5, 4, 3)
        acc = rng.normal(0, 1, (3, 4))
        one = orc.merge(ms, ls, acc)
        # left: ((a (+) b) (+) c) built explicitly
        ab = orc.merge(ms[:2], ls[:2], acc[:2])
        left = orc.merge([ab[0], ms[2]], [ab[1], ls[2]], np.stack([ab[2], acc[2]]))
        bc = orc.merge(ms[1:], ls[1:], acc[1:])
        right = orc.merge([ms[0], bc[0]], [ls[0], bc[1]], np.stack([acc[0], bc[2]]))
        perm = [2, 0, 1]
        swapped = orc.merge(ms[perm], ls[perm], acc[perm])
        for other in (left, right, swapped):
            assert abs(other[0] - one[0]) == 0.0
            assert abs(other[1] - one[1]) <= 1e-12 * abs(one[1])
            assert np.allclose(other[2], one[2], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Summaries: splitting the keys and merging equals the unsplit summary, and
# the summary normalizes to the attention output
# --------------------------------------------------------------------------
def pin_split_merge(orc):
    B, Hq, Hkv, M, N, D = 1, 2, 1, 5, 23, 6
    q, k, v = _rand((B, Hq, M, D), 1), _rand((B, Hkv, N, D), 2), _rand((B, Hkv, N, D), 3)
    for causal, window in ((False, 0), (True, 0), (True, 7)):
        out = orc.attention(q, k, v, causal=causal, window=window)
        for row in range(B * Hq * M):
            m, l, a = orc.partial(q, k, v, row, 0, N, causal, window)
            assert np.allclose(a / l, out.reshape(-1, D)[row], rtol=1e-12, atol=1e-13)
            cuts = [0, 4, 5, 11, 17, 23]
            parts = [orc.partial(q, k, v, row, c0, c1, causal, window) for c0, c1 in zip(cuts, cuts[1:])]
            mm, ll, aa = orc.merge([p[0] for p in parts], [p[1] for p in parts], np.stack([p[2] for p in parts]))
            assert mm == m and abs(ll - l) <= 1e-12 * l and np.allclose(aa, a, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Independent library formula on tiny inputs (all masks, GQA, ragged)
# --------------------------------------------------------------------------
def library_attention(q, k, v, causal, window, scale):
    """softmax(scale Q K^T + mask) V with torch float64 routines; masks from
    triangular library routines; rows with no allowed key give 0."""
    q, k, v = (torch.from_numpy(np.asarray(x)) for x in (q, k, v))
    B, Hq, M, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    v = v.repeat_interleave(Hq // Hkv, dim=1)
    keep = torch.ones(M, N, dtype=torch.bool)
    if causal:
        keep &= torch.ones(M, N, dtype=torch.bool).tril(diagonal=N - M)
    if window > 0:
        keep &= torch.ones(M, N, dtype=torch.bool).triu(diagonal=N - M - window + 1)
    s = torch.matmul(q, k.transpose(-1, -2)) * scale
    s = s.masked_fill(~keep, float("-inf"))
    w = torch.softmax(s, dim=-1)
    w = torch.nan_to_num(w, nan=0.0)  # rows with every key masked
    return torch.matmul(w, v).numpy()


def pin_bruteforce(orc):
    rng = np.random.default_rng(11)
    for trial in range(40):
        Hkv = int(rng.integers(1, 4))
        Hq = Hkv * int(rng.integers(1, 4))
        B, M, N = int(rng.integers(1, 3)), int(rng.integers(1, 9)), int(rng.integers(1, 9))
        D = int(rng.choice([1, 3, 8, 16]))
        causal = bool(rng.integers(0, 2))
        window = int(rng.choice([0, 0, 1, 2, 5]))
        q = _rand((B, Hq, M, D), 100 + trial)
        k = _rand((B, Hkv, N, D), 200 + trial)
        v = _rand((B, Hkv, N, D), 300 + trial)
        scale = 1.0 / math.sqrt(D)
        got = orc.attention(q, k, v, causal=causal, window=window)
        want = library_attention(q, k, v, causal, window, scale)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (B, Hq, Hkv, M, N, D, causal, window)


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------
def pin_invariants(orc):
    B, Hq, Hkv, M, N, D = 1, 2, 2, 9, 13, 5
    q, k, v = _rand((B, Hq, M, D), 21), _rand((B, Hkv, N, D), 22), _rand((B, Hkv, N, D), 23)
    for causal, window in ((False, 0), (True, 0), (True, 4), (False, 6)):
        out = orc.attention(q, k, v, causal=causal, window=window).reshape(-1, D)
        for row in range(B * Hq * M):
            w = orc.weights(q, k, row, causal, window)
            assert abs(w.sum() - 1.0) < 1e-13 and np.all(w >= 0)
            bh, i = divmod(row, M)
            vh = v[0, bh % Hq]
            allowed = w > 0
            lo, hi = vh[allowed].min(axis=0), vh[allowed].max(axis=0)
            assert np.all(out[row] >= lo - 1e-12) and np.all(out[row] <= hi + 1e-12)
        # adding a per-row constant to every logit changes nothing: one extra
        # coordinate with q' = c_row / scale and k' = 1 adds c_row to the row
        scale = 1.0 / math.sqrt(D)
        c = np.arange(B * Hq * M, dtype=np.float64).reshape(B, Hq, M, 1) * 3.7 - 11.0
        q2 = np.concatenate([q, c / scale], axis=-1)
        k2 = np.concatenate([k, np.ones((B, Hkv, N, 1))], axis=-1)
        v2 = np.concatenate([v, np.zeros((B, Hkv, N, 1))], axis=-1)
        out2 = orc.attention(q2, k2, v2, causal=causal, window=window, scale=scale)[..., :D]
        assert np.allclose(out2.reshape(-1, D), out, rtol=1e-10, atol=1e-11)
    # noncausal output is equivariant to permuting keys and values together
    perm = np.random.default_rng(3).permutation(N)
    a = orc.attention(q, k, v)
    b = orc.attention(q, k[:, :, perm], v[:, :, perm])
    assert np.allclose(a, b, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
def pin_closed_forms(orc):
    D = 4
    q, k, v = _rand((1, 1, 6, D), 31), _rand((1, 1, 6, D), 32), _rand((1, 1, 6, D), 33)
    # N = 1: every row returns v_0
    o = orc.attention(q, k[:, :, :1], v[:, :, :1])
    assert np.allclose(o, np.broadcast_to(v[:, :, :1], o.shape), rtol=0, atol=1e-15)
    # q = 0: uniform weights over the allowed keys
    o = orc.attention(np.zeros_like(q), k, v, causal=True)
    for i in range(6):
        assert np.allclose(o[0, 0, i], v[0, 0, : i + 1].mean(axis=0), rtol=1e-13, atol=1e-14)
    # causal with M == N: row 0 sees only key 0
    o = orc.attention(q, k, v, causal=True)
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    # window = 1: each row sees only its own position
    o = orc.attention(q, k, v, causal=True, window=1)
    assert np.allclose(o[0, 0], v[0, 0], rtol=0, atol=1e-15)
    # identical key rows: uniform weights
    o = orc.attention(q, np.broadcast_to(k[:, :, :1], k.shape).copy(), v)
    assert np.allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (6, D)), rtol=1e-13, atol=1e-14)
    # one query (decode) sits at position N-1: causal equals noncausal
    a = orc.attention(q[:, :, :1], k, v, causal=True)
    b = orc.attention(q[:, :, :1], k, v, causal=False)
    assert np.allclose(a, b, rtol=0, atol=0)
    # M > N causal: rows i < M-N have no allowed key and give 0
    o = orc.attention(q, k[:, :, :2], v[:, :, :2], causal=True)
    assert np.all(o[0, 0, :4] == 0.0) and np.allclose(o[0, 0, 4], v[0, 0, 0], atol=1e-15)
    # N = 0 gives zeros, M = 0 gives an empty output
    o = orc.attention(q, k[:, :, :0], v[:, :, :0])
    assert o.shape == (1, 1, 6, D) and np.all(o == 0.0)
    o = orc.attention(q[:, :, :0], k, v)
    assert o.shape == (1, 1, 0, D)
    # D = 1 with logits [0, ln 3] under scale 1: weights 1/4 and 3/4
    o = orc.attention(np.ones((1, 1, 1, 1)), np.array([0.0, math.log(3.0)]).reshape(1, 1, 2, 1),
                      np.array([8.0, 4.0]).reshape(1, 1, 2, 1), scale=1.0)
    assert abs(o[0, 0, 0, 0] - 5.0) < 1e-14
    # the default scale is 1/sqrt(D): scaling q by 2 and passing scale/2 is the same
    a = orc.attention(q, k, v)
    b = orc.attention(2.0 * q, k, v, scale=0.5 / math.sqrt(D))
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)


def pin_gqa_map(orc):
    """Hq=4 over Hkv=2: heads 0,1 read KV head 0 and heads 2,3 read KV head 1."""
    D, N = 3, 5
    q = _rand((1, 4, 2, D), 41)
    k = np.broadcast_to(_rand((1, 2, 1, D), 42), (1, 2, N, D)).copy()  # uniform weights within a head
    v = np.zeros((1, 2, N, D))
    v[0, 0] = 1.0
    v[0, 1] = 2.0
    o = orc.attention(q, k, v)
    assert np.allclose(o[0, 0], 1.0) and np.allclose(o[0, 1], 1.0)
    assert np.allclose(o[0, 2], 2.0) and np.allclose(o[0, 3], 2.0)


# --------------------------------------------------------------------------
# Row sampling and the weight vector against the same torch float64 formula
# --------------------------------------------------------------------------
def library_weights(q, k, causal, window, scale):
    """softmax(scale Q K^T + mask) with torch float64 routines, [B, Hq, M, N]."""
    q, k = (torch.from_numpy(np.asarray(x)) for x in (q, k))
    B, Hq, M, D = q.shape
    Hkv, N = k.shape[1], k.shape[2]
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    keep = torch.ones(M, N, dtype=torch.bool)
    if causal:
        keep &= torch.ones(M, N, dtype=torch.bool).tril(diagonal=N - M)
    if window > 0:
        keep &= torch.ones(M, N, dtype=torch.bool).triu(diagonal=N - M - window + 1)
    s = (torch.matmul(q, k.transpose(-1, -2)) * scale).masked_fill(~keep, float("-inf"))
    return torch.nan_to_num(torch.softmax(s, dim=-1), nan=0.0).numpy()


def pin_rows_and_weights(orc):
    rng = np.random.default_rng(17)
    for trial in range(12):
        Hkv = int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 4))
        B, M, N, D = int(rng.integers(1, 3)), int(rng.integers(1, 7)), int(rng.integers(1, 9)), 4
        causal, window = bool(rng.integers(0, 2)), int(rng.choice([0, 2, 3]))
        q, k, v = _rand((B, Hq, M, D), 400 + trial), _rand((B, Hkv, N, D), 500 + trial), _rand((B, Hkv, N, D), 600 + trial)
        scale = 1.0 / math.sqrt(D)
        want_o = library_attention(q, k, v, causal, window, scale).reshape(-1, D)
        want_w = library_weights(q, k, causal, window, scale).reshape(-1, N)
        rows = rng.integers(0, B * Hq * M, 7)
        got = orc.attention_rows(q, k, v, rows, causal=causal, window=window)
        assert np.allclose(got, want_o[rows], rtol=1e-12, atol=1e-12)
        for r in rows:
            assert np.allclose(orc.weights(q, k, int(r), causal, window), want_w[r], rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Paged KV cache: pages cut from a contiguous cache, in any order, with a
# length per sequence, against the torch float64 formula on the truncated
# contiguous cache
# --------------------------------------------------------------------------
def to_pages(k, page_size, rng=None):
    """[B, Hkv, N, D] -> pool [B * N / page_size, Hkv, page_size, D] and block
    table [B, N / page_size]; with rng the pool's pages are shuffled."""
    B, Hkv, N, D = k.shape
    npg = N // page_size
    pool = k.reshape(B, Hkv, npg, page_size, D).transpose(0, 2, 1, 3, 4).reshape(B * npg, Hkv, page_size, D)
    table = np.arange(B * npg, dtype=np.int64).reshape(B, npg)
    if rng is not None:
        perm = rng.permutation(B * npg)  # page i moves to slot perm[i]
        moved = np.empty_like(pool)
        moved[perm] = pool
        pool, table = moved, perm[table]
    return np.ascontiguousarray(pool), table


def pin_paged(orc):
    rng = np.random.default_rng(29)
    B, Hq, Hkv, M, D, ps, npg = 3, 4, 2, 2, 5, 4, 6
    N = ps * npg
    q, k, v = _rand((B, Hq, M, D), 41), _rand((B, Hkv, N, D), 42), _rand((B, Hkv, N, D), 43)
    scale = 1.0 / math.sqrt(D)
    for shuffle in (False, True):
        r = np.random.default_rng(5) if shuffle else None
        kp, table = to_pages(k, ps, r)
        r = np.random.default_rng(5) if shuffle else None
        vp, table_v = to_pages(v, ps, r)
        assert np.array_equal(table, table_v)
        for causal, window in ((True, 0), (False, 0), (True, 7), (False, 5)):
            # every sequence full: the contiguous attention
            full = orc.attention_paged(q, kp, vp, table, [N] * B, N, causal, window)
            assert np.allclose(full, library_attention(q, k, v, causal, window, scale), rtol=1e-12, atol=1e-12)
            # ragged lengths, one empty sequence, one past the table (clamped)
            lens = [0, 13, N + 9]
            got = orc.attention_paged(q, kp, vp, table, lens, N + 9, causal, window)
            for b, L in enumerate(lens):
                L = min(L, N)
                want = library_attention(q[b:b + 1], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal, window, scale)
                assert np.allclose(got[b:b + 1], want, rtol=1e-12, atol=1e-12), (shuffle, causal, window, b)
            # max_seq_len below the lengths cuts every sequence there
            cut = orc.attention_paged(q, kp, vp, table, [N] * B, 9, causal, window)
            want = library_attention(q, k[:, :, :9], v[:, :, :9], causal, window, scale)
            assert np.allclose(cut, want, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Log-sum-exp of each row
# --------------------------------------------------------------------------
def pin_lse(orc):
    # A3 worked example: logits 0, 0, ln 2 -> ln(1 + 1 + 2) = ln 4
    fx, q, k, v = a3_inputs()
    _, lse = orc.attention_lse(q, k, v, scale=1.0)
    assert abs(lse[0, 0, 0] - math.log(4.0)) < 1e-12
    # library formula (torch.logsumexp over masked float64 logits), all masks, GQA
    rng = np.random.default_rng(23)
    for trial in range(20):
        Hkv = int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 3))
        B, M, N, D = 1, int(rng.integers(1, 7)), int(rng.integers(1, 9)), 3
        causal, window = bool(rng.integers(0, 2)), int(rng.choice([0, 1, 3]))
        q, k, v = _rand((B, Hq, M, D), 700 + trial), _rand((B, Hkv, N, D), 800 + trial), _rand((B, Hkv, N, D), 900 + trial)
        scale = 1.0 / math.sqrt(D)
        o, lse = orc.attention_lse(q, k, v, causal=causal, window=window)
        qt, kt = torch.from_numpy(q), torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
        keep = torch.ones(M, N, dtype=torch.bool)
        if causal:
            keep &= torch.ones(M, N, dtype=torch.bool).tril(diagonal=N - M)
        if window > 0:
            keep &= torch.ones(M, N, dtype=torch.bool).triu(diagonal=N - M - window + 1)
        s = (torch.matmul(qt, kt.transpose(-1, -2)) * scale).masked_fill(~keep, float("-inf"))
        want = torch.logsumexp(s, dim=-1).numpy()
        assert np.array_equal(np.isinf(lse), np.isinf(want))
        fin = np.isfinite(want)
        assert np.allclose(lse[fin], want[fin], rtol=1e-12, atol=1e-12)
        assert np.allclose(o, library_attention(q, k, v, causal, window, scale), rtol=1e-12, atol=1e-12)
    # q = 0: every visible logit is 0, so lse = ln(number of visible keys)
    q0 = np.zeros((1, 1, 6, 2))
    k0, v0 = _rand((1, 1, 6, 2), 1), _rand((1, 1, 6, 2), 2)
    _, lse = orc.attention_lse(q0, k0, v0, causal=True, window=4)
    assert np.allclose(lse[0, 0], np.log([1, 2, 3, 4, 4, 4]), rtol=0, atol=1e-14)
    # a row with no visible key: -inf
    _, lse = orc.attention_lse(_rand((1, 1, 3, 2), 3), _rand((1, 1, 1, 2), 4), _rand((1, 1, 1, 2), 5), causal=True)
    assert lse[0, 0, 0] == -np.inf and lse[0, 0, 1] == -np.inf and np.isfinite(lse[0, 0, 2])


# --------------------------------------------------------------------------
# Backward pass
# --------------------------------------------------------------------------
def pin_backward_i2_example(orc):
    """The answer key's I2 worked answer inside attention: one query row (q = 1,
    D = 1, scale 1) over two keys with logits ln 0.25 and ln 0.75 has weights
    y = (0.25, 0.75); values (2, -1) and do = 1 make dP = g = (2, -1), so the
    logit gradient is the softmax input gradient, and dK = dS * q = dx."""
    fx = _golden("i2_softmax_vjp_example.json")
    y, g = np.array(fx["y"]), np.array(fx["g"])
    q = np.ones((1, 1, 1, 1))
    k = np.log(y).reshape(1, 1, 2, 1)
    v = g.reshape(1, 1, 2, 1)
    do = np.ones((1, 1, 1, 1))
    dq, dk, dv = orc_backward(q, k, v, do, False, 0, 1.0)
    assert np.allclose(dk.reshape(-1), fx["dx"], rtol=0, atol=fx["tol"])
    assert np.allclose(dv.reshape(-1), y, rtol=0, atol=1e-15)            # dv = P^T do
    assert abs(dq.reshape(-1)[0] - float(np.dot(fx["dx"], np.log(y)))) < 1e-12  # dq = dS k
    # the same worked answer's second point: a gradient that is constant along
    # a row (here dP = do . v_j, constant when every value row is the same)
    # gives a zero logit gradient, since the weights sum to one; so dq = dk = 0,
    # with every mask and GQA, while dv = P^T do stays nonzero
    for causal, window, Hq, Hkv in ((False, 0, 2, 1), (True, 0, 2, 2), (True, 3, 4, 2)):
        q, k = _rand((1, Hq, 5, 3), 61), _rand((1, Hkv, 6, 3), 62)
        v = np.broadcast_to(_rand((1, Hkv, 1, 3), 63), (1, Hkv, 6, 3)).copy()
        do = _rand((1, Hq, 5, 3), 64)
        dq, dk, dv = orc_backward(q, k, v, do, causal, window, 1.0 / math.sqrt(3))
        assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13, (causal, window)
        assert np.abs(dv).max() > 0.1


def orc_backward(q, k, v, do, causal, window, scale):
    import oracle
    return oracle.attention_backward(q, k, v, do, causal=causal, window=window, scale=scale)


def pin_backward_finite_differences(orc):
    """Central differences of the forward oracle (L = sum do * o) against the
    backward oracle, for every input element of small cases with every mask."""
    rng = np.random.default_rng(31)
    h = 1e-6
    for causal, window, Hq, Hkv in ((False, 0, 2, 1), (True, 0, 2, 2), (True, 3, 4, 2), (False, 2, 1, 1)):
        B, M, N, D = 1, 4, 5, 3
        q, k, v = _rand((B, Hq, M, D), 51), _rand((B, Hkv, N, D), 52), _rand((B, Hkv, N, D), 53)
        do = rng.standard_normal((B, Hq, M, D))
        scale = 1.0 / math.sqrt(D)
        dq, dk, dv = orc_backward(q, k, v, do, causal, window, scale)

        def loss(q_, k_, v_):
            return float((orc.attention(q_, k_, v_, causal=causal, window=window) * do).sum())

        for x, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = [q, k, v]
                args_m = [q, k, v]
                args_p[which], args_m[which] = xp, xm
                fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
                assert abs(fd - grad[idx]) < 1e-6, (causal, window, which, idx, fd, grad[idx])


def pin_backward_autograd(orc):
    """torch.autograd in float64 (masked softmax built from library routines)."""
    rng = np.random.default_rng(37)
    for trial in range(10):
        Hkv = int(rng.integers(1, 3))
        Hq = Hkv * int(rng.integers(1, 3))
        B, M, N, D = int(rng.integers(1, 3)), int(rng.integers(1, 7)), int(rng.integers(1, 8)), 4
        causal, window = bool(rng.integers(0, 2)), int(rng.choice([0, 2, 3]))
        q, k, v = _rand((B, Hq, M, D), 60 + trial), _rand((B, Hkv, N, D), 70 + trial), _rand((B, Hkv, N, D), 80 + trial)
        do = rng.standard_normal((B, Hq, M, D))
        scale = 1.0 / math.sqrt(D)
        qt, kt, vt = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
        kk, vv = kt.repeat_interleave(Hq // Hkv, dim=1), vt.repeat_interleave(Hq // Hkv, dim=1)
        keep = torch.ones(M, N, dtype=torch.bool)
        if causal:
            keep &= torch.ones(M, N, dtype=torch.bool).tril(diagonal=N - M)
        if window > 0:
            keep &= torch.ones(M, N, dtype=torch.bool).triu(diagonal=N - M - window + 1)
        s = (torch.matmul(qt, kk.transpose(-1, -2)) * scale).masked_fill(~keep, float("-inf"))
        w = torch.nan_to_num(torch.softmax(s, dim=-1), nan=0.0)
        o = torch.matmul(w, vv)
        (o * torch.from_numpy(do)).sum().backward()
        dq, dk, dv = orc_backward(q, k, v, do, causal, window, scale)
        for got, want in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
            assert np.allclose(got, want.numpy(), rtol=1e-11, atol=1e-12), (trial, causal, window)


# --------------------------------------------------------------------------
# Row softmax (wide-row split softmax oracle)
# --------------------------------------------------------------------------
def pin_softmax_rows(orc):
    import oracle
    rng = np.random.default_rng(41)
    x = rng.standard_normal((6, 37)) * 5
    got = oracle.softmax_rows(x)
    want = torch.softmax(torch.from_numpy(x), dim=-1).numpy()  # library routine, float64
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)
    assert np.allclose(got.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(oracle.softmax_rows(x + rng.standard_normal((6, 1)) * 100), got, rtol=1e-12, atol=1e-15)
    assert np.allclose(oracle.softmax_rows(np.full((2, 8), 3.5)), 1.0 / 8, rtol=0, atol=1e-16)  # constant row
    one = np.zeros((1, 5)); one[0, 2] = 1000.0
    assert np.allclose(oracle.softmax_rows(one), [[0, 0, 1, 0, 0]], rtol=0, atol=1e-300)
    assert oracle.softmax_rows(np.zeros((0, 4))).shape == (0, 4)


# --------------------------------------------------------------------------
# E4M3 inputs: the code table and the dequantized attention
# --------------------------------------------------------------------------
def pin_e4m3_decode(orc):
    import oracle
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes)
    # closed forms of the encoding (bias 7, 3 mantissa bits, subnormals below 2^-6)
    want = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0, 0x01: 2.0 ** -9,
            0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x3F: 1.875, 0x40: 2.0, 0x30: 0.5, 0x3C: 1.5, 0x77: 240.0}
    for c, val in want.items():
        assert got[c] == val, (hex(c), got[c], val)
    assert np.signbit(got[0x80]) and got[0x80] == 0.0
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2
    # magnitudes strictly increase with the code; the sign bit mirrors them
    assert np.all(np.diff(got[:0x7F]) > 0)
    assert np.array_equal(got[0x80:0xFF], -got[:0x7F])
    # the library's own E4M3 conversion agrees on every code
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(lib), np.isnan(got))
    assert np.array_equal(lib[~np.isnan(lib)], got[~np.isnan(got)])
    # and rounding each finite value back to E4M3 returns its code
    fin = ~np.isnan(got)
    back = torch.from_numpy(got[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(back, codes[fin])


def pin_attention_fp8(orc):
    import oracle
    g = torch.Generator().manual_seed(44)
    f8 = torch.float8_e4m3fn
    B, Hq, Hkv, M, N, D = 1, 4, 2, 9, 13, 16
    q = (torch.randn(B, Hq, M, D, generator=g) * 2).to(f8)
    k = (torch.randn(B, Hkv, N, D, generator=g) * 3).to(f8)
    v = (torch.randn(B, Hkv, N, D, generator=g) * 4).to(f8)
    qd, kd, vd, scale = 0.5, 0.125, 0.25, 0.3
    for causal, window in ((False, 0), (True, 0), (True, 5)):
        got = oracle.attention_fp8(q, k, v, qd, kd, vd, causal=causal, window=window, scale=scale)
        # a library formula on the library's own FP8 -> FP64 conversion
        want = library_attention(q.to(torch.float64).numpy() * qd, k.to(torch.float64).numpy() * kd,
                                 v.to(torch.float64).numpy() * vd, causal, window, scale)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-13), (causal, window)
        # homogeneity: the Q and K factors only rescale the logits, the V factor the output
        plain = oracle.attention_fp8(q, k, v, 1.0, 1.0, 1.0, causal=causal, window=window, scale=scale * qd * kd)
        assert np.allclose(got, vd * plain, rtol=1e-12, atol=1e-14)
    # all-zero queries weight every visible key equally: the mean of V's rows
    z = torch.zeros(B, Hq, M, D).to(f8)
    got = oracle.attention_fp8(z, k, v, 1.0, 1.0, vd, causal=False)
    vv = vd * v.to(torch.float64).numpy()
    want = np.repeat(vv.mean(axis=2, keepdims=True), Hq // Hkv, axis=1).repeat(M, axis=2)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-14)


ALL_PINS = [
    pin_a3_worked_example,
    pin_a1_merge_example,
    pin_merge_empty,
    pin_merge_algebra,
    pin_split_merge,
    pin_bruteforce,
    pin_invariants,
    pin_closed_forms,
    pin_gqa_map,
    pin_rows_and_weights,
    pin_paged,
    pin_lse,
    pin_backward_i2_example,
    pin_backward_finite_differences,
    pin_backward_autograd,
    pin_softmax_rows,
    pin_e4m3_decode,
    pin_attention_fp8,
]
