"""The oracle against its pins (CPU only), and planted mistakes against the pins."""
import math
import os
import tempfile

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def _stream(logits, values, tile, rescale_numerator=True):
    """Running (m, l, a) over key tiles, as the A3 row of the answer key
    describes; with rescale_numerator=False it reproduces the unrescaled-accumulator mistake."""
    m, l, a = -math.inf, 0.0, 0.0
    for t0 in range(0, len(logits), tile):
        s = logits[t0:t0 + tile]
        m_new = max(m, max(s))
        alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
        p = [math.exp(x - m_new) for x in s]
        l = l * alpha + sum(p)
        a = (a * alpha if rescale_numerator else a) + sum(pi * vi for pi, vi in zip(p, values[t0:t0 + tile]))
        m = m_new
    return a / l


def test_a3_fixture_discriminates_missing_alpha():
    fx, q, k, v = P.a3_inputs()
    logits = list(k.reshape(-1))
    values = list(v.reshape(-1))
    assert abs(_stream(logits, values, tile=2) - fx["expected"]) < 1e-12
    assert abs(_stream(logits, values, tile=2, rescale_numerator=False) - fx["missing_alpha_bug"]) < 1e-12


# Each planted mistake (compiled with ORACLE_MUTANT=n) must fail at least one pin.
MUTANTS = {
    1: "causal mask drops the diagonal",
    2: "window keeps W+1 keys",
    3: "GQA strided head map",
    4: "top-left causal alignment",
    5: "output not normalized",
    6: "scale dropped",
    7: "K read transposed",
    8: "last head dimension dropped",
    9: "merge sums denominators without rescaling",
    10: "merge without the empty guard",
}


@pytest.fixture(scope="module")
def mutant_dir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda n: f"m{n}")
def test_planted_mistake_is_caught(mutant, mutant_dir):
    orc = oracle.Oracle(mutant, out_dir=mutant_dir)
    assert orc.lib.oracle_mutant_id() == mutant
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


# Planted mistakes in the Python functions (oracle.PY_MUTANT = n), each of
# which must also fail at least one pin.
PY_MUTANTS = {
    11: "backward: softmax VJP without its row-sum term",
    12: "backward: GQA dk/dv keep one query head's share",
    13: "backward: dq without the scale",
    14: "backward: top-left causal alignment",
    15: "row softmax normalized over columns",
    16: "E4M3 exponent bias 8",
    17: "E4M3 subnormals with an implicit one",
    18: "E4M3 attention drops the V factor",
    19: "paged: lengths not cut at max_seq_len",
    20: "paged: pages taken in pool order, not through the block table",
}


@pytest.mark.parametrize("mutant", sorted(PY_MUTANTS), ids=lambda n: f"m{n}")
def test_planted_python_mistake_is_caught(mutant, oracle_lib, monkeypatch):
    monkeypatch.setattr(oracle, "PY_MUTANT", mutant)
    failed = []
    for pin in P.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(oracle_lib)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({PY_MUTANTS[mutant]}) passed every pin"
