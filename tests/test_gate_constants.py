"""CPU pin of the constants behind the decode's gate exponential (`gate` in decode.cu).

The kernel evaluates e^g as 2^m * 2^(j/64) * e^r with g = (64m + j) ln2/64 + r. Its correctness
argument rests on these facts about the constants in the source, checked here in high precision:
  - each table pair hi + lo is within 2^-48 (relative) of 2^(j/64), hi the float32 nearest to it;
  - ln2/64 = A + B + C to 2^-66, with A of at most 11 significant bits (n*A exact for |n| < 2^13)
    and |ln2/64 - A| <= 2^-18 (so g - n*A is exact for every g in [-87, 88]);
  - kInv is the float32 nearest to 64/ln2.
"""

from __future__ import annotations

import os
import re
from fractions import Fraction

import numpy as np
import pytest

mp = pytest.importorskip("mpmath")

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "decode_state_gb300", "csrc", "decode.cu")
HEX = r"(-?0x[0-9a-fA-F]+(?:\.[0-9a-fA-F]*)?p[-+]?\d+)f"


def _source() -> str:
    with open(SRC) as f:
        return f.read()


def _hex(s: str) -> float:
    return float.fromhex(s)


def _table():
    body = re.search(r"kExp2Tab\[64\] = \{(.*?)\n\};", _source(), re.S).group(1)
    pairs = re.findall(r"\{([^,{}]+)f, ([^,{}]+)f\}", body)
    return [(float(a) if a == "0.0" else _hex(a), float(b) if b == "0.0" else _hex(b)) for a, b in pairs]


def _const(name: str) -> float:
    return _hex(re.search(name + r" = " + HEX, _source()).group(1))


def _is_f32(x: float) -> bool:
    return float(np.float32(x)) == x


def _nearest_f32(x) -> float:
    f = np.float32(float(x))
    cands = [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    return float(min(cands, key=lambda c: abs(mp.mpf(float(c)) - x)))


def test_table_pairs_are_the_powers():
    mp.mp.prec = 200
    tab = _table()
    assert len(tab) == 64
    for j, (hi, lo) in enumerate(tab):
        assert _is_f32(hi) and _is_f32(lo)
        exact = mp.mpf(2) ** (mp.mpf(j) / 64)
        assert hi == _nearest_f32(exact), j
        assert abs((mp.mpf(hi) + mp.mpf(lo)) - exact) <= exact * mp.mpf(2) ** -48, j


def test_reduction_constants():
    mp.mp.prec = 200
    A, B, C, inv = _const("kA"), _const("kB"), _const("kC"), _const("kInv")
    assert all(_is_f32(x) for x in (A, B, C, inv))
    step = mp.log(2) / 64
    assert abs(mp.mpf(A) + mp.mpf(B) + mp.mpf(C) - step) <= mp.mpf(2) ** -66
    assert abs(mp.mpf(A) - step) <= mp.mpf(2) ** -18
    # significant bits of A: the odd part of its numerator (A is a dyadic rational)
    mant = abs(Fraction(A).numerator)
    while mant % 2 == 0:
        mant //= 2
    assert mant.bit_length() <= 11
    assert inv == _nearest_f32(64 / mp.log(2))


def test_largest_reduction_index_fits():
    """|n| = |rint(g * kInv)| stays below 2^13 over the fast range [-87, 88], so n*A is exact."""
    inv = np.float32(_const("kInv"))
    for g in (np.float32(-87.0), np.float32(88.0)):
        n = int(np.rint(np.float32(g * inv)))
        assert abs(n) < 1 << 13
