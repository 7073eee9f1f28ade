"""The oracle reproduces the digests its committed golden file recorded (cross-platform check)."""

import json
import os

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _load():
    import sys
    sys.path.insert(0, os.path.join(HERE, "golden"))
    import make_oracle_golden
    with open(os.path.join(HERE, "golden", "oracle_golden.json")) as f:
        return make_oracle_golden, json.load(f)["cases"]


MOD, CASES = _load()


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_oracle_matches_golden(case):
    got = MOD.run_case(oracle.default(), {k: v for k, v in case.items() if k != "digests"})
    assert got == case["digests"]
