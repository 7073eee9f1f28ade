"""Writes oracle_golden.json: digests of the oracle's outputs on small seeded inputs.

Run from the repository root: ``python tests/golden/make_oracle_golden.py``. It calls only the
oracle package and numpy. The inputs come from numpy's PCG64 generator (the same bits on every
platform), so the test that reads the file checks that the oracle built on another machine (the
Arm GPU host, for one) reproduces the same bits as the one that wrote it.
"""

from __future__ import annotations

import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

CASES = [
    dict(name="decode_f32_i32", kind="decode", dtype="f32", idx="i32", S=3, P=50, hd=24, W=8, R=8, G=1, T=5, seed=101),
    dict(name="decode_bf16_i64_gw", kind="decode", dtype="bf16", idx="i64", S=4, P=64, hd=40, W=16, R=12, G=16, T=6,
         seed=102),
    dict(name="gather_bf16_2op", kind="gather", dtype="bf16", wdtype="bf16", idx="i64", n_slots=300, hd=48, tokens=24,
         chunk=8, widths=[16, 9], seed=103),
    dict(name="gather_f32_1op", kind="gather", dtype="f32", wdtype="f32", idx="i32", n_slots=100, hd=20, tokens=12,
         chunk=4, widths=[7], seed=104),
]


def _bits_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even, in numpy (input drawing only)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def _u(rng, lo, hi, shape) -> np.ndarray:
    """float32 uniform on [lo, hi): PCG64 integer bits only, no libm call, same on every platform."""
    return (lo + (hi - lo) * rng.random(shape)).astype(np.float32)


def make_inputs(case: dict) -> dict:
    rng = np.random.default_rng(case["seed"])
    idt = np.int32 if case["idx"] == "i32" else np.int64
    if case["kind"] == "decode":
        S, P, hd, W, R, G, T = (case[k] for k in ("S", "P", "hd", "W", "R", "G", "T"))
        bank = _u(rng, -1.0, 1.0, (S * P, hd))
        bank = _bits_bf16(bank) if case["dtype"] == "bf16" else bank
        k_idx = np.stack([np.stack([rng.permutation(P)[:W] + s * P for s in range(S)]) for _ in range(T)]).astype(idt)
        k_val = _u(rng, -0.5, 0.5, (T, S, W))
        v = _u(rng, -2.0, 2.0, (T, S, hd))
        beta = _u(rng, 0.05, 0.95, (T, S))
        g = _u(rng, -2.0, 0.0, (T, S, G))
        q_idx = (rng.integers(0, P, (T, S, R)) + (np.arange(S) * P)[None, :, None]).astype(idt)
        q_val = _u(rng, -0.5, 0.5, (T, S, R))
        return dict(bank=bank, k_idx=k_idx, k_val=k_val, v=v, beta=beta, g=g, q_idx=q_idx, q_val=q_val)
    n, hd, tokens, chunk = case["n_slots"], case["hd"], case["tokens"], case["chunk"]
    bank = _u(rng, -2.0, 2.0, (n, hd))
    bank = _bits_bf16(bank) if case["dtype"] == "bf16" else bank
    ops = []
    for width in case["widths"]:
        idx = rng.integers(0, n, (tokens, width)).astype(idt)
        w = _u(rng, -0.5, 0.5, (tokens, width))
        ops.append((idx, _bits_bf16(w) if case["wdtype"] == "bf16" else w))
    chunk_valid = rng.integers(0, chunk + 1, tokens // chunk).astype(np.int32)
    return dict(bank=bank, ops=ops, chunk_valid=chunk_valid)


def run_case(orc, case: dict) -> dict:
    x = make_inputs(case)
    if case["kind"] == "decode":
        bank = x["bank"].copy()
        out = orc.decode_seq(bank, x["k_idx"], x["k_val"], x["v"], x["beta"], x["g"], x["q_idx"], x["q_val"])
        arrays = {"bank": bank, "out": out}
    else:
        ops = x["ops"]
        a = ops[0] + (ops[1] if len(ops) > 1 else (None, None))
        o0, o1, st = orc.gather(x["bank"], *a, chunk=case["chunk"], chunk_valid=x["chunk_valid"])
        arrays = {"out0": o0, "stash": st}
        if o1 is not None:
            arrays["out1"] = o1
    return {k: hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest() for k, v in arrays.items()}


def main():
    import oracle

    orc = oracle.default()
    result = {"note": "sha256 of the oracle's outputs; written by tests/golden/make_oracle_golden.py",
              "cases": [dict(case, digests=run_case(orc, case)) for case in CASES]}
    with open(os.path.join(HERE, "oracle_golden.json"), "w") as f:
        json.dump(result, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
