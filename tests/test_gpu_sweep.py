"""Seeded random sweep of decode and gather shapes on the GPU against the CPU oracle.

Shapes are drawn once from a fixed numpy seed (so every run checks the same cases): both bank
dtypes and index dtypes, shared and per-write gates, widths up to 256, head dims from 1 to 512
(16-byte and ragged rows, so the staged, streamed and plain-load kernel paths all appear), and for
the gather one or two operands with a stash, no stash or a compact snapshot. Tolerances are the
ones in parity.py; the gather is compared bit for bit.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from decode_state_gb300 import sdm, workloads
from parity import DECODE_KEYS, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
HDS = [1, 2, 3, 8, 16, 24, 48, 64, 96, 100, 128, 136, 200, 256, 264, 384, 512]


def _width(rng) -> int:
    return int(rng.choice([rng.integers(1, 9), rng.integers(9, 65), rng.integers(65, 257)]))


def _decode_cases(n=40, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        W, R = _width(rng), _width(rng)
        out.append(dict(dtype=str(rng.choice(["bf16", "f32"])), idx=str(rng.choice(["i32", "i64"])),
                        hd=int(rng.choice(HDS)), W=W, R=R, G=W if rng.random() < 0.4 else 1,
                        S=int(rng.integers(1, 40)), T=int(rng.integers(1, 5)), P=int(W + rng.integers(0, 300)),
                        seed=int(rng.integers(0, 1 << 30))))
    return out


def _gather_cases(n=24, seed=2025):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        chunk = int(rng.choice([1, 3, 8, 16, 64]))
        mode = str(rng.choice(["stash", "nostash", "kpos"]))
        n_ops = int(rng.integers(1, 3))
        out.append(dict(dtype=str(rng.choice(["bf16", "f32"])), wdtype=str(rng.choice(["bf16", "f32"])),
                        idx=str(rng.choice(["i32", "i64"])), hd=int(rng.choice(HDS)),
                        n_slots=int(rng.integers(1, 3000)), tokens=chunk * int(rng.integers(1, 12)), chunk=chunk,
                        widths=tuple(_width(rng) for _ in range(n_ops)), mode=mode,
                        per_chunk=bool(rng.random() < 0.6), seed=int(rng.integers(0, 1 << 30))))
    return out


DECODE = _decode_cases()
GATHER = _gather_cases()


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0


@pytest.mark.parametrize("c", DECODE, ids=[f"d{i}-{c['dtype']}-{c['idx']}-hd{c['hd']}-W{c['W']}R{c['R']}-"
                                         f"G{c['G']}-S{c['S']}-T{c['T']}" for i, c in enumerate(DECODE)])
def test_decode_sweep(c):
    wl = workloads.DecodeWorkload("sweep", c["dtype"], c["S"], c["hd"], c["P"], c["W"], c["R"], c["G"], c["T"],
                                  c["idx"], 0.35, bank_std=0.5, seed=c["seed"])
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    out_ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), out_ref, c["dtype"], "readings")
    assert_close(to_np(x["bank"]), bank_ref, c["dtype"], "bank")


def _kpos_first(idx: np.ndarray, chunk: int) -> np.ndarray:
    tokens, W0 = idx.shape
    kpos = np.full((tokens, W0), -1, np.int32)
    for ch in range(tokens // chunk):
        ent = idx[ch * chunk:(ch + 1) * chunk].ravel()
        order = np.sort(ent)
        _, first = np.unique(ent, return_index=True)
        for e in first:
            kpos[ch * chunk + e // W0, e % W0] = int(np.searchsorted(order, ent[e]))
    return kpos


@pytest.mark.parametrize("c", GATHER, ids=[f"g{i}-{c['dtype']}-w{c['wdtype']}-{c['idx']}-hd{c['hd']}-"
                                         f"{'x'.join(map(str, c['widths']))}-{c['mode']}" for i, c in enumerate(GATHER)])
def test_gather_sweep(c):
    wl = workloads.GatherWorkload("sweep", c["dtype"], c["n_slots"], c["hd"], c["tokens"], c["chunk"], c["widths"],
                                  c["idx"], c["wdtype"], 0.25, stash=c["mode"] == "stash",
                                  per_chunk_valid=c["per_chunk"], seed=c["seed"])
    g = workloads.make_gather_inputs(wl, device=DEV)
    cv = g["chunk_valid"]
    a = [to_np(g["ops"][0][0]), to_np(g["ops"][0][1])]
    if len(g["ops"]) == 2:
        a += [to_np(g["ops"][1][0]), to_np(g["ops"][1][1])]
    cv_h = None if cv is None else to_np(cv)
    r0, r1, rs = oracle.gather(to_np(g["bank"]), *a, chunk=c["chunk"], chunk_valid=cv_h, stash=c["mode"] == "stash")
    if c["mode"] == "kpos":
        kpos = _kpos_first(a[0], c["chunk"])
        compact = torch.full((c["tokens"] // c["chunk"], c["chunk"] * c["widths"][0], c["hd"]), float("nan"),
                             dtype=g["bank"].dtype, device=DEV)
        ref_compact = oracle.gather_kpos(to_np(g["bank"]), a[0], kpos, to_np(compact), chunk=c["chunk"],
                                         chunk_valid=cv_h)
        outs, _ = sdm.gather(g["bank"], g["ops"], chunk=c["chunk"], chunk_valid=cv,
                             kpos=torch.from_numpy(kpos).to(DEV), compact=compact)
        torch.cuda.synchronize()
        assert bits_equal(to_np(compact), ref_compact)
    else:
        outs, stash = sdm.gather(g["bank"], g["ops"], chunk=c["chunk"], chunk_valid=cv,
                                 with_stash=c["mode"] == "stash")
        torch.cuda.synchronize()
        if c["mode"] == "stash":
            assert bits_equal(to_np(stash), rs)
    assert bits_equal(to_np(outs[0]), r0)
    if len(c["widths"]) == 2:
        assert bits_equal(to_np(outs[1]), r1)
