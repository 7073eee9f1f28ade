"""GPU parity of the staged decode's write-back by 16-byte pieces.

The launcher writes back by pieces (each thread one 16-byte piece of every few rows, with the delta
pairs published by the column owners) on every grid where the pieces tile the block's threads. These
cases cover grids of several blocks per SM and of a few blocks in all, with rows of 128 to 512 bytes
in both bank dtypes, both index dtypes, shared and per-write gates, and write widths that the row
groups do not divide evenly.
"""

from __future__ import annotations

import pytest
import torch

import oracle
from decode_state_gb300 import sdm, workloads
from parity import DECODE_KEYS, assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# (bank dtype, idx dtype, head_dim, W, R, G, streams, slots per stream, T)
CASES = [
    ("bf16", "i64", 128, 24, 24, 24, 640, 64, 3),
    ("f32", "i32", 64, 20, 33, 1, 700, 48, 2),
    ("bf16", "i32", 256, 8, 8, 1, 620, 16, 2),
    ("f32", "i64", 32, 5, 5, 5, 700, 8, 4),
    ("bf16", "i64", 64, 16, 16, 16, 700, 32, 2),   # 128-byte rows: the one-column-per-thread instance
    ("bf16", "i32", 128, 24, 20, 1, 9, 64, 5),     # a few blocks in all
    ("f32", "i64", 64, 13, 7, 13, 5, 32, 4),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}-hd{c[2]}-W{c[3]}R{c[4]}G{c[5]}-S{c[6]}" for c in CASES])
def test_piece_write_matches_oracle(case):
    dt, idt, hd, W, R, G, S, P, T = case
    wl = workloads.DecodeWorkload("piece", dt, S, hd, P, W, R, G, T, idt, 0.35, bank_std=0.5, seed=hd + W)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, dt, "readings")
    assert_close(to_np(x["bank"]), bank_ref, dt, "bank")
    assert sdm.device_status() == 0
