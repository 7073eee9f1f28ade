"""GPU checks of the decode's degenerate cases, on each kernel path, against closed forms.

The oracle pins these properties on the CPU; here the CUDA path must satisfy them directly:
  - beta = 0 and g = 0: the write changes nothing (d = 1, delta = 0), so the bank stays bit-identical;
  - beta = 0 (decay only): every written row becomes round(row * d) with d the float32 nearest to e^g;
  - W = 1, k_val = 1, g = 0, beta = 1 on a bf16 bank: the written row becomes round(v) exactly
    (row + (v - row) is exact in float32 for bf16 operands);
  - G = W with all of a token's gates equal gives the bits of G = 1.
Paths: staged rows (bf16, 256-byte rows), streamed rows (float32, 1 KiB rows, W = R = 256) and
plain loads (bf16 rows of 13 elements).
"""

from __future__ import annotations

import pytest
import torch

from decode_state_gb300 import sdm, workloads
from parity import DECODE_KEYS, bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# (name, bank dtype, head_dim, W, R, streams, slots per stream, T)
PATHS = [
    ("staged", "bf16", 128, 16, 12, 24, 96, 3),
    ("streamed", "f32", 256, 256, 256, 6, 512, 2),
    ("plain", "bf16", 13, 6, 5, 10, 40, 3),
]
PIDS = [p[0] for p in PATHS]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0


def _inputs(dt, hd, W, R, S, P, T, G=1, seed=0):
    wl = workloads.DecodeWorkload("degenerate", dt, S, hd, P, W, R, G, T, "i32", 0.35, bank_std=0.5, seed=seed)
    x = workloads.make_decode_inputs(wl, device=DEV)
    x["bank"][x["bank"] == 0] = 0.25  # a zero-free bank: a written +0 and -0 would differ bit-wise
    return x


def _run(x):
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("path", PATHS, ids=PIDS)
def test_no_write_leaves_the_bank_bit_identical(path):
    _, dt, hd, W, R, S, P, T = path
    x = _inputs(dt, hd, W, R, S, P, T, seed=1)
    x["beta"].zero_()
    x["g"].zero_()
    before = to_np(x["bank"])
    _run(x)
    assert bits_equal(to_np(x["bank"]), before)


@pytest.mark.parametrize("path", PATHS, ids=PIDS)
def test_decay_only_writes_round_row_times_d(path):
    _, dt, hd, W, R, S, P, T = path
    x = _inputs(dt, hd, W, R, S, P, 1, seed=2)
    x["beta"].zero_()
    before = x["bank"].clone()
    _run(x)
    d = torch.exp(x["g"][0, :, 0].double()).float()  # [S]: the float32 nearest to e^g
    rows = x["k_idx"][0].long()  # [S, W]
    expect = (before[rows].float() * d.view(S, 1, 1)).to(before.dtype)
    assert bits_equal(to_np(x["bank"][rows]), to_np(expect))
    untouched = torch.ones(x["bank"].shape[0], dtype=torch.bool, device=DEV)
    untouched[rows.flatten()] = False
    assert bits_equal(to_np(x["bank"][untouched]), to_np(before[untouched]))


@pytest.mark.parametrize("path", [p for p in PATHS if p[1] == "bf16"], ids=[p[0] for p in PATHS if p[1] == "bf16"])
def test_single_unit_write_stores_v(path):
    _, dt, hd, _, R, S, P, T = path
    x = _inputs(dt, hd, 1, R, S, P, 1, seed=3)
    x["k_val"].fill_(1.0)
    x["g"].zero_()
    x["beta"].fill_(1.0)
    x["v"] = (x["v"] * 0.5).to(torch.bfloat16).float()  # values already representable in bf16
    _run(x)
    rows = x["k_idx"][0, :, 0].long()
    assert bits_equal(to_np(x["bank"][rows]), to_np(x["v"][0].to(torch.bfloat16)))


@pytest.mark.parametrize("path", PATHS, ids=PIDS)
def test_equal_per_write_gates_match_one_gate(path):
    _, dt, hd, W, R, S, P, T = path
    x1 = _inputs(dt, hd, W, R, S, P, T, G=1, seed=4)
    xw = {k: v.clone() for k, v in x1.items()}
    xw["g"] = x1["g"].expand(T, S, W).contiguous()
    out1, outw = _run(x1), _run(xw)
    assert bits_equal(to_np(out1), to_np(outw))
    assert bits_equal(to_np(x1["bank"]), to_np(xw["bank"]))
