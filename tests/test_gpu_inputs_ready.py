"""GPU parity of single-token steps launched with SDM_INPUTS_READY (sdm_decode_step_ex).

With the flag a step loads its metadata and warms L2 with its rows before it waits for the step
ahead of it, which may still be writing those rows. The steps here draw their slots from a few
more slots than they write per token, so nearly every row a step reads or writes was written by
the step just before. Launched back to back (a DecodeStepPlan, each launch chained to the previous
one by programmatic dependent launch) and replayed from a graph, they must give the bits of one
sdm_decode_seq launch over the same tokens, and match the oracle. Every kernel path is covered:
staged (paired and one-column, with and without the write-back by pieces), streamed (paired and
one-column) and plain loads (which ignore the flag).
"""

from __future__ import annotations

import pytest
import torch

import oracle
from decode_state_gb300 import sdm, workloads
from parity import DECODE_KEYS, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None

# (name, dtype, idx, streams, slots/stream, head_dim, W, R, G, T)
CASES = [
    ("staged-one-column", "bf16", "i64", 16, 40, 128, 32, 32, "W", 24),
    ("staged-pairs", "f32", "i32", 24, 30, 96, 24, 20, 1, 16),
    ("staged-pieces", "bf16", "i32", 700, 72, 128, 64, 64, 1, 6),
    ("streamed-pairs", "bf16", "i64", 3, 260, 512, 200, 200, "W", 4),
    ("streamed-one-column", "f32", "i32", 8, 280, 128, 256, 200, "W", 4),
    ("plain", "bf16", "i32", 12, 12, 13, 8, 6, 1, 12),
]
IDS = [c[0] for c in CASES]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0


def _inputs(case, seed):
    _, dt, idx, S, P, hd, W, R, G, T = case
    wl = workloads.DecodeWorkload("inputs_ready", dt, S, hd, P, W, R, W if G == "W" else G, T, idx, 0.35,
                                  bank_std=0.5, seed=seed)
    return wl, workloads.make_decode_inputs(wl, device=DEV)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_chained_steps_equal_one_seq_launch(case):
    wl, x = _inputs(case, 41)
    bank_seq, bank_plan = x["bank"].clone(), x["bank"].clone()
    ref_bank = to_np(x["bank"])
    out_seq = sdm.decode_seq(bank_seq, *(x[k] for k in DECODE_KEYS))
    plan = sdm.DecodeStepPlan(bank_plan, {k: x[k] for k in DECODE_KEYS}, inputs_ready=True)
    for t in range(wl.T):
        plan.launch(t)
    torch.cuda.synchronize()
    assert bits_equal(to_np(plan.out), to_np(out_seq))
    assert bits_equal(to_np(bank_plan), to_np(bank_seq))
    ref_out = oracle.decode_seq(ref_bank, *(to_np(x[k]) for k in DECODE_KEYS))
    assert_close(to_np(plan.out), ref_out, wl.bank_dtype, "readings")
    assert_close(to_np(bank_plan), ref_bank, wl.bank_dtype, "bank")


@pytest.mark.parametrize("case", CASES[:2], ids=IDS[:2])
def test_graph_of_chained_steps_equals_one_seq_launch(case):
    from decode_state_gb300.graphs import DecodeStepGraph

    wl, x = _inputs(case, 42)
    bank_seq, bank_g = x["bank"].clone(), x["bank"].clone()
    out_seq = sdm.decode_seq(bank_seq, *(x[k] for k in DECODE_KEYS))
    gr = DecodeStepGraph(bank_g, x)
    for k in DECODE_KEYS:
        gr.inputs[k].copy_(x[k])
    out_g = gr.replay()
    torch.cuda.synchronize()
    assert bits_equal(to_np(out_g), to_np(out_seq))
    assert bits_equal(to_np(bank_g), to_np(bank_seq))


def test_flagged_step_after_a_kernel_that_writes_the_bank():
    """The kernel just ahead rewrites the rows this step reads (a torch multiply on the same stream):
    the flag only promises the inputs, so the step must still see the new bank."""
    wl, x = _inputs(CASES[0], 43)
    t0 = {k: x[k][0] for k in DECODE_KEYS}
    bank_a, bank_b = x["bank"].clone(), x["bank"].clone()
    bank_a.mul_(0.5)
    out_a = sdm.decode_step(bank_a, *(t0[k] for k in DECODE_KEYS), inputs_ready=True)
    bank_b.mul_(0.5)
    out_b = sdm.decode_step(bank_b, *(t0[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert bits_equal(to_np(out_a), to_np(out_b))
    assert bits_equal(to_np(bank_a), to_np(bank_b))
