"""GPU parity of the gather launch plan (sdm_gather_plan_init / sdm_gather_plan_launch).

A plan checks a no-stash gather once and is then launched per slab: launch (row0, valid) gathers
index rows [row0, row0 + tokens) with `valid` live tokens per chunk. Every launch must equal the
oracle's gather of that slab with a scalar `valid` (bit for bit, as sdm_gather is) and the
direct sdm_gather call on the same slab.
"""

from __future__ import annotations

import pytest
import torch

import oracle
from decode_state_gb300 import sdm, workloads
from parity import bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
EROW, ECHUNK = -13, -8


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0


def _inputs(bank, wdt, idx, n_slots, hd, rows, widths, seed):
    wl = workloads.GatherWorkload(f"plan_{bank}_{hd}", bank, n_slots, hd, rows, 1, tuple(widths), idx, wdt, 0.125,
                                  stash=False, per_chunk_valid=False, seed=seed)
    return workloads.make_gather_inputs(wl, device=DEV)


def _slab_oracle(g, row0, tokens, chunk, valid):
    a = []
    for idx, w in g["ops"]:
        a += [to_np(idx[row0:row0 + tokens]), to_np(w[row0:row0 + tokens])]
    return oracle.gather(to_np(g["bank"]), *a, chunk=chunk, valid=valid, chunk_valid=None, stash=False)


# (bank dtype, weight dtype, idx dtype, n_slots, head_dim, index rows, tokens per launch, chunk, widths)
CASES = [
    ("bf16", "bf16", "i64", 5000, 128, 320, 64, 16, (64, 64)),   # the gather workload's row shape
    ("f32", "f32", "i32", 3000, 200, 90, 30, 10, (30,)),         # one operand (the backward shape)
    ("bf16", "f32", "i32", 700, 13, 48, 12, 4, (5, 7)),          # 26-byte rows: plain-load path
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-hd{c[4]}-{'x'.join(map(str, c[8]))}" for c in CASES])
def test_plan_launches_match_oracle(case):
    bank_dt, wdt, idt, n_slots, hd, rows, tokens, chunk, widths = case
    g = _inputs(bank_dt, wdt, idt, n_slots, hd, rows, widths, seed=11)
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=tokens, chunk=chunk)
    assert plan.row0_max == rows - tokens
    for row0, valid in ((0, chunk), (5, 0), (rows // 3, chunk // 2 + 1), (rows - tokens, chunk), (1, 1)):
        outs = plan.launch(row0, valid)
        torch.cuda.synchronize()
        ref = _slab_oracle(g, row0, tokens, chunk, valid)
        for o in range(len(widths)):
            assert bits_equal(to_np(outs[o]), ref[o]), (row0, valid, o)
        direct, _ = sdm.gather(g["bank"], [(i[row0:row0 + tokens], w[row0:row0 + tokens]) for i, w in g["ops"]],
                               chunk=chunk, valid=valid, with_stash=False)
        torch.cuda.synchronize()
        for o in range(len(widths)):
            assert bits_equal(to_np(outs[o]), to_np(direct[o]))


def test_plan_launches_replay_in_a_graph():
    g = _inputs("bf16", "bf16", "i32", 4000, 128, 256, (24, 8), seed=3)
    tokens, chunk = 64, 16
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=tokens, chunk=chunk)
    steps = [(0, 16), (64, 9), (192, 16), (17, 0)]
    dst = torch.empty((len(steps), 2, tokens, 128), dtype=torch.float32, device=DEV)
    plan.launch(0)  # first launch outside capture
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i, (row0, valid) in enumerate(steps):
                outs = plan.launch(row0, valid)
                dst[i, 0].copy_(outs[0])
                dst[i, 1].copy_(outs[1])
    torch.cuda.current_stream(DEV).wait_stream(side)
    dst.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    for i, (row0, valid) in enumerate(steps):
        ref = _slab_oracle(g, row0, tokens, chunk, valid)
        assert bits_equal(to_np(dst[i, 0]), ref[0]) and bits_equal(to_np(dst[i, 1]), ref[1]), (row0, valid)


def test_plan_launch_checks_row0_and_valid():
    g = _inputs("f32", "f32", "i64", 500, 64, 40, (8,), seed=4)
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=16, chunk=8, row0_max=20)
    for row0, valid, code in ((21, 8, EROW), (-1, 8, EROW), (0, 9, ECHUNK), (0, -1, ECHUNK)):
        with pytest.raises(sdm.SDMError) as e:
            plan.launch(row0, valid)
        assert e.value.status == code
    plan.launch(20, 8)  # the largest planned row0 is fine
    torch.cuda.synchronize()


def test_plan_init_checks_rows():
    g = _inputs("bf16", "bf16", "i32", 500, 64, 40, (8,), seed=4)
    with pytest.raises(sdm.SDMError) as e:
        sdm.GatherPlan(g["bank"], g["ops"], tokens=16, chunk=8, row0_max=25)  # 25 + 16 > 40 rows
    assert e.value.status == EROW


def test_empty_plan_launches_nothing():
    g = _inputs("bf16", "bf16", "i32", 500, 64, 40, (8,), seed=4)
    outs = [torch.full((0, 64), 7.0, device=DEV)]
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=0, chunk=8, outs=outs)
    plan.launch(40, 0)
    torch.cuda.synchronize()


def test_flagged_launches_after_decode_steps_see_their_writes():
    """Plan launches with SDM_INPUTS_READY (the index and weight rows were made up front) chained
    after decode steps that rewrite the very rows they gather: each launch may warm L2 with its
    rows while the step ahead still writes them, and must still read the written rows. The same
    sequence without the flag (checked against the oracle above) gives the reference bits."""
    from parity import DECODE_KEYS

    S, P, hd, W, T = 16, 64, 128, 32, 6
    dwl = workloads.DecodeWorkload("plan_after_decode", "bf16", S, hd, P, W, W, 1, T, "i32", 0.35, bank_std=0.5,
                                   seed=21)
    x = workloads.make_decode_inputs(dwl, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(22)
    rows, tokens, chunk = 6 * 64, 64, 16
    ops = [(torch.randint(0, S * P, (rows, w), generator=gen, device=DEV, dtype=torch.int32),
            (torch.randn((rows, w), generator=gen, device=DEV) * 0.125).to(torch.bfloat16)) for w in (48, 16)]
    results = []
    for flag in (False, True):
        bank = x["bank"].clone()
        plan = sdm.GatherPlan(bank, ops, tokens=tokens, chunk=chunk)
        got = []
        for t in range(T):
            sdm.decode_step(bank, *(x[k][t] for k in DECODE_KEYS))
            outs = plan.launch(t * 64, chunk - t, inputs_ready=flag)
            got.append([o.clone() for o in outs])
        torch.cuda.synchronize()
        results.append((got, bank))
    (plain, bank_p), (flagged, bank_f) = results
    assert bits_equal(to_np(bank_p), to_np(bank_f))
    for a, b in zip(plain, flagged):
        assert bits_equal(to_np(a[0]), to_np(b[0])) and bits_equal(to_np(a[1]), to_np(b[1]))


def test_plan_walk_applies_each_slab():
    """sdm_gather_plan_walk: slab i of a walk is launch(row0[i], valid[i]); the outputs hold the last
    slab's gather, for walks ending at every slab of the list (and with inputs_ready)."""
    g = _inputs("bf16", "bf16", "i64", 5000, 128, 320, (64, 64), seed=21)
    tokens, chunk = 64, 16
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=tokens, chunk=chunk)
    row0s, valids = [0, 200, 37, 256, 5], [16, 3, 0, 16, 11]
    for end in range(1, len(row0s) + 1):
        for ready in (False, True):
            for o in plan.outs:
                o.fill_(float("nan"))
            outs = plan.walk(row0s[:end], valids[:end], inputs_ready=ready)
            torch.cuda.synchronize()
            ref = _slab_oracle(g, row0s[end - 1], tokens, chunk, valids[end - 1])
            for o in range(2):
                assert bits_equal(to_np(outs[o]), ref[o]), (end, ready, o)
    outs = plan.walk([7, 96])  # valid omitted: every slab full
    torch.cuda.synchronize()
    ref = _slab_oracle(g, 96, tokens, chunk, chunk)
    assert bits_equal(to_np(outs[0]), ref[0]) and bits_equal(to_np(outs[1]), ref[1])


def test_plan_walk_checks_every_slab_before_launching():
    g = _inputs("f32", "f32", "i64", 500, 64, 40, (8,), seed=4)
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=16, chunk=8, row0_max=20)
    plan.outs[0].fill_(float("nan"))
    torch.cuda.synchronize()
    for row0s, valids, code in (([0, 8, 21], None, EROW), ([0, 4], [8, 9], ECHUNK), ([3, -1], [1, 1], EROW)):
        with pytest.raises(sdm.SDMError) as e:
            plan.walk(row0s, valids)
        assert e.value.status == code
    torch.cuda.synchronize()
    assert torch.isnan(plan.outs[0]).all()  # no slab of a refused walk was launched
    plan.walk([], [])  # an empty walk launches nothing
    torch.cuda.synchronize()
    assert torch.isnan(plan.outs[0]).all()
