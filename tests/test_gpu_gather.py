"""GPU parity of sdm_gather against the CPU oracle, through the C ABI.

The kernel sums each column over the entries in ascending order with fmaf, which is the
oracle's one-group order, so outputs are compared bit for bit; stash rows and padding zeros are
bit-exact by definition.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from decode_state_gb300 import sdm, workloads
from parity import bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield


def _gw(bank, wdt, idx, n_slots, hd, tokens, chunk, widths, stash, per_chunk, seed=0):
    return workloads.GatherWorkload(f"t_{bank}_{hd}_{widths}", bank, n_slots, hd, tokens, chunk, tuple(widths), idx,
                                    wdt, 0.125, stash=stash, per_chunk_valid=per_chunk, seed=seed)


# (bank dtype, weight dtype, idx dtype, n_slots, head_dim, tokens, chunk, widths, stash, per-chunk valid)
CASES = [
    ("bf16", "bf16", "i64", 5000, 128, 192, 64, (64, 64), True, True),  # the gather workload's shape, fewer tokens
    ("f32", "f32", "i32", 3000, 64, 96, 32, (17,), True, False),
    ("bf16", "f32", "i32", 2000, 200, 40, 8, (9, 30), False, True),    # no stash
    ("f32", "bf16", "i64", 1000, 520, 16, 4, (256, 3), True, True),    # widest operand, rows cut into slices
    ("bf16", "bf16", "i32", 700, 13, 24, 6, (5, 7), True, True),       # 26-byte rows: plain-load path
    ("f32", "f32", "i64", 100, 1, 8, 8, (1, 1), True, False),          # head_dim 1, width 1
]
IDS = [f"{c[0]}-w{c[1]}-{c[2]}-hd{c[4]}-{'x'.join(map(str, c[7]))}-{'stash' if c[8] else 'nostash'}" for c in CASES]


def _oracle(g, wl, valid=None, chunk_valid="auto"):
    ops = g["ops"]
    cv = g["chunk_valid"] if chunk_valid == "auto" else chunk_valid
    a = [to_np(ops[0][0]), to_np(ops[0][1])]
    if len(ops) == 2:
        a += [to_np(ops[1][0]), to_np(ops[1][1])]
    return oracle.gather(to_np(g["bank"]), *a, chunk=wl.chunk, valid=-1 if valid is None else valid,
                         chunk_valid=None if cv is None else to_np(cv), stash=wl.stash)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_gather_matches_oracle(case):
    wl = _gw(*case)
    g = workloads.make_gather_inputs(wl, device=DEV)
    outs, stash = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], with_stash=wl.stash)
    torch.cuda.synchronize()
    r0, r1, rs = _oracle(g, wl)
    assert bits_equal(to_np(outs[0]), r0)
    if len(wl.widths) == 2:
        assert bits_equal(to_np(outs[1]), r1)
    if wl.stash:
        assert bits_equal(to_np(stash), rs)
    else:
        assert stash is None
    assert sdm.device_status() == 0


@pytest.mark.parametrize("valid", [0, 1, 37, 64])
def test_gather_scalar_valid(valid):
    wl = _gw("bf16", "bf16", "i32", 4000, 128, 128, 64, (20, 11), True, False, seed=5)
    g = workloads.make_gather_inputs(wl, device=DEV)
    outs, stash = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, valid=valid)
    torch.cuda.synchronize()
    r0, r1, rs = _oracle(g, wl, valid=valid, chunk_valid=None)
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1) and bits_equal(to_np(stash), rs)
    if valid == 0:
        assert not outs[0].any() and not stash.view(torch.int16).any()


def test_gather_reuses_outputs_with_garbage():
    """Outputs and stash filled with NaN bits beforehand are fully overwritten (padding included)."""
    wl = _gw("bf16", "f32", "i64", 3000, 64, 64, 16, (8, 8), True, True, seed=6)
    g = workloads.make_gather_inputs(wl, device=DEV)
    outs = [torch.full((64, 64), float("nan"), device=DEV) for _ in range(2)]
    stash = torch.full((64, 8, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], stash=stash, outs=outs)
    torch.cuda.synchronize()
    r0, r1, rs = _oracle(g, wl)
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1) and bits_equal(to_np(stash), rs)


def test_gather_empty():
    wl = _gw("f32", "f32", "i32", 10, 8, 0, 4, (3,), True, False)
    bank = torch.zeros((10, 8), device=DEV)
    ops = [(torch.zeros((0, 3), dtype=torch.int32, device=DEV), torch.zeros((0, 3), device=DEV))]
    outs, stash = sdm.gather(bank, ops, chunk=wl.chunk)
    assert outs[0].shape == (0, 8) and stash.shape == (0, 3, 8)


def test_gather_out_of_range_index_is_skipped_and_flagged():
    wl = _gw("bf16", "bf16", "i64", 1000, 128, 16, 16, (6,), True, False, seed=7)
    g = workloads.make_gather_inputs(wl, device=DEV)
    idx, w = g["ops"][0]
    idx[3, 2] = wl.n_slots  # one past the end
    sdm.device_status(clear=True)
    outs, stash = sdm.gather(g["bank"], [(idx, w)], chunk=wl.chunk)
    torch.cuda.synchronize()
    assert sdm.device_status(clear=True) & sdm.SDM_DEV_BAD_INDEX
    assert not stash[3, 2].view(torch.int16).any()
    # the skipped entry contributes nothing: the oracle with that entry's weight set to zero
    idx_ok, w_ok = idx.clone(), w.clone()
    idx_ok[3, 2] = 0
    w_ok[3, 2] = 0
    r0, _, rs = oracle.gather(to_np(g["bank"]), to_np(idx_ok), to_np(w_ok), chunk=wl.chunk)
    assert np.array_equal(to_np(outs[0]), r0)  # value equality (an exact zero's sign may differ)
    rs[3, 2] = 0
    assert bits_equal(to_np(stash), rs)


def test_gather_full_size():
    """The full gather workload in the benchmark's launch configuration: sampled tokens against the
    oracle bit for bit, every stash row against torch's own row indexing, every padding token zero,
    and every output within the float32 summation bound of a float64 evaluation."""
    wl = workloads.C4
    g = workloads.make_gather_inputs(wl, device=DEV)
    outs, stash = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"])
    torch.cuda.synchronize()
    assert sdm.device_status() == 0
    live = (torch.arange(wl.tokens, device=DEV) % wl.chunk) < g["chunk_valid"].repeat_interleave(wl.chunk)
    (i0, w0), (i1, w1) = g["ops"]
    # stash: raw rows, bit-exact (torch's indexing as the independent reference); padding rows zero
    ref_stash = g["bank"][i0[live]]
    assert torch.equal(stash[live].view(torch.int16), ref_stash.view(torch.int16))
    assert not stash[~live].view(torch.int16).any()
    for o, (idx, w) in enumerate(g["ops"]):
        out = outs[o]
        assert not out[~live].any()
        rows = g["bank"][idx[live]].double()
        wd = w[live].double()
        ref = torch.einsum("tn,tnc->tc", wd, rows)
        bound = idx.shape[1] * 2.0 ** -24 * torch.einsum("tn,tnc->tc", wd.abs(), rows.abs()) * 1.01
        assert bool(((out[live].double() - ref).abs() <= bound).all())
    # sampled tokens against the oracle, bit for bit
    bank_h = to_np(g["bank"])
    sample = torch.nonzero(live).flatten()[:: max(1, int(live.sum()) // 256)][:256]
    for o, (idx, w) in enumerate(g["ops"]):
        ref, _, _ = oracle.gather(bank_h, to_np(idx[sample]), to_np(w[sample]), chunk=1, stash=False)
        assert bits_equal(to_np(outs[o][sample]), ref)
