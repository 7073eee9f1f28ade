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
    ("bf16", "bf16", "i32", 3000, 136, 64, 16, (13, 21), True, True),  # column pairs, a last slice of 8 columns
    ("bf16", "bf16", "i64", 2000, 264, 32, 8, (8, 1), False, True),    # three slices; a one-entry operand
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


def test_device_status_waits_for_side_streams():
    """sdm_device_status synchronises the device: a gather still running on a non-blocking side
    stream has raised its bit before the word is read, with no synchronisation by the caller."""
    wl = _gw("bf16", "bf16", "i64", 1 << 16, 128, 4096, 64, (64, 64), True, False, seed=11)
    g = workloads.make_gather_inputs(wl, device=DEV)
    idx, w = g["ops"][0]
    idx[wl.tokens - 1, wl.widths[0] - 1] = -5  # the very last entry of the launch
    torch.cuda.synchronize()
    sdm.device_status(clear=True)
    side = torch.cuda.Stream(DEV)
    with torch.cuda.stream(side):
        for _ in range(4):  # several launches queued behind one another on the side stream
            sdm.gather(g["bank"], [(idx, w), g["ops"][1]], chunk=wl.chunk)
    assert sdm.device_status(clear=True) & sdm.SDM_DEV_BAD_INDEX
    assert sdm.device_status(clear=True) == 0  # cleared after every launch had finished


@pytest.mark.parametrize("wl", [workloads.C4, workloads.C4_BWD], ids=lambda w: w.name)
def test_gather_full_size(wl):
    """A full gather workload in the benchmark's launch configuration (the two-operand forward
    shape and the one-operand backward shape): every token's outputs and stash rows against the
    oracle run over the whole launch, bit for bit; every stash row also against torch's own row
    indexing, every padding token zero, and every output within the float32 summation bound of a
    float64 evaluation."""
    g = workloads.make_gather_inputs(wl, device=DEV)
    outs, stash = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"])
    torch.cuda.synchronize()
    assert sdm.device_status() == 0
    live = (torch.arange(wl.tokens, device=DEV) % wl.chunk) < g["chunk_valid"].repeat_interleave(wl.chunk)
    i0 = g["ops"][0][0]
    bits = torch.int16 if wl.bank_dtype == "bf16" else torch.int32
    # stash: raw rows, bit-exact (torch's indexing as the independent reference); padding rows zero
    ref_stash = g["bank"][i0[live]]
    assert torch.equal(stash[live].view(bits), ref_stash.view(bits))
    assert not stash[~live].view(bits).any()
    for o, (idx, w) in enumerate(g["ops"]):
        out = outs[o]
        assert not out[~live].any()
        rows = g["bank"][idx[live]].double()
        wd = w[live].double()
        ref = torch.einsum("tn,tnc->tc", wd, rows)
        bound = idx.shape[1] * 2.0 ** -24 * torch.einsum("tn,tnc->tc", wd.abs(), rows.abs()) * 1.01
        assert bool(((out[live].double() - ref).abs() <= bound).all())
    # the whole launch against the oracle, bit for bit
    ref = _oracle(g, wl)
    for o in range(len(g["ops"])):
        assert bits_equal(to_np(outs[o]), ref[o]), f"operand {o} outputs differ from the oracle"
    assert bits_equal(to_np(stash), ref[2]), "stash differs from the oracle"


def _first_occurrence_kpos(idx: np.ndarray, chunk: int, live: np.ndarray) -> np.ndarray:
    """kpos of each chunk's first occurrences: position in the chunk's sorted entries (numpy)."""
    tokens, W0 = idx.shape
    kpos = np.full((tokens, W0), -1, np.int32)
    for c in range(tokens // chunk):
        ent = idx[c * chunk:(c + 1) * chunk].ravel()
        order = np.sort(ent)
        _, first = np.unique(ent, return_index=True)
        for e in first:
            t = c * chunk + e // W0
            kpos[t, e % W0] = int(np.searchsorted(order, ent[e]))
    kpos[~live] = np.where(kpos[~live] >= 0, 0, -1)  # padding tokens name rows too; they must store nothing
    return kpos


KPOS_CASES = [
    ("bf16", "bf16", "i64", 3000, 128, 128, 16, (32, 32)),
    ("f32", "f32", "i32", 500, 520, 16, 4, (12,)),       # rows cut into slices
    ("bf16", "f32", "i32", 300, 13, 24, 6, (5, 7)),       # 26-byte rows: plain-load path
    ("bf16", "bf16", "i32", 800, 136, 32, 8, (11, 6)),    # column pairs, a last slice of 8 columns
]


@pytest.mark.parametrize("case", KPOS_CASES, ids=[f"{c[0]}-hd{c[4]}-{'x'.join(map(str, c[7]))}" for c in KPOS_CASES])
def test_gather_kpos_matches_oracle(case):
    bank_dt, w_dt, idx_dt, n_slots, hd, tokens, chunk, widths = case
    wl = _gw(bank_dt, w_dt, idx_dt, n_slots, hd, tokens, chunk, widths, True, True, seed=21)
    g = workloads.make_gather_inputs(wl, device=DEV)
    idx0 = to_np(g["ops"][0][0])
    live = (np.arange(tokens) % chunk) < np.repeat(to_np(g["chunk_valid"]), chunk)
    kpos = _first_occurrence_kpos(idx0, chunk, live)
    W0 = widths[0]
    compact = torch.full((tokens // chunk, chunk * W0, hd), float("nan"), dtype=g["bank"].dtype, device=DEV)
    ref_compact = to_np(compact)
    outs, comp = sdm.gather(g["bank"], g["ops"], chunk=chunk, chunk_valid=g["chunk_valid"],
                            kpos=torch.from_numpy(kpos).to(DEV), compact=compact)
    torch.cuda.synchronize()
    assert comp is compact
    oracle.gather_kpos(to_np(g["bank"]), idx0, kpos, ref_compact, chunk=chunk, chunk_valid=to_np(g["chunk_valid"]))
    assert bits_equal(to_np(compact), ref_compact)
    r0, r1, _ = _oracle(g, wl)
    assert bits_equal(to_np(outs[0]), r0)
    if len(widths) == 2:
        assert bits_equal(to_np(outs[1]), r1)
    assert sdm.device_status() == 0


def test_gather_kpos_out_of_range_is_skipped_and_flagged():
    wl = _gw("bf16", "bf16", "i64", 800, 64, 16, 8, (4,), True, False, seed=22)
    g = workloads.make_gather_inputs(wl, device=DEV)
    kpos = torch.full((16, 4), -1, dtype=torch.int32, device=DEV)
    kpos[0, 0] = 0
    kpos[1, 2] = 8 * 4  # one past the chunk's snapshot
    compact = torch.zeros((2, 32, 64), dtype=torch.bfloat16, device=DEV)
    sdm.device_status(clear=True)
    sdm.gather(g["bank"], g["ops"], chunk=8, kpos=kpos, compact=compact)
    torch.cuda.synchronize()
    assert sdm.device_status(clear=True) & sdm.SDM_DEV_BAD_INDEX
    assert torch.equal(compact[0, 0], g["bank"][g["ops"][0][0][0, 0]])
    assert not compact[0, 1:].view(torch.int16).any() and not compact[1].view(torch.int16).any()


def test_gather_kpos_full_size():
    """The full gather workload with a compact snapshot: every named row equals torch's own row
    indexing, every other snapshot row keeps its sentinel bits, outputs equal the stash form's."""
    wl = workloads.C4
    g = workloads.make_gather_inputs(wl, device=DEV)
    live = ((torch.arange(wl.tokens, device=DEV) % wl.chunk) < g["chunk_valid"].repeat_interleave(wl.chunk))
    idx0 = g["ops"][0][0]
    W0 = idx0.shape[1]
    # first occurrence of each row within its chunk (torch on the GPU): sort each chunk's entries
    ent = idx0.view(wl.tokens // wl.chunk, wl.chunk * W0)
    srt, order = ent.sort(dim=1, stable=True)
    first_sorted = torch.ones_like(srt, dtype=torch.bool)
    first_sorted[:, 1:] = srt[:, 1:] != srt[:, :-1]
    pos = torch.arange(srt.shape[1], device=DEV).expand_as(srt)
    first_pos = torch.cummax(torch.where(first_sorted, pos, torch.zeros_like(pos)), dim=1).values
    kp_sorted = torch.where(first_sorted, first_pos, torch.full_like(first_pos, -1))
    kpos = torch.empty_like(kp_sorted).scatter_(1, order, kp_sorted).view(wl.tokens, W0).to(torch.int32)
    compact = torch.full((wl.tokens // wl.chunk, wl.chunk * W0, wl.hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    sentinel = compact[0, 0].clone()
    outs, _ = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], kpos=kpos,
                         compact=compact)
    outs_ref, _ = sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], with_stash=False)
    torch.cuda.synchronize()
    named = (kpos >= 0) & live[:, None]
    t_idx, n_idx = torch.nonzero(named, as_tuple=True)
    rows = compact[t_idx // wl.chunk, kpos[t_idx, n_idx].long()]
    assert torch.equal(rows.view(torch.int16), g["bank"][idx0[t_idx, n_idx]].view(torch.int16))
    mask = torch.zeros(compact.shape[:2], dtype=torch.bool, device=DEV)
    mask[t_idx // wl.chunk, kpos[t_idx, n_idx].long()] = True
    assert torch.equal(compact[~mask].view(torch.int16), sentinel.expand(int((~mask).sum()), -1).view(torch.int16))
    for a, b in zip(outs, outs_ref):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert sdm.device_status() == 0
    # the whole launch against the oracle, bit for bit: the snapshot (sentinel rows included) and
    # both operands' outputs
    bank_h = to_np(g["bank"])
    ref_compact = np.full(compact.shape, to_np(sentinel)[0], dtype=np.uint16)
    oracle.gather_kpos(bank_h, to_np(idx0), to_np(kpos), ref_compact, chunk=wl.chunk,
                       chunk_valid=to_np(g["chunk_valid"]), check=False)
    assert bits_equal(to_np(compact), ref_compact), "compact snapshot differs from the oracle"
    del ref_compact
    (i0, w0), (i1, w1) = g["ops"]
    r0, r1, _ = oracle.gather(bank_h, to_np(i0), to_np(w0), to_np(i1), to_np(w1), chunk=wl.chunk,
                              chunk_valid=to_np(g["chunk_valid"]), stash=False, check=False)
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1), "outputs differ from the oracle"
