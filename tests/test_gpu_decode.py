"""GPU parity of sdm_decode_step / sdm_decode_seq against the CPU oracle, through the C ABI.

Every case, small or at the full size of a workload (in the launch configuration the benchmark
times), compares every reading and every bank element with the oracle run over the same inputs.
Tolerances are in parity.py: 1e-5*(1+|ref|) for float32, 2 bf16 ulps for bfloat16; beside them
every comparison also requires the oracle's bits, since the kernels take its rounding steps in
its order.
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0, "a kernel raised the device status word"


def _wl(dtype, idx, S, P, hd, W, R, G, T, seed=0):
    return workloads.DecodeWorkload(f"t_{dtype}_{S}x{hd}_w{W}r{R}", dtype, S, hd, P, W, R, W if G == "W" else G, T,
                                    idx, 0.35, bank_std=0.5, seed=seed)


# (dtype, idx, streams, slots/stream, head_dim, W, R, G, T)
SMALL = [
    ("f32", "i32", 4, 1024, 64, 8, 8, 1, 16),       # the float32 decode workload's shape
    ("bf16", "i64", 5, 300, 200, 16, 12, "W", 3),   # several column slices, ragged last slice, per-write gates
    ("f32", "i64", 3, 700, 37, 5, 9, 1, 4),         # 148-byte rows: plain-load path
    ("bf16", "i32", 2, 600, 13, 3, 256, "W", 2),    # odd bf16 rows, R at its maximum
    ("f32", "i32", 7, 520, 256, 256, 256, 1, 2),    # W = R = 256, 1 KiB rows cut into slices
    ("bf16", "i32", 33, 128, 128, 64, 64, 1, 5),    # the serving shape, fewer streams
    ("bf16", "i64", 1, 64, 8, 1, 1, 1, 3),          # W = R = 1, 16-byte rows
    ("f32", "i32", 2, 16, 1, 4, 4, "W", 3),         # head_dim 1
    ("f32", "i64", 5, 300, 256, 40, 7, 1, 3),       # streamed rows: 3 write chunks, 1 read chunk
    ("bf16", "i32", 3, 400, 512, 70, 200, "W", 2),  # streamed rows: 1 KiB rows in 512-byte slices
]
IDS = [f"{c[0]}-{c[1]}-S{c[2]}-hd{c[4]}-W{c[5]}R{c[6]}G{c[7]}-T{c[8]}" for c in SMALL]


def _oracle_seq(x: dict):
    bank = to_np(x["bank"])
    out = oracle.decode_seq(bank, *(to_np(x[k]) for k in DECODE_KEYS))
    return bank, out


@pytest.mark.parametrize("case", SMALL, ids=IDS)
def test_decode_seq_matches_oracle(case):
    wl = _wl(*case)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref, out_ref = _oracle_seq(x)
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), out_ref, wl.bank_dtype, "readings")
    assert_close(to_np(x["bank"]), bank_ref, wl.bank_dtype, "bank")


@pytest.mark.parametrize("case", SMALL, ids=IDS)
def test_decode_step_matches_oracle(case):
    wl = _wl(*case, seed=1)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref, out_ref = _oracle_seq(x)
    for t in range(wl.T):
        out = sdm.decode_step(x["bank"], *(x[k][t] for k in DECODE_KEYS))
        assert_close(to_np(out), out_ref[t], wl.bank_dtype, f"readings of token {t}")
    assert_close(to_np(x["bank"]), bank_ref, wl.bank_dtype, "bank")


@pytest.mark.parametrize("case", SMALL[:6], ids=IDS[:6])
def test_seq_equals_steps_bitwise(case):
    """One persistent launch of T tokens gives the same bits as T single-token launches."""
    wl = _wl(*case, seed=2)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank2 = x["bank"].clone()
    out_seq = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    outs = [sdm.decode_step(bank2, *(x[k][t] for k in DECODE_KEYS)) for t in range(wl.T)]
    torch.cuda.synchronize()
    assert torch.equal(out_seq.view(torch.int16 if wl.bank_dtype == "bf16" else torch.int32),
                       torch.stack(outs).view(torch.int16 if wl.bank_dtype == "bf16" else torch.int32))
    assert bits_equal(to_np(x["bank"]), to_np(bank2))


def test_deterministic():
    wl = _wl("bf16", "i32", 16, 256, 128, 32, 32, 1, 6, seed=3)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank0 = x["bank"].clone()
    o1 = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    b1 = x["bank"].clone()
    x["bank"].copy_(bank0)
    o2 = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert bits_equal(to_np(o1), to_np(o2)) and bits_equal(to_np(b1), to_np(x["bank"]))


def test_empty_launches_are_noops():
    wl = _wl("f32", "i32", 2, 16, 8, 2, 2, 1, 2)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank0 = x["bank"].clone()
    sdm.decode_seq(x["bank"], *(x[k][:0] for k in DECODE_KEYS))  # T = 0
    sdm.decode_step(x["bank"], *(x[k][0, :0] for k in DECODE_KEYS))  # no streams
    torch.cuda.synchronize()
    assert torch.equal(bank0, x["bank"])


def test_read_slot_written_this_token():
    """Readings of a slot written in the same token see the new row (read after write)."""
    wl = _wl("bf16", "i64", 8, 64, 128, 4, 1, 1, 2, seed=4)
    x = workloads.make_decode_inputs(wl, device=DEV)
    x["q_idx"][:, :, 0] = x["k_idx"][:, :, 2]
    x["q_val"][:] = 1.0
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    last_rows = x["bank"][x["k_idx"][-1, :, 2].long()]
    assert torch.equal(out[-1].view(torch.int16), last_rows.view(torch.int16))


# ---------------------------------------------------------------- full-size workloads


@pytest.mark.parametrize("wl", [workloads.C0, workloads.C2, workloads.C3], ids=lambda w: w.name)
def test_full_size_seq(wl):
    """The multi-token workloads as the benchmark launches them (one sdm_decode_seq call), compared
    with the oracle run over the whole workload: every stream's readings of every token and the
    whole bank, within the tolerance and bit for bit."""
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS), check=False)
    assert_close(to_np(out), ref, wl.bank_dtype, "readings")
    del ref
    assert_close(to_np(x["bank"]), bank_ref, wl.bank_dtype, "bank")


def test_full_size_steps_bf16_gw():
    """The 256-step bf16 workload with per-write gates, as single-token launches: every step's
    readings of every stream and the whole final bank against one oracle run over all 256 steps
    from the same start (no re-seeding), within the tolerance and bit for bit."""
    wl = workloads.C1
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    outs = torch.empty((wl.T, wl.n_streams, wl.hd), dtype=torch.bfloat16, device=DEV)
    for t in range(wl.T):
        sdm.decode_step(x["bank"], *(x[k][t] for k in DECODE_KEYS), out=outs[t])
    torch.cuda.synchronize()
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS), check=False)
    got = to_np(outs)
    for t0 in range(0, wl.T, 16):
        assert_close(got[t0:t0 + 16], ref[t0:t0 + 16], "bf16", f"tokens {t0}..{t0 + 15}")
    assert_close(to_np(x["bank"]), bank_ref, "bf16", "bank")


def test_layer_state_steps_match_seq_and_oracle():
    from decode_state_gb300.state import SDMLayerState

    wl = _wl("bf16", "i64", 6, 96, 64, 8, 5, "W", 4, seed=9)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref, out_ref = _oracle_seq(x)
    st = SDMLayerState(x["bank"].clone())
    outs = [st.step(*(x[k][t] for k in DECODE_KEYS)) for t in range(wl.T)]
    assert st.cache_len == wl.T
    seq = SDMLayerState(x["bank"].clone(), seq_len=2)
    out_seq = seq.steps(*(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert seq.cache_len == 2 + wl.T
    assert torch.equal(torch.stack(outs).view(torch.int16), out_seq.view(torch.int16))
    assert torch.equal(st.memory.view(torch.int16), seq.memory.view(torch.int16))
    assert_close(to_np(out_seq), out_ref, "bf16", "readings")
    assert_close(to_np(seq.memory), bank_ref, "bf16", "bank")


def test_host_fed_decoder_matches_sequential_calls():
    """Pipelined host-fed steps (double-buffered inputs, copies on their own streams) give the same
    bank and readings, bit for bit, as the same steps run one after another on the device."""
    from decode_state_gb300.hostfed import HostFedDecoder

    wl = _wl("bf16", "i32", 40, 128, 128, 16, 16, 1, 4, seed=11)
    steps = [workloads.make_decode_inputs(wl, device=DEV, seed=100 + n) for n in range(5)]
    bank0 = steps[0]["bank"].clone()
    ref_bank = bank0.clone()
    refs = [sdm.decode_seq(ref_bank, *(x[k] for k in DECODE_KEYS)).clone() for x in steps]
    dec = HostFedDecoder(bank0, steps[0], depth=2)
    host = [{k: x[k].cpu().pin_memory() for k in DECODE_KEYS} for x in steps]
    outs = [torch.empty(refs[0].shape, dtype=torch.bfloat16, pin_memory=True) for _ in steps]
    for h, o in zip(host, outs):
        dec.submit(h, o)
    dec.synchronize()
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs):
        assert torch.equal(o.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(bank0.view(torch.int16), ref_bank.view(torch.int16))


def test_step_graph_matches_eager_steps():
    """T single-token launches replayed from one captured graph equal the same launches run eagerly."""
    from decode_state_gb300.graphs import DecodeStepGraph

    wl = _wl("bf16", "i64", 16, 256, 128, 32, 32, "W", 6, seed=12)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_g = x["bank"].clone()
    gr = DecodeStepGraph(bank_g, x)
    for k in DECODE_KEYS:
        gr.inputs[k].copy_(x[k])
    out_g = gr.replay()
    eager = [sdm.decode_step(x["bank"], *(x[k][t] for k in DECODE_KEYS)) for t in range(wl.T)]
    torch.cuda.synchronize()
    assert torch.equal(out_g.view(torch.int16), torch.stack(eager).view(torch.int16))
    assert torch.equal(bank_g.view(torch.int16), x["bank"].view(torch.int16))


def test_decode_step_plan_matches_eager_steps():
    """T single-token launches through a DecodeStepPlan (checked once, pointers precomputed) equal
    the same launches through decode_step, on the default stream and on a given one."""
    wl = _wl("f32", "i32", 16, 256, 96, 24, 40, 1, 5, seed=13)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_p = x["bank"].clone()
    plan = sdm.DecodeStepPlan(bank_p, {k: x[k] for k in DECODE_KEYS})
    for t in range(wl.T):
        if t == 2:
            side = torch.cuda.Stream(DEV)
            side.wait_stream(torch.cuda.current_stream(DEV))
            with torch.cuda.stream(side):
                plan.launch(t, stream=side)
            torch.cuda.current_stream(DEV).wait_stream(side)
        else:
            plan.launch(t)
    eager = [sdm.decode_step(x["bank"], *(x[k][t] for k in DECODE_KEYS)) for t in range(wl.T)]
    torch.cuda.synchronize()
    assert torch.equal(plan.out.view(torch.int32), torch.stack(eager).view(torch.int32))
    assert torch.equal(bank_p.view(torch.int32), x["bank"].view(torch.int32))


@pytest.mark.parametrize("case", [SMALL[1], SMALL[5], SMALL[8]], ids=[IDS[1], IDS[5], IDS[8]])
def test_decode_plan_walk_matches_seq_and_oracle(case):
    """sdm_decode_plan_walk: a walk over all T steps (in two parts, one with SDM_INPUTS_READY)
    gives the bits of one sdm_decode_seq launch and of the oracle, on the staged, narrow-slice and
    streamed kernels."""
    wl = _wl(*case)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref, out_ref = _oracle_seq(x)
    bank_s = x["bank"].clone()
    out_s = sdm.decode_seq(bank_s, *(x[k] for k in DECODE_KEYS))
    plan = sdm.DecodeStepPlan(x["bank"], {k: x[k] for k in DECODE_KEYS})
    plan.walk(0, 1)
    ready = sdm.DecodeStepPlan(x["bank"], {k: x[k] for k in DECODE_KEYS}, out=plan.out, inputs_ready=True)
    ready.walk(1)
    torch.cuda.synchronize()
    assert bits_equal(to_np(plan.out), to_np(out_s)) and bits_equal(to_np(x["bank"]), to_np(bank_s))
    assert_close(to_np(plan.out), out_ref, wl.bank_dtype, "readings")
    assert_close(to_np(x["bank"]), bank_ref, wl.bank_dtype, "bank")


def test_decode_plan_checks_steps_before_launching():
    wl = _wl("bf16", "i32", 4, 64, 128, 8, 8, 1, 4, seed=5)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank0 = x["bank"].clone()
    plan = sdm.DecodeStepPlan(x["bank"], {k: x[k] for k in DECODE_KEYS})
    for t0, n, code in ((3, 2, -13), (-1, 1, -13), (4, 1, -13), (0, -1, -7)):
        with pytest.raises(sdm.SDMError) as e:
            plan.walk(t0, n)
        assert e.value.status == code
    with pytest.raises(sdm.SDMError) as e:
        plan.launch(4)
    assert e.value.status == -13
    plan.walk(4, 0)  # an empty walk past the end launches nothing
    torch.cuda.synchronize()
    assert torch.equal(x["bank"].view(torch.int16), bank0.view(torch.int16))  # nothing was launched


def test_gather_after_decode_sees_its_writes():
    """A gather launched right after a decode on the same stream (no host synchronisation) reads
    the rows the decode wrote: the overlapped launch waits for its predecessor before reading."""
    wl = _wl("bf16", "i32", 64, 128, 128, 16, 16, 1, 1, seed=13)
    x = workloads.make_decode_inputs(wl, device=DEV)
    idx = x["k_idx"][0].reshape(-1, 1).contiguous()  # every written row, one per token
    w = torch.ones(idx.shape, dtype=torch.float32, device=DEV)
    outs = [torch.empty((idx.shape[0], wl.hd), device=DEV)]
    stash = torch.empty((idx.shape[0], 1, wl.hd), dtype=torch.bfloat16, device=DEV)
    out = torch.empty((1, wl.n_streams, wl.hd), dtype=torch.bfloat16, device=DEV)
    sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS), out=out)
    sdm.gather(x["bank"], [(idx, w)], chunk=1, outs=outs, stash=stash)  # launched directly after the decode
    torch.cuda.synchronize()
    assert torch.equal(stash[:, 0].view(torch.int16), x["bank"][idx[:, 0].long()].view(torch.int16))
    assert torch.equal(outs[0], x["bank"][idx[:, 0].long()].float())


@pytest.mark.parametrize("streams", [512, 320, 160, 64])
def test_streamed_decode_many_streams_matches_oracle(streams):
    """Wide rows over grids of several sizes: 1 KiB float32 rows with W = R = 256, which the
    streaming kernel cuts into whole, half or quarter rows with rings of different depths (two
    stages of up to 128 rows where few blocks share an SM, two waves of blocks at 320 streams);
    compared with the oracle on every stream."""
    wl = workloads.DecodeWorkload("wide_many", "f32", streams, 256, 300, 256, 256, 1, 2, "i64", 1 / 16, bank_std=0.5,
                                  seed=9)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, "f32", "readings")
    assert_close(to_np(x["bank"]), bank_ref, "f32", "bank")
    assert sdm.device_status() == 0


@pytest.mark.parametrize("streams,W,R,idx", [(16, 256, 256, "i32"), (3, 200, 256, "i64"), (40, 256, 120, "i32")])
def test_streamed_decode_per_write_gates_and_ragged_passes(streams, W, R, idx):
    """The streaming kernel with per-write gates (G = W), 32-bit slots, and write / read passes whose
    last chunk is short (W or R not a multiple of the chunk height), against the oracle."""
    wl = workloads.DecodeWorkload("wide_gw", "f32", streams, 256, 400, W, R, W, 3, idx, 1 / 16, bank_std=0.5,
                                  seed=17)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, "f32", "readings")
    assert_close(to_np(x["bank"]), bank_ref, "f32", "bank")


@pytest.mark.parametrize("hd,idx", [(60, "i64"), (64, "i64"), (60, "i32")])
def test_streamed_decode_slot_widths(hd, idx):
    """The streaming kernel keeps 64-bit slots as 64-bit row indices for float32 rows of fewer than
    64 columns and as 32-bit ones from 64 columns on (and for 32-bit slots): rows of 60 and 64
    columns, W = 256, slots spread over the whole bank, against the oracle."""
    wl = workloads.DecodeWorkload("wide_slots", "f32", 12, hd, 2000, 256, 96, 256, 3, idx, 1 / 16, bank_std=0.5,
                                  seed=23)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, "f32", "readings")
    assert_close(to_np(x["bank"]), bank_ref, "f32", "bank")
    assert sdm.device_status() == 0


def test_concurrent_calls_on_two_streams_match_sequential():
    """The library keeps no state between calls: a decode of one bank and a gather of another,
    launched on two CUDA streams without synchronising between them, give the same bits as the same
    calls run one after the other."""
    wd = workloads.C2.scaled(n_streams=256, T=16)
    wg = workloads.C4.scaled(tokens=8192)
    xd = workloads.make_decode_inputs(wd, device=DEV)
    g = workloads.make_gather_inputs(wg, device=DEV)
    bank0 = xd["bank"].clone()
    ref_out = sdm.decode_seq(xd["bank"], *(xd[k] for k in DECODE_KEYS))
    ref_g, ref_stash = sdm.gather(g["bank"], g["ops"], chunk=wg.chunk, chunk_valid=g["chunk_valid"])
    torch.cuda.synchronize()
    ref_bank = xd["bank"].clone()
    xd["bank"].copy_(bank0)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)
    with torch.cuda.stream(s1):
        out = sdm.decode_seq(xd["bank"], *(xd[k] for k in DECODE_KEYS), stream=s1)
    with torch.cuda.stream(s2):
        outs, stash = sdm.gather(g["bank"], g["ops"], chunk=wg.chunk, chunk_valid=g["chunk_valid"], stream=s2)
    torch.cuda.synchronize()
    assert bits_equal(to_np(out), to_np(ref_out)) and bits_equal(to_np(xd["bank"]), to_np(ref_bank))
    assert all(bits_equal(to_np(a), to_np(b)) for a, b in zip(outs, ref_g))
    assert bits_equal(to_np(stash), to_np(ref_stash))


def test_streamed_bf16_four_stage_ring_matches_oracle():
    """bf16 wide rows in a large grid: 400 streams of 1 KiB rows with W = R = 256 stream through
    half-row slices (800 blocks) with 16-row chunks in a four-stage ring, on the column-pair
    streaming kernel; compared with the oracle on every stream."""
    wl = workloads.DecodeWorkload("wide_bf16_many", "bf16", 400, 512, 300, 256, 256, 1, 2, "i32", 1 / 16,
                                  bank_std=0.5, seed=17)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    out = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, "bf16", "readings")
    assert_close(to_np(x["bank"]), bank_ref, "bf16", "bank")
    assert sdm.device_status() == 0


def test_prompt_stream_major_matches_staged_and_oracle():
    """A prompt in the layer's own stream-major layout [S, T, .] (64 streams x 1024 tokens of the
    serving geometry): sdm_decode_seq_ex with SDM_STREAM_MAJOR gives, bit for bit, the readings
    and bank of sdm_decode_seq on the same arrays staged to time-major, and both equal the oracle."""
    wl = workloads.PROMPT
    x = workloads.make_decode_inputs(wl, device=DEV)  # time-major draw: the staged form
    bank0 = x["bank"].clone()
    xs = {k: x[k].transpose(0, 1).contiguous() for k in DECODE_KEYS}  # the stream-major layout
    out_sm = sdm.decode_seq(x["bank"], *(xs[k] for k in DECODE_KEYS), stream_major=True)
    assert out_sm.shape == (wl.n_streams, wl.T, wl.hd)
    bank_sm = x["bank"].clone()
    x["bank"].copy_(bank0)
    out_tm = sdm.decode_seq(x["bank"], *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert torch.equal(out_sm.transpose(0, 1).view(torch.int16), out_tm.view(torch.int16))
    assert torch.equal(bank_sm.view(torch.int16), x["bank"].view(torch.int16))
    bank_ref = to_np(bank0)
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS), check=False)
    assert_close(to_np(out_tm), ref, "bf16", "readings")
    assert_close(to_np(bank_sm), bank_ref, "bf16", "bank")
    assert sdm.device_status() == 0


@pytest.mark.parametrize("case", [SMALL[1], SMALL[2], SMALL[8]], ids=[IDS[1], IDS[2], IDS[8]])
def test_stream_major_small_paths(case):
    """The stream-major layout on the staged (sliced, per-write gates), plain-load and streamed
    kernel paths, with and without the inputs-ready promise, equal to the oracle."""
    wl = _wl(*case, seed=5)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank_ref, out_ref = _oracle_seq(x)
    bank0 = x["bank"].clone()
    xs = {k: x[k].transpose(0, 1).contiguous() for k in DECODE_KEYS}
    for ready in (False, True):
        x["bank"].copy_(bank0)
        out = sdm.decode_seq(x["bank"], *(xs[k] for k in DECODE_KEYS), stream_major=True, inputs_ready=ready)
        torch.cuda.synchronize()
        assert_close(to_np(out.transpose(0, 1).contiguous()), out_ref, wl.bank_dtype, f"readings (ready={ready})")
        assert_close(to_np(x["bank"]), bank_ref, wl.bank_dtype, f"bank (ready={ready})")
