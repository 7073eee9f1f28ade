"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
entry point include/sdm.h declares, and rejects bad arguments with the documented negative codes
before touching CUDA. Every call here fails validation, so nothing is ever launched."""

from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

from decode_state_gb300 import build, sdm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdm.h")


def _codes():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (SDM_E\w+) \((-\d+)\)", text)}


CODES = _codes()


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sdm.library()


def test_header_declares_the_entry_points():
    text = open(HEADER).read()
    declared = set(re.findall(r"^(?:int|const char\*) (sdm_\w+)\(", text, flags=re.M))
    assert declared == set(sdm.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(lib):
    for name in sdm.ENTRY_POINTS:
        assert hasattr(lib, name), name
    assert sdm.version() == 200


def test_status_strings(lib):
    for name, code in CODES.items():
        s = sdm.status_string(code)
        assert s and s != "unknown status", name
    assert sdm.status_string(0) == "ok"


FAKE = 0x10000000  # never dereferenced: every call below fails validation first


def _decode(lib, **kw):
    a = dict(bank=FAKE, k_idx=FAKE, k_val=FAKE, v=FAKE, beta=FAKE, g=FAKE, q_idx=FAKE, q_val=FAKE, out=FAKE + 4096,
             n_streams=4, hd=64, W=8, R=8, G=1, T=2, bank_dtype=0, idx_dtype=0)
    a.update(kw)
    return lib.sdm_decode_seq(a["bank"], a["k_idx"], a["k_val"], a["v"], a["beta"], a["g"], a["q_idx"], a["q_val"],
                              a["out"], a["n_streams"], a["hd"], a["W"], a["R"], a["G"], a["T"], a["bank_dtype"],
                              a["idx_dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(bank_dtype=2), "SDM_EDTYPE"), (dict(idx_dtype=5), "SDM_EIDX"), (dict(hd=0), "SDM_EHD"),
    (dict(hd=70000), "SDM_EHD"), (dict(W=0), "SDM_EWIDTH"), (dict(W=257), "SDM_EWIDTH"), (dict(R=0), "SDM_EWIDTH"),
    (dict(R=300), "SDM_EWIDTH"), (dict(G=3), "SDM_EGATES"), (dict(W=4, G=8), "SDM_EGATES"),
    (dict(n_streams=-1), "SDM_ECOUNT"), (dict(T=-2), "SDM_ECOUNT"), (dict(bank=0), "SDM_ENULL"),
    (dict(q_val=0), "SDM_ENULL"), (dict(out=0), "SDM_ENULL"), (dict(bank=FAKE + 1), "SDM_EALIGN"),
    (dict(bank=FAKE + 2, bank_dtype=1), "SDM_EALIGN"), (dict(k_idx=FAKE + 4, idx_dtype=1), "SDM_EALIGN"),
    (dict(v=FAKE + 2), "SDM_EALIGN"),
])
def test_decode_argument_errors(lib, kw, code):
    assert _decode(lib, **kw) == CODES[code]


def test_decode_step_ex_flags(lib):
    """Unknown flag bits are refused before anything else; the known flag validates like the step."""
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 8, 1, 0, 0)
    assert lib.sdm_decode_step_ex(*args, 2, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_decode_step_ex(*args, 0x80000000, None) == CODES["SDM_EFLAGS"]
    bad = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 0, 8, 1, 0, 0)
    assert lib.sdm_decode_step_ex(*bad, sdm.SDM_INPUTS_READY, None) == CODES["SDM_EWIDTH"]
    assert lib.sdm_decode_step_ex(*args[:9], 0, *args[10:], sdm.SDM_INPUTS_READY, None) == 0  # no streams


def test_decode_seq_ex_flags(lib):
    """Unknown flag bits are refused first; the stream-major layout and the inputs-ready promise
    validate like sdm_decode_seq."""
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 8, 8, 1, 3, 0, 0)
    assert lib.sdm_decode_seq_ex(*args, 4, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_decode_seq_ex(*args, sdm.SDM_STREAM_MAJOR | 8, None) == CODES["SDM_EFLAGS"]
    bad = args[:11] + (257,) + args[12:]
    for flags in (0, sdm.SDM_STREAM_MAJOR, sdm.SDM_INPUTS_READY, sdm.SDM_STREAM_MAJOR | sdm.SDM_INPUTS_READY):
        assert lib.sdm_decode_seq_ex(*bad, flags, None) == CODES["SDM_EWIDTH"]
        assert lib.sdm_decode_seq_ex(*args[:9], 0, *args[10:], flags, None) == 0  # no streams
        assert lib.sdm_decode_seq_ex(*args[:14], 0, *args[15:], flags, None) == 0  # no tokens


def test_decode_step_validates_like_seq(lib):
    assert lib.sdm_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 0, 8, 1, 0, 0,
                               None) == CODES["SDM_EWIDTH"]


def test_decode_empty_is_ok_without_pointers(lib):
    assert _decode(lib, n_streams=0, bank=0, out=0) == 0
    assert _decode(lib, T=0, bank=0, out=0) == 0


def _gather(lib, **kw):
    a = dict(bank=FAKE, n_slots=1000, hd=64, bank_dtype=0, n_ops=2, idx=(FAKE + (1 << 24), FAKE + (2 << 24)),
             w=(FAKE + (3 << 24), FAKE + (4 << 24)), out=(FAKE + (5 << 24), FAKE + (6 << 24)), width=(8, 4),
             idx_dtype=1, w_dtype=0, stash=FAKE + (8 << 24), tokens=64, chunk=16, valid=16, chunk_valid=None)
    a.update(kw)
    vp = ctypes.c_void_p
    idx = (vp * 2)(*a["idx"])
    w = (vp * 2)(*a["w"])
    out = (vp * 2)(*a["out"])
    width = (ctypes.c_int * 2)(*a["width"])
    return lib.sdm_gather(a["bank"], a["n_slots"], a["hd"], a["bank_dtype"], a["n_ops"], idx, w, out, width,
                          a["idx_dtype"], a["w_dtype"], a["stash"], a["tokens"], a["chunk"], a["valid"],
                          a["chunk_valid"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(bank_dtype=7), "SDM_EDTYPE"), (dict(w_dtype=3), "SDM_EDTYPE"), (dict(idx_dtype=-1), "SDM_EIDX"),
    (dict(hd=0), "SDM_EHD"), (dict(n_ops=0), "SDM_ENOPS"), (dict(n_ops=3), "SDM_ENOPS"),
    (dict(width=(0, 4)), "SDM_EWIDTH"), (dict(width=(8, 257)), "SDM_EWIDTH"), (dict(n_slots=0), "SDM_ECOUNT"),
    (dict(n_slots=1 << 31), "SDM_ECOUNT"), (dict(tokens=-16), "SDM_ECOUNT"), (dict(chunk=0), "SDM_ECHUNK"),
    (dict(tokens=60), "SDM_ECHUNK"), (dict(valid=17), "SDM_ECHUNK"), (dict(valid=-1), "SDM_ECHUNK"),
    (dict(bank=0), "SDM_ENULL"), (dict(idx=(0, FAKE)), "SDM_ENULL"), (dict(out=(FAKE, 0)), "SDM_ENULL"),
    (dict(bank=FAKE + 1), "SDM_EALIGN"), (dict(stash=FAKE + 1), "SDM_EALIGN"),
    (dict(idx=(FAKE + 4, FAKE), idx_dtype=1), "SDM_EALIGN"), (dict(w=(FAKE + 1, FAKE)), "SDM_EALIGN"),
    (dict(out=(FAKE + 64, FAKE + (6 << 24))), "SDM_EOVERLAP"), (dict(stash=FAKE + 128), "SDM_EOVERLAP"),
])
def test_gather_argument_errors(lib, kw, code):
    assert _gather(lib, **kw) == CODES[code]


def test_gather_second_operand_ignored_for_one_op(lib):
    # with one operand, a NULL second operand is fine: the failure comes from the bad chunk
    assert _gather(lib, n_ops=1, idx=(FAKE, 0), w=(FAKE, 0), out=(FAKE + (5 << 24), 0), chunk=0) == CODES["SDM_ECHUNK"]


def test_gather_empty_is_ok(lib):
    assert _gather(lib, tokens=0, bank=0) == 0


def test_binding_rejects_host_tensors():
    bank = torch.zeros((16, 8))
    k = torch.zeros((2, 3), dtype=torch.int32)
    f = torch.zeros((2, 3))
    with pytest.raises(ValueError):
        sdm.decode_step(bank, k, f, torch.zeros((2, 8)), torch.zeros(2), torch.zeros((2, 1)), k, f)


def test_binding_rejects_bad_dtypes():
    with pytest.raises(TypeError):
        sdm.decode_step(torch.zeros((4, 4), dtype=torch.float16), *([torch.zeros(1)] * 7))


def _gather_kpos(lib, **kw):
    a = dict(bank=FAKE, n_slots=1000, hd=64, bank_dtype=0, n_ops=1, idx=(FAKE + (1 << 24), 0),
             w=(FAKE + (3 << 24), 0), out=(FAKE + (5 << 24), 0), width=(8, 0), idx_dtype=1, w_dtype=0,
             compact=FAKE + (8 << 24), kpos=FAKE + (9 << 24), tokens=64, chunk=16, valid=16, chunk_valid=None)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.sdm_gather_kpos(a["bank"], a["n_slots"], a["hd"], a["bank_dtype"], a["n_ops"], (vp * 2)(*a["idx"]),
                               (vp * 2)(*a["w"]), (vp * 2)(*a["out"]), (ctypes.c_int * 2)(*a["width"]),
                               a["idx_dtype"], a["w_dtype"], a["compact"], a["kpos"], a["tokens"], a["chunk"],
                               a["valid"], a["chunk_valid"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(compact=0), "SDM_ENULL"), (dict(kpos=0), "SDM_ENULL"), (dict(kpos=FAKE + (9 << 24) + 2), "SDM_EALIGN"),
    (dict(compact=FAKE + 64), "SDM_EOVERLAP"), (dict(chunk=5), "SDM_ECHUNK"), (dict(width=(300, 0)), "SDM_EWIDTH"),
])
def test_gather_kpos_argument_errors(lib, kw, code):
    assert _gather_kpos(lib, **kw) == CODES[code]


def _plan_init(lib, record, **kw):
    a = dict(bank=FAKE, n_slots=1000, hd=64, bank_dtype=0, n_ops=1, idx=(FAKE + (1 << 24), 0),
             w=(FAKE + (3 << 24), 0), out=(FAKE + (5 << 24), 0), width=(8, 0), idx_dtype=1, w_dtype=0, rows=256,
             row0_max=192, tokens=64, chunk=16)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.sdm_gather_plan_init(record, a["bank"], a["n_slots"], a["hd"], a["bank_dtype"], a["n_ops"],
                                    (vp * 2)(*a["idx"]), (vp * 2)(*a["w"]), (vp * 2)(*a["out"]),
                                    (ctypes.c_int * 2)(*a["width"]), a["idx_dtype"], a["w_dtype"], a["rows"],
                                    a["row0_max"], a["tokens"], a["chunk"])


def test_plan_record_size_matches_header():
    text = open(HEADER).read()
    assert int(re.search(r"#define SDM_GATHER_PLAN_BYTES (\d+)", text).group(1)) == sdm.GATHER_PLAN_BYTES


@pytest.mark.parametrize("kw,code", [
    (dict(row0_max=-1), "SDM_EROW"), (dict(row0_max=193), "SDM_EROW"), (dict(rows=63, row0_max=0), "SDM_EROW"),
    (dict(chunk=5), "SDM_ECHUNK"), (dict(width=(0, 0)), "SDM_EWIDTH"), (dict(n_ops=3), "SDM_ENOPS"),
    (dict(idx=(0, 0)), "SDM_ENULL"), (dict(out=(FAKE + 64, 0)), "SDM_EOVERLAP"), (dict(bank_dtype=4), "SDM_EDTYPE"),
])
def test_gather_plan_init_argument_errors(lib, kw, code):
    record = ctypes.create_string_buffer(sdm.GATHER_PLAN_BYTES)
    assert _plan_init(lib, record, **kw) == CODES[code]
    assert record.raw == bytes(sdm.GATHER_PLAN_BYTES)  # nothing written on an error


def test_gather_plan_init_null_record(lib):
    assert _plan_init(lib, None) == CODES["SDM_ENULL"]


def test_gather_plan_launch_ex_flags(lib):
    """Unknown flag bits are refused before the record is looked at; the known flag checks as usual."""
    zero = ctypes.create_string_buffer(sdm.GATHER_PLAN_BYTES)
    assert lib.sdm_gather_plan_launch_ex(None, 0, 16, 4, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_gather_plan_launch_ex(zero, 0, 16, 3, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_gather_plan_launch_ex(None, 0, 16, sdm.SDM_INPUTS_READY, None) == CODES["SDM_ENULL"]
    assert lib.sdm_gather_plan_launch_ex(zero, 0, 16, sdm.SDM_INPUTS_READY, None) == CODES["SDM_EPLAN"]


def test_decode_plan_argument_errors(lib):
    """The decode-step plan refuses unknown flags, a NULL record, a negative count and a foreign
    record before launching anything; init checks its arguments like sdm_decode_seq."""
    zero = ctypes.create_string_buffer(sdm.DECODE_PLAN_BYTES)
    assert lib.sdm_decode_plan_walk(zero, 0, 1, 4, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_decode_plan_launch(zero, 0, 2, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_decode_plan_walk(None, 0, 1, 0, None) == CODES["SDM_ENULL"]
    assert lib.sdm_decode_plan_walk(zero, 0, -1, 0, None) == CODES["SDM_ECOUNT"]
    assert lib.sdm_decode_plan_walk(zero, 0, 1, sdm.SDM_INPUTS_READY, None) == CODES["SDM_EPLAN"]
    assert lib.sdm_decode_plan_launch(zero, 0, 0, None) == CODES["SDM_EPLAN"]
    junk = ctypes.create_string_buffer(bytes(range(256)) * 2)
    assert lib.sdm_decode_plan_launch(junk, 0, 0, None) == CODES["SDM_EPLAN"]
    record = ctypes.create_string_buffer(sdm.DECODE_PLAN_BYTES)
    p = [FAKE] * 9
    assert lib.sdm_decode_plan_init(None, *p, 4, 64, 8, 8, 1, 2, 0, 0) == CODES["SDM_ENULL"]
    assert lib.sdm_decode_plan_init(record, *p, 4, 64, 8, 8, 3, 2, 0, 0) == CODES["SDM_EGATES"]
    assert lib.sdm_decode_plan_init(record, *p, 4, 64, 0, 8, 1, 2, 0, 0) == CODES["SDM_EWIDTH"]
    assert lib.sdm_decode_plan_init(record, *p, 4, 64, 8, 8, 1, 2, 7, 0) == CODES["SDM_EDTYPE"]
    assert record.raw == bytes(sdm.DECODE_PLAN_BYTES)  # nothing written on an error


def test_gather_plan_walk_argument_errors(lib):
    """The walk refuses unknown flags, a NULL record or row list, a negative count and a foreign
    record before launching anything."""
    zero = ctypes.create_string_buffer(sdm.GATHER_PLAN_BYTES)
    rows = (ctypes.c_int64 * 2)(0, 1)
    assert lib.sdm_gather_plan_walk(zero, rows, None, 2, 4, None) == CODES["SDM_EFLAGS"]
    assert lib.sdm_gather_plan_walk(None, rows, None, 2, 0, None) == CODES["SDM_ENULL"]
    assert lib.sdm_gather_plan_walk(zero, None, None, 2, 0, None) == CODES["SDM_ENULL"]
    assert lib.sdm_gather_plan_walk(zero, rows, None, -1, 0, None) == CODES["SDM_ECOUNT"]
    assert lib.sdm_gather_plan_walk(zero, rows, None, 2, sdm.SDM_INPUTS_READY, None) == CODES["SDM_EPLAN"]
    assert lib.sdm_gather_plan_walk(zero, None, None, 0, 0, None) == CODES["SDM_EPLAN"]


def test_gather_plan_launch_refuses_a_foreign_record(lib):
    zero = ctypes.create_string_buffer(sdm.GATHER_PLAN_BYTES)
    assert lib.sdm_gather_plan_launch(zero, 0, 16, None) == CODES["SDM_EPLAN"]
    junk = ctypes.create_string_buffer(bytes(range(256)) * 2)
    assert lib.sdm_gather_plan_launch(junk, 0, 16, None) == CODES["SDM_EPLAN"]
    assert lib.sdm_gather_plan_launch(None, 0, 16, None) == CODES["SDM_ENULL"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_gather_plan_init_without_a_device_reports_the_cuda_error(lib):
    record = ctypes.create_string_buffer(sdm.GATHER_PLAN_BYTES)
    rc = _plan_init(lib, record)
    assert rc > 0 and sdm.status_string(rc)
    assert record.raw == bytes(sdm.GATHER_PLAN_BYTES)
