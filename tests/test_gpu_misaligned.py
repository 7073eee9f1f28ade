"""GPU parity when the bank or the outputs start off a 16-byte boundary.

The ABI only requires element alignment; the 16-byte copy paths need 16-byte aligned rows, so the
launcher must fall back to the plain-load kernels. These cases take views one element into a
larger buffer (contiguous, element-aligned, not 16-byte aligned) and compare with the oracle.
"""

from __future__ import annotations

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
    assert sdm.device_status(clear=True) == 0


def _shifted(t: torch.Tensor) -> torch.Tensor:
    """A copy of t that starts one element into a fresh buffer (contiguous, not 16-byte aligned)."""
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
    view = flat[1:].view(t.shape)
    view.copy_(t)
    assert view.is_contiguous() and view.data_ptr() % 16 != 0
    return view


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_decode_on_a_misaligned_bank_and_output(dt):
    wl = workloads.DecodeWorkload("misaligned", dt, 12, 128, 80, 10, 7, 1, 3, "i32", 0.35, bank_std=0.5, seed=21)
    x = workloads.make_decode_inputs(wl, device=DEV)
    bank = _shifted(x["bank"])
    out = _shifted(torch.zeros((wl.T, wl.n_streams, wl.hd), dtype=bank.dtype, device=DEV))
    bank_ref = to_np(x["bank"])
    ref = oracle.decode_seq(bank_ref, *(to_np(x[k]) for k in DECODE_KEYS))
    sdm.decode_seq(bank, *(x[k] for k in DECODE_KEYS), out=out)
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, dt, "readings")
    assert_close(to_np(bank), bank_ref, dt, "bank")


def test_gather_on_a_misaligned_bank_and_stash():
    wl = workloads.GatherWorkload("misaligned", "bf16", 900, 128, 48, 16, (20, 9), "i64", "bf16", 0.125, seed=22)
    g = workloads.make_gather_inputs(wl, device=DEV)
    bank = _shifted(g["bank"])
    stash = _shifted(torch.zeros((wl.tokens, wl.widths[0], wl.hd), dtype=bank.dtype, device=DEV))
    outs, _ = sdm.gather(bank, g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], stash=stash)
    torch.cuda.synchronize()
    (i0, w0), (i1, w1) = g["ops"]
    r0, r1, rs = oracle.gather(to_np(g["bank"]), to_np(i0), to_np(w0), to_np(i1), to_np(w1), chunk=wl.chunk,
                               chunk_valid=to_np(g["chunk_valid"]))
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1)
    assert bits_equal(to_np(stash), rs)


@pytest.mark.parametrize("wdt", ["bf16", "f32"])
def test_gather_aligned_bank_misaligned_stash_and_outputs(wdt):
    """An aligned bank keeps the 16-byte row copies (and the 128-column instance) while the stash and
    the outputs start off a 16-byte boundary: the stash leaves shared memory column by column
    instead of as one bulk store, and padding tokens zero it the same way; with bf16 weights the
    column-pair sums meet outputs 4 bytes off an 8-byte boundary and store one float at a time."""
    wl = workloads.GatherWorkload("misaligned_stash", "bf16", 900, 128, 48, 16, (20, 9), "i64", wdt, 0.125, seed=23)
    g = workloads.make_gather_inputs(wl, device=DEV)
    stash = _shifted(torch.full((wl.tokens, wl.widths[0], wl.hd), 3.0, dtype=g["bank"].dtype, device=DEV))
    outs = [_shifted(torch.full((wl.tokens, wl.hd), 5.0, device=DEV)) for _ in range(2)]
    assert g["bank"].data_ptr() % 16 == 0
    sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], stash=stash, outs=outs)
    torch.cuda.synchronize()
    (i0, w0), (i1, w1) = g["ops"]
    r0, r1, rs = oracle.gather(to_np(g["bank"]), to_np(i0), to_np(w0), to_np(i1), to_np(w1), chunk=wl.chunk,
                               chunk_valid=to_np(g["chunk_valid"]))
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1)
    assert bits_equal(to_np(stash), rs)
