"""GPU parity at the size limits of the C ABI: slot indices at and past 2^31 (64-bit row offsets in
every kernel path), the largest gather bank (n_slots = 2^31 - 1) and the largest head dimension
(65536 elements per row).

The GPU runs on the real bank: 2^31 + 1024 rows of 16 bytes (32 GiB). The oracle runs on a compact
bank holding only the rows the calls touch, with the indices remapped onto it; the arithmetic is the
same, so the usual tolerances apply. Guard rows around every touched range are checked to be left
untouched.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from decode_state_gb300 import sdm
from parity import assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
BIG_ROWS = (1 << 31) + 1024
GUARD = 16


@pytest.fixture(scope="module")
def big_bank():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    bank = torch.empty((BIG_ROWS, 8), dtype=torch.bfloat16, device=DEV)
    yield bank
    del bank
    torch.cuda.empty_cache()


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _fill(bank, lo, hi, gen):
    bank[lo:hi] = (torch.randn((hi - lo, bank.shape[1]), generator=gen, device=DEV) * 0.5).to(bank.dtype)


def _decode_inputs(S, P, hd, W, R, G, T, bases, gen, idx_dtype):
    """Time-major decode inputs for S streams whose slots are [bases[s], bases[s] + P)."""
    f32 = torch.float32
    base = torch.tensor(bases, dtype=torch.int64, device=DEV).view(1, S, 1)
    k_idx = torch.stack([torch.stack([torch.randperm(P, generator=gen, device=DEV)[:W] for _ in range(S)])
                         for _ in range(T)]) + base
    q_idx = torch.randint(0, P, (T, S, R), generator=gen, device=DEV) + base
    x = dict(k_idx=k_idx.to(idx_dtype), k_val=torch.randn((T, S, W), generator=gen, device=DEV) * 0.35,
             v=torch.randn((T, S, hd), generator=gen, device=DEV),
             beta=torch.sigmoid(torch.randn((T, S), generator=gen, device=DEV)),
             g=-torch.nn.functional.softplus(torch.randn((T, S, G), generator=gen, device=DEV)),
             q_idx=q_idx.to(idx_dtype), q_val=torch.randn((T, S, R), generator=gen, device=DEV) * 0.35)
    assert all(t.dtype in (f32, idx_dtype) for t in x.values())
    return x


KEYS = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")


def _check_decode_on_compact(bank, x, bases, P, dtype):
    """Run the decode on `bank` and the oracle on a compact copy of the streams' slot ranges."""
    S = len(bases)
    compact = np.concatenate([to_np(bank[b:b + P]) for b in bases])
    shift = torch.tensor([b - s * P for s, b in enumerate(bases)], dtype=torch.int64, device=DEV).view(1, S, 1)
    guards = [(to_np(bank[b - GUARD:b]), to_np(bank[b + P:b + P + GUARD])) for b in bases]
    ref = oracle.decode_seq(compact, to_np((x["k_idx"].to(torch.int64) - shift).to(torch.int64)),
                            to_np(x["k_val"]), to_np(x["v"]), to_np(x["beta"]), to_np(x["g"]),
                            to_np((x["q_idx"].to(torch.int64) - shift).to(torch.int64)), to_np(x["q_val"]))
    out = sdm.decode_seq(bank, *(x[k] for k in KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, dtype, "readings")
    got = np.concatenate([to_np(bank[b:b + P]) for b in bases])
    assert_close(got, compact, dtype, "touched rows")
    for b, (lo, hi) in zip(bases, guards):
        assert bits_equal(to_np(bank[b - GUARD:b]), lo) and bits_equal(to_np(bank[b + P:b + P + GUARD]), hi)
    assert sdm.device_status() == 0


def test_decode_slots_past_2_31(big_bank):
    """int64 slots on both sides of 2^31: the top of the int32 range and past it."""
    P, gen = 256, _gen(1)
    bases = [(1 << 31) - P - GUARD, (1 << 31) + 256]
    for b in bases:
        _fill(big_bank, b - GUARD, b + P + GUARD, gen)
    x = _decode_inputs(2, P, 8, 24, 20, 1, 3, bases, gen, torch.int64)
    _check_decode_on_compact(big_bank, x, bases, P, "bf16")


def test_decode_int32_slots_at_the_top(big_bank):
    """int32 slots up to 2^31 - 1, the largest the index type holds (the byte offset needs 64 bits)."""
    P, gen = 128, _gen(2)
    bases = [(1 << 31) - P, (1 << 31) - 4 * P]
    for b in bases:
        _fill(big_bank, b - GUARD, min(b + P + GUARD, BIG_ROWS), gen)
    x = _decode_inputs(2, P, 8, 16, 16, 16, 2, bases, gen, torch.int32)
    _check_decode_on_compact(big_bank, x, bases, P, "bf16")


def test_gather_largest_bank(big_bank):
    """n_slots = 2^31 - 1 (the largest the ABI takes); rows drawn near the top of the bank."""
    n_slots, gen = (1 << 31) - 1, _gen(3)
    bank = big_bank[:n_slots]
    lo = n_slots - 4096
    _fill(big_bank, lo, n_slots, gen)
    tokens, chunk = 24, 8
    ops = [(torch.randint(lo, n_slots, (tokens, w), generator=gen, device=DEV),
            (torch.randn((tokens, w), generator=gen, device=DEV) * 0.25).to(torch.bfloat16)) for w in (12, 5)]
    cv = torch.tensor([8, 3, 6], dtype=torch.int32, device=DEV)
    outs, stash = sdm.gather(bank, ops, chunk=chunk, chunk_valid=cv)
    torch.cuda.synchronize()
    compact = to_np(big_bank[lo:n_slots])
    r0, r1, rs = oracle.gather(compact, to_np(ops[0][0] - lo), to_np(ops[0][1]), to_np(ops[1][0] - lo),
                               to_np(ops[1][1]), chunk=chunk, chunk_valid=to_np(cv))
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1)
    assert bits_equal(to_np(stash), rs)
    assert sdm.device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_largest_head_dim(dtype):
    """hd = 65536 (the ABI's limit): rows of 128 or 256 KiB, cut into many column slices."""
    from decode_state_gb300 import build

    build.build()
    gen, hd, S, P = _gen(4), 65536, 2, 6
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    bank = (torch.randn((S * P, hd), generator=gen, device=DEV) * 0.5).to(tdt)
    x = _decode_inputs(S, P, hd, 3, 4, 3, 2, [0, P], gen, torch.int32)
    ref_bank = to_np(bank)
    ref = oracle.decode_seq(ref_bank, *(to_np(x[k]) for k in KEYS))
    out = sdm.decode_seq(bank, *(x[k] for k in KEYS))
    torch.cuda.synchronize()
    assert_close(to_np(out), ref, dtype, "readings")
    assert_close(to_np(bank), ref_bank, dtype, "bank")


def test_gather_largest_head_dim():
    gen, hd, n_slots = _gen(5), 65536, 40
    bank = (torch.randn((n_slots, hd), generator=gen, device=DEV)).to(torch.bfloat16)
    ops = [(torch.randint(0, n_slots, (8, w), generator=gen, device=DEV, dtype=torch.int64).to(torch.int32),
            torch.randn((8, w), generator=gen, device=DEV) * 0.25) for w in (3, 2)]
    outs, stash = sdm.gather(bank, ops, chunk=4, valid=3)
    torch.cuda.synchronize()
    r0, r1, rs = oracle.gather(to_np(bank), to_np(ops[0][0]), to_np(ops[0][1]), to_np(ops[1][0]), to_np(ops[1][1]),
                               chunk=4, valid=3)
    assert bits_equal(to_np(outs[0]), r0) and bits_equal(to_np(outs[1]), r1)
    assert bits_equal(to_np(stash), rs)
