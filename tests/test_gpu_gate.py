"""GPU pin of the decode's gates: d, the float32 nearest to e^g, bit for bit on every kernel path.

With a float32 bank of ones, beta = 0 and k_val = 0, the write reduces to bank[k_w] = 1 * d[w]
(retrieved and delta are zero), so the written rows read back the gates the kernel applied. They
must carry the bits of the float32 rounding of the double-precision exponential (torch's, on the
same device) for every input:
  - every float of four whole binades ([1, 2), [-2, -1), [-64, -32), [-2^-7, -2^-8));
  - seeded random values over [-87, 88] and log-uniform small magnitudes of both signs;
  - the edges of the table evaluation (|g| around 2^-30, -87, 88, the reduction's interval ends
    n ln2/64 and their midpoints) and the range the double-precision exponential takes alone
    (subnormal, zero and near-overflow results, -inf).
numpy's exponential must round the same way except where e^g lies within 2^-45 (relative) of a
float32 rounding midpoint, where two correct double-precision exponentials may round apart.
Paths: staged rows (16-byte float32 rows), plain loads (12-byte rows), streamed rows (1 KiB rows),
and the shared gate of G = 1 over several tokens (the rows then hold the running float32 product).
"""

from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from decode_state_gb300 import sdm
from parity import DECODE_KEYS, bits_equal, to_np

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0") if torch.cuda.is_available() else None
CHUNK = 1 << 22  # gates per launch


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_state_gb300 import build

    build.build()
    sdm.device_status(clear=True)
    yield
    assert sdm.device_status(clear=True) == 0


def _binade(lo_bits: int, hi_bits: int) -> np.ndarray:
    return np.arange(lo_bits, hi_bits, dtype=np.uint32).view(np.float32)


def _edges() -> np.ndarray:
    f = np.float32
    up = lambda x: np.nextafter(f(x), f(np.inf))  # noqa: E731
    dn = lambda x: np.nextafter(f(x), f(-np.inf))  # noqa: E731
    e = [0.0, -0.0, 2.0 ** -30, -(2.0 ** -30), dn(2.0 ** -30), up(-(2.0 ** -30)), 2.0 ** -24, -(2.0 ** -24),
         1e-45, -1e-45, 1e-38, -1e-38, 1.0, -1.0, 0.5, -0.5, -87.0, dn(-87.0), up(-87.0), 88.0, up(88.0), dn(88.0),
         88.5, 88.72, -87.5, -100.0, -103.97, -104.5, -110.0, -200.0, -1e30, -np.inf]
    step = math.log(2) / 64
    n = np.arange(-8200, 8200, dtype=np.float64)
    ends = np.concatenate([n * step, (n + 0.5) * step]).astype(np.float32)
    ends = ends[(ends >= -87.0) & (ends <= 88.0)]
    near = np.concatenate([ends, np.nextafter(ends, np.float32(np.inf)), np.nextafter(ends, np.float32(-np.inf))])
    return np.concatenate([np.asarray(e, dtype=np.float32), near])


def _gates(seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    mags = np.exp2(rng.uniform(-40, -5, 1 << 20)).astype(np.float32)
    return np.concatenate([
        _binade(0x3F800000, 0x40000000),  # [1, 2)
        _binade(0xBF800000, 0xC0000000),  # [-2, -1)
        _binade(0xC2000000, 0xC2800000),  # [-64, -32)
        _binade(0xBB800000, 0xBC000000),  # [-2^-7, -2^-8)
        rng.uniform(-87.0, 88.0, 1 << 22).astype(np.float32),
        mags, -mags, _edges(),
    ])


def _applied(g: torch.Tensor, hd: int, W: int) -> torch.Tensor:
    """The gates one single-token launch applies, one gate per write and W writes per stream."""
    n = g.numel()
    S = -(-n // W)
    gp = torch.zeros(S * W, dtype=torch.float32, device=DEV)
    gp[:n] = g
    bank = torch.ones((S * W, hd), dtype=torch.float32, device=DEV)
    rows = torch.arange(S * W, dtype=torch.int32, device=DEV).view(1, S, W)
    z = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=DEV)  # noqa: E731
    x = dict(k_idx=rows, k_val=z(1, S, W), v=z(1, S, hd), beta=z(1, S), g=gp.view(1, S, W),
             q_idx=rows[:, :, :1].contiguous(), q_val=z(1, S, 1))
    sdm.decode_seq(bank, *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    assert bits_equal(to_np(bank[:n]), to_np(bank[:n, :1].expand(n, hd)))  # every column the same
    return bank[:n, 0]


def _check(g_np: np.ndarray, got: np.ndarray):
    g = torch.from_numpy(g_np).to(DEV)
    expect = torch.exp(g.double()).float()
    assert bits_equal(got, to_np(expect)), f"{int((got.view(np.uint32) != to_np(expect).view(np.uint32)).sum())} gates"
    ref = np.exp(g_np.astype(np.float64))
    ref32 = ref.astype(np.float32)
    off = np.flatnonzero(ref32.view(np.uint32) != got.view(np.uint32))
    if off.size:
        lo = np.minimum(ref32[off], got[off]).astype(np.float64)
        hi = np.maximum(ref32[off], got[off]).astype(np.float64)
        mid = (lo + hi) / 2  # exact in float64
        assert off.size <= 8 and (np.abs(ref[off] - mid) <= mid * 2.0 ** -45).all(), (g_np[off], got[off], ref[off])


@pytest.mark.parametrize("path", [("staged", 4, 256), ("plain", 3, 64)], ids=["staged", "plain"])
def test_gates_are_the_nearest_float32(path):
    _, hd, W = path
    if hd == 4:
        g_all = _gates(31)
    else:  # a lighter set for the plain-load kernel
        rng = np.random.default_rng(32)
        g_all = np.concatenate([rng.uniform(-87.0, 88.0, 1 << 20).astype(np.float32),
                                _binade(0xBF800000, 0xC0000000)[::8], _edges()])
    got = np.empty_like(g_all)
    for lo in range(0, g_all.size, CHUNK):
        part = torch.from_numpy(g_all[lo:lo + CHUNK]).to(DEV)
        got[lo:lo + CHUNK] = to_np(_applied(part, hd, W))
    _check(g_all, got)


def test_gates_on_streamed_rows():
    rng = np.random.default_rng(33)
    g_all = np.concatenate([rng.uniform(-87.0, 88.0, 1 << 17).astype(np.float32), _edges()])
    got = to_np(_applied(torch.from_numpy(g_all).to(DEV), 256, 256))
    _check(g_all, got)


def test_shared_gate_over_tokens():
    """G = 1, T = 8: each token's shared gate (computed ahead by one thread) multiplies the rows."""
    T, S, W, hd = 8, 4096, 8, 4
    gen = torch.Generator(device=DEV)
    gen.manual_seed(34)
    g = torch.rand((T, S, 1), generator=gen, device=DEV) * 5.5 - 5.0
    bank = torch.ones((S * W, hd), dtype=torch.float32, device=DEV)
    rows = torch.arange(S * W, dtype=torch.int32, device=DEV).view(1, S, W).expand(T, S, W).contiguous()
    z = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=DEV)  # noqa: E731
    x = dict(k_idx=rows, k_val=z(T, S, W), v=z(T, S, hd), beta=z(T, S), g=g,
             q_idx=rows[:, :, :1].contiguous(), q_val=z(T, S, 1))
    sdm.decode_seq(bank, *(x[k] for k in DECODE_KEYS))
    torch.cuda.synchronize()
    d = torch.exp(g[:, :, 0].double()).float()  # [T, S]
    expect = torch.ones(S, dtype=torch.float32, device=DEV)
    for t in range(T):
        expect = expect * d[t]  # one float32 rounding per token, as the write does
    assert bits_equal(to_np(bank), to_np(expect.repeat_interleave(W).view(S * W, 1).expand(S * W, hd)))
