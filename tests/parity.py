"""Helpers for comparing the CUDA path with the oracle (bit views, tolerances, stream slicing).

Tolerances (stated once, used by every parity test):
  float32 banks and readings: |gpu - ref| <= 1e-5 * (1 + |ref|)
  bfloat16 banks and readings: at most 2 bf16 ulps apart (distance on the ordered bit line)
  gather outputs: bit-identical to the oracle's one-chain order; stash and padding bit-identical

The tolerance is the contract. The kernels also claim more: they take every rounding step of the
oracle in the oracle's order (the same fma chains over ascending entries, the same products
rounded first, gates that are the float32 nearest to e^g on both sides), so decode results are
also bit-identical to the oracle. assert_close checks the tolerance first and then, unless
exact=False, the bit identity, with messages that tell the two apart.
"""

from __future__ import annotations

import numpy as np
import torch

DECODE_KEYS = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")


def to_np(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy; bfloat16 becomes its uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def ordered_bf16(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def max_bf16_ulps(a: np.ndarray, b: np.ndarray) -> int:
    if a.size == 0:
        return 0
    return int(np.abs(ordered_bf16(a) - ordered_bf16(b)).max())


def max_f32_excess(a: np.ndarray, b: np.ndarray) -> float:
    """max of |a-b| - 1e-5 (1 + |b|); <= 0 means within tolerance."""
    if a.size == 0:
        return -1.0
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    return float((np.abs(a64 - b64) - 1e-5 * (1 + np.abs(b64))).max())


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str, exact: bool = True):
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    if dtype == "bf16":
        assert got.dtype == np.uint16
        d = max_bf16_ulps(got, ref)
        assert d <= 2, f"{what}: {d} bf16 ulps from the oracle (beyond the contract tolerance)"
    else:
        assert not np.isnan(got).any(), f"{what}: NaN"
        e = max_f32_excess(got, ref)
        assert e <= 0, f"{what}: exceeds 1e-5*(1+|ref|) by {e} (beyond the contract tolerance)"
    if exact and not bits_equal(got, ref):
        u = f"u{got.itemsize}"
        bad = np.flatnonzero(np.ascontiguousarray(got).reshape(-1).view(u) != np.ascontiguousarray(ref).reshape(-1).view(u))
        raise AssertionError(f"{what}: within the tolerance but not bit-identical to the oracle's operation "
                             f"order: {bad.size} of {got.size} elements differ, first at flat index {bad[0]}")


def bits_equal(a: np.ndarray, b: np.ndarray) -> bool:
    """Same shape and the same bytes (compared in 64 MiB pieces, so that multi-GiB banks need no
    temporary of their own size)."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.shape != b.shape or a.nbytes != b.nbytes:
        return False
    av, bv = a.reshape(-1).view(np.uint8), b.reshape(-1).view(np.uint8)
    step = 64 << 20
    return all(np.array_equal(av[i:i + step], bv[i:i + step]) for i in range(0, av.size, step))


def stream_slice(x: dict, s: int, P: int) -> dict:
    """Host copies of stream s's inputs (time-major, one stream) with slots rebased to its own
    bank rows [s*P, (s+1)*P), plus that bank slice."""
    out = {}
    for k in DECODE_KEYS:
        v = x[k][:, s:s + 1]
        if k in ("k_idx", "q_idx"):
            v = v - s * P
        out[k] = to_np(v)
    out["bank"] = to_np(x["bank"][s * P:(s + 1) * P])
    return out
