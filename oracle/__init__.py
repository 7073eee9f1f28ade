"""CPU oracle for the SDM decode step, multi-token decode and token gather (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use this package.
It wraps ``sdm_oracle.c`` (plain C, built with gcc) through ctypes and works on numpy arrays:
bfloat16 data travels as raw ``uint16`` bits. It shares nothing with the CUDA library.

The arithmetic it follows is described at the top of ``sdm_oracle.c`` (decode.py's
``sdm_decode_step`` docstring and kernel; gather_cuda.py's module docstring and kernel).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "sdm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

BF16, F32 = 0, 1
I32, I64 = 0, 1

OK, EARG, EDUP, ERANGE, ENOMEM = 0, -1, -2, -3, -4


class OracleError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"{fn} returned {rc}")
        self.rc = rc


def build_command(src: str = SOURCE, out: str = _LIB_PATH) -> list[str]:
    """gcc command that builds the oracle library; -ffp-contract=off keeps every product unfused."""
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
            "-Wall", "-Wextra", "-o", out, src, "-lm"]


def build(force: bool = False) -> str:
    """Compile the oracle if needed and return the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(build_command(SOURCE, tmp), check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _sentinel(shape, dtype) -> np.ndarray:
    """Output buffer filled with all-ones bits (a NaN pattern), so every element must be written."""
    a = np.empty(shape, dtype=dtype)
    a.view(np.uint8).fill(0xFF)
    return a


def _bank_code(bank: np.ndarray) -> int:
    if bank.dtype == np.uint16:
        return BF16
    if bank.dtype == np.float32:
        return F32
    raise TypeError(f"bank must be uint16 (bf16 bits) or float32, got {bank.dtype}")


def _idx_code(idx: np.ndarray) -> int:
    if idx.dtype == np.int32:
        return I32
    if idx.dtype == np.int64:
        return I64
    raise TypeError(f"indices must be int32 or int64, got {idx.dtype}")


class Oracle:
    """One loaded copy of the oracle library (the default one, or a test's own build)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_sdm_decode_seq.argtypes = [vp, i32, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                              i64, i32, i32, i32, i32, i64, i32]
        lib.oracle_sdm_decode_seq.restype = i32
        lib.oracle_sdm_gather.argtypes = [vp, i32, i64, i64, i32, vp, vp, vp, i32, vp, vp, vp, i32,
                                          i32, i32, vp, i64, i32, i32, vp, i32, i32]
        lib.oracle_sdm_gather.restype = i32
        lib.oracle_sdm_gather_kpos.argtypes = [vp, i32, i64, i64, vp, i32, i32, vp, vp, i64, i32, i32, vp, i32]
        lib.oracle_sdm_gather_kpos.restype = i32
        lib.oracle_f32_to_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_f32_to_bf16_array.restype = None
        lib.oracle_bf16_to_f32_array.argtypes = [vp, vp, i64]
        lib.oracle_bf16_to_f32_array.restype = None
        self.lib = lib
        self.path = lib_path

    def decode_seq(self, bank, k_idx, k_val, v, beta, g, q_idx, q_val, *, check: bool = True) -> np.ndarray:
        """Run T tokens for every stream, in place on ``bank``; returns readings [T, S, hd].

        Per-token arrays are time-major: k_idx/k_val [T, S, W], v [T, S, hd], beta [T, S] (or
        [T, S, 1]), g [T, S, G], q_idx/q_val [T, S, R]; k_val, v, q_val, beta, g are float32.
        """
        if not bank.flags["C_CONTIGUOUS"]:
            raise ValueError("bank must be C-contiguous (it is updated in place)")
        T, S, W = k_idx.shape
        R = q_idx.shape[-1]
        G = g.shape[-1]
        n_slots, hd = bank.shape
        out = _sentinel((T, S, hd), bank.dtype)
        k_idx, k_val, v, beta, g, q_idx, q_val = (np.ascontiguousarray(x) for x in
                                                  (k_idx, k_val, v, beta, g, q_idx, q_val))
        for x in (k_val, v, beta, g, q_val):
            if x.dtype != np.float32:
                raise TypeError("k_val, v, beta, g, q_val must be float32")
        if k_idx.dtype != q_idx.dtype:
            raise TypeError("k_idx and q_idx must share one dtype")
        rc = self.lib.oracle_sdm_decode_seq(_ptr(bank), _bank_code(bank), n_slots, hd, _ptr(k_idx), _ptr(k_val),
                                            _ptr(v), _ptr(beta), _ptr(g), _ptr(q_idx), _ptr(q_val), _ptr(out), S, W,
                                            R, G, _idx_code(k_idx), T, 1 if check else 0)
        if rc != OK:
            raise OracleError("oracle_sdm_decode_seq", rc)
        return out

    def decode_step(self, bank, k_idx, k_val, v, beta, g, q_idx, q_val, *, check: bool = True) -> np.ndarray:
        """One token for every stream (arrays [S, .]); returns readings [S, hd]."""
        return self.decode_seq(bank, k_idx[None], k_val[None], v[None], np.asarray(beta)[None], g[None],
                               q_idx[None], q_val[None], check=check)[0]

    def gather(self, bank, idx0, w0, idx1=None, w1=None, *, chunk: int, valid: int = -1, chunk_valid=None,
               stash: bool = True, groups: int = 1, check: bool = True):
        """Token gather. Returns (out0, out1 or None, stash or None).

        bank [n_slots, hd] uint16 (bf16 bits) or float32; idx_o [tokens, width_o]; w_o like idx_o,
        uint16 (bf16 bits) or float32. ``valid`` is the scalar count (default: chunk), or
        ``chunk_valid`` [tokens / chunk] int32 gives one count per chunk.
        """
        n_slots, hd = bank.shape
        tokens, width0 = idx0.shape
        n_ops = 1 if idx1 is None else 2
        width1 = idx1.shape[1] if n_ops == 2 else 0
        if valid < 0:
            valid = chunk
        wd = BF16 if w0.dtype == np.uint16 else F32
        out0 = _sentinel((tokens, hd), np.float32)
        out1 = _sentinel((tokens, hd), np.float32) if n_ops == 2 else None
        st = _sentinel((tokens, width0, hd), bank.dtype) if stash else None
        cv = None if chunk_valid is None else np.ascontiguousarray(chunk_valid, dtype=np.int32)
        bank = np.ascontiguousarray(bank)
        idx0, w0 = np.ascontiguousarray(idx0), np.ascontiguousarray(w0)
        if n_ops == 2:
            idx1, w1 = np.ascontiguousarray(idx1), np.ascontiguousarray(w1)
        rc = self.lib.oracle_sdm_gather(_ptr(bank), _bank_code(bank), n_slots, hd, n_ops, _ptr(idx0), _ptr(w0),
                                        _ptr(out0), width0, _ptr(idx1), _ptr(w1), _ptr(out1), width1,
                                        _idx_code(idx0), wd, _ptr(st), tokens, chunk, valid, _ptr(cv), groups,
                                        1 if check else 0)
        if rc != OK:
            raise OracleError("oracle_sdm_gather", rc)
        return out0, out1, st

    def gather_kpos(self, bank, idx0, kpos, compact, *, chunk: int, valid: int = -1, chunk_valid=None,
                    check: bool = True):
        """Compact snapshot of operand 0 (kpos form), written into ``compact`` in place.

        compact [tokens / chunk, chunk * width0, hd] in the bank dtype; kpos [tokens, width0] int32,
        -1 for entries that store nothing. Returns ``compact``.
        """
        n_slots, hd = bank.shape
        tokens, width0 = idx0.shape
        if valid < 0:
            valid = chunk
        if not compact.flags["C_CONTIGUOUS"] or compact.dtype != bank.dtype:
            raise ValueError("compact must be C-contiguous in the bank dtype")
        if compact.size != (tokens // chunk) * chunk * width0 * hd:
            raise ValueError("compact must hold tokens / chunk blocks of chunk * width0 rows")
        cv = None if chunk_valid is None else np.ascontiguousarray(chunk_valid, dtype=np.int32)
        bank = np.ascontiguousarray(bank)
        idx0 = np.ascontiguousarray(idx0)
        kpos = np.ascontiguousarray(kpos, dtype=np.int32)
        rc = self.lib.oracle_sdm_gather_kpos(_ptr(bank), _bank_code(bank), n_slots, hd, _ptr(idx0), width0,
                                             _idx_code(idx0), _ptr(kpos), _ptr(compact), tokens, chunk, valid,
                                             _ptr(cv), 1 if check else 0)
        if rc != OK:
            raise OracleError("oracle_sdm_gather_kpos", rc)
        return compact

    def f32_to_bf16(self, x) -> np.ndarray:
        """float32 array -> bf16 bits (uint16), round to nearest even."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
        return y

    def bf16_to_f32(self, x) -> np.ndarray:
        """bf16 bits (uint16) -> float32 array."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        y = np.empty(x.shape, dtype=np.float32)
        self.lib.oracle_bf16_to_f32_array(_ptr(x), _ptr(y), x.size)
        return y


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``sdm_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def decode_seq(*a, **kw):
    return default().decode_seq(*a, **kw)


def decode_step(*a, **kw):
    return default().decode_step(*a, **kw)


def gather(*a, **kw):
    return default().gather(*a, **kw)


def gather_kpos(*a, **kw):
    return default().gather_kpos(*a, **kw)


def f32_to_bf16(x):
    return default().f32_to_bf16(x)


def bf16_to_f32(x):
    return default().bf16_to_f32(x)
