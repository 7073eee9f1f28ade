"""Python binding of the SDM C ABI (``include/sdm.h``): argument marshalling only.

Every operation runs in the CUDA library ``_build/libsdm.so``; these wrappers check shapes and
dtypes of PyTorch CUDA tensors, pass raw device pointers and the current CUDA stream, and raise
``SDMError`` on a non-zero status. There is no fallback: without the built library every call
raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libsdm.so")

SDM_BF16, SDM_F32 = 0, 1
SDM_I32, SDM_I64 = 0, 1
SDM_DEV_TIMEOUT, SDM_DEV_BAD_INDEX = 1, 2

ENTRY_POINTS = ("sdm_decode_step", "sdm_decode_step_ex", "sdm_decode_seq", "sdm_decode_seq_ex",
                "sdm_decode_plan_init", "sdm_decode_plan_launch", "sdm_decode_plan_walk", "sdm_gather",
                "sdm_gather_kpos",
                "sdm_gather_plan_init", "sdm_gather_plan_launch", "sdm_gather_plan_launch_ex", "sdm_gather_plan_walk",
                "sdm_status_string",
                "sdm_device_status", "sdm_version")
SDM_INPUTS_READY = 1  # flag of the _ex calls: the inputs predate the kernel launched just before
SDM_STREAM_MAJOR = 2  # flag of sdm_decode_seq_ex: per-token arrays are [S, T, .] instead of [T, S, .]
GATHER_PLAN_BYTES = 512  # SDM_GATHER_PLAN_BYTES
DECODE_PLAN_BYTES = 512  # SDM_DECODE_PLAN_BYTES

_BANK_CODES = {torch.bfloat16: SDM_BF16, torch.float32: SDM_F32}
_IDX_CODES = {torch.int32: SDM_I32, torch.int64: SDM_I64}

_lock = threading.Lock()
_lib = None


class SDMError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"the SDM CUDA library is not built ({_LIB_PATH} is missing); "
                                   "run decode_state_gb300.build.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            dec = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32]
            lib.sdm_decode_step.argtypes = dec + [i32, i32, vp]
            lib.sdm_decode_step.restype = i32
            lib.sdm_decode_step_ex.argtypes = dec + [i32, i32, ctypes.c_uint, vp]
            lib.sdm_decode_step_ex.restype = i32
            lib.sdm_decode_seq.argtypes = dec + [i32, i32, i32, vp]
            lib.sdm_decode_seq.restype = i32
            lib.sdm_decode_seq_ex.argtypes = dec + [i32, i32, i32, ctypes.c_uint, vp]
            lib.sdm_decode_seq_ex.restype = i32
            lib.sdm_decode_plan_init.argtypes = [vp] + dec + [i32, i32, i32]
            lib.sdm_decode_plan_init.restype = i32
            lib.sdm_decode_plan_launch.argtypes = [vp, i32, ctypes.c_uint, vp]
            lib.sdm_decode_plan_launch.restype = i32
            lib.sdm_decode_plan_walk.argtypes = [vp, i32, i32, ctypes.c_uint, vp]
            lib.sdm_decode_plan_walk.restype = i32
            lib.sdm_gather.argtypes = [vp, i64, i32, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                       ctypes.POINTER(vp), ctypes.POINTER(i32), i32, i32, vp, i64, i32, i32, vp, vp]
            lib.sdm_gather.restype = i32
            lib.sdm_gather_kpos.argtypes = [vp, i64, i32, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                            ctypes.POINTER(vp), ctypes.POINTER(i32), i32, i32, vp, vp, i64, i32, i32,
                                            vp, vp]
            lib.sdm_gather_kpos.restype = i32
            lib.sdm_gather_plan_init.argtypes = [vp, vp, i64, i32, i32, i32, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                                 ctypes.POINTER(vp), ctypes.POINTER(i32), i32, i32, i64, i64, i64, i32]
            lib.sdm_gather_plan_init.restype = i32
            lib.sdm_gather_plan_launch.argtypes = [vp, i64, i32, vp]
            lib.sdm_gather_plan_launch.restype = i32
            lib.sdm_gather_plan_launch_ex.argtypes = [vp, i64, i32, ctypes.c_uint, vp]
            lib.sdm_gather_plan_launch_ex.restype = i32
            lib.sdm_gather_plan_walk.argtypes = [vp, vp, vp, i32, ctypes.c_uint, vp]
            lib.sdm_gather_plan_walk.restype = i32
            lib.sdm_status_string.argtypes = [i32]
            lib.sdm_status_string.restype = ctypes.c_char_p
            lib.sdm_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
            lib.sdm_device_status.restype = i32
            lib.sdm_version.argtypes = []
            lib.sdm_version.restype = i32
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().sdm_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != 0:
        raise SDMError(fn, status, status_string(status))


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, name: str, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t: torch.Tensor, name: str, shape: tuple):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")


def _decode_args(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, lead: tuple, stream):
    if bank.dtype not in _BANK_CODES:
        raise TypeError(f"bank must be bfloat16 or float32, got {bank.dtype}")
    if bank.dim() != 2:
        raise ValueError("bank must be [n_slots, head_dim]")
    dev = bank.device
    if k_idx.dtype not in _IDX_CODES or q_idx.dtype != k_idx.dtype:
        raise TypeError(f"k_idx and q_idx must share one dtype, int32 or int64; got {k_idx.dtype}, {q_idx.dtype}")
    hd = bank.shape[1]
    W, R, G = k_idx.shape[-1], q_idx.shape[-1], g.shape[-1]
    for name, t, shp in (("k_idx", k_idx, (*lead, W)), ("k_val", k_val, (*lead, W)), ("v", v, (*lead, hd)),
                         ("beta", beta, lead), ("g", g, (*lead, G)), ("q_idx", q_idx, (*lead, R)),
                         ("q_val", q_val, (*lead, R))):
        _need(t, name, dev)
        _shape(t, name, shp)
    for name, t in (("k_val", k_val), ("v", v), ("beta", beta), ("g", g), ("q_val", q_val)):
        _f32(t, name)
    _need(bank, "bank", dev)
    if out is None:
        out = torch.empty((*lead, hd), dtype=bank.dtype, device=dev)
    _need(out, "out", dev)
    _shape(out, "out", (*lead, hd))
    if out.dtype != bank.dtype:
        raise TypeError("out must have the bank dtype")
    return out, (bank.data_ptr(), k_idx.data_ptr(), k_val.data_ptr(), v.data_ptr(), beta.data_ptr(), g.data_ptr(),
                 q_idx.data_ptr(), q_val.data_ptr(), out.data_ptr()), hd, W, R, G, _stream_handle(stream, dev)


def decode_step(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out=None, stream=None,
                inputs_ready: bool = False) -> torch.Tensor:
    """One write-then-read token for every stream (sdm_decode_step). Per-stream arrays are [S, .],
    beta is [S]; the bank is updated in place; returns the readings [S, hd] in the bank dtype.

    ``inputs_ready`` (sdm_decode_step_ex with SDM_INPUTS_READY) promises that the inputs were
    complete before the kernel enqueued just ahead of this call began; the launch then loads them
    and warms L2 with the step's rows while that kernel still runs. Same results."""
    S = k_idx.shape[0]
    out, ptrs, hd, W, R, G, st = _decode_args(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, (S,), stream)
    codes = (_BANK_CODES[bank.dtype], _IDX_CODES[k_idx.dtype])
    if inputs_ready:
        rc = library().sdm_decode_step_ex(*ptrs, S, hd, W, R, G, *codes, SDM_INPUTS_READY, st)
        _check("sdm_decode_step_ex", rc)
    else:
        rc = library().sdm_decode_step(*ptrs, S, hd, W, R, G, *codes, st)
        _check("sdm_decode_step", rc)
    return out


def decode_seq(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out=None, stream=None, *, stream_major: bool = False,
               inputs_ready: bool = False) -> torch.Tensor:
    """T tokens for every stream in one launch (sdm_decode_seq). Arrays are time-major [T, S, .],
    beta is [T, S]; returns the readings [T, S, hd].

    ``stream_major`` (sdm_decode_seq_ex with SDM_STREAM_MAJOR): the arrays are in the layer's own
    prompt layout [S, T, .] (beta [S, T]) and the readings come back as [S, T, hd]; no staging copy
    is made. ``inputs_ready``: SDM_INPUTS_READY, as for decode_step."""
    lead = tuple(k_idx.shape[:2])
    S, T = lead if stream_major else lead[::-1]
    out, ptrs, hd, W, R, G, st = _decode_args(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, lead, stream)
    codes = (_BANK_CODES[bank.dtype], _IDX_CODES[k_idx.dtype])
    flags = (SDM_STREAM_MAJOR if stream_major else 0) | (SDM_INPUTS_READY if inputs_ready else 0)
    if flags:
        rc = library().sdm_decode_seq_ex(*ptrs, S, hd, W, R, G, T, *codes, flags, st)
        _check("sdm_decode_seq_ex", rc)
    else:
        rc = library().sdm_decode_seq(*ptrs, S, hd, W, R, G, T, *codes, st)
        _check("sdm_decode_seq", rc)
    return out


def gather(bank, ops, *, chunk: int, valid: int | None = None, chunk_valid=None, stash=None, with_stash=True,
           outs=None, kpos=None, compact=None, stream=None):
    """Token gather (sdm_gather) with one or two operands ``ops = [(idx, w), ...]``.

    idx [tokens, width] int32/int64, w [tokens, width] bf16/float32. Returns (outs, stash):
    outs is a list of [tokens, hd] float32 tensors; stash [tokens, width0, hd] in the bank dtype
    (allocated when ``with_stash`` and not given), or None. ``valid`` is the scalar count
    (default: chunk) unless ``chunk_valid`` [tokens / chunk] int32 gives one per chunk.

    With ``kpos`` [tokens, width0] int32 the call is sdm_gather_kpos: operand 0's rows go to the
    compact snapshot ``compact`` [tokens / chunk, chunk * width0, hd] (written in place; only the
    rows kpos names), which is returned in place of the stash.
    """
    if bank.dtype not in _BANK_CODES or bank.dim() != 2:
        raise TypeError("bank must be a [n_slots, head_dim] bfloat16 or float32 tensor")
    dev = bank.device
    _need(bank, "bank", dev)
    if len(ops) not in (1, 2):
        raise ValueError("gather takes one or two operands")
    n_slots, hd = bank.shape
    tokens = ops[0][0].shape[0]
    idx_dt, w_dt = ops[0][0].dtype, ops[0][1].dtype
    if idx_dt not in _IDX_CODES or w_dt not in _BANK_CODES:
        raise TypeError("indices must be int32/int64 and weights bfloat16/float32")
    for o, (idx, w) in enumerate(ops):
        _need(idx, f"idx[{o}]", dev)
        _need(w, f"w[{o}]", dev)
        if idx.dtype != idx_dt or w.dtype != w_dt:
            raise TypeError("both operands must share the index dtype and the weight dtype")
        if idx.dim() != 2 or idx.shape[0] != tokens or tuple(w.shape) != tuple(idx.shape):
            raise ValueError(f"operand {o}: idx and w must both be [tokens, width]")
    if outs is None:
        outs = [torch.empty((tokens, hd), dtype=torch.float32, device=dev) for _ in ops]
    for o, out in enumerate(outs):
        _need(out, f"out[{o}]", dev)
        _f32(out, f"out[{o}]")
        _shape(out, f"out[{o}]", (tokens, hd))
    if kpos is not None:
        _need(kpos, "kpos", dev)
        if kpos.dtype != torch.int32:
            raise TypeError("kpos must be int32")
        _shape(kpos, "kpos", tuple(ops[0][0].shape))
        if compact is None:
            raise ValueError("kpos needs the compact snapshot tensor")
        _need(compact, "compact", dev)
        if compact.dtype != bank.dtype:
            raise TypeError("compact must have the bank dtype")
        if tokens % chunk == 0:
            _shape(compact, "compact", (tokens // chunk, chunk * ops[0][0].shape[1], hd))
        stash, with_stash = None, False
    if stash is None and with_stash:
        stash = torch.empty((tokens, ops[0][0].shape[1], hd), dtype=bank.dtype, device=dev)
    if stash is not None:
        _need(stash, "stash", dev)
        _shape(stash, "stash", (tokens, ops[0][0].shape[1], hd))
        if stash.dtype != bank.dtype:
            raise TypeError("stash must have the bank dtype")
    if chunk_valid is not None:
        _need(chunk_valid, "chunk_valid", dev)
        if chunk_valid.dtype != torch.int32:
            raise TypeError("chunk_valid must be int32")
        if tokens % chunk == 0:
            _shape(chunk_valid, "chunk_valid", (tokens // chunk,))
    if valid is None:
        valid = chunk
    vp = ctypes.c_void_p
    n = len(ops)
    idx_arr = (vp * 2)(*[vp(op[0].data_ptr()) for op in ops], *([vp(0)] * (2 - n)))
    w_arr = (vp * 2)(*[vp(op[1].data_ptr()) for op in ops], *([vp(0)] * (2 - n)))
    out_arr = (vp * 2)(*[vp(o.data_ptr()) for o in outs], *([vp(0)] * (2 - n)))
    width_arr = (ctypes.c_int * 2)(*[op[0].shape[1] for op in ops], *([0] * (2 - n)))
    cv_ptr = chunk_valid.data_ptr() if chunk_valid is not None else None
    if kpos is not None:
        rc = library().sdm_gather_kpos(bank.data_ptr(), n_slots, hd, _BANK_CODES[bank.dtype], n, idx_arr, w_arr,
                                       out_arr, width_arr, _IDX_CODES[idx_dt], _BANK_CODES[w_dt], compact.data_ptr(),
                                       kpos.data_ptr(), tokens, chunk, valid, cv_ptr, _stream_handle(stream, dev))
        _check("sdm_gather_kpos", rc)
        return outs, compact
    rc = library().sdm_gather(bank.data_ptr(), n_slots, hd, _BANK_CODES[bank.dtype], n, idx_arr, w_arr, out_arr,
                              width_arr, _IDX_CODES[idx_dt], _BANK_CODES[w_dt],
                              stash.data_ptr() if stash is not None else None, tokens, chunk, valid, cv_ptr,
                              _stream_handle(stream, dev))
    _check("sdm_gather", rc)
    return outs, stash


class DecodeStepPlan:
    """Single-token decode steps over fixed device buffers, checked once (sdm_decode_plan_init).

    ``inputs`` maps the names of ``DECODE_KEYS`` to time-major device tensors [T, S, .] (beta
    [T, S]) that the caller fills; ``launch(t)`` runs sdm_decode_step on step t's slabs and writes
    the readings into ``out[t]`` ([T, S, hd], allocated when not given); ``walk(t0, n)`` runs steps
    t0 .. t0 + n - 1 from one foreign call. Shapes, dtypes, devices and the launch are settled in a
    plan record made here, so a launch is one foreign call with four arguments. The plan keeps
    references to its tensors; they must not be resized or reallocated in place.

    With ``inputs_ready`` every launch passes SDM_INPUTS_READY: the caller fills all T slabs before
    the launches, not between them.
    """

    DECODE_KEYS = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")

    def __init__(self, bank, inputs: dict, out=None, stream=None, inputs_ready: bool = False):
        T = inputs["k_idx"].shape[0]
        if out is None:
            out = torch.empty((T, inputs["k_idx"].shape[1], bank.shape[1]), dtype=bank.dtype, device=bank.device)
        args = [inputs[k] for k in self.DECODE_KEYS]
        self.out, _, hd, W, R, G, _ = _decode_args(bank, *args, out, (T, inputs["k_idx"].shape[1]), stream)
        S = inputs["k_idx"].shape[1]
        self._record = ctypes.create_string_buffer(DECODE_PLAN_BYTES)
        rc = library().sdm_decode_plan_init(self._record, bank.data_ptr(), *(a.data_ptr() for a in args),
                                            self.out.data_ptr(), S, hd, W, R, G, T, _BANK_CODES[bank.dtype],
                                            _IDX_CODES[inputs["k_idx"].dtype])
        _check("sdm_decode_plan_init", rc)
        self._flags = SDM_INPUTS_READY if inputs_ready else 0
        self._launch = library().sdm_decode_plan_launch
        self._stream = _stream_handle(stream, bank.device) if stream is not None else None
        self._keep = (bank, inputs)
        self.device, self.T = bank.device, T

    def launch(self, t: int, stream=None) -> torch.Tensor:
        """Step t (0 <= t < T) on the bank; returns the readings out[t]."""
        st = self._stream if stream is None and self._stream is not None else _stream_handle(stream, self.device)
        rc = self._launch(self._record, t, self._flags, st)
        if rc != 0:
            _check("sdm_decode_plan_launch", rc)
        return self.out[t]

    def walk(self, t0: int = 0, n: int | None = None, stream=None) -> torch.Tensor:
        """Steps t0 .. t0 + n - 1 (n: all the rest when None) from one call; returns ``out``."""
        n = self.T - t0 if n is None else n
        st = self._stream if stream is None and self._stream is not None else _stream_handle(stream, self.device)
        rc = library().sdm_decode_plan_walk(self._record, t0, n, self._flags, st)
        _check("sdm_decode_plan_walk", rc)
        return self.out


class GatherPlan:
    """A checked no-stash gather launch replayed per slab (sdm_gather_plan_init / _launch).

    ``ops = [(idx, w), ...]`` are the WHOLE index and weight tensors [rows, width]; every
    ``launch(row0, valid)`` gathers their rows [row0, row0 + tokens) into ``outs`` (one [tokens,
    hd] float32 tensor per operand, allocated when not given), with ``valid`` live tokens per
    chunk. The plan keeps references to every tensor it was made with, so they stay alive while
    it exists; they must not be resized or reallocated in place.
    """

    def __init__(self, bank, ops, *, tokens: int, chunk: int, row0_max: int | None = None, outs=None):
        if bank.dtype not in _BANK_CODES or bank.dim() != 2:
            raise TypeError("bank must be a [n_slots, head_dim] bfloat16 or float32 tensor")
        dev = bank.device
        _need(bank, "bank", dev)
        if len(ops) not in (1, 2):
            raise ValueError("gather takes one or two operands")
        n_slots, hd = bank.shape
        rows = ops[0][0].shape[0]
        idx_dt, w_dt = ops[0][0].dtype, ops[0][1].dtype
        if idx_dt not in _IDX_CODES or w_dt not in _BANK_CODES:
            raise TypeError("indices must be int32/int64 and weights bfloat16/float32")
        for o, (idx, w) in enumerate(ops):
            _need(idx, f"idx[{o}]", dev)
            _need(w, f"w[{o}]", dev)
            if idx.dtype != idx_dt or w.dtype != w_dt:
                raise TypeError("both operands must share the index dtype and the weight dtype")
            if idx.dim() != 2 or idx.shape[0] != rows or tuple(w.shape) != tuple(idx.shape):
                raise ValueError(f"operand {o}: idx and w must both be [rows, width] with the same rows")
        if outs is None:
            outs = [torch.empty((tokens, hd), dtype=torch.float32, device=dev) for _ in ops]
        for o, out in enumerate(outs):
            _need(out, f"out[{o}]", dev)
            _f32(out, f"out[{o}]")
            _shape(out, f"out[{o}]", (tokens, hd))
        if row0_max is None:
            row0_max = rows - tokens
        vp = ctypes.c_void_p
        n = len(ops)
        idx_arr = (vp * 2)(*[vp(op[0].data_ptr()) for op in ops], *([vp(0)] * (2 - n)))
        w_arr = (vp * 2)(*[vp(op[1].data_ptr()) for op in ops], *([vp(0)] * (2 - n)))
        out_arr = (vp * 2)(*[vp(o.data_ptr()) for o in outs], *([vp(0)] * (2 - n)))
        width_arr = (ctypes.c_int * 2)(*[op[0].shape[1] for op in ops], *([0] * (2 - n)))
        self._record = ctypes.create_string_buffer(GATHER_PLAN_BYTES)
        with torch.cuda.device(dev):
            rc = library().sdm_gather_plan_init(self._record, bank.data_ptr(), n_slots, hd, _BANK_CODES[bank.dtype], n,
                                                idx_arr, w_arr, out_arr, width_arr, _IDX_CODES[idx_dt],
                                                _BANK_CODES[w_dt], rows, row0_max, tokens, chunk)
        _check("sdm_gather_plan_init", rc)
        self._keep = (bank, tuple(tuple(op) for op in ops))
        self.outs, self.device, self.tokens, self.chunk, self.row0_max = outs, dev, tokens, chunk, row0_max

    def launch(self, row0: int, valid: int | None = None, stream=None, inputs_ready: bool = False) -> list:
        """The planned gather over index rows [row0, row0 + tokens); returns ``outs``.

        ``inputs_ready`` (sdm_gather_plan_launch_ex with SDM_INPUTS_READY) promises that those index
        and weight rows were complete before the kernel enqueued just ahead of this launch began;
        the launch then reads them and warms L2 with their rows while that kernel still runs."""
        v = self.chunk if valid is None else valid
        st = _stream_handle(stream, self.device)
        if inputs_ready:
            rc = library().sdm_gather_plan_launch_ex(self._record, row0, v, SDM_INPUTS_READY, st)
            _check("sdm_gather_plan_launch_ex", rc)
        else:
            rc = library().sdm_gather_plan_launch(self._record, row0, v, st)
            _check("sdm_gather_plan_launch", rc)
        return self.outs

    def walk(self, row0s, valids=None, *, inputs_ready: bool = False, stream=None):
        """Every slab of a walk from one foreign call (sdm_gather_plan_walk): slab i is
        ``launch(row0s[i], valids[i])``, in order; ``outs`` holds the last slab's result.
        ``row0s`` and ``valids`` are host integer sequences (``valids`` None: every slab full).
        For a walk replayed many times, pass the arrays from ``walk_arrays`` to skip the
        conversion."""
        r, v = row0s, valids
        if not (isinstance(r, ctypes.Array) and (v is None or isinstance(v, ctypes.Array))):
            r, v = self.walk_arrays(row0s, valids)
        n = len(r)
        if v is not None and len(v) != n:
            raise ValueError("row0s and valids must have the same length")
        st = _stream_handle(stream, self.device)
        rc = library().sdm_gather_plan_walk(self._record, r, v, n, SDM_INPUTS_READY if inputs_ready else 0, st)
        _check("sdm_gather_plan_walk", rc)
        return self.outs

    @staticmethod
    def walk_arrays(row0s, valids=None):
        """Host arrays for ``walk``: (int64 row offsets, int32 valid counts or None)."""
        r = (ctypes.c_int64 * len(row0s))(*row0s)
        v = None if valids is None else (ctypes.c_int32 * len(valids))(*valids)
        return r, v


def device_status(clear: bool = True) -> int:
    """OR of the SDM_DEV_* bits kernels raised on the current device since the last clear."""
    word = ctypes.c_uint(0)
    rc = library().sdm_device_status(ctypes.byref(word), 1 if clear else 0)
    _check("sdm_device_status", rc)
    return int(word.value)


def version() -> int:
    return int(library().sdm_version())
