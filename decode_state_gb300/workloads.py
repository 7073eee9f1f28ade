"""Seeded synthetic workloads for the SDM decode step, multi-token decode and token gather.

This module only draws inputs; it holds none of the method's arithmetic. Both the CUDA path and
the CPU oracle consume what it draws (the oracle through host copies), so neither side ever
produces the other's inputs.

Every tensor of a workload is drawn from one ``torch.Generator`` seeded once, in a fixed order:
bank, k_idx, k_val, v, beta, g, q_idx, q_val (decode) or bank, valid, idx0, w0, idx1, w1 (gather).
The same seed on the same device type gives the same tensors.

Distributions (the SDM decode and gather workloads):
  bank       N(0, bank_std) rounded to the bank dtype; stream s owns rows [s*P, (s+1)*P)
  k_idx      W distinct slots drawn uniformly from the stream's own P slots
  q_idx      R slots drawn uniformly (repeats allowed) from the stream's own P slots
  k_val,q_val N(0,1) * kq_scale (float32)
  v          N(0,1) (float32);  beta = sigmoid(N(0,1));  g = -softplus(N(0,1))  (float32)
  gather     idx uniform over the whole bank; weights N(0,1) * w_scale in the weight dtype;
             valid ~ Uniform{1..chunk} per chunk
"""

from __future__ import annotations

import dataclasses
import math

import torch

BANK_DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}
IDX_DTYPES = {"i32": torch.int32, "i64": torch.int64}


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    bank_dtype: str  # "bf16" | "f32"
    n_streams: int
    hd: int
    slots_per_stream: int
    W: int
    R: int
    G: int  # 1 or W
    T: int  # tokens per stream
    idx_dtype: str  # "i32" | "i64"
    kq_scale: float
    bank_std: float = 0.02
    mode: str = "seq"  # how the benchmark drives it: "seq" (one persistent launch) or "step"
    seed: int = 0

    @property
    def n_slots(self) -> int:
        return self.n_streams * self.slots_per_stream

    def scaled(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class GatherWorkload:
    name: str
    bank_dtype: str
    n_slots: int
    hd: int
    tokens: int
    chunk: int
    widths: tuple  # (W0,) or (W0, W1)
    idx_dtype: str
    w_dtype: str  # "bf16" | "f32"
    w_scale: float
    stash: bool = True
    bank_std: float = 1.0
    per_chunk_valid: bool = True
    seed: int = 0

    def scaled(self, **kw) -> "GatherWorkload":
        return dataclasses.replace(self, **kw)


# The five workloads: four decode shapes and one gather shape (plus the gather's backward shape).
C0 = DecodeWorkload("decode_f32_s4_hd64_w8_t16", "f32", 4, 64, 1024, 8, 8, 1, 16, "i32", 1 / math.sqrt(8))
C1 = DecodeWorkload("decode_bf16_s64_hd128_w32_gw_256steps", "bf16", 64, 128, 65536, 32, 32, 32, 256, "i64",
                    1 / math.sqrt(8), mode="step")
C2 = DecodeWorkload("decode_bf16_s1024_hd128_w64_seq64", "bf16", 1024, 128, 16384, 64, 64, 1, 64, "i32",
                    1 / math.sqrt(8))
C3 = DecodeWorkload("decode_f32_s256_hd256_w256_t8", "f32", 256, 256, 8192, 256, 256, 1, 8, "i64", 1 / 16)
C4 = GatherWorkload("gather_bf16_4M_hd128_65536tok_2x64_stash", "bf16", 4194304, 128, 65536, 64, (64, 64), "i64",
                    "bf16", 1 / 8)

# The backward's one-operand shape of the same gather: bank-gradient rows (float32) at the write
# slots weighted by the write weights, plus the stash of those rows.
C4_BWD = GatherWorkload("gather_bwd_f32_4M_hd128_65536tok_1x64_stash", "f32", 4194304, 128, 65536, 64, (64,), "i64",
                        "f32", 1 / 8)

# A prompt run through the recurrent form: the serving geometry per stream (bf16, hd 128,
# W = R = 64, one gate per token, 16384 slots each) for 64 streams of 1024 tokens, with every
# per-token array in the layer's own stream-major layout [S, T, .] (the benchmark transposes the
# time-major draw once, before timing).
PROMPT = DecodeWorkload("prompt_bf16_s64_hd128_w64_t1024_stream_major", "bf16", 64, 128, 16384, 64, 64, 1, 1024,
                        "i32", 1 / math.sqrt(8), mode="seq_stream_major")

DECODE_WORKLOADS = {w.name: w for w in (C0, C1, C2, C3, PROMPT)}
GATHER_WORKLOADS = {w.name: w for w in (C4, C4_BWD)}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal_bank(n_rows: int, hd: int, std: float, dtype, device, gen, block_rows: int = 1 << 20):
    """[n_rows, hd] ~ N(0, std) in `dtype`, drawn in row blocks to bound temporary memory."""
    bank = torch.empty((n_rows, hd), dtype=dtype, device=device)
    for r0 in range(0, n_rows, block_rows):
        r1 = min(n_rows, r0 + block_rows)
        x = torch.randn((r1 - r0, hd), generator=gen, device=device, dtype=torch.float32)
        bank[r0:r1] = (x * std).to(dtype)
    return bank


def distinct_slots(rows: int, k: int, n: int, device, gen) -> torch.Tensor:
    """[rows, k] int64: each row holds k distinct values drawn uniformly from [0, n).

    Oversample-and-deduplicate: draw m >= 2k candidates per row, keep each value's first
    occurrence, take the first k survivors. Rows with fewer than k survivors are redrawn with a
    larger m. For n <= 4k a random permutation per row is used instead.
    """
    if k > n:
        raise ValueError(f"cannot draw {k} distinct slots from {n}")
    if rows == 0:
        return torch.empty((0, k), dtype=torch.int64, device=device)
    if n <= 4 * k:
        keys = torch.rand((rows, n), generator=gen, device=device)
        return keys.argsort(dim=1)[:, :k].contiguous()
    out = torch.empty((rows, k), dtype=torch.int64, device=device)
    todo = torch.arange(rows, device=device)
    m = 2 * k
    while todo.numel() > 0:
        cand = torch.randint(0, n, (todo.numel(), m), generator=gen, device=device)
        srt, order = cand.sort(dim=1, stable=True)
        dup_sorted = torch.zeros_like(srt, dtype=torch.bool)
        dup_sorted[:, 1:] = srt[:, 1:] == srt[:, :-1]
        dup = torch.empty_like(dup_sorted).scatter_(1, order, dup_sorted)
        keep = ~dup
        enough = keep.sum(dim=1) >= k
        ok_rows = todo[enough]
        if ok_rows.numel() > 0:
            kk = keep[enough]
            sel = kk & (kk.cumsum(dim=1) <= k)
            out[ok_rows] = cand[enough][sel].view(-1, k)
        todo = todo[~enough]
        m *= 2
    return out


def make_decode_inputs(wl: DecodeWorkload, device="cpu", seed: int | None = None) -> dict:
    """Draw one decode workload. Per-token tensors are time-major [T, S, ...]."""
    seed = wl.seed if seed is None else seed
    gen = _gen(device, seed)
    T, S, W, R, G, hd, P = wl.T, wl.n_streams, wl.W, wl.R, wl.G, wl.hd, wl.slots_per_stream
    bdt, idt = BANK_DTYPES[wl.bank_dtype], IDX_DTYPES[wl.idx_dtype]
    bank = _normal_bank(S * P, hd, wl.bank_std, bdt, device, gen)
    base = (torch.arange(S, device=device, dtype=torch.int64) * P).view(1, S, 1)
    k_idx = (distinct_slots(T * S, W, P, device, gen).view(T, S, W) + base).to(idt)
    f32 = torch.float32
    k_val = torch.randn((T, S, W), generator=gen, device=device, dtype=f32) * wl.kq_scale
    v = torch.randn((T, S, hd), generator=gen, device=device, dtype=f32)
    beta = torch.sigmoid(torch.randn((T, S), generator=gen, device=device, dtype=f32))
    g = -torch.nn.functional.softplus(torch.randn((T, S, G), generator=gen, device=device, dtype=f32))
    q_idx = (torch.randint(0, P, (T, S, R), generator=gen, device=device) + base).to(idt)
    q_val = torch.randn((T, S, R), generator=gen, device=device, dtype=f32) * wl.kq_scale
    return dict(bank=bank, k_idx=k_idx, k_val=k_val.contiguous(), v=v, beta=beta.contiguous(), g=g.contiguous(),
                q_idx=q_idx, q_val=q_val.contiguous())


SHARD_BLOCK = 64  # streams per independently seeded block of a partitioned decode workload


def shard_blocks(n_streams: int, block: int = SHARD_BLOCK) -> int:
    return (n_streams + block - 1) // block


def make_decode_shard(wl: DecodeWorkload, lo: int, hi: int, device="cpu", seed: int | None = None,
                      block: int = SHARD_BLOCK) -> dict:
    """Streams [lo, hi) of decode workload ``wl`` drawn as one job that any set of processes can
    split: the job's streams form blocks of ``block`` streams (the last may be shorter), block b
    drawn by make_decode_inputs from its own seed (seed + 7919 * b), with its slots offset to the
    block's own bank rows. ``lo`` and ``hi`` must be block boundaries (or n_streams). Returns the
    shard with the layout of make_decode_inputs over hi - lo streams: its bank holds the shard's
    rows [lo * P, hi * P) of the job's bank, and its slots are rebased to that local bank."""
    seed = wl.seed if seed is None else seed
    if lo % block or (hi % block and hi != wl.n_streams) or not 0 <= lo <= hi <= wl.n_streams:
        raise ValueError(f"shard [{lo}, {hi}) is not on {block}-stream block boundaries of {wl.n_streams} streams")
    parts = []
    for b in range(lo // block, shard_blocks(hi, block)):
        n = min(block, wl.n_streams - b * block)
        x = make_decode_inputs(wl.scaled(n_streams=n), device=device, seed=seed + 7919 * b)
        off = (b * block - lo) * wl.slots_per_stream  # the block's first row in the shard's bank
        x["k_idx"] += off
        x["q_idx"] += off
        parts.append(x)
    if not parts:
        return make_decode_inputs(wl.scaled(n_streams=0), device=device, seed=seed)
    out = {"bank": torch.cat([x["bank"] for x in parts])}
    for k in ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val"):
        out[k] = torch.cat([x[k] for x in parts], dim=1).contiguous()
    return out


def make_gather_inputs(wl: GatherWorkload, device="cpu", seed: int | None = None) -> dict:
    """Draw one gather workload: bank, per-chunk valid counts, and one or two operands."""
    seed = wl.seed if seed is None else seed
    gen = _gen(device, seed)
    bdt, idt = BANK_DTYPES[wl.bank_dtype], IDX_DTYPES[wl.idx_dtype]
    wdt = BANK_DTYPES[wl.w_dtype]
    if wl.tokens % wl.chunk:
        raise ValueError("tokens must be a multiple of chunk")
    bank = _normal_bank(wl.n_slots, wl.hd, wl.bank_std, bdt, device, gen)
    n_chunks = wl.tokens // wl.chunk
    if wl.per_chunk_valid:
        chunk_valid = torch.randint(1, wl.chunk + 1, (n_chunks,), generator=gen, device=device).to(torch.int32)
    else:
        chunk_valid = None
    ops = []
    for width in wl.widths:
        idx = torch.randint(0, wl.n_slots, (wl.tokens, width), generator=gen, device=device).to(idt)
        w = (torch.randn((wl.tokens, width), generator=gen, device=device, dtype=torch.float32) * wl.w_scale).to(wdt)
        ops.append((idx, w))
    return dict(bank=bank, chunk_valid=chunk_valid, ops=ops)


def decode_bytes_per_stream_token(wl: DecodeWorkload) -> int:
    """Algorithmic bytes of one stream-token: gathered and written rows, v (float32) and out."""
    es = 2 if wl.bank_dtype == "bf16" else 4
    return (wl.W + wl.R) * wl.hd * es + wl.W * wl.hd * es + wl.hd * 4 + wl.hd * es


def gather_bytes(wl: GatherWorkload, chunk_valid) -> int:
    """Algorithmic bytes of one gather call: live-token row reads, stash writes (zero rows for
    padding tokens too) and the float32 outputs."""
    es = 2 if wl.bank_dtype == "bf16" else 4
    if chunk_valid is None:
        live = wl.tokens
    else:
        live = int(chunk_valid.to(torch.int64).sum().item())
    reads = live * sum(wl.widths) * wl.hd * es
    stash = wl.tokens * wl.widths[0] * wl.hd * es if wl.stash else 0
    outs = wl.tokens * len(wl.widths) * wl.hd * 4
    return reads + stash + outs
