#!/usr/bin/env python
"""Benchmark of the SDM decode hot path on GB300.

A step is one sdm_decode_seq launch over the serving-scale decode workload: 1024 streams (batch 64
x 16 heads), head_dim 128, a bf16 bank of 16384 private slots per stream (4 GiB), W = R = 64
writes and reads per token, one gate per token, int32 slots, T = 64 tokens per stream.
The metric is stream-tokens per second (whole job over all ranks) with the effective bank
bandwidth as a fraction of the measured HBM peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

--impl reference times the CPU oracle on the host cores instead (the reference arm: bounded
samples of the same workload per step). Under torch.distributed.run every rank runs its own
shard (weak scaling); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from decode_state_gb300 import dist as sdist  # noqa: E402
from decode_state_gb300 import workloads  # noqa: E402

METRIC = "SDM stream-tokens/sec and effective bank GB/s as fraction of GB300 HBM peak"
UNIT = "stream-tokens/s"
WL = workloads.C2
DECODE_KEYS = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--no-extras", action="store_true", help="skip the secondary workloads")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget of the CPU baseline")
    p.add_argument("--workload", default=WL.name,
                   choices=sorted(list(workloads.DECODE_WORKLOADS) + list(workloads.GATHER_WORKLOADS)),
                   help="workload of the timed step (default: the serving-scale decode)")
    p.add_argument("--streams", type=int, default=0, help="override the decode stream count (smaller cases)")
    p.add_argument("--tokens", type=int, default=0, help="override T (decode) or the token count (gather)")
    p.add_argument("--gather-form", choices=("stash", "compact", "none"), default="stash",
                   help="gather workloads: the stash (as the workload names it), a compact snapshot of operand 0 "
                        "(sdm_gather_kpos) in its place, or outputs only")
    a = p.parse_args()
    a.warmup = max(3, a.warmup)
    a.steps = max(1, a.steps)
    return a


# ---------------------------------------------------------------- peaks, clocks, profiles


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(files) -> str:
    """sha256 over the named kernel source files (name, NUL, bytes; sorted by name)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_state_gb300", "csrc")
    for f in sorted(files):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu record, if it was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
        if not rec or rec.get("kernel_source_sha256") != kernel_source_hash(rec["files"]):
            return None
    except (OSError, ValueError, KeyError):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples (100 ms) with host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.samples = []
        self.proc = None
        self.error = None
        try:
            props = torch.cuda.get_device_properties(device)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            sel = ["-i", bus]
        except Exception:  # older torch: no PCI ids
            sel = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", *sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError as e:
            self.error = f"nvidia-smi unavailable: {e}"
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": self.error}
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        note = None
        if len(inside) < 3:  # a short timed region: use the samples around it too
            inside = [p for (t, p) in self.samples if t0 - 0.5 <= t <= t1 + 0.5]
            note = "few samples inside the timed region; includes samples within 0.5 s of it"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for p in inside for n, v in zip(names, p[5:9]) if v.lower() == "active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------- workloads as timed cases


def _np(t):
    import numpy as np

    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def oracle_stream_tokens(x: dict, streams, P: int):
    """Oracle run over whole streams of a decode workload (host copies); returns (stream-tokens, seconds)."""
    import oracle

    orc = oracle.default()
    done, secs = 0, 0.0
    for s in streams:
        args = []
        for k in DECODE_KEYS:
            v = x[k][:, s:s + 1]
            args.append(_np(v - s * P if k in ("k_idx", "q_idx") else v))
        bank = _np(x["bank"][s * P:(s + 1) * P])
        t0 = time.perf_counter()
        orc.decode_seq(bank, *args, check=False)
        secs += time.perf_counter() - t0
        done += x["k_idx"].shape[0]
    return done, secs


def _oracle_worker(job):
    """One process of the all-cores CPU baseline: the oracle `reps` times over `streams` streams of
    the decode workload, drawn on the host from the job's own seed. Returns (stream-tokens, start,
    end), wall-clock seconds around the oracle calls."""
    fields, seed, streams, reps = job
    wl = workloads.DecodeWorkload(**fields).scaled(n_streams=streams)
    x = workloads.make_decode_inputs(wl, device="cpu", seed=seed)
    oracle_stream_tokens(x, [0], wl.slots_per_stream)  # loads the oracle library
    t0 = time.time()
    done = 0
    for _ in range(reps):
        done += oracle_stream_tokens(x, range(streams), wl.slots_per_stream)[0]
    return done, t0, time.time()


def oracle_gather_tokens(bank_h, g: dict, tokens, chunk: int):
    """Oracle run over a list of gather tokens (host copies); returns (tokens, seconds)."""
    import oracle

    orc = oracle.default()
    tok = torch.as_tensor(tokens, dtype=torch.int64)
    (i0, w0), *rest = g["ops"]
    a = [_np(i0[tok]), _np(w0[tok])]
    if rest:
        a += [_np(rest[0][0][tok]), _np(rest[0][1][tok])]
    cv = g["chunk_valid"]
    valid_t = (cv[tok // chunk] if cv is not None else torch.full((len(tokens),), chunk, dtype=torch.int32))
    # one token per chunk of one: a live token has valid 1, a padding token valid 0
    per_token = _np(((tok % chunk) < valid_t.cpu().to(torch.int64)).to(torch.int32))
    t0 = time.perf_counter()
    orc.gather(bank_h, *a, chunk=1, chunk_valid=per_token, check=False)
    return len(tokens), time.perf_counter() - t0


def decode_config(wl, r: sdist.Rank) -> dict:
    """The config object of a decode workload's JSON line (wl: one rank's share); both arms use
    it, so that they name the same workload with the same keys and values (the entry point each
    arm calls is the line's own `call` key)."""
    bank_gib = wl.n_slots * wl.hd * (2 if wl.bank_dtype == "bf16" else 4) / 2 ** 30
    return {"workload": wl.name, "streams": wl.n_streams, "head_dim": wl.hd,
            "slots_per_stream": wl.slots_per_stream, "W": wl.W, "R": wl.R, "G": wl.G, "T": wl.T,
            "bank_dtype": wl.bank_dtype, "idx_dtype": wl.idx_dtype,
            "l2": (f"inputs larger than L2 ({bank_gib:.2f} GiB bank), no flush" if bank_gib > 0.2 else
                   f"L2-resident ({bank_gib * 1024:.0f} MiB bank)"),
            "parallelism": (f"weak: a job of {wl.n_streams * r.world} streams split into {r.world} contiguous "
                            f"stream range(s) of {wl.n_streams}, each rank holding its streams' bank rows; no "
                            f"collective in the data path")}


class Case:
    """One timed workload: its step, its units and bytes, its end-to-end form and its oracle."""

    def __init__(self, args, dev, r: sdist.Rank):
        from decode_state_gb300 import sdm

        self.sdm = sdm
        name = args.workload
        self.dev = dev
        if name in workloads.DECODE_WORKLOADS:
            wl = workloads.DECODE_WORKLOADS[name]
            if args.streams:
                wl = wl.scaled(n_streams=args.streams)
            if args.tokens:
                wl = wl.scaled(T=args.tokens)
            self.kind = "decode_" + wl.mode
            # weak scaling: the job holds wl.n_streams streams per rank, split into contiguous
            # stream ranges; this rank draws only its own streams and their bank rows
            job = wl.scaled(n_streams=wl.n_streams * r.world)
            lo, hi = sdist.stream_shard(job.n_streams, r, workloads.SHARD_BLOCK)
            self.x = workloads.make_decode_shard(job, lo, hi, device=dev)
            self.shard = (lo, hi, job.n_streams)
            wl = wl.scaled(n_streams=hi - lo)
            bdt = workloads.BANK_DTYPES[wl.bank_dtype]
            self.out = torch.empty((wl.T, wl.n_streams, wl.hd), dtype=bdt, device=dev)
            if self.kind == "decode_seq_stream_major":  # the prompt's own layout [S, T, .], made once
                self.x = {k: (v.transpose(0, 1).contiguous() if k in DECODE_KEYS else v) for k, v in self.x.items()}
                self.out = torch.empty((wl.n_streams, wl.T, wl.hd), dtype=bdt, device=dev)
            self.units = wl.n_streams * wl.T
            self.unit = UNIT
            self.launches = 1 if wl.mode.startswith("seq") else wl.T
            self.nbytes = workloads.decode_bytes_per_stream_token(wl) * wl.n_streams * wl.T
            # float32 rows that cannot all be staged stream through a ring (decode_wide_kernel)
            wide = wl.bank_dtype == "f32" and max(wl.W, wl.R) * min(wl.hd, 256) * 4 > 32768
            self.kernel = f"{'decode_wide_kernel' if wide else 'decode_vec_kernel'}<{wl.bank_dtype},{wl.idx_dtype}>"
            self.metric = METRIC
        else:
            wl = workloads.GATHER_WORKLOADS[name]
            if args.tokens:
                wl = wl.scaled(tokens=args.tokens)
            self.kind = "gather"
            self.g = workloads.make_gather_inputs(wl, device=dev, seed=sdist.shard_seed(wl.seed, r))
            self.outs = [torch.empty((wl.tokens, wl.hd), device=dev) for _ in wl.widths]
            bdt = workloads.BANK_DTYPES[wl.bank_dtype]
            self.form = args.gather_form if wl.stash else "none"
            self.stash = (torch.empty((wl.tokens, wl.widths[0], wl.hd), dtype=bdt, device=dev)
                          if self.form == "stash" else None)
            self.kpos, self.compact, written = (compact_snapshot(wl, self.g, dev) if self.form == "compact"
                                                else (None, None, 0))
            self.units = wl.tokens
            self.unit = "tokens/s"
            self.launches = 1
            self.nbytes = gather_form_bytes(wl, self.g, self.form, written)
            self.kernel = f"gather_kernel<{wl.bank_dtype},{wl.idx_dtype},{wl.w_dtype},vector rows>"
            self.metric = "SDM token-gather tokens/sec and effective bank GB/s as fraction of GB300 HBM peak"
        self.wl = wl

    # device-resident step
    def step(self):
        wl, sdm = self.wl, self.sdm
        if self.kind == "decode_seq":
            sdm.decode_seq(self.x["bank"], *(self.x[k] for k in DECODE_KEYS), out=self.out)
        elif self.kind == "decode_seq_stream_major":
            sdm.decode_seq(self.x["bank"], *(self.x[k] for k in DECODE_KEYS), out=self.out, stream_major=True)
        elif self.kind == "decode_step":
            for t in range(wl.T):
                sdm.decode_step(self.x["bank"], *(self.x[k][t] for k in DECODE_KEYS), out=self.out[t])
        else:
            sdm.gather(self.g["bank"], self.g["ops"], chunk=wl.chunk, chunk_valid=self.g["chunk_valid"],
                       stash=self.stash, outs=self.outs, with_stash=self.stash is not None, kpos=self.kpos,
                       compact=self.compact)

    def config(self, r: sdist.Rank) -> dict:
        wl = self.wl
        par = f"weak: {r.world} independent token shard(s), bank drawn per rank, no collective in the data path"
        if self.kind == "gather":
            gib = wl.n_slots * wl.hd * (2 if wl.bank_dtype == "bf16" else 4) / 2 ** 30
            return {"workload": wl.name, "n_slots": wl.n_slots, "head_dim": wl.hd, "tokens": wl.tokens,
                    "chunk": wl.chunk, "widths": list(wl.widths), "bank_dtype": wl.bank_dtype,
                    "idx_dtype": wl.idx_dtype, "w_dtype": wl.w_dtype, "stash": self.form == "stash",
                    "form": self.form,
                    "l2": f"inputs larger than L2 ({gib:.0f} GiB bank), no flush", "parallelism": par}
        return decode_config(wl, r)

    def call(self) -> str:
        """The library entry point the timed step calls."""
        if self.kind == "gather":
            return "sdm_gather_kpos" if self.form == "compact" else "sdm_gather"
        return {"decode_seq": "sdm_decode_seq", "decode_seq_stream_major": "sdm_decode_seq_ex (SDM_STREAM_MAJOR)",
                "decode_step": "sdm_decode_step x T"}[self.kind]

    # end to end: host inputs in, results out, every step
    def e2e(self, steps: int, r: sdist.Rank) -> dict:
        dev, wl, sdm = self.dev, self.wl, self.sdm
        stream = torch.cuda.current_stream(dev)
        if self.kind == "decode_seq":
            # the package's host-fed decoder: double-buffered device inputs, copies on their own streams
            from decode_state_gb300.hostfed import HostFedDecoder

            host_in = {k: self.x[k].cpu().pin_memory() for k in DECODE_KEYS}
            outs_h = [torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True) for _ in range(2)]
            dec = HostFedDecoder(self.x["bank"], self.x, depth=2)
            h2d = sum(t.numel() * t.element_size() for t in host_in.values())
            d2h = outs_h[0].numel() * outs_h[0].element_size()
            for i in range(3):
                dec.submit(host_in, outs_h[i % 2])
            dec.synchronize()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            sdist.barrier(r, dev)
            e0.record(dec.h2d)
            for i in range(steps):
                dec.submit(host_in, outs_h[i % 2])
            e1.record(dec.d2h)
            dec.synchronize()
            torch.cuda.synchronize()
            ms = sdist.max_over_ranks(r, e0.elapsed_time(e1), dev)
            return {"value": self.units * steps * r.world / (ms / 1e3), "unit": self.unit, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
                    "api": "decode_state_gb300.hostfed.HostFedDecoder (depth 2)"}
        if self.kind.startswith("decode"):
            host_in = [self.x[k].cpu().pin_memory() for k in DECODE_KEYS]
            dev_in = [torch.empty_like(self.x[k]) for k in DECODE_KEYS]
            host_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
            d2h = host_out.numel() * host_out.element_size()

            def step():
                for d, h in zip(dev_in, host_in):
                    d.copy_(h, non_blocking=True)
                if self.kind == "decode_seq":
                    sdm.decode_seq(self.x["bank"], *dev_in, out=self.out)
                elif self.kind == "decode_seq_stream_major":
                    sdm.decode_seq(self.x["bank"], *dev_in, out=self.out, stream_major=True)
                else:
                    for t in range(wl.T):
                        sdm.decode_step(self.x["bank"], *(d[t] for d in dev_in), out=self.out[t])
                host_out.copy_(self.out, non_blocking=True)
        else:
            g = self.g
            flat = [t for op in g["ops"] for t in op] + ([g["chunk_valid"]] if g["chunk_valid"] is not None else [])
            flat += [self.kpos] if self.kpos is not None else []
            host_in = [t.cpu().pin_memory() for t in flat]
            dev_in = [torch.empty_like(t) for t in flat]
            host_outs = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in self.outs]
            d2h = sum(o.numel() * o.element_size() for o in host_outs)
            n_ops = len(g["ops"])

            def step():
                for d, h in zip(dev_in, host_in):
                    d.copy_(h, non_blocking=True)
                ops = [(dev_in[2 * o], dev_in[2 * o + 1]) for o in range(n_ops)]
                cv = dev_in[2 * n_ops] if g["chunk_valid"] is not None else None
                kp = dev_in[-1] if self.kpos is not None else None
                sdm.gather(g["bank"], ops, chunk=wl.chunk, chunk_valid=cv, stash=self.stash, outs=self.outs,
                           with_stash=self.stash is not None, kpos=kp, compact=self.compact)
                for h, o in zip(host_outs, self.outs):
                    h.copy_(o, non_blocking=True)
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sdist.barrier(r, dev)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = sdist.max_over_ranks(r, e0.elapsed_time(e1), dev)
        return {"value": self.units * steps * r.world / (ms / 1e3), "unit": self.unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps}

    # the oracle on the host cores, on a time-bounded sample of this workload's own inputs
    def cpu_baseline(self, budget_s: float) -> dict:
        if self.kind.startswith("decode"):
            S, P = self.wl.n_streams, self.wl.slots_per_stream
            order = torch.randperm(S, generator=torch.Generator().manual_seed(0)).tolist()
            done, secs, n = 0, 0.0, 0
            xt = self.x  # the oracle takes time-major arrays: a stream-major case is viewed back
            if self.kind == "decode_seq_stream_major":
                xt = {k: (v.transpose(0, 1) if k in DECODE_KEYS else v) for k, v in self.x.items()}
            for s in order:
                d, t = oracle_stream_tokens(xt, [s], P)
                done, secs, n = done + d, secs + t, n + 1
                if secs >= budget_s:
                    break
            sample = (f"{n} of {S} streams x {self.wl.T} tokens of the benchmark's own inputs "
                      f"({done} stream-tokens, {secs:.1f} s single-threaded)")
        else:
            bank_h = _np(self.g["bank"])
            order = torch.randperm(self.wl.tokens, generator=torch.Generator().manual_seed(0))
            done, secs, i = 0, 0.0, 0
            while secs < budget_s and i < self.wl.tokens:
                d, t = oracle_gather_tokens(bank_h, self.g, order[i:i + 256].tolist(), self.wl.chunk)
                done, secs, i = done + d, secs + t, i + 256
            sample = (f"{done} of {self.wl.tokens} tokens of the benchmark's own inputs "
                      f"(padding included, {secs:.1f} s single-threaded"
                      + ("" if self.form == "stash" else "; the oracle's outputs-and-stash form") + ")")
        return {"value": done / secs, "unit": self.unit, "cores": 1, "kind": "oracle", "sample": sample}

    def cpu_baseline_all_cores(self, budget_s: float, single: dict):
        """The oracle on every host core at once: one process per core (spawn: CUDA is already
        initialised here), each over its own streams of the same workload recipe. The value is all
        processes' stream-tokens over the wall-clock span from the first start to the last end."""
        if not self.kind.startswith("decode"):
            return None
        import dataclasses
        import multiprocessing as mp

        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        streams = min(8, self.wl.n_streams)
        per_rep_s = streams * self.wl.T / max(single["value"], 1e-9)
        reps = max(1, int(budget_s / per_rep_s))
        jobs = [(dataclasses.asdict(self.wl), 1000 + i, streams, reps) for i in range(cores)]
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_worker, jobs)
        done = sum(r[0] for r in res)
        span = max(r[2] for r in res) - min(r[1] for r in res)
        sample = (f"{cores} processes at once, each {reps} passes over {streams} streams x {self.wl.T} tokens drawn "
                  f"with the workload's recipe (seeds 1000..{999 + cores}); {done} stream-tokens in {span:.1f} s "
                  f"of wall clock")
        return {"value": done / span, "unit": self.unit, "cores": cores, "kind": "oracle", "sample": sample}


# ---------------------------------------------------------------- our arm


def run_ours(args, r: sdist.Rank):
    from decode_state_gb300 import sdm

    dev = torch.device("cuda", r.local_rank)
    torch.cuda.set_device(dev)
    sdm.library()
    case = Case(args, dev, r)
    for _ in range(args.warmup):
        case.step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(dev)
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sdist.barrier(r, dev)
    torch.cuda.synchronize()
    h0 = time.time()
    e0.record(stream)
    for a, b in ev:
        a.record(stream)
        case.step()
        b.record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    h1 = time.time()
    sdist.barrier(r, dev)
    time.sleep(0.2)
    sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    step_ms = statistics.fmean(a.elapsed_time(b) for a, b in ev)
    max_ms = sdist.max_over_ranks(r, elapsed_ms, dev)
    value = case.units * args.steps * r.world / (max_ms / 1e3)
    peak, peak_kind = hbm_peak()
    launch_ms = step_ms / case.launches
    achieved = case.nbytes / case.launches / (launch_ms / 1e3) / 1e9
    res = {
        "metric": case.metric, "value": value, "unit": case.unit, "n_gpus": r.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": case.config(r), "call": case.call(),
        "effective_gbs": case.nbytes * args.steps * r.world / (max_ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(case.wl.name), "peak_kind": peak_kind, "kernel": case.kernel,
                     "algorithmic_bytes_per_launch": case.nbytes // case.launches, "avg_launch_ms": launch_ms},
        "gpu_launches": args.steps * case.launches,
        "clocks": sampler.summary(h0, h1),
    }
    res["e2e"] = case.e2e(max(3, min(args.steps, 200)), r)
    res["device_status"] = sdm.device_status()
    return res, case


def _time_calls(fn, reps: int, warm: int = 3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def extras(args, dev, r: sdist.Rank, peak: float, skip: str):
    """The other workloads (parity cases of the test suite), timed briefly for context."""
    res = {}
    for name in list(workloads.DECODE_WORKLOADS) + list(workloads.GATHER_WORKLOADS):
        if name == skip or name == workloads.C0.name:
            continue
        a = argparse.Namespace(**vars(args))
        a.workload, a.streams, a.tokens = name, 0, 0
        case = Case(a, dev, r)
        reps = 5 if case.kind == "decode_step" else 20
        ms = _time_calls(case.step, reps)
        item = {"unit_per_s": case.units / (ms / 1e3), "unit": case.unit, "ms_per_step": ms,
                "effective_gbs": case.nbytes / (ms / 1e3) / 1e9, "frac_of_hbm_peak": case.nbytes / (ms / 1e3) / 1e9 / peak,
                "launches_per_step": case.launches}
        if case.kind == "decode_step":  # the same single-token launches replayed from a CUDA graph
            graph = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream(dev)
            s.wait_stream(torch.cuda.current_stream(dev))
            with torch.cuda.stream(s):
                case.step()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=s):
                    case.step()
            torch.cuda.current_stream(dev).wait_stream(s)
            gms = _time_calls(graph.replay, reps, 1)
            item.update({"graph_unit_per_s": case.units / (gms / 1e3), "graph_ms_per_step": gms,
                         "graph_us_per_launch": gms * 1e3 / case.launches})
            del graph
            from decode_state_gb300 import sdm

            # the graph again with every launch promising its inputs staged ahead (SDM_INPUTS_READY,
            # as DecodeStepGraph does): the inputs are written before the replay starts
            def ready_steps():
                for t in range(case.wl.T):
                    sdm.decode_step(case.x["bank"], *(case.x[k][t] for k in DECODE_KEYS), out=case.out[t],
                                    inputs_ready=True)

            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                ready_steps()
                torch.cuda.synchronize()
                with torch.cuda.graph(graph, stream=s):
                    ready_steps()
            torch.cuda.current_stream(dev).wait_stream(s)
            rgms = _time_calls(graph.replay, reps, 1)
            item.update({"graph_ready_unit_per_s": case.units / (rgms / 1e3), "graph_ready_ms_per_step": rgms,
                         "graph_ready_us_per_launch": rgms * 1e3 / case.launches})
            del graph
            # the same launches eagerly through a plan (checked once, pointers precomputed)

            plan = sdm.DecodeStepPlan(case.x["bank"], {k: case.x[k] for k in DECODE_KEYS}, out=case.out,
                                      stream=torch.cuda.current_stream(dev))

            def plan_steps():
                for t in range(case.wl.T):
                    plan.launch(t)

            pms = _time_calls(plan_steps, reps)
            item.update({"plan_unit_per_s": case.units / (pms / 1e3), "plan_ms_per_step": pms,
                         "plan_us_per_launch": pms * 1e3 / case.launches})
            # the same plan promising inputs staged ahead (SDM_INPUTS_READY): each launch loads its
            # metadata and warms L2 while the launch ahead of it still runs
            plan = sdm.DecodeStepPlan(case.x["bank"], {k: case.x[k] for k in DECODE_KEYS}, out=case.out,
                                      stream=torch.cuda.current_stream(dev), inputs_ready=True)
            rms = _time_calls(plan_steps, reps)
            item.update({"plan_ready_unit_per_s": case.units / (rms / 1e3), "plan_ready_ms_per_step": rms,
                         "plan_ready_us_per_launch": rms * 1e3 / case.launches})
            # every step of the plan from one call into the library's own loop (sdm_decode_plan_walk)
            wms = _time_calls(plan.walk, reps)
            item.update({"plan_walk_ready_unit_per_s": case.units / (wms / 1e3), "plan_walk_ready_ms_per_step": wms,
                         "plan_walk_ready_us_per_launch": wms * 1e3 / case.launches})
            del plan
        res[name] = item
        del case
        torch.cuda.empty_cache()
    return res


def plan_slabs(dev, slab: int = 256) -> dict:
    """The gather workload's index tensor walked in slabs of `slab` tokens: one launch per slab
    through a gather plan (checked once) against direct sdm_gather calls on the same slabs (no
    stash). Device time per walk and host time per call, for the launch-overhead comparison."""
    from decode_state_gb300 import sdm

    wl = workloads.C4.scaled(stash=False, per_chunk_valid=False)
    g = workloads.make_gather_inputs(wl, device=dev)
    n = wl.tokens // slab
    plan = sdm.GatherPlan(g["bank"], g["ops"], tokens=slab, chunk=wl.chunk)
    outs = plan.outs
    slabs = [[(i[k * slab:(k + 1) * slab], w[k * slab:(k + 1) * slab]) for i, w in g["ops"]] for k in range(n)]

    def via_plan():
        for k in range(n):
            plan.launch(k * slab)

    def via_plan_ready():  # the index rows exist before the walk: SDM_INPUTS_READY holds
        for k in range(n):
            plan.launch(k * slab, inputs_ready=True)

    def direct():
        for k in range(n):
            sdm.gather(g["bank"], slabs[k], chunk=wl.chunk, outs=outs, with_stash=False)

    walk_rows, _ = sdm.GatherPlan.walk_arrays([k * slab for k in range(n)])

    def native_walk():  # every slab from one call into the library's own loop
        plan.walk(walk_rows)

    def native_walk_ready():
        plan.walk(walk_rows, inputs_ready=True)

    res = {"slab_tokens": slab, "launches_per_walk": n}
    for name, fn in (("plan", via_plan), ("plan_ready", via_plan_ready), ("plan_walk", native_walk),
                     ("plan_walk_ready", native_walk_ready), ("direct", direct)):
        ms = _time_calls(fn, 5)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fn()
        host_us = (time.perf_counter() - t0) * 1e6 / n
        torch.cuda.synchronize()
        res[name] = {"ms_per_walk": ms, "us_per_launch": ms * 1e3 / n, "host_us_per_launch": host_us}
    # the plan walks replayed from CUDA graphs: device time per launch without the host calls
    side = torch.cuda.Stream(dev)
    for name, fn in (("plan_graph", via_plan), ("plan_ready_graph", via_plan_ready)):
        graph = torch.cuda.CUDAGraph()
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                fn()
        torch.cuda.current_stream(dev).wait_stream(side)
        ms = _time_calls(graph.replay, 5, 1)
        res[name] = {"ms_per_walk": ms, "us_per_launch": ms * 1e3 / n}
        del graph
    return res


def compact_snapshot(wl, g: dict, dev):
    """Inputs of the compact-snapshot form of a gather workload: operand 0's rows are stored once
    per chunk, at the first position of each distinct row among the chunk's sorted entries. Returns
    (kpos [tokens, W0] int32, the zeroed snapshot [chunks, chunk * W0, hd], rows written by live
    tokens), prepared on the device."""
    idx0 = g["ops"][0][0]
    W0, n_chunks = idx0.shape[1], wl.tokens // wl.chunk
    ent = idx0.view(n_chunks, wl.chunk * W0)
    srt, order = ent.sort(dim=1, stable=True)
    first = torch.ones_like(srt, dtype=torch.bool)
    first[:, 1:] = srt[:, 1:] != srt[:, :-1]
    pos = torch.arange(srt.shape[1], device=dev).expand_as(srt)
    first_pos = torch.cummax(torch.where(first, pos, torch.zeros_like(pos)), dim=1).values
    kpos = torch.empty_like(srt).scatter_(1, order, torch.where(first, first_pos, torch.full_like(pos, -1)))
    kpos = kpos.view(wl.tokens, W0).to(torch.int32)
    compact = torch.zeros((n_chunks, wl.chunk * W0, wl.hd), dtype=workloads.BANK_DTYPES[wl.bank_dtype], device=dev)
    live = (torch.arange(wl.tokens, device=dev) % wl.chunk) < g["chunk_valid"].repeat_interleave(wl.chunk)
    written = int(((kpos >= 0) & live[:, None]).sum().item())
    return kpos, compact, written


def gather_form_bytes(wl, g: dict, form: str, written: int = 0) -> int:
    """Algorithmic bytes of one gather call in the given form: the workload's own (stash), or
    live-token row reads and outputs plus the compact rows written (compact), or without them (none)."""
    if form == "stash":
        return workloads.gather_bytes(wl, g["chunk_valid"])
    es = 2 if wl.bank_dtype == "bf16" else 4
    live = int(g["chunk_valid"].to(torch.int64).sum().item()) if g["chunk_valid"] is not None else wl.tokens
    return live * sum(wl.widths) * wl.hd * es + written * wl.hd * es + wl.tokens * len(wl.widths) * wl.hd * 4


def kpos_gather(dev, peak: float) -> dict:
    """The gather workload with a compact snapshot (sdm_gather_kpos) in place of the stash."""
    from decode_state_gb300 import sdm

    wl = workloads.C4
    g = workloads.make_gather_inputs(wl, device=dev)
    kpos, compact, written = compact_snapshot(wl, g, dev)
    outs = [torch.empty((wl.tokens, wl.hd), device=dev) for _ in wl.widths]
    nbytes = gather_form_bytes(wl, g, "compact", written)

    def step():
        sdm.gather(g["bank"], g["ops"], chunk=wl.chunk, chunk_valid=g["chunk_valid"], kpos=kpos, compact=compact,
                   outs=outs)

    ms = _time_calls(step, 20)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": wl.name + " with a compact snapshot", "unit_per_s": wl.tokens / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "compact_rows_written": written, "algorithmic_bytes": nbytes, "effective_gbs": gbs,
            "frac_of_hbm_peak": gbs / peak}


# ---------------------------------------------------------------- reference arm (the oracle)


def run_reference(args, r: sdist.Rank):
    """The CPU oracle on the host cores: each step is the oracle over a bounded sample of whole
    streams of the same workload: the first streams of the benchmark's own job (its first block of
    streams, drawn on the host with the same recipe and seed)."""
    if args.workload not in workloads.DECODE_WORKLOADS:
        raise SystemExit("--impl reference times the decode workloads")
    base = workloads.DECODE_WORKLOADS[args.workload]
    n_pool = min(8, base.n_streams)
    wl = base.scaled(n_streams=n_pool)
    xb = workloads.make_decode_shard(base, 0, min(workloads.SHARD_BLOCK, base.n_streams), device="cpu")
    x = {k: (v[:, :n_pool] if k in DECODE_KEYS else v[:n_pool * base.slots_per_stream]) for k, v in xb.items()}
    del xb
    _, per_stream_s = oracle_stream_tokens(x, [0], wl.slots_per_stream)
    total = args.steps + args.warmup
    budget = 90.0
    per_step_streams = max(1, min(n_pool, int(budget / total / max(per_stream_s, 1e-6))))
    T_used = wl.T
    if per_stream_s * total > budget:  # even one whole stream per step is too long: a prefix of its tokens
        T_used = max(1, int(wl.T * budget / total / per_stream_s))
    xs = {k: (v[:T_used] if k in DECODE_KEYS else v) for k, v in x.items()}

    def step(i):
        lo = (i * per_step_streams) % n_pool
        return oracle_stream_tokens(xs, [(lo + j) % n_pool for j in range(per_step_streams)], wl.slots_per_stream)

    for i in range(args.warmup):
        step(i)
    done, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        done += step(i)[0]
    secs = time.perf_counter() - t0
    value = done / secs
    sample = (f"{per_step_streams} whole stream(s) x {T_used} token(s) per step, cycling over the first {n_pool} "
              f"streams of the benchmark's own job")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": r.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": decode_config(base, r), "call": "oracle_sdm_decode_seq (CPU)",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    r = sdist.init_from_env()
    try:
        if args.impl == "reference":
            if r.is_root:
                print(json.dumps(run_reference(args, r)), flush=True)
            return
        res, case = run_ours(args, r)
        if r.is_root:
            res["cpu_baseline"] = case.cpu_baseline(args.cpu_seconds)
        if r.is_root and r.world == 1 and not args.no_extras:
            res["cpu_baseline_all_cores"] = case.cpu_baseline_all_cores(args.cpu_seconds / 2, res["cpu_baseline"])
        del case
        torch.cuda.empty_cache()
        if r.is_root and r.world == 1 and not args.no_extras:
            res["other_workloads"] = extras(args, torch.device("cuda", r.local_rank), r, res["roofline"]["peak"],
                                            res["config"]["workload"])
            res["other_workloads"]["gather_plan_slabs"] = plan_slabs(torch.device("cuda", r.local_rank))
            torch.cuda.empty_cache()
            res["other_workloads"]["gather_kpos"] = kpos_gather(torch.device("cuda", r.local_rank),
                                                                res["roofline"]["peak"])
            torch.cuda.empty_cache()
        if r.is_root:
            print(json.dumps(res), flush=True)
    finally:
        sdist.shutdown(r)


if __name__ == "__main__":
    main()
