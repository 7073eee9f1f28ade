"""Host-fed decode: per-step inputs arrive from pinned host memory and the readings go back to it.

``HostFedDecoder`` keeps ``depth`` sets of device input/output buffers. For step n (buffer set
i = n % depth) it copies the step's inputs host->device on a copy stream, runs ``sdm_decode_seq`` on
the compute stream once they have landed, and copies the readings device->host on a third stream.
The bank is only touched by the compute stream, so steps apply in submission order; with two or
more buffer sets the copies of one step overlap the kernel of the previous one. PyTorch provides
the streams, events and buffers; every decode runs in the CUDA library.
"""

from __future__ import annotations

import torch

from . import sdm

DECODE_INPUTS = ("k_idx", "k_val", "v", "beta", "g", "q_idx", "q_val")


class HostFedDecoder:
    """Pipelined multi-token decode of one bank from pinned host inputs.

    ``like`` maps each name of ``DECODE_INPUTS`` to a tensor with the per-step shape and dtype
    (time-major [T, S, .], beta [T, S]); only shapes and dtypes are used.
    """

    def __init__(self, bank: torch.Tensor, like: dict, depth: int = 2):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.bank = bank
        dev = bank.device
        self.device = dev
        self.depth = depth
        self.inputs = [{k: torch.empty(like[k].shape, dtype=like[k].dtype, device=dev) for k in DECODE_INPUTS}
                       for _ in range(depth)]
        T, S = like["k_idx"].shape[:2]
        self.outs = [torch.empty((T, S, bank.shape[1]), dtype=bank.dtype, device=dev) for _ in range(depth)]
        self.h2d = torch.cuda.Stream(dev)
        self.compute = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.loaded = [torch.cuda.Event() for _ in range(depth)]
        self.used = [torch.cuda.Event() for _ in range(depth)]
        self.returned = [torch.cuda.Event() for _ in range(depth)]
        self.n = 0

    def submit(self, host_inputs: dict, host_out: torch.Tensor) -> torch.cuda.Event:
        """Queue one step: host_inputs (pinned, per-step shapes) in, readings into host_out (pinned).
        Returns the event that completes when host_out holds the readings."""
        i = self.n % self.depth
        self.n += 1
        ins, out = self.inputs[i], self.outs[i]
        with torch.cuda.stream(self.h2d):
            self.h2d.wait_event(self.used[i])  # the kernel that last read buffer set i has finished
            for k in DECODE_INPUTS:
                ins[k].copy_(host_inputs[k], non_blocking=True)
            self.loaded[i].record(self.h2d)
        with torch.cuda.stream(self.compute):
            self.compute.wait_event(self.loaded[i])
            self.compute.wait_event(self.returned[i])  # its readings buffer has been copied out
            sdm.decode_seq(self.bank, *(ins[k] for k in DECODE_INPUTS), out=out, stream=self.compute)
            self.used[i].record(self.compute)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.used[i])
            host_out.copy_(out, non_blocking=True)
            self.returned[i].record(self.d2h)
        return self.returned[i]

    def synchronize(self):
        for s in (self.h2d, self.compute, self.d2h):
            s.synchronize()
