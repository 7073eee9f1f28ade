"""Host-side decode state of one SDM layer: the memory bank and the number of tokens consumed.

Mirrors ``SDMLayerState`` of the sparse-delta-memory 2.0.0 wheel (cache.py): the state is the bank
(a device tensor updated in place by every decode call) plus a running token count; ``update_``
swaps in a new bank and advances the count, ``reset`` zeroes the bank and the count. ``step`` and
``steps`` advance the state through the C ABI (``sdm_decode_step`` / ``sdm_decode_seq``).
"""

from __future__ import annotations

import torch

from . import sdm


class SDMLayerState:
    """Decode state: ``memory`` [num_slots, head_dim] (bf16 or float32, on the GPU) and ``cache_len``."""

    def __init__(self, memory: torch.Tensor, seq_len: int = 0) -> None:
        self.memory = memory
        self._cache_len = int(seq_len)

    def __getitem__(self, key_idx: int) -> torch.Tensor:
        if key_idx == 0:
            return self.memory
        raise KeyError(key_idx)

    def __len__(self) -> int:
        return 1

    @property
    def cache_len(self) -> int:
        return self._cache_len

    def reset(self) -> None:
        """Zero the bank and the token count."""
        self.memory.zero_()
        self._cache_len = 0

    def update_(self, new_memory: torch.Tensor, seq_len: int = 1) -> "SDMLayerState":
        """Take ``new_memory`` as the bank and count ``seq_len`` more tokens."""
        if self.memory is None:
            raise RuntimeError("the state has no bank")
        self.memory = new_memory.detach()
        self._cache_len += int(seq_len)
        return self

    def step(self, k_idx, k_val, v, beta, g, q_idx, q_val, out=None, stream=None) -> torch.Tensor:
        """One token for every stream (arrays [S, .], beta [S]); returns the readings [S, head_dim]."""
        readings = sdm.decode_step(self.memory, k_idx, k_val, v, beta, g, q_idx, q_val, out=out, stream=stream)
        self._cache_len += 1
        return readings

    def steps(self, k_idx, k_val, v, beta, g, q_idx, q_val, out=None, stream=None) -> torch.Tensor:
        """T tokens for every stream in one launch (time-major arrays [T, S, .], beta [T, S]);
        returns the readings [T, S, head_dim]."""
        readings = sdm.decode_seq(self.memory, k_idx, k_val, v, beta, g, q_idx, q_val, out=out, stream=stream)
        self._cache_len += int(k_idx.shape[0])
        return readings
