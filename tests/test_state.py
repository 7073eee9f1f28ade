"""Host-side decode state holder (bank + token count): bookkeeping on the CPU; the GPU test
checks that stepping it equals the multi-token call and the oracle."""

import pytest
import torch

from decode_state_gb300.state import SDMLayerState


def test_bookkeeping():
    bank = torch.ones((8, 4))
    st = SDMLayerState(bank, seq_len=3)
    assert st.cache_len == 3 and len(st) == 1 and st[0] is bank
    with pytest.raises(KeyError):
        st[1]
    other = torch.full((8, 4), 2.0)
    assert st.update_(other, seq_len=5) is st
    assert st.cache_len == 8 and torch.equal(st.memory, other)
    st.reset()
    assert st.cache_len == 0 and not st.memory.any()


def test_step_rejects_host_tensors_and_keeps_count():
    st = SDMLayerState(torch.zeros((16, 8)))
    k = torch.zeros((2, 3), dtype=torch.int32)
    f = torch.zeros((2, 3))
    with pytest.raises(ValueError):
        st.step(k, f, torch.zeros((2, 8)), torch.zeros(2), torch.zeros((2, 1)), k, f)
    assert st.cache_len == 0
