"""GB300-native sparse delta-memory (SDM) decode state: decode step, multi-token decode, token gather.

The compute runs in the C-ABI CUDA library ``libsdm.so`` (built from ``csrc/``); this package is a
thin binding over it. See ``sdm.py`` for the Python entry points.
"""
