"""GB300-native KDA (Kimi Delta Attention) layer step.

The compute path lives in ``libkda.so`` (C ABI, hand-written sm_103a CUDA
kernels, sources under ``csrc/``, declarations in ``include/kda.h``).
``hybrid_linear_attention_03_gb300.kda`` is the thin ctypes binding with the
same entry-point names; ``inputs`` holds the seeded synthetic workloads.
Importing the package loads nothing; the binding loads the library on first
use and raises if it is missing.
"""
