"""Decode-time Mixture-of-Experts layer with GPU expert slots, for GB300 (sm_103a).

The compute path lives in ``libmoe.so`` (CUDA kernels behind a C ABI, declared
in ``include/moe.h``); ``expert_offload_moe_gb300.moe`` is the thin ctypes
binding with the same call names.  ``synth`` draws the seeded inputs.
Importing this package loads nothing; ``moe.lib()`` loads the library and
raises if it has not been built.
"""
