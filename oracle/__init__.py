"""CPU oracle of the scaled FP8 cast -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import, call or link anything here.  It shares no code with the CUDA
library ``tensor_scaling_cast_gb300`` and never imports it.

  spec.py     exact Fraction + explicit-sign definition (tiny inputs)
  oracle.c    plain C, integer bit manipulation (used at scale)
  coracle.py  ctypes binding of oracle.c
  policy.py   per-tensor window / margin / hysteresis state machine
"""
