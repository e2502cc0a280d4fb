"""GB300-native speculative-decoding verify step (W4A16 target, int8 lm_head).

The compute path is the C-ABI library ``libw4v.so`` (hand-written CUDA for
sm_103a, built from ``csrc/``); ``w4v`` is its thin ctypes binding and
``inputs`` the seeded synthetic-input generators.  Submodules load lazily so
that importing ``inputs`` needs no GPU.
"""
