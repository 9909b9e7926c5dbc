"""GB300-native (sm_103a) training step of a Qwen3-style decoder block stack.

The compute path lives in ``librdt.so`` (hand-written CUDA kernels behind a
C ABI declared in ``include/rdt.h``); ``rdt`` is its thin ctypes binding and
``step`` drives one full training step through it. ``synth`` draws the seeded
synthetic inputs.
"""
