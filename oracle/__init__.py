"""CPU fp64 oracle for GPTQ's per-layer quantization — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct NumPy restatement of what the GPTQ pages compute,
used to check the CUDA path. Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does, and it
shares no code with the CUDA library (the two only share the seeded input
generators in `synth`).

Every pinned function is checked in `tests/test_oracle_pins.py` against facts
that do not come from this module: printed page values, closed forms, brute
force, and limit cases that reduce to round-to-nearest.
"""
from .gptq_oracle import *  # noqa: F401,F403
from .gptq_oracle import __all__  # noqa: F401
