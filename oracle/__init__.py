"""CPU oracle for one Transformer layer forward -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 NumPy statement of what the layer computes, written from
the Megatron pages.  Only the tests, the smoke check and the bench's CPU-baseline
and reference legs may import it; the product path never does.  It shares no
code with the CUDA library: its only dependency inside this repository is the
seeded input generator (``synth``), which holds no layer arithmetic.

Parity status of each function is listed in ``oracle.layer``'s header.
"""
from .layer import *  # noqa: F401,F403
