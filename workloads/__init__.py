"""Seeded synthetic workloads for speculative-decoding verify attention and sampling.

This package only draws random inputs with the shapes and value distributions of the
workloads described on the pages (LLaMA-3-8B / 70B-shaped layers, MagicDec long context,
Medusa-style trees).  It holds none of the method's arithmetic: no attention, no softmax,
no accept/reject.  Both the CUDA path's tests/bench and the CPU oracle's tests consume it.
"""

from .configs import CONFIGS, WorkloadConfig, get_config  # noqa: F401
