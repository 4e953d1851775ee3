"""Q8_0 GEMV for batch-1 / small-batch LLM decode, hand-written for GB300 (sm_103a).

The compute path is the C-ABI library liblk.so (include/lk.h), built in-tree
by ``q8_quantized_gemv_gb300.build.build()``; ``q8_quantized_gemv_gb300.lk``
is its thin binding.  ``synth`` draws the seeded synthetic inputs.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "lk", "build"]
