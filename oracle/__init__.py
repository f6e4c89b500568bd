"""fp64 CPU oracle for the Flux MMDiT block forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The library never does, and the
oracle imports nothing from the library.

Modules: ``flux`` (the blocks, the whole model, rectified flow, sampling step),
``e4m3`` (E4M3 and delayed scaling), ``e5m2`` (the gradient format), ``fp8_recipes``
(tensorwise, blockwise, MXFP8), ``fp8_attention``, ``backward`` (block and whole-model
gradients), ``fp8_backward`` (the FP8 linear backward).
"""
from . import flux, e4m3  # noqa: F401
