"""GB300 (sm_103a) Flux MMDiT block forward: CUDA kernels behind a C ABI (libmmdit.so).

``build_ext`` compiles the library, ``_lib`` is its ctypes binding (argument marshalling only)
and ``synth`` draws the seeded synthetic inputs.  Importing the package loads nothing; the
library is loaded on first use of ``_lib`` and there is no CPU fallback.
"""
__all__ = ["build_ext", "synth"]
