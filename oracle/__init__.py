"""fp64 CPU oracle for the Flux MMDiT block forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The library never does, and the
oracle imports nothing from the library.
"""
from . import flux, e4m3  # noqa: F401
