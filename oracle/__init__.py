"""CPU fp64 oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this package.  It shares no code with the CUDA library.
"""

from .ref import ref_decode, ref_prefill  # noqa: F401
