"""CPU oracle for the owner-rank Muon update (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import this package. It shares no code with the CUDA library: see ``ns64`` (float64) and
``exact`` (exact rationals on tiny inputs).
"""
from . import exact, ns64  # noqa: F401
