"""CPU oracle for the owner-rank Muon update (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm may
import this package. It shares no code with the CUDA library: see ``ns64`` (float64) and
``exact`` (exact rationals on tiny inputs). ``fp16_model`` is not an oracle but the fp16 error floor
the GPU's error is judged against (tests only).
"""
from . import exact, fp16_model, ns64  # noqa: F401
