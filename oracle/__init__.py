"""CPU oracle for continuous depth batching (test infrastructure only).

This package is the plain, slow reference that the CUDA library is checked
against.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline may import it; the library itself never does and shares no code with
it.
"""

from .model import (  # noqa: F401
    OracleModel,
    SeqTrace,
    decode_sequence,
    iter_decode,
    decode_workload,
)
