"""fp64 CPU oracle for exact attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path.
"""

from .attention import (  # noqa: F401
    ROW_STRIPE,
    attention_backward,
    attention_forward,
    head_backward,
    head_forward,
    head_probabilities,
    varlen_backward,
    varlen_forward,
)
