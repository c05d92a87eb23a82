"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The library never calls it, and it shares
no code with the CUDA path.  See ``oracle/attention.py`` for the functions and
the passages each one follows.
"""
from .attention import (  # noqa: F401
    EXP2_POLY, attention_backward, attention_forward, exp2_cubic,
    head_backward, head_backward_from_saved, head_forward, online_softmax_forward,
    softmax_probs,
)
