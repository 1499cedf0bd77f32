"""CPU oracle for the skinny decode projection -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.  See ``oracle.c`` for the definition it computes and
the passages of "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and
Responsibly" it follows.
"""
from .oracle import (  # noqa: F401
    build,
    bf16_decode,
    bf16_round,
    ulp_bf16,
    linear,
    linear_points,
    max_threads,
    library_path,
)
