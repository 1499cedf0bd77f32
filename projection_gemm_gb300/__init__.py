"""Skinny decode projection GEMM for one GB300 (sm_103a).

y = x.W^T (+ residual), M = 1..64 tokens, bf16 operands, fp32 accumulation,
computed by the CUDA kernels of ``lib/libskg.so`` behind the C ABI of
``include/skg.h``.  ``skg`` is the ctypes binding; ``inputs`` draws seeded
synthetic operands; ``build`` compiles the library.
"""
from . import skg  # noqa: F401
from .skg import Plan, SkgError  # noqa: F401
