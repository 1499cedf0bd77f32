"""Python binding of libskg.so (see include/skg.h) -- argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but convert arguments: torch tensors become device pointers, streams
become cudaStream_t handles, statuses become exceptions.  All computation
happens in the library's CUDA kernels; if the library is missing this module
raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libskg.so")

SKG_OK = 0
SKG_ERR_INVALID_ARG = 1
SKG_ERR_UNSUPPORTED = 2
SKG_ERR_ALIGNMENT = 3
SKG_ERR_CUDA = 4
SKG_ERR_DEVICE_TIMEOUT = 5

SKG_EPI_BF16 = 0
SKG_EPI_BF16_RESIDUAL = 1
SKG_EPI_FP32 = 2
EPILOGUES = {"bf16": SKG_EPI_BF16, "bf16_residual": SKG_EPI_BF16_RESIDUAL, "fp32": SKG_EPI_FP32}

CANONICAL_CHUNKS = 16     # SKG_CANONICAL_CHUNKS of include/skg.h

SKG_KERNEL_GEMV = 1
SKG_KERNEL_SPLITK_TC = 2
KERNEL_NAMES = {SKG_KERNEL_GEMV: "gemv", SKG_KERNEL_SPLITK_TC: "splitk_tc"}

# Every symbol include/skg.h declares.
EXPORTS = (
    "skg_plan_query", "skg_plan", "skg_plan_force", "skg_plan_force_kernel", "skg_plan_set_pdl", "skg_run",
    "skg_prefetch_l2", "skg_plan_set_prefetch_fraction", "skg_plan_info", "skg_plan_check",
    "skg_plan_destroy", "skg_debug_wait_timeout", "skg_last_error", "skg_version",
    "skg_run_noalloc", "skg_noalloc_check", "skg_plan_set_k_shard", "skg_combine_partials", "skg_plan_set_l2_ahead", "skg_plan_set_next_weight",
    "skg_plan_set_reducers",
    "skg_group", "skg_group_run", "skg_group_info", "skg_group_check", "skg_group_destroy",
)


class SkgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"skg status {status}: {message}")
        self.status = status


class skg_plan_desc(ctypes.Structure):
    _fields_ = [
        ("kernel_kind", ctypes.c_int), ("M", ctypes.c_int), ("N", ctypes.c_int),
        ("K", ctypes.c_int), ("epilogue", ctypes.c_int), ("split_k", ctypes.c_int),
        ("tile_n", ctypes.c_int), ("m_pad", ctypes.c_int), ("stages", ctypes.c_int),
        ("tma_burst", ctypes.c_int),
        ("grid", ctypes.c_int), ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_int),
        ("from_table", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
        ("prefetch_bytes", ctypes.c_size_t), ("pdl", ctypes.c_int), ("l2_ahead", ctypes.c_int),
        ("reducers", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
    ]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["kernel"] = KERNEL_NAMES.get(self.kernel_kind, "?")
        return d


_lib = None


def load(path: str = LIB_PATH):
    """Load libskg.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m projection_gemm_gb300.build` "
                           "(there is no other implementation of the projection)")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    lib.skg_plan_query.argtypes = [i, i, i, i, i, sz, P(skg_plan_desc)]
    lib.skg_plan.argtypes = [i, i, i, i, P(vp)]
    lib.skg_plan_force.argtypes = [vp, i, i, i, i]
    lib.skg_plan_set_pdl.argtypes = [vp, i]
    lib.skg_plan_force_kernel.argtypes = [vp, i]
    lib.skg_run.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.skg_prefetch_l2.argtypes = [vp, vp, vp]
    lib.skg_plan_set_prefetch_fraction.argtypes = [vp, ctypes.c_double]
    lib.skg_plan_info.argtypes = [vp, P(skg_plan_desc)]
    lib.skg_plan_check.argtypes = [vp]
    lib.skg_plan_destroy.argtypes = [vp]
    lib.skg_debug_wait_timeout.argtypes = [vp, ctypes.c_ulonglong, vp]
    lib.skg_run_noalloc.argtypes = [i, i, i, i, vp, vp, vp, vp, vp]
    lib.skg_noalloc_check.argtypes = [vp]
    lib.skg_plan_set_k_shard.argtypes = [vp, i, i]
    lib.skg_combine_partials.argtypes = [i, i, i, P(vp), vp, vp, i, vp]
    lib.skg_plan_set_l2_ahead.argtypes = [vp, i]
    lib.skg_plan_set_reducers.argtypes = [vp, i]
    lib.skg_plan_set_next_weight.argtypes = [vp, vp, sz]
    lib.skg_group.argtypes = [i, i, P(i), P(i), P(i), P(i), P(vp)]
    lib.skg_group_run.argtypes = [vp, P(vp), P(vp), P(vp), P(vp), vp]
    lib.skg_group_info.argtypes = [vp, P(i), P(i), P(i), P(i)]
    lib.skg_group_check.argtypes = [vp]
    lib.skg_group_destroy.argtypes = [vp]
    for name in EXPORTS:
        getattr(lib, name).restype = ctypes.c_int
    lib.skg_last_error.restype = ctypes.c_char_p
    lib.skg_last_error.argtypes = []
    lib.skg_version.argtypes = []
    _lib = lib
    return lib


def _check(status: int):
    if status != SKG_OK:
        raise SkgError(status, load().skg_last_error().decode(errors="replace"))


def _epi(epilogue) -> int:
    return EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def skg_version() -> int:
    return int(load().skg_version())


def skg_last_error() -> str:
    return load().skg_last_error().decode(errors="replace")


def skg_plan_query(M: int, N: int, K: int, epilogue, num_sms: int, l2_bytes: int) -> dict:
    d = skg_plan_desc()
    _check(load().skg_plan_query(M, N, K, _epi(epilogue), num_sms, l2_bytes, ctypes.byref(d)))
    return d.as_dict()


def skg_plan(M: int, N: int, K: int, epilogue) -> int:
    h = ctypes.c_void_p()
    _check(load().skg_plan(M, N, K, _epi(epilogue), ctypes.byref(h)))
    return h.value


def skg_plan_force(plan: int, split_k: int = 0, stages: int = 0, grid: int = 0, tma_burst: int = 0):
    _check(load().skg_plan_force(plan, split_k, stages, grid, tma_burst))


def skg_plan_force_kernel(plan: int, kind: int):
    _check(load().skg_plan_force_kernel(plan, kind))


def skg_plan_set_pdl(plan: int, enable: bool):
    _check(load().skg_plan_set_pdl(plan, 1 if enable else 0))


def skg_plan_set_next_weight(plan: int, W_next, nbytes: int):
    _check(load().skg_plan_set_next_weight(plan, _ptr(W_next), int(nbytes)))


def skg_plan_set_l2_ahead(plan: int, ahead: int):
    _check(load().skg_plan_set_l2_ahead(plan, int(ahead)))


def skg_plan_set_reducers(plan: int, reducers: int):
    _check(load().skg_plan_set_reducers(plan, int(reducers)))


def skg_plan_set_prefetch_fraction(plan: int, fraction: float):
    _check(load().skg_plan_set_prefetch_fraction(plan, float(fraction)))


def skg_plan_set_k_shard(plan: int, rank: int, ranks: int):
    _check(load().skg_plan_set_k_shard(plan, int(rank), int(ranks)))


def skg_combine_partials(M: int, N: int, partials, residual, y, epilogue="bf16", stream=None):
    """partials: R fp32 [M, N] device tensors (or addresses), in rank order."""
    arr = (ctypes.c_void_p * len(partials))(*[_ptr(t) for t in partials])
    _check(load().skg_combine_partials(M, N, len(partials), arr, _ptr(residual), _ptr(y), _epi(epilogue),
                                       _stream(stream)))


def skg_plan_info(plan: int) -> dict:
    d = skg_plan_desc()
    _check(load().skg_plan_info(plan, ctypes.byref(d)))
    return d.as_dict()


def skg_run(plan: int, x, W, residual, y, stream=None):
    _check(load().skg_run(plan, _ptr(x), _ptr(W), _ptr(residual), _ptr(y), _stream(stream)))


def skg_prefetch_l2(plan_next: int, W_next, side_stream=None):
    _check(load().skg_prefetch_l2(plan_next, _ptr(W_next), _stream(side_stream)))


def skg_plan_check(plan: int):
    _check(load().skg_plan_check(plan))


def skg_plan_destroy(plan: int):
    _check(load().skg_plan_destroy(plan))


def skg_debug_wait_timeout(plan, timeout_ns: int, stream=None):
    """plan None: the timeout word of the allocation-free entry point."""
    _check(load().skg_debug_wait_timeout(plan, int(timeout_ns), _stream(stream)))


def skg_run_noalloc(M: int, N: int, K: int, epilogue, x, W, residual, y, stream=None):
    """The split-K projection without a plan and without allocating (fixed
    in-library scratch); see include/skg.h for its limits."""
    _check(load().skg_run_noalloc(M, N, K, _epi(epilogue), _ptr(x), _ptr(W), _ptr(residual), _ptr(y),
                                  _stream(stream)))


def skg_noalloc_check(stream=None):
    """Synchronise the stream; raise SKG_ERR_DEVICE_TIMEOUT if a kernel of
    skg_run_noalloc ran out of a bounded wait since the last check."""
    _check(load().skg_noalloc_check(_stream(stream)))


class Plan:
    """Owns one skg plan handle; methods forward to the C entry points."""

    def __init__(self, M: int, N: int, K: int, epilogue="bf16"):
        self.M, self.N, self.K = M, N, K
        self.epilogue = _epi(epilogue)
        self.handle = skg_plan(M, N, K, self.epilogue)

    def info(self) -> dict:
        return skg_plan_info(self.handle)

    def force(self, split_k: int = 0, stages: int = 0, grid: int = 0, tma_burst: int = 0):
        skg_plan_force(self.handle, split_k, stages, grid, tma_burst)

    def force_kernel(self, kind: int):
        skg_plan_force_kernel(self.handle, kind)

    def set_pdl(self, enable: bool):
        skg_plan_set_pdl(self.handle, enable)

    def set_next_weight(self, W_next, nbytes: int):
        skg_plan_set_next_weight(self.handle, W_next, nbytes)

    def set_l2_ahead(self, ahead: int):
        skg_plan_set_l2_ahead(self.handle, ahead)

    def set_reducers(self, reducers: int):
        skg_plan_set_reducers(self.handle, reducers)

    def set_k_shard(self, rank: int, ranks: int):
        skg_plan_set_k_shard(self.handle, rank, ranks)

    def run(self, x, W, residual, y, stream=None):
        skg_run(self.handle, x, W, residual, y, stream)

    def prefetch(self, W, side_stream=None):
        skg_prefetch_l2(self.handle, W, side_stream)

    def check(self):
        skg_plan_check(self.handle)

    def close(self):
        if self.handle:
            skg_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------- groups
def _ints(vals):
    return (ctypes.c_int * len(vals))(*[int(v) for v in vals])


def _ptrs(vals):
    return (ctypes.c_void_p * len(vals))(*[_ptr(v) for v in vals])


def skg_group(M: int, N, K, epilogue, dep=None) -> int:
    g = ctypes.c_void_p()
    n = len(N)
    _check(load().skg_group(n, M, _ints(N), _ints(K), _ints([_epi(e) for e in epilogue]),
                            _ints(dep) if dep is not None else None, ctypes.byref(g)))
    return g.value


def skg_group_run(group: int, x, W, residual, y, stream=None):
    res = None if residual is None else _ptrs(residual)
    _check(load().skg_group_run(group, _ptrs(x), _ptrs(W), res, _ptrs(y), _stream(stream)))


def skg_group_info(group: int, n: int) -> dict:
    grid, stages, units = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    split = (ctypes.c_int * n)()
    _check(load().skg_group_info(group, ctypes.byref(grid), ctypes.byref(stages), ctypes.byref(units), split))
    return {"grid": grid.value, "stages": stages.value, "units": units.value, "split": list(split)}


def skg_group_check(group: int):
    _check(load().skg_group_check(group))


def skg_group_destroy(group: int):
    _check(load().skg_group_destroy(group))


class Group:
    """Several projections of one M in one persistent launch (skg_group)."""

    def __init__(self, M: int, N, K, epilogue, dep=None):
        self.n = len(N)
        self.handle = skg_group(M, N, K, epilogue, dep)

    def run(self, x, W, residual, y, stream=None):
        skg_group_run(self.handle, x, W, residual, y, stream)

    def info(self) -> dict:
        return skg_group_info(self.handle, self.n)

    def check(self):
        skg_group_check(self.handle)

    def close(self):
        if self.handle:
            skg_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
