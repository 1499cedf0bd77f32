"""The scratch-free entry point, checked against the plan-based one.

skg_run_noalloc is for callers that may not allocate device memory (a
runtime that owns the whole memory budget, or code that must not enter the
CUDA allocator): it needs no plan and keeps the split-K kernel's partials,
counters and timeout word in a fixed array inside the library.  Its outputs
must meet the same acceptance bound against the oracle as skg_run's and,
since it runs the same kernel with the same reduction order, equal them bit
for bit -- on two calls in a row, because the array keeps whatever the
previous call left in it.

This file is named to be collected last; it passes on its own in a fresh
process as well as after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import Projection
from tests import tolerance as T
from tests.gpu_util import DeviceCase, out_bits, out_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()
    assert torch.cuda.is_available()


CASES = [
    (8, 1000, 1048, "bf16_residual"),
    (64, 7168, 7168, "bf16"),
    (16, 384, 7168, "fp32"),
    (33, 12288, 7168, "bf16"),
    (64, 32512, 64, "bf16"),      # the largest N whose partials fit the array at M = 64
]


def _poison(y, epi):
    if epi == "fp32":
        y.fill_(float("nan"))
    else:
        y.view(torch.int16).fill_(0x7FC0)


@pytest.mark.parametrize("M,N,K,epi", CASES, ids=lambda v: str(v))
def test_noalloc_matches_skg_run_two_calls(M, N, K, epi):
    for call, seed in enumerate((11, 12)):       # two calls in a row, different operands
        case = DeviceCase(Projection(M, N, K, epi, seed=seed + M))
        try:
            ref = case.run_bits()                 # the plan-based entry point
            y = out_tensor(M, N, epi)
            _poison(y, epi)
            skg.skg_run_noalloc(M, N, K, epi, case.x, case.W, case.res, y)
            skg.skg_noalloc_check()
            got = out_bits(y)
            xb, wb, rb = case.host_bits()
            y_ref, s1, _ = O.linear(xb, wb, rb)   # every output against the oracle
            T.check(got, y_ref, s1, K, fp32=epi == "fp32", what=f"noalloc call {call}")
            assert np.array_equal(got, ref), f"call {call}: skg_run_noalloc differs from skg_run"
        finally:
            case.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    # partials of 2 * 256 tiles * 64 * 128 * 4 bytes (16 MiB) exceed the array: rejected before any launch
    for N in (32768, 40000):
        with pytest.raises(skg.SkgError) as e:
            skg.skg_run_noalloc(64, N, 64, "bf16", x, W, None, y)
        assert e.value.status == skg.SKG_ERR_UNSUPPORTED and "scratch" in str(e.value)
    with pytest.raises(skg.SkgError) as e:
        skg.skg_run_noalloc(2, 64, 64, "bf16", x, W, None, y)
    assert e.value.status == skg.SKG_ERR_UNSUPPORTED


def test_noalloc_check_reports_a_timeout_once():
    """A bounded wait that runs out sets the array's timeout word (here the
    self-test kernel, which waits 2 ms on a barrier nothing arrives at);
    skg_noalloc_check reports it once and clears it, and the next call
    computes the same bits as skg_run."""
    skg.skg_noalloc_check()                      # nothing pending
    skg.skg_debug_wait_timeout(None, 2_000_000)
    with pytest.raises(skg.SkgError) as e:
        skg.skg_noalloc_check()
    assert e.value.status == skg.SKG_ERR_DEVICE_TIMEOUT
    skg.skg_noalloc_check()                      # cleared
    M, N, K = 24, 2000, 2048
    case = DeviceCase(Projection(M, N, K, "bf16", seed=5))
    try:
        ref = case.run_bits()
        y = out_tensor(M, N, "bf16")
        _poison(y, "bf16")
        skg.skg_run_noalloc(M, N, K, "bf16", case.x, case.W, None, y)
        skg.skg_noalloc_check()
        assert np.array_equal(out_bits(y), ref)
    finally:
        case.close()
