"""Failure detection without a GPU fault.

Every wait in the library's kernels is bounded by %globaltimer and reports
expiry through the plan's error word.  The self-test kernel waits on a
shared-memory barrier that nothing arrives at, with a 2 ms limit: it must
record the timeout and return normally, the host must see
SKG_ERR_DEVICE_TIMEOUT once, and the context must stay usable.
"""
import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import Projection
from tests import tolerance as T
from tests.gpu_util import DeviceCase

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()


def test_bounded_wait_reports_and_context_survives():
    case = DeviceCase(Projection(8, 512, 1024, "bf16", seed=3))
    try:
        skg.skg_debug_wait_timeout(case.plan.handle, 2_000_000)
        with pytest.raises(skg.SkgError) as e:
            case.plan.check()
        assert e.value.status == skg.SKG_ERR_DEVICE_TIMEOUT
        case.plan.check()                     # reported once, then cleared

        # the next skg_run reports a timeout recorded since the last call
        skg.skg_debug_wait_timeout(case.plan.handle, 1_000_000)
        torch.cuda.synchronize()
        with pytest.raises(skg.SkgError) as e:
            case.run()
        assert e.value.status == skg.SKG_ERR_DEVICE_TIMEOUT

        # and the context still computes correctly
        y = case.run_bits()
        xb, wb, rb = case.host_bits()
        y_ref, s1, _ = O.linear(xb, wb, rb)
        T.check(y, y_ref, s1, case.p.K, what="after timeout")
        case.plan.check()
    finally:
        case.close()
