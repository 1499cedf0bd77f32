"""The kernel kind the picker should choose, read from the compiled-in table.

M <= 2 runs the GEMV unless the measured table holds a tensor-core row for
exactly that (M, N, K, epilogue); M > 2 always runs the tensor-core kernel.
"""
from __future__ import annotations

import os
import re

_INC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "projection_gemm_gb300", "csrc", "skg_plan_table.inc")
_EPI = {"bf16": 0, "bf16_residual": 1, "fp32": 2}


def _tc_rows():
    rows = set()
    for line in open(_INC):
        m = re.match(r"^\{([-\d, ]+)\}", line)
        if m:
            v = [int(a) for a in m.group(1).split(",")]
            if v[0] == 2:
                rows.add((v[1], v[2], v[3], v[4]))
    return rows


_TC = _tc_rows()


def expected_kind(M: int, N: int, K: int, epilogue: str) -> str:
    if M > 2 or (M, N, K, _EPI[epilogue]) in _TC:
        return "splitk_tc"
    return "gemv"
