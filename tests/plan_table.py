"""The kernel kind the picker should choose, read from the compiled-in table.

M <= 2 runs the GEMV unless the measured table holds a tensor-core row for
exactly that (M, N, K, epilogue), x (M x K bf16) does not fit the GEMV's
226 KB of shared memory, or M = 2 with N >= 2048 and no GEMV row for exactly
that shape; M > 2 always runs the tensor-core kernel.
"""
from __future__ import annotations

import os
import re

_INC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "projection_gemm_gb300", "csrc", "skg_plan_table.inc")
_EPI = {"bf16": 0, "bf16_residual": 1, "fp32": 2}


def table_rows():
    """Every row of the table: (kind, M, N, K, epilogue, split, stages, grid, aux, ahead, reducers)."""
    rows = []
    for line in open(_INC):
        m = re.match(r"^\{([-\d, ]+)\}", line)
        if m:
            rows.append(tuple(int(a) for a in m.group(1).split(",")))
    return rows


_TC = {(r[1], r[2], r[3], r[4]) for r in table_rows() if r[0] == 2}
_GEMV = {(r[1], r[2], r[3], r[4]) for r in table_rows() if r[0] == 1}


def expected_kind(M: int, N: int, K: int, epilogue: str) -> str:
    key = (M, N, K, _EPI[epilogue])
    if M > 2 or key in _TC or M * K * 2 > 226 * 1024:
        return "splitk_tc"
    if M == 2 and N >= 2048 and key not in _GEMV:
        return "splitk_tc"
    return "gemv"
