"""Acceptance test of a GPU output against the oracle.

Per output element, with y_ref the oracle's fp64 value (residual included),
S1 = sum_k |x_mk| |W_nk| and K the reduction length:

  bf16 outputs:  |y_gpu - round_bf16(y_ref)| <= ulp_bf16(|y_ref|) + 1e-3 * S1 / sqrt(K)
  fp32 outputs:  |y_gpu - y_ref|             <= ulp_bf16(|y_ref|) + 1e-3 * S1 / sqrt(K)
                 and, stricter, |y_gpu - y_ref| <= 2^-16 * S1 + 2^-23 * |y_ref|

The first bound is the projection's stated acceptance criterion; for an fp32
output the rounding to bf16 is replaced by the identity.  The extra fp32
bound follows from fp32 accumulation: each of the at most 16 chunk sums and
the tree over them carries a relative error of a few units of 2^-24 of S1,
far below 2^-16 * S1.  ulp_bf16(v) = 2^(floor(log2 v) - 7) for normal v, and
2^-133 for zero and subnormal v.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.oracle as O


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """GPU output bits -> fp64 via torch's own conversion (not the oracle's)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def bound(y_ref: np.ndarray, s1: np.ndarray, K: int) -> np.ndarray:
    return O.ulp_bf16(np.abs(y_ref)) + 1e-3 * s1 / math.sqrt(K)


def check(y_gpu, y_ref, s1, K: int, fp32: bool = False, what: str = ""):
    """Assert the acceptance bound element-wise; returns the worst ratio
    error / bound (<= 1 passes)."""
    y_ref = np.asarray(y_ref, dtype=np.float64)
    s1 = np.asarray(s1, dtype=np.float64)
    tol = bound(y_ref, s1, K)
    if fp32:
        yg = np.asarray(y_gpu, dtype=np.float64)
        err = np.abs(yg - y_ref)
        strict = 2.0 ** -16 * s1 + 2.0 ** -23 * np.abs(y_ref)
        bad2 = ~(err <= strict)
        assert not bad2.any(), (f"{what}: {bad2.sum()} fp32 outputs exceed the fp32 accumulation bound; "
                                f"worst at {np.unravel_index(np.argmax(err - strict), err.shape)}")
    else:
        yg = decode_bf16(np.asarray(y_gpu, dtype=np.uint16))
        want = decode_bf16(O.bf16_round(y_ref))
        err = np.abs(yg - want)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), float(yg[tuple(i)]), float(y_ref[tuple(i)]), float(tol[tuple(i)])) for i in idx]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outputs outside tolerance; "
                             f"(index, gpu, oracle, bound): {detail}")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(tol > 0, err / tol, 0.0)
    return float(np.max(ratio)) if ratio.size else 0.0
