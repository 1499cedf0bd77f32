"""Checks that pin the CPU oracle to facts other than itself.

Each check takes a loaded oracle library (so the mutation tests can run the
same checks against deliberately broken copies of the oracle) and raises
AssertionError when the oracle disagrees with:
  * exact integer arithmetic (Python ints) on tiny shapes,
  * the closed forms W = I and W = a permutation matrix,
  * exact power-of-two scaling (of x, and of chosen W rows by 16),
  * linearity in x and invariance to cutting K into slices (fp64 bound),
  * numpy's fp64 matmul (a library routine with another summation order),
  * hand-worked IEEE round-to-nearest-even cases and torch's own bf16
    conversions (decode of every bit pattern, encode of float32 values).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle.oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS64 = 2.0 ** -53


def _bf16_bits_from_float(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand_bf16(rng, shape, scale=1.0) -> np.ndarray:
    return _bf16_bits_from_float(rng.standard_normal(shape) * scale)


def _int_bf16(rng, shape, lo=-8, hi=8):
    vals = rng.integers(lo, hi + 1, size=shape)
    return vals, _bf16_bits_from_float(vals.astype(np.float32))


def load_golden_rne():
    cases = []
    with open(os.path.join(GOLDEN, "bf16_rne_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            v, b = line.split()
            cases.append((float.fromhex(v), int(b, 16)))
    return cases


# ----------------------------------------------------------------- bf16 codec
def check_decode_all_patterns(lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.bf16_decode(pats, lib=lib)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert math.copysign(1.0, ours[0x8000]) == -1.0


def check_round_golden(lib):
    cases = load_golden_rne()
    vals = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases], dtype=np.uint16)
    got = O.bf16_round(vals, lib=lib)
    bad = [(vals[i].hex(), hex(got[i]), hex(want[i])) for i in range(len(cases)) if got[i] != want[i]]
    assert not bad, f"RNE mismatches (value, got, want): {bad}"


def check_round_matches_torch(lib, n=200000, seed=1):
    """float32 inputs (exact in fp64), so torch's single RNE step is the truth.
    Includes exact ties: midpoints of adjacent bf16 values."""
    rng = np.random.default_rng(seed)
    with np.errstate(over="ignore"):
        f = (rng.standard_normal(n) * np.exp2(rng.integers(-140, 128, n))).astype(np.float32)
    f = f[np.isfinite(f)]
    lo = _bf16_bits_from_float(rng.standard_normal(20000).astype(np.float32))
    lo = lo[(lo & 0x7F80) != 0x7F80]
    a = torch.from_numpy(lo.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    b = torch.from_numpy((lo + 1).astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    mids = ((a + b) / 2).astype(np.float32)   # exact in float32
    allv = np.concatenate([f, mids]).astype(np.float32)
    ours = O.bf16_round(allv.astype(np.float64), lib=lib)
    ref = _bf16_bits_from_float(allv)
    assert np.array_equal(ours, ref)


def check_ulp(lib):
    one = O.ulp_bf16(np.array([1.0, 1.99, 2.0, -3.0, 0.0, 2.0 ** -126, 2.0 ** -127]), lib=lib)
    assert list(one) == [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -6, 2.0 ** -133, 2.0 ** -133, 2.0 ** -133]
    # the spacing of consecutive positive finite bf16 patterns is the ulp
    pats = np.arange(0x0001, 0x7F7F, dtype=np.uint16)
    v0 = O.bf16_decode(pats, lib=lib)
    v1 = O.bf16_decode(pats + 1, lib=lib)
    assert np.array_equal(v1 - v0, O.ulp_bf16(v0, lib=lib))


# ------------------------------------------------------------ the projection
def check_brute_force_integers(lib, trials=60, seed=2):
    rng = np.random.default_rng(seed)
    for t in range(trials):
        M, N, K = int(rng.integers(1, 5)), int(rng.integers(1, 9)), int(rng.integers(1, 17))
        xv, xb = _int_bf16(rng, (M, K))
        wv, wb = _int_bf16(rng, (N, K))
        use_res = t % 2 == 1
        rv, rb = _int_bf16(rng, (M, N), -64, 64) if use_res else (None, None)
        y, s1, yb = O.linear(xb, wb, rb, lib=lib)
        for m in range(M):
            for n in range(N):
                exact = sum(int(xv[m, k]) * int(wv[n, k]) for k in range(K))
                mag = sum(abs(int(xv[m, k])) * abs(int(wv[n, k])) for k in range(K))
                if use_res:
                    exact += int(rv[m, n])
                assert y[m, n] == exact, (M, N, K, m, n, y[m, n], exact)
                assert s1[m, n] == mag
        # the bf16 output is the library RNE of the exact integer
        assert np.array_equal(yb, _bf16_bits_from_float(y.astype(np.float32)))


def check_identity(lib, seed=3):
    rng = np.random.default_rng(seed)
    for M, K in ((1, 64), (5, 40), (64, 136)):
        xb = _rand_bf16(rng, (M, K))
        eye = _bf16_bits_from_float(np.eye(K, dtype=np.float32))
        y, s1, yb = O.linear(xb, eye, lib=lib)
        assert np.array_equal(yb, xb)
        assert np.array_equal(y, O.bf16_decode(xb, lib=lib))
        rb = _rand_bf16(rng, (M, K))
        y2, _, _ = O.linear(xb, eye, rb, lib=lib)
        assert np.array_equal(y2, O.bf16_decode(xb, lib=lib) + O.bf16_decode(rb, lib=lib))


def check_permutation(lib, seed=4):
    rng = np.random.default_rng(seed)
    for M, K in ((1, 32), (3, 96), (17, 24)):
        xb = _rand_bf16(rng, (M, K))
        perm = rng.permutation(K)
        P = np.zeros((K, K), dtype=np.float32)
        P[np.arange(K), perm] = 1.0        # row n of W picks column perm[n]
        y, _, yb = O.linear(xb, _bf16_bits_from_float(P), lib=lib)
        assert np.array_equal(yb, xb[:, perm])
        assert np.array_equal(y, O.bf16_decode(xb[:, perm], lib=lib))


def check_power_of_two_scaling(lib, seed=5):
    rng = np.random.default_rng(seed)
    M, N, K = 3, 50, 72
    xb = _rand_bf16(rng, (M, K))
    wb = _rand_bf16(rng, (N, K), 1 / math.sqrt(K))
    y, s1, _ = O.linear(xb, wb, lib=lib)
    x4 = _bf16_bits_from_float(O.bf16_decode(xb, lib=lib).astype(np.float32) * 4)
    y4, s14, _ = O.linear(x4, wb, lib=lib)
    assert np.array_equal(y4, 4 * y) and np.array_equal(s14, 4 * s1)
    rows = rng.choice(N, size=5, replace=False)
    wf = O.bf16_decode(wb, lib=lib).astype(np.float32)
    wf[rows] *= 16
    y16, _, _ = O.linear(xb, _bf16_bits_from_float(wf), lib=lib)
    keep = np.setdiff1d(np.arange(N), rows)
    assert np.array_equal(y16[:, rows], 16 * y[:, rows])
    assert np.array_equal(y16[:, keep], y[:, keep])


def check_linearity(lib, seed=6):
    """x = x1 + x2 with disjoint supports (even / odd k), exact in bf16."""
    rng = np.random.default_rng(seed)
    M, N, K = 4, 33, 400
    xf = rng.standard_normal((M, K)).astype(np.float32)
    x1f, x2f = xf.copy(), xf.copy()
    x1f[:, 1::2] = 0
    x2f[:, 0::2] = 0
    wb = _rand_bf16(rng, (N, K), 1 / math.sqrt(K))
    y, s1, _ = O.linear(_bf16_bits_from_float(xf), wb, lib=lib)
    y1, _, _ = O.linear(_bf16_bits_from_float(x1f), wb, lib=lib)
    y2, _, _ = O.linear(_bf16_bits_from_float(x2f), wb, lib=lib)
    assert np.all(np.abs(y - (y1 + y2)) <= K * EPS64 * 2 * s1 + 1e-300)
    # and it is not trivially zero
    assert np.max(np.abs(y)) > 0.1


def check_k_split(lib, seed=7):
    rng = np.random.default_rng(seed)
    M, N, K = 5, 40, 1000
    xb = _rand_bf16(rng, (M, K))
    wb = _rand_bf16(rng, (N, K), 1 / math.sqrt(K))
    y, s1, _ = O.linear(xb, wb, lib=lib)
    cuts = [0, 7, 300, 301, 640, 1000]
    acc = np.zeros_like(y)
    for a, b in zip(cuts[:-1], cuts[1:]):
        ys, _, _ = O.linear(np.ascontiguousarray(xb[:, a:b]), np.ascontiguousarray(wb[:, a:b]), lib=lib)
        acc += ys
    assert np.all(np.abs(acc - y) <= 2 * K * EPS64 * s1)


def check_against_numpy(lib, seed=8):
    rng = np.random.default_rng(seed)
    for M, N, K in ((1, 256, 512), (7, 129, 264), (64, 70, 1024)):
        xb = _rand_bf16(rng, (M, K))
        wb = _rand_bf16(rng, (N, K), 1 / math.sqrt(K))
        rb = _rand_bf16(rng, (M, N))
        xf = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        wf = torch.from_numpy(wb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        rf = torch.from_numpy(rb.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
        ref = xf @ wf.T
        y, s1, yb = O.linear(xb, wb, lib=lib)
        assert np.all(np.abs(y - ref) <= 2 * K * EPS64 * s1)
        assert np.allclose(s1, np.abs(xf) @ np.abs(wf).T, rtol=4 * K * EPS64, atol=0)
        yr, _, _ = O.linear(xb, wb, rb, lib=lib)
        assert np.all(np.abs(yr - (ref + rf)) <= 2 * K * EPS64 * s1 + EPS64 * np.abs(ref + rf))
        # the residual is one fp64 add on top of the finished sum
        assert np.array_equal(yr, y + rf)


def check_points(lib, seed=9):
    rng = np.random.default_rng(seed)
    M, N, K = 6, 90, 200
    xb = _rand_bf16(rng, (M, K))
    wb = _rand_bf16(rng, (N, K), 1 / math.sqrt(K))
    rb = _rand_bf16(rng, (M, N))
    y, s1, _ = O.linear(xb, wb, rb, lib=lib)
    ms = rng.integers(0, M, 50)
    ns = rng.integers(0, N, 50)
    yp, sp = O.linear_points(xb, wb, ms, ns, rb, lib=lib)
    assert np.array_equal(yp, y[ms, ns]) and np.array_equal(sp, s1[ms, ns])


ALL_CHECKS = [
    check_decode_all_patterns,
    check_round_golden,
    check_round_matches_torch,
    check_ulp,
    check_brute_force_integers,
    check_identity,
    check_permutation,
    check_power_of_two_scaling,
    check_linearity,
    check_k_split,
    check_against_numpy,
    check_points,
]
