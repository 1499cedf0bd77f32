"""GPU kernels against the CPU oracle, through the C ABI.

Small shapes (the oracle computes every output) span several tiles with
ragged tails in M, N and K for both kernels and all three epilogues; every
allowed split must reproduce the default plan's bits exactly.  Full-size
workloads (every named configuration) are checked on every output.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import (CHAIN_M, DEEPK_M, SWEEP_M, WIDE_M, Projection, bits,
                                          chain, deepk, generate, pr1, sweep, wide)
from tests import tolerance as T
from tests.gpu_util import DeviceCase, out_bits, out_tensor
from tests.plan_table import expected_kind

pytestmark = pytest.mark.gpu

GEMV_SPLITS = (1, 2, 4, 8)
TC_SPLITS = (2, 4, 8, 16)
REDUCERS = (1, 2, 4, 8)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()
    assert torch.cuda.is_available()


def force_each_split(case: DeviceCase, base, M):
    """Run every split the plan accepts (the split-K kernel at every reducer
    count per tile); each must reproduce `base` exactly.  The GEMV rejects
    splits whose per-warp K slice exceeds its register budget
    (SKG_ERR_UNSUPPORTED); those are skipped."""
    ran = []
    for s in (GEMV_SPLITS if M <= 2 else TC_SPLITS):
        try:
            case.plan.force(split_k=s)
        except skg.SkgError as e:
            assert e.status == skg.SKG_ERR_UNSUPPORTED, e
            continue
        for r in (REDUCERS if case.plan.info()["kernel"] == "splitk_tc" else (None,)):
            if r:
                case.plan.set_reducers(r)
            got = case.run_bits()
            assert np.array_equal(got, base), f"split {s}, reducers {r} changed the bits of {case.p}"
        ran.append(s)
    return ran


def full_check(case: DeviceCase, y_bits, what=""):
    xb, wb, rb = case.host_bits()
    y_ref, s1, _ = O.linear(xb, wb, rb)
    return T.check(y_bits, y_ref, s1, case.p.K, fp32=case.p.epilogue == "fp32", what=what)


SMALL = [
    # GEMV (M <= 2)
    (1, 1000, 1048, "bf16"), (2, 1000, 1048, "bf16_residual"), (1, 384, 7168, "fp32"),
    (2, 130, 8, "bf16"), (1, 1, 8, "bf16_residual"), (2, 4096, 520, "fp32"), (1, 3000, 4104, "bf16"),
    # split-K tensor-core kernel (M > 2)
    (3, 1000, 1048, "bf16"), (5, 257, 1048, "bf16_residual"), (8, 384, 7168, "fp32"),
    (16, 1024, 1024, "bf16_residual"), (17, 640, 2056, "bf16"), (33, 300, 200, "bf16"),
    (48, 1000, 1048, "fp32"), (63, 129, 72, "bf16_residual"), (64, 1000, 1048, "bf16"),
    (64, 128, 8, "bf16"), (4, 1, 64, "bf16"), (32, 2000, 3080, "bf16_residual"),
    # M = 2 at the kind boundary of the default rule: the split-K kernel from N = 2048, the GEMV below
    (2, 2048, 1024, "bf16_residual"), (2, 2047, 1000, "bf16"), (2, 3000, 264, "fp32"),
    # the default rule's deeper ring and its one-wave split at m_pad 32 and 48
    (32, 4100, 2048, "bf16"), (48, 1030, 4096, "bf16_residual"),
]


@pytest.mark.parametrize("M,N,K,epi", SMALL, ids=lambda v: str(v))
def test_small_shapes_all_splits(M, N, K, epi):
    p = Projection(M, N, K, epi, seed=1000 + M + N + K, residual_var=1.0)
    case = DeviceCase(p)
    try:
        info = case.plan.info()
        assert info["kernel"] == expected_kind(M, N, K, epi)
        base = case.run_bits()
        full_check(case, base, what=f"{p} default split {info['split_k']}")
        ran = force_each_split(case, base, M)
        assert len(ran) >= 2 or (M <= 2 and len(ran) >= 1), ran
    finally:
        case.close()


GEMV_FORM_SHAPES = [sh for sh in SMALL if sh[0] <= 2] + [
    (1, 7168, 7168, "bf16"), (2, 7168, 7168, "bf16"), (2, 12288, 7168, "bf16"),
    (1, 7168, 16384, "bf16_residual"), (2, 4096, 7168, "bf16"), (1, 384, 7168, "fp32"),
]


@pytest.mark.parametrize("M,N,K,epi", GEMV_FORM_SHAPES, ids=lambda v: str(v))
def test_gemv_row_forms_bit_identical(M, N, K, epi):
    """Split 1 of the M <= 2 kernel has two forms -- weights loaded into
    registers (stages 1) and, for K % 256 == 0, weights streamed by the copy
    engine through a ring of 16 KB shared-memory slots (stages = slots, a
    multiple of 7, the consumer warps).  Every form, ring depth and grid reproduces the bits of
    the default plan, which meet the oracle."""
    p = Projection(M, N, K, epi, seed=2000 + M + N + K, residual_var=1.0)
    case = DeviceCase(p)
    try:
        if case.plan.info()["kernel"] != "gemv":      # the table gave this shape to the tensor-core kernel
            case.plan.force_kernel(skg.SKG_KERNEL_GEMV)
        base = case.run_bits()
        full_check(case, base, what=f"{p} default")
        ran = []
        for stages, grid, batch in ((1, 0, 0), (2, 0, 8), (2, 0, 4), (1, 5, 0), (2, 1, 8), (2, 7, 4), (2, N, 8),
                                    (3, 0, 8), (3, 0, 4), (3, 1, 8), (3, 7, 4), (3, N, 8)):
            try:
                case.plan.force(split_k=1, stages=stages, grid=grid, tma_burst=batch)
            except skg.SkgError as e:
                # the copy-engine form needs K % 256 == 0 and rings that fit
                assert e.status == skg.SKG_ERR_UNSUPPORTED and stages >= 2, e
                continue
            info = case.plan.info()
            assert info["kernel"] == "gemv" and info["split_k"] == 1
            assert info["stages"] == (0 if stages == 1 else stages)
            assert info["tma_burst"] == batch
            assert 1 <= info["grid"] <= N and info["threads"] == 256
            got = case.run_bits()
            assert np.array_equal(got, base), f"stages {stages} grid {grid} changed the bits of {p}"
            ran.append((stages, grid, batch))
        assert len(ran) >= (10 if K % 256 == 0 else 2), ran
        case.plan.check()
    finally:
        case.close()


@pytest.mark.parametrize("M,N,K,epi", [(1, 1000, 1048, "bf16"), (2, 129, 72, "bf16_residual"),
                                       (1, 384, 7168, "fp32"), (2, 7168, 7168, "bf16")], ids=lambda v: str(v))
def test_tensor_core_kernel_at_m_le_2(M, N, K, epi):
    """skg_plan_force_kernel puts an M <= 2 plan on the tensor-core kernel
    (tokens padded to 16 columns): it meets the oracle, and every split
    gives the same bits; back on the GEMV it meets the oracle too."""
    p = Projection(M, N, K, epi, seed=2100 + M + N + K, residual_var=1.0)
    case = DeviceCase(p)
    try:
        case.plan.force_kernel(skg.SKG_KERNEL_SPLITK_TC)
        info = case.plan.info()
        assert info["kernel"] == "splitk_tc" and info["m_pad"] == 16
        base = case.run_bits()
        full_check(case, base, what=f"{p} tensor-core kernel")
        for split in (2, 4, 8, 16):
            case.plan.force(split_k=split)
            assert np.array_equal(case.run_bits(), base), f"split {split} changed the bits of {p}"
        case.plan.force_kernel(skg.SKG_KERNEL_GEMV)
        assert case.plan.info()["kernel"] == "gemv"
        full_check(case, case.run_bits(), what=f"{p} back on the GEMV")
        case.plan.check()
    finally:
        case.close()


def test_pr1_config():
    p = pr1()
    case = DeviceCase(p)
    try:
        assert case.plan.info()["kernel"] == "gemv"
        y = case.run_bits()
        r = full_check(case, y, what="PR1")
        assert r <= 1.0
    finally:
        case.close()


@pytest.mark.parametrize("M", (1, 2, 8, 64))
def test_determinism_20_runs(M):
    case = DeviceCase(Projection(M, 7168, 7168, "bf16", seed=77))
    try:
        first = case.run_bits()
        for _ in range(19):
            assert np.array_equal(case.run_bits(), first)
    finally:
        case.close()


@pytest.mark.parametrize("M", (1, 8, 64))
@pytest.mark.parametrize("kind", ("identity", "permutation"))
def test_closed_forms_bit_exact(M, kind):
    K = 1024
    g = torch.Generator().manual_seed(5 + M)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    if kind == "identity":
        W = torch.eye(K, dtype=torch.bfloat16)
        want = bits(x)
    else:
        perm = torch.randperm(K, generator=g)
        W = torch.zeros(K, K, dtype=torch.bfloat16)
        W[torch.arange(K), perm] = 1
        want = bits(x[:, perm])
    from projection_gemm_gb300.inputs import Tensors
    case = DeviceCase(Projection(M, K, K, "bf16"), Tensors(x=x, W=W, res=None, outlier_rows=None))
    try:
        assert np.array_equal(case.run_bits(), want)
    finally:
        case.close()


@pytest.mark.parametrize("M", (1, 2, 16, 64))
def test_zero_weight_gives_residual_exactly(M):
    from projection_gemm_gb300.inputs import Tensors
    N, K = 700, 520
    g = torch.Generator().manual_seed(M)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    res = torch.randn(M, N, generator=g).to(torch.bfloat16)
    W = torch.zeros(N, K, dtype=torch.bfloat16)
    case = DeviceCase(Projection(M, N, K, "bf16_residual"), Tensors(x=x, W=W, res=res, outlier_rows=None))
    try:
        assert np.array_equal(case.run_bits(), bits(res))
    finally:
        case.close()


def _full_size_check(p: Projection):
    """A full-size launch checked against the oracle on every output (the
    oracle's fp64 loop over all host cores takes about a second per
    projection here)."""
    case = DeviceCase(p)
    try:
        y = case.run_bits()
        return full_check(case, y, what=f"{p.name} all outputs"), case.plan.info()
    finally:
        case.close()


@pytest.mark.parametrize("M", SWEEP_M)
def test_sweep_full_size(M):
    ratio, info = _full_size_check(sweep(M))
    assert info["kernel"] == expected_kind(M, 7168, 7168, "bf16")


@pytest.mark.parametrize("M", WIDE_M)
def test_wide_full_size(M):
    """Includes the 1% outlier rows scaled by 16."""
    _full_size_check(wide(M))


@pytest.mark.parametrize("M", DEEPK_M)
def test_deepk_residual_full_size(M):
    _full_size_check(deepk(M))


@pytest.mark.parametrize("M", CHAIN_M)
def test_chain_stages_full_size(M):
    for p in chain(M):
        _full_size_check(p)


@pytest.mark.parametrize("M,N,K,epi,kind", [
    (64, 32768, 16384, "bf16_residual", "splitk_tc"),   # 1 GiB of weights, the largest M
    (64, 1, 16384, "bf16", "splitk_tc"),                # a single output row
    (3, 1, 8, "fp32", "splitk_tc"),                     # the smallest split-K problem
    (1, 300, 115200, "bf16", "gemv"),                   # the longest K whose x the GEMV stages
    (1, 512, 131072, "bf16_residual", "splitk_tc"),     # longer K at M = 1: the split-K kernel
    (2, 700, 65536, "fp32", "splitk_tc"),
], ids=lambda v: str(v))
def test_extreme_sizes(M, N, K, epi, kind):
    """Sizes at the edges of what the kernels take, every output against the
    oracle; at M <= 2 a K too long for the GEMV's shared-memory x runs the
    split-K kernel."""
    case = DeviceCase(Projection(M, N, K, epi, seed=3000 + M + N))
    try:
        assert case.plan.info()["kernel"] == kind
        full_check(case, case.run_bits(), what=f"M={M} N={N} K={K}")
        case.plan.check()
    finally:
        case.close()


@pytest.mark.parametrize("M", (1, 2, 8, 64))
def test_full_size_splits_bit_identical(M):
    case = DeviceCase(sweep(M))
    try:
        base = case.run_bits()
        assert len(force_each_split(case, base, M)) >= 2
    finally:
        case.close()


@pytest.mark.parametrize("M", (8, 64))
def test_chain_reducers_bit_identical(M):
    """The decode-layer chain's split-K stages at every reducer count per
    tile: the bits of the default plan, which meet the oracle."""
    for p in chain(M):
        case = DeviceCase(p)
        try:
            if case.plan.info()["kernel"] != "splitk_tc":
                continue
            base = case.run_bits()
            full_check(case, base, what=f"{p.name} default reducers")
            for r in REDUCERS:
                case.plan.set_reducers(r)
                assert np.array_equal(case.run_bits(), base), f"{p.name}: reducers {r} changed the bits"
            case.plan.check()
        finally:
            case.close()


# ---------------------------------------------------------------- errors
def test_rejections_launch_nothing():
    p = skg.Plan(4, 256, 256, "bf16")
    try:
        x = torch.zeros(4 * 256 + 8, dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
        y = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(skg.SkgError) as e:
            p.run(x.data_ptr() + 2, W, None, y)
        assert e.value.status == skg.SKG_ERR_ALIGNMENT
        with pytest.raises(skg.SkgError) as e:
            p.run(x, W, y, y)
        assert e.value.status == skg.SKG_ERR_INVALID_ARG
        with pytest.raises(skg.SkgError) as e:
            p.run(x, 0, None, y)
        assert e.value.status == skg.SKG_ERR_INVALID_ARG
    finally:
        p.close()
    for bad in ((0, 128, 128), (65, 128, 128), (4, 0, 128), (4, 128, 12), (4, 128, 0)):
        with pytest.raises(skg.SkgError):
            skg.Plan(*bad, "bf16")
    with pytest.raises(skg.SkgError):
        skg.Plan(4, 128, 128, 7)


def test_force_kernel_rejections_keep_the_plan():
    """The GEMV takes M <= 2 only; an unknown kind is an argument error; a
    rejected request leaves the plan as it was, still runnable."""
    p = Projection(4, 300, 1048, "bf16", seed=2200)
    case = DeviceCase(p)
    try:
        before = case.plan.info()
        base = case.run_bits()
        with pytest.raises(skg.SkgError) as e:
            case.plan.force_kernel(skg.SKG_KERNEL_GEMV)
        assert e.value.status == skg.SKG_ERR_UNSUPPORTED
        with pytest.raises(skg.SkgError) as e:
            case.plan.force_kernel(7)
        assert e.value.status == skg.SKG_ERR_INVALID_ARG
        assert case.plan.info() == before
        assert np.array_equal(case.run_bits(), base)
        case.plan.force_kernel(skg.SKG_KERNEL_SPLITK_TC)      # the kind it already has: same bits
        assert np.array_equal(case.run_bits(), base)
        case.plan.check()
    finally:
        case.close()


def test_forced_one_wave_grid_keeps_rows_per_cta_bounded():
    """The one-wave GEMV form, forced on a very tall weight, takes at most 256
    rows per CTA: its grid grows past one wave (no launch needed)."""
    p = skg.Plan(1, 300000, 1024, "bf16")
    try:
        p.force(split_k=1, stages=3)
        d = p.info()
        assert d["stages"] == 3 and -(-300000 // d["grid"]) <= 256
    finally:
        p.close()


def test_reducer_rejections_and_bounds():
    """Reducers per tile: 1, 2, 4 or 8 on a split-K plan; a GEMV plan rejects
    them; the plan reports the count a launch uses -- at most the split, and
    1 while the grid is more than one wave of the CTAs the SMs hold."""
    tc = skg.Plan(64, 7168, 4096, "bf16")
    gemv = skg.Plan(1, 7168, 4096, "bf16")
    try:
        gemv.force_kernel(skg.SKG_KERNEL_GEMV)
        for bad in (0, 3, 16, -1):
            with pytest.raises(skg.SkgError) as e:
                tc.set_reducers(bad)
            assert e.value.status == skg.SKG_ERR_INVALID_ARG
        with pytest.raises(skg.SkgError) as e:
            gemv.set_reducers(2)
        assert e.value.status == skg.SKG_ERR_UNSUPPORTED
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert tc.info()["reducers"] == 4                       # the default at M = 64, split 4, 56 tiles
        tc.force(split_k=2)
        assert tc.info()["reducers"] == 1                       # a forced split takes its own default
        tc.force(split_k=4)
        assert tc.info()["reducers"] == 4
        tc.set_reducers(8)
        assert tc.info()["reducers"] == 4                       # at most the split
        tc.force(split_k=16)
        tc.set_reducers(8)
        assert tc.info()["reducers"] == 1                       # splits of 16 reduce in one CTA
        tc.force(split_k=8, stages=4)
        # m_pad 64, a 4-stage ring: registers, shared memory and TMEM each
        # allow 2 CTAs per SM (the profiler's launch statistics agree)
        assert tc.info()["ctas_per_sm"] == 2
        tc.set_reducers(8)
        assert 56 * 8 > 2 * sms and tc.info()["reducers"] == 1    # 448 CTAs: more than one wave
        tc.force(split_k=4)
        assert tc.info()["reducers"] == 4                       # 224 CTAs: one wave, the request returns
    finally:
        tc.close()
        gemv.close()
    narrow = skg.Plan(64, 4096, 4096, "bf16")
    try:
        narrow.force(split_k=8, stages=4)
        narrow.set_reducers(8)
        assert narrow.info()["reducers"] == 8                   # 32 tiles x 8: one wave
    finally:
        narrow.close()


def test_table_reducers_reach_the_plan():
    """A split-K table row's reducers per tile are what the plan launches,
    within the bound on waiting CTAs (tiles x (R - 1) below the CTAs the SMs
    hold) for the row's launch shape."""
    from tests.plan_table import table_rows
    rows = [r for r in table_rows() if r[0] == skg.SKG_KERNEL_SPLITK_TC]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for kind, M, N, K, epi, split, stages, grid, aux, ahead, reducers in rows:
        p = skg.Plan(M, N, K, epi)
        try:
            i = p.info()
            assert i["from_table"] == 1 and i["ctas_per_sm"] >= 1
            tiles, slots = -(-N // 128), sms * i["ctas_per_sm"]
            want = reducers if reducers else (4 if M >= 16 and split >= 4 and tiles <= 56 else 1)
            r = min(want, split) if split <= 8 and tiles * split <= slots else 1
            assert i["reducers"] == r, (M, N, K, i["reducers"], r)
        finally:
            p.close()


def test_table_rows_launch_what_the_tuner_measured():
    """A measured GEMV row whose warps share rows (split > 1) leaves the grid
    to the library: the plan must launch the grid the tuner timed, one wave
    at that ring depth's occupancy -- the same as forcing the row's split and
    ring."""
    from tests.plan_table import table_rows
    rows = [r for r in table_rows() if r[0] == skg.SKG_KERNEL_GEMV and r[5] > 1 and r[7] == 0]
    assert rows, "no GEMV row with warps sharing rows to check"
    for kind, M, N, K, epi, split, stages, grid, aux, ahead, _reducers in rows:
        a = skg.Plan(M, N, K, epi)
        b = skg.Plan(M, N, K, epi)
        try:
            b.force(split_k=split, stages=stages)
            ia, ib = a.info(), b.info()
            assert ia["from_table"] == 1 and (ia["split_k"], ia["stages"]) == (split, stages)
            assert ia["grid"] == ib["grid"], (M, N, K, ia["grid"], ib["grid"])
        finally:
            a.close()
            b.close()
