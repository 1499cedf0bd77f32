"""The C ABI on the CPU: it builds, loads, exports what include/skg.h declares,
and its host-only picker makes the documented choices (no GPU needed)."""
import os
import re

import pytest

from projection_gemm_gb300 import build, skg
from tests.plan_table import expected_kind

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skg.h")
SMS, L2 = 152, 126 * 2 ** 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    skg.load()


def header_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"SKG_API\s+[\w\s\*]*?\b(skg_\w+)\s*\(", src)))


def test_header_and_binding_agree():
    hs = header_symbols()
    assert len(hs) >= 12
    assert sorted(skg.EXPORTS) == hs


def test_library_exports_every_declared_symbol():
    lib = skg.load()
    for name in header_symbols():
        assert hasattr(lib, name), name
    assert skg.skg_version() == 3


def test_library_is_sm103a_only():
    out = build.ARCH
    assert out == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("M", range(1, 65))
def test_kernel_kind_follows_batch(M):
    d = skg.skg_plan_query(M, 7168, 7168, "bf16", SMS, L2)
    assert d["kernel"] == expected_kind(M, 7168, 7168, "bf16")
    s = d["split_k"]
    assert s & (s - 1) == 0 and 16 % s == 0
    if d["kernel"] == "splitk_tc":
        assert s >= 2
        assert d["m_pad"] == (M + 15) // 16 * 16
        assert d["grid"] == 56 * s
        assert d["workspace_bytes"] == s * M * 7168 * 4 + 56 * 4
        assert d["smem_bytes"] <= 232448
        assert d["reducers"] in (1, 2, 4, 8)
    else:
        assert d["workspace_bytes"] == 0 and d["reducers"] == 0


@pytest.mark.parametrize("N,K,epi", [(384, 7168, "fp32"), (12288, 7168, "bf16"), (7168, 16384, "bf16_residual"),
                                     (4096, 7168, "bf16"), (1, 8, "bf16"), (129, 72, "bf16_residual")])
def test_query_shapes(N, K, epi):
    for M in (1, 2, 3, 16, 64):
        d = skg.skg_plan_query(M, N, K, epi, SMS, L2)
        assert d["N"] == N and d["K"] == K and d["epilogue"] == skg.EPILOGUES[epi]
        assert d["prefetch_bytes"] == min(2 * N * K, L2 // 2) // 16 * 16
        assert d["grid"] >= 1


@pytest.mark.parametrize("args,status", [
    ((0, 128, 128, 0), skg.SKG_ERR_UNSUPPORTED),
    ((65, 128, 128, 0), skg.SKG_ERR_UNSUPPORTED),
    ((4, 0, 128, 0), skg.SKG_ERR_INVALID_ARG),
    ((4, 128, 12, 0), skg.SKG_ERR_UNSUPPORTED),
    ((4, 128, 0, 0), skg.SKG_ERR_UNSUPPORTED),
    ((4, 128, 128, 3), skg.SKG_ERR_INVALID_ARG),
])
def test_query_rejections(args, status):
    with pytest.raises(skg.SkgError) as e:
        skg.skg_plan_query(*args, SMS, L2)
    assert e.value.status == status
    assert skg.skg_last_error()


def test_null_arguments_are_rejected():
    lib = skg.load()
    assert lib.skg_run(None, None, None, None, None, None) == skg.SKG_ERR_INVALID_ARG
    assert lib.skg_plan_info(None, None) == skg.SKG_ERR_INVALID_ARG
    assert lib.skg_plan_destroy(None) == skg.SKG_OK
    assert lib.skg_plan_query(4, 128, 128, 0, SMS, L2, None) == skg.SKG_ERR_INVALID_ARG
    assert lib.skg_prefetch_l2(None, None, None) == skg.SKG_ERR_INVALID_ARG


@pytest.mark.parametrize("N,K", [(5120, 5120), (8192, 2048), (4608, 3072), (2048, 8192), (1024, 4096),
                                 (28672, 8192)])
def test_default_rule_for_shapes_outside_the_table(N, K):
    """Shapes the measured table does not list fall back to the documented
    rules.  At M = 1 from N = 1024 the bulk-copy GEMV: in one balanced wave
    where rows are long (K >= 5120) and fewer than 16384, whole rows per warp
    elsewhere (both need K % 256 == 0).  At M = 2 the split-K kernel from
    N = 2048, below that whole rows per warp.  For M > 2 the split-K kernel
    with its W tiles after the ring requested into L2 before the wait for the
    previous kernel."""
    d1 = skg.skg_plan_query(1, N, K, "bf16", SMS, L2)
    assert d1["from_table"] == 0 and d1["kernel"] == "gemv" and d1["split_k"] == 1 and d1["threads"] == 256
    if K >= 5120 and N < 16384:
        assert d1["stages"] == 3
        assert 1 <= d1["grid"] <= 4 * SMS and d1["tile_n"] == -(-N // d1["grid"])
    else:
        assert d1["stages"] == 2 and d1["grid"] == -(-N // 8)
    d2 = skg.skg_plan_query(2, N, K, "bf16", SMS, L2)
    assert d2["from_table"] == 0
    if N >= 2048:
        assert d2["kernel"] == "splitk_tc"
    else:
        assert d2["kernel"] == "gemv" and d2["stages"] == 2 and d2["tma_burst"] in (4, 8)
        assert d2["grid"] == -(-N // 8)
    d8 = skg.skg_plan_query(8, N, K, "bf16", SMS, L2)
    assert d8["from_table"] == 0 and d8["kernel"] == "splitk_tc" and d8["l2_ahead"] == 2


@pytest.mark.parametrize("M,N,K,split,stages,reducers", [
    (8, 5120, 5120, 8, 4, 1),      # 40 tiles: split 8 fills one wave only at 3 CTAs per SM (4 stages)
    (8, 8192, 2048, 4, 6, 1),      # 64 tiles: split 4 either way, so the deeper ring at 2 per SM
    (8, 4608, 3072, 8, 6, 1),      # 36 x 8 = 288 CTAs fit 2 per SM: the deeper ring
    (16, 4096, 4096, 8, 6, 4),     # from M = 16, four reducers over few tiles
    (32, 5120, 5120, 8, 3, 4),     # m_pad 32: 3 stages at 3 per SM keep split 8
    (32, 4096, 14336, 8, 4, 4),    # ... 4 stages where 2 per SM keep it
    (32, 14336, 4096, 4, 3, 1),    # 112 tiles: one reducer
    (48, 6144, 4096, 4, 4, 4),     # m_pad 48 and 64: 4 stages, 2 per SM
    (64, 28672, 8192, 2, 4, 1),    # 224 tiles x 2 is two waves: the last arrival reduces alone
    (64, 1024, 512, 8, 4, 4),      # K = 512: 8 chunks, split 8
    (64, 1024, 256, 4, 4, 4),      # K = 256: 4 chunks, no split finer than 4
])
def test_default_split_k_shape(M, N, K, split, stages, reducers):
    """The measured default for split-K shapes outside the table: split K as
    finely as one wave of CTAs at the ring's occupancy holds (at most 8, no
    finer than K's chunks), the deeper ring where 2 CTAs per SM keep that
    split, and four reducers per tile from M = 16 at splits of 4-8 over at
    most 56 tiles."""
    d = skg.skg_plan_query(M, N, K, "bf16", SMS, L2)
    assert d["from_table"] == 0 and d["kernel"] == "splitk_tc"
    assert (d["split_k"], d["stages"], d["reducers"], d["l2_ahead"]) == (split, stages, reducers, 2)


def test_register_loads_when_k_is_not_a_multiple_of_256():
    d = skg.skg_plan_query(1, 5120, 5128, "bf16", SMS, L2)
    assert d["kernel"] == "gemv" and d["split_k"] == 1 and d["stages"] == 0


def test_tall_weights_take_whole_rows_per_warp():
    """From N = 16384 rows (and for K < 5120) M = 1 runs whole rows per warp,
    one row per warp, however tall the weight."""
    for N, K in ((300000, 8192), (16384, 7168), (300000, 1024)):
        d = skg.skg_plan_query(1, N, K, "bf16", SMS, L2)
        assert d["kernel"] == "gemv" and d["stages"] == 2 and d["grid"] == -(-N // 8)


def test_plan_table_rows_are_well_formed():
    """The measured table (rewritten by tune.py, partly with --only-m): one row
    per (M, N, K, epilogue), valid kinds and launch fields, and every row's
    shape picks that row's kernel kind."""
    from projection_gemm_gb300 import tune
    rows = tune.read_rows(tune.INC)
    assert rows
    keys = [(r[1], r[2], r[3], r[4]) for r in rows]
    assert len(keys) == len(set(keys))
    for kind, M, N, K, epi, split, stages, grid, burst, ahead, reducers, us, gbs in rows:
        assert kind in (skg.SKG_KERNEL_GEMV, skg.SKG_KERNEL_SPLITK_TC)
        assert 1 <= M <= 64 and N >= 1 and K % 8 == 0 and epi in (0, 1, 2)
        assert split & (split - 1) == 0 and 16 % split == 0
        if kind == skg.SKG_KERNEL_GEMV:
            assert M <= 2 and split <= 8
        else:
            assert split >= 2 and 2 <= stages <= 16 and burst >= 1 and 0 <= ahead <= 64
            assert reducers in (0, 1, 2, 4, 8) and reducers <= split
        assert us > 0 and 0 < gbs < 8000          # no launch streams faster than the HBM
        epi_name = {0: "bf16", 1: "bf16_residual", 2: "fp32"}[epi]
        d = skg.skg_plan_query(M, N, K, epi_name, SMS, L2)
        assert d["kernel"] == ("gemv" if kind == skg.SKG_KERNEL_GEMV else "splitk_tc")
        assert d["split_k"] == split and d["from_table"] == 1


def test_long_k_at_small_m_takes_the_split_k_kernel():
    """x must fit the GEMV's shared memory (M x K x 2 bytes); longer K at
    M <= 2 is planned on the split-K kernel instead of being rejected."""
    assert skg.skg_plan_query(1, 4096, 115200, "bf16", SMS, L2)["kernel"] == "gemv"
    for M, K in ((1, 116736), (1, 1 << 20), (2, 65536)):
        d = skg.skg_plan_query(M, 4096, K, "bf16", SMS, L2)
        assert d["kernel"] == "splitk_tc" and d["m_pad"] == 16
