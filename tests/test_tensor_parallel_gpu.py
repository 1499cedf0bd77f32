"""Tensor-parallel projections, with the ranks run one after another on one GPU.

Row-parallel: K split across R ranks along canonical chunks; each rank's
skg_run leaves its fp32 subtree value and skg_combine_partials adds the top
levels of the tree, the residual and the one rounding -- the bits must equal
one launch of the split-K kernel over the whole K, and meet the oracle.
Column-parallel: each rank runs one group launch over its rows of the router
and latent weights (same x); the gathered slices must equal the unsharded
launches bit for bit.  (Moving the partials and slices between GPUs is the
all-gather exercised on CPU ranks in test_tensor_parallel_dist.py.)
"""
import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300 import tensor_parallel as tp
from projection_gemm_gb300.inputs import Projection, bits, generate
from tests import tolerance as T
from tests.gpu_util import out_bits, out_tensor, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()


ROW_CASES = [
    (8, 7168, 8192, "bf16_residual"),    # the decode layer's output projection
    (64, 7168, 4096, "bf16_residual"),
    (1, 1000, 2048, "bf16"),
    (33, 300, 1024, "fp32"),
]


@pytest.mark.parametrize("M,N,K,epi", ROW_CASES, ids=lambda v: str(v))
@pytest.mark.parametrize("ranks", (2, 4, 8))
def test_row_parallel_equals_one_launch(M, N, K, epi, ranks):
    t = generate(Projection(M, N, K, epi, seed=700 + M + ranks))
    x, W, res = to_dev(t.x), to_dev(t.W), to_dev(t.res)
    ref_plan = skg.Plan(M, N, K, epi)
    try:
        ref_plan.force_kernel(skg.SKG_KERNEL_SPLITK_TC)        # the same kernel and tree at every M
        y_ref = out_tensor(M, N, epi)
        ref_plan.run(x, W, res, y_ref)
        torch.cuda.synchronize()
        ref_plan.check()
    finally:
        ref_plan.close()
    ref = out_bits(y_ref)
    ranks_ = [tp.RowParallelProjection(M, N, K, epi, r, ranks) for r in range(ranks)]
    try:
        partials = []
        for rp in ranks_:
            c0, c1 = rp.columns
            part = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
            rp.partial(x[:, c0:c1].contiguous(), W[:, c0:c1].contiguous(), part)
            partials.append(part)
        y = out_tensor(M, N, epi)
        y.fill_(float("nan")) if epi == "fp32" else y.view(torch.int16).fill_(0x7FC0)
        ranks_[0].combine(partials, res, y)
        torch.cuda.synchronize()
        for rp in ranks_:
            rp.plan.check()
        got = out_bits(y)
        assert np.array_equal(got, ref), f"{ranks} ranks differ from one launch"
        y_ref64, s1, _ = O.linear(bits(t.x), bits(t.W), None if t.res is None else bits(t.res))
        T.check(got, y_ref64, s1, K, fp32=epi == "fp32", what=f"row-parallel x{ranks}")
    finally:
        for rp in ranks_:
            rp.close()


def test_k_shard_rejections():
    p = skg.Plan(8, 256, 1024, "bf16")
    try:
        with pytest.raises(skg.SkgError) as e:
            p.set_k_shard(0, 2)                     # a partial is fp32
        assert e.value.status == skg.SKG_ERR_UNSUPPORTED
    finally:
        p.close()
    p = skg.Plan(8, 256, 1000, "fp32")
    try:
        with pytest.raises(skg.SkgError) as e:
            p.set_k_shard(0, 2)                     # K % 1024 != 0
        assert e.value.status == skg.SKG_ERR_UNSUPPORTED
        for bad in ((0, 3), (2, 2), (-1, 2)):
            with pytest.raises(skg.SkgError) as e:
                p.set_k_shard(*bad)
            assert e.value.status == skg.SKG_ERR_INVALID_ARG
    finally:
        p.close()
    y = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    part = torch.zeros(8, 256, dtype=torch.float32, device="cuda")
    with pytest.raises(skg.SkgError) as e:
        skg.skg_combine_partials(8, 256, [part] * 3, None, y, "bf16")
    assert e.value.status == skg.SKG_ERR_INVALID_ARG
    with pytest.raises(skg.SkgError) as e:
        skg.skg_combine_partials(8, 256, [part] * 2, None, y, "bf16_residual")
    assert e.value.status == skg.SKG_ERR_INVALID_ARG


@pytest.mark.parametrize("M", (1, 8, 64))
@pytest.mark.parametrize("ranks", (2, 4))
def test_column_parallel_router_and_latent(M, ranks):
    """Router scores (N = 384, fp32) and the latent input projection
    (N = 4096) of one hidden state: each rank one group launch over its rows."""
    K, Ns, epis = 7168, [384, 4096], ["fp32", "bf16"]
    ts = [generate(Projection(M, n, K, e, seed=800 + M + i)) for i, (n, e) in enumerate(zip(Ns, epis))]
    x = to_dev(ts[0].x)
    Ws = [to_dev(t.W) for t in ts]
    full = skg.Group(M, Ns, [K, K], epis, None)
    try:
        y_full = [out_tensor(M, n, e) for n, e in zip(Ns, epis)]
        full.run([x, x], Ws, None, y_full)
        torch.cuda.synchronize()
        full.check()
    finally:
        full.close()
    slices = [[] for _ in Ns]
    for r in range(ranks):
        cg = tp.ColumnParallelGroup(M, Ns, K, epis, r, ranks)
        try:
            ys = [out_tensor(M, n1 - n0, e) for (n0, n1), e in zip(cg.rows, epis)]
            cg.run_local(x, [W[n0:n1].contiguous() for W, (n0, n1) in zip(Ws, cg.rows)], ys)
            torch.cuda.synchronize()
            cg.group.check()
            for i, y in enumerate(ys):
                slices[i].append(y)
        finally:
            cg.close()
    for i, (n, e) in enumerate(zip(Ns, epis)):
        got = out_bits(torch.cat(slices[i], dim=1))
        assert got.shape == (M, n)
        # a row of y depends only on its row of W, and every split gives the
        # same bits: the gathered slices equal the whole launch exactly
        assert np.array_equal(got, out_bits(y_full[i])), f"projection {i}: slices differ from the whole launch"
        y_ref, s1, _ = O.linear(bits(ts[0].x), bits(ts[i].W))      # both read the same x
        T.check(got, y_ref, s1, K, fp32=e == "fp32", what=f"column-parallel projection {i} x{ranks}")
