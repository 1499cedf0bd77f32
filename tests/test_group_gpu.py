"""Groups: several projections of one M in one persistent split-K launch.

Every projection of a group must have exactly the bits of skg_run at the
same split (the arithmetic per work unit is the one-projection kernel's),
and meet the oracle.  A projection with dep set reads the previous
projection's output: with that output first poisoned with NaN, the group
must reproduce the two-launch chain, run after run (the on-device counters
return to zero at the end of every launch).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import CHAIN_STAGES, Projection, bits, generate
from tests import tolerance as T
from tests.gpu_util import out_bits, out_tensor, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()
    assert torch.cuda.is_available()


def _single(M, N, K, epi, split, x, W, res):
    p = skg.Plan(M, N, K, epi)
    try:
        p.force_kernel(skg.SKG_KERNEL_SPLITK_TC)       # groups run the split-K kernel at every M
        p.force(split_k=split)
        y = out_tensor(M, N, epi)
        p.run(x, W, res, y)
        torch.cuda.synchronize()
        p.check()
        return out_bits(y)
    finally:
        p.close()


def _group_case(M, shapes, dep, seed, runs=3):
    """shapes: [(K, N, epilogue)]; independent seeded operands per projection."""
    ts = [generate(Projection(M, N, K, epi, seed=seed + i)) for i, (K, N, epi) in enumerate(shapes)]
    xs = [to_dev(t.x) for t in ts]
    Ws = [to_dev(t.W) for t in ts]
    rs = [to_dev(t.res) for t in ts]
    ys = [out_tensor(M, N, epi) for (K, N, epi) in shapes]
    g = skg.Group(M, [N for _, N, _ in shapes], [K for K, _, _ in shapes], [e for _, _, e in shapes], dep)
    try:
        info = g.info()
        assert info["units"] == sum(-(-N // 128) * s for (_, N, _), s in zip(shapes, info["split"]))
        assert 1 <= info["grid"] <= info["units"]
        for _ in range(runs):
            for y in ys:
                y.fill_(float("nan"))
            g.run(xs, Ws, rs, ys)
            torch.cuda.synchronize()
            g.check()
        got = [out_bits(y) for y in ys]
    finally:
        g.close()
    for i, ((K, N, epi), t) in enumerate(zip(shapes, ts)):
        want = _single(M, N, K, epi, info["split"][i], xs[i], Ws[i], rs[i])
        assert np.array_equal(got[i], want), f"projection {i} ({K}->{N} {epi}) differs from skg_run"
        xb, wb, rb = bits(t.x), bits(t.W), None if t.res is None else bits(t.res)
        y_ref, s1, _ = O.linear(xb, wb, rb)
        T.check(got[i], y_ref, s1, K, fp32=epi == "fp32", what=f"group projection {i} all outputs")
    return info


@pytest.mark.parametrize("M", (8, 33, 64))
def test_decode_layer_group_matches_skg_run(M):
    """The five decode-layer stages in one launch (each ordered after the previous one)."""
    info = _group_case(M, list(CHAIN_STAGES), dep=[0, 1, 1, 1, 1], seed=300 + M)
    assert all(s in (2, 4, 8) for s in info["split"])


@pytest.mark.parametrize("M,shapes", [
    (1, [(1048, 1000, "bf16"), (72, 129, "bf16_residual"), (7168, 384, "fp32")]),
    (2, [(4096, 7168, "bf16_residual"), (7168, 4096, "bf16")]),
    (3, [(1048, 1000, "bf16"), (72, 129, "bf16_residual"), (2056, 640, "fp32")]),
    (17, [(200, 300, "bf16"), (1024, 1024, "bf16_residual")]),
    (64, [(8, 128, "bf16"), (7168, 384, "fp32"), (520, 4096, "bf16_residual"), (1048, 1, "bf16")]),
    (48, [(4096, 7168, "bf16_residual")]),
    # the router and latent projections: one unit per CTA, several reducers per tile
    (64, [(7168, 384, "fp32"), (7168, 4096, "bf16")]),
    (16, [(7168, 384, "fp32"), (7168, 4096, "bf16")]),
])
def test_ragged_groups_without_dependencies(M, shapes):
    """Groups without dependencies: every output equals skg_run's and meets
    the oracle; where the grid holds every unit, the last arrivals of a tile
    share its reduction (the bits do not depend on how many share it)."""
    _group_case(M, shapes, dep=None, seed=400 + M, runs=2)


@pytest.mark.parametrize("M", (1, 5, 16, 64))
def test_dependent_chain_reads_the_previous_output(M):
    """x of projection 1 is y of projection 0 (dep set), y0 poisoned before every run."""
    t0 = generate(Projection(M, 4096, 7168, "bf16", seed=500 + M))
    t1 = generate(Projection(M, 7168, 4096, "bf16_residual", seed=501 + M))
    t2 = generate(Projection(M, 2048, 7168, "bf16", seed=502 + M))
    x0, W0, W1, r1, W2 = to_dev(t0.x), to_dev(t0.W), to_dev(t1.W), to_dev(t1.res), to_dev(t2.W)
    y0 = torch.empty(M, 4096, dtype=torch.bfloat16, device="cuda")
    y1 = torch.empty(M, 7168, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(M, 2048, dtype=torch.bfloat16, device="cuda")
    g = skg.Group(M, [4096, 7168, 2048], [7168, 4096, 7168], ["bf16", "bf16_residual", "bf16"], [0, 1, 1])
    try:
        split = g.info()["split"]
        # the reference: three separate launches at the same splits
        want = []
        ref_y = [torch.empty_like(y0), torch.empty_like(y1), torch.empty_like(y2)]
        chain = [(4096, 7168, "bf16", x0, W0, None), (7168, 4096, "bf16_residual", ref_y[0], W1, r1),
                 (2048, 7168, "bf16", ref_y[1], W2, None)]
        for i, (N, K, epi, x, W, r) in enumerate(chain):
            p = skg.Plan(M, N, K, epi)
            try:
                p.force_kernel(skg.SKG_KERNEL_SPLITK_TC)
                p.force(split_k=split[i])
                p.run(x, W, r, ref_y[i])
                torch.cuda.synchronize()
            finally:
                p.close()
            want.append(out_bits(ref_y[i]))
        for _ in range(5):
            for y in (y0, y1, y2):
                y.view(torch.int16).fill_(0x7FC0)
            g.run([x0, y0, y1], [W0, W1, W2], [None, r1, None], [y0, y1, y2])
            torch.cuda.synchronize()
            g.check()
            for a, b in zip((y0, y1, y2), want):
                got = out_bits(a)
                assert not np.any((got & 0x7FFF) > 0x7F80), "NaN: a projection read its input too early"
                assert np.array_equal(got, b)
        # each stage against the oracle, fed the previous stage's GPU output
        xin = bits(t0.x)
        for i, (W, r, yb) in enumerate(zip((t0.W, t1.W, t2.W), (None, t1.res, None), want)):
            y_ref, s1, _ = O.linear(xin, bits(W), None if r is None else bits(r))
            T.check(yb, y_ref, s1, xin.shape[1], what=f"dependent group stage {i}")
            xin = yb
    finally:
        g.close()


def test_group_captures_into_a_cuda_graph():
    M = 8
    shapes = [(7168, 4096, "bf16"), (4096, 7168, "bf16_residual")]
    ts = [generate(Projection(M, N, K, epi, seed=600 + i)) for i, (K, N, epi) in enumerate(shapes)]
    xs, Ws, rs = [to_dev(t.x) for t in ts], [to_dev(t.W) for t in ts], [to_dev(t.res) for t in ts]
    ys = [out_tensor(M, N, epi) for (K, N, epi) in shapes]
    g = skg.Group(M, [4096, 7168], [7168, 4096], ["bf16", "bf16_residual"], [0, 1])
    try:
        g.run(xs, Ws, rs, ys)
        torch.cuda.synchronize()
        want = [out_bits(y) for y in ys]
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            g.run(xs, Ws, rs, ys, s)
        for y in ys:
            y.view(torch.int16).fill_(0x7FC0)
        for _ in range(4):
            graph.replay()
        torch.cuda.synchronize()
        g.check()
        assert all(np.array_equal(out_bits(y), w) for y, w in zip(ys, want))
        for i, ((K, N, epi), t) in enumerate(zip(shapes, ts)):
            y_ref, s1, _ = O.linear(bits(t.x), bits(t.W), None if t.res is None else bits(t.res))
            T.check(out_bits(ys[i]), y_ref, s1, K, what=f"graph-replayed group projection {i}")
    finally:
        g.close()


def test_group_rejections():
    with pytest.raises(skg.SkgError) as e:
        skg.Group(65, [128], [128], ["bf16"])
    assert e.value.status == skg.SKG_ERR_UNSUPPORTED
    with pytest.raises(skg.SkgError) as e:
        skg.Group(8, [128] * 9, [128] * 9, ["bf16"] * 9)
    assert e.value.status == skg.SKG_ERR_UNSUPPORTED
    with pytest.raises(skg.SkgError):
        skg.Group(8, [128], [12], ["bf16"])
    g = skg.Group(8, [256, 256], [256, 256], ["bf16", "bf16_residual"])
    try:
        x = torch.zeros(8 * 256 + 8, dtype=torch.bfloat16, device="cuda")
        W = torch.zeros(256, 256, dtype=torch.bfloat16, device="cuda")
        y = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(skg.SkgError) as e:        # residual missing for projection 1
            g.run([x, x], [W, W], None, [y, y])
        assert e.value.status == skg.SKG_ERR_INVALID_ARG
        with pytest.raises(skg.SkgError) as e:        # misaligned x
            g.run([x.data_ptr() + 2, x], [W, W], [None, y], [y, y])
        assert e.value.status == skg.SKG_ERR_ALIGNMENT
    finally:
        g.close()


def test_groups_between_other_launches_complete():
    """The decode-layer chain as launched back to back: five M = 1 GEMV
    launches, then the M = 8 group, then the M = 64 group, repeated without
    a host sync.  The groups start while the previous kernels still hold
    SMs, so only part of a group's grid may be resident at first; every
    launch must still complete (no bounded wait runs out) and the last run
    of each group must equal skg_run at the same splits."""
    def stage_tensors(M, seed):
        ts = [generate(Projection(M, N, K, epi, seed=seed + i)) for i, (K, N, epi) in enumerate(CHAIN_STAGES)]
        return ([to_dev(t.x) for t in ts], [to_dev(t.W) for t in ts], [to_dev(t.res) for t in ts],
                [out_tensor(M, N, epi) for (K, N, epi) in CHAIN_STAGES])

    dims = ([N for _, N, _ in CHAIN_STAGES], [K for K, _, _ in CHAIN_STAGES], [e for _, _, e in CHAIN_STAGES])
    gemv = stage_tensors(1, 700)
    plans = [skg.Plan(1, N, K, epi) for (K, N, epi) in CHAIN_STAGES]
    groups = {M: (skg.Group(M, *dims, [0, 1, 1, 1, 1]), stage_tensors(M, 710 + M)) for M in (8, 64)}
    try:
        s = torch.cuda.Stream()
        for _ in range(300):
            for i, p in enumerate(plans):
                p.run(gemv[0][i], gemv[1][i], gemv[2][i], gemv[3][i], s)
            for M in (8, 64):
                g, (xs, Ws, rs, ys) = groups[M]
                g.run(xs, Ws, rs, ys, s)
        s.synchronize()
        for p in plans:
            p.check()
        for M in (8, 64):
            g, (xs, Ws, rs, ys) = groups[M]
            g.check()
            split = g.info()["split"]
            for i, (K, N, epi) in enumerate(CHAIN_STAGES):
                assert np.array_equal(out_bits(ys[i]), _single(M, N, K, epi, split[i], xs[i], Ws[i], rs[i])), \
                    f"M={M} projection {i} differs from skg_run"
    finally:
        for p in plans:
            p.close()
        for g, _ in groups.values():
            g.close()
