"""Launch ordering and the side-stream prefetch.

"Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly" (background
2, validate correctness systematically) reports a compiler that hoisted an
activation read above a synchronisation wait, fixed by allowing early loads
of static weights only.  Under programmatic dependent launch the kernels here
may start before the previous kernel finished; these tests chain projections
whose x is the previous projection's y, with the intermediate buffers first
filled with NaN, and require the bits of a fully serialised run.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.oracle as O
from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import Projection, bits, generate
from tests import tolerance as T
from tests.gpu_util import out_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from projection_gemm_gb300 import build
    build.build()
    skg.load()


class Reference:
    """The oracle's values for one projection's operands (computed once),
    and the acceptance check of a GPU output against them."""

    def __init__(self, x, W, res=None, fp32=False):
        self.K = x.shape[1]
        self.fp32 = fp32
        self.y, self.s1, _ = O.linear(bits(x.cpu()), bits(W.cpu()), None if res is None else bits(res.cpu()))

    def check(self, y_bits, what):
        T.check(y_bits, self.y, self.s1, self.K, fp32=self.fp32, what=what)


def check_chain(x0, Ws, y_bits, what):
    """Each stage of a chain against the oracle, fed the bits the GPU's
    previous stage produced."""
    x = bits(x0.cpu())
    for i, (W, yb) in enumerate(zip(Ws, y_bits)):
        y_ref, s1, _ = O.linear(x, bits(W.cpu()))
        T.check(yb, y_ref, s1, x.shape[1], what=f"{what} stage {i}")
        x = yb


def _chain_run(plans, Ws, x0, ys, pdl: bool, serialize: bool):
    for p in plans:
        p.set_pdl(pdl)
    for y in ys:
        y.view(torch.int16).fill_(0x7FC0)   # NaN: any early read shows up
    torch.cuda.synchronize()
    x = x0
    for p, W, y in zip(plans, Ws, ys):
        p.run(x, W, None, y)
        if serialize:
            torch.cuda.synchronize()
        x = y
    torch.cuda.synchronize()
    return [out_bits(y) for y in ys]


@pytest.mark.parametrize("M", (1, 2, 8, 64))
def test_pdl_chain_reads_activations_after_wait(M):
    dims = [4096, 7168, 4096, 7168, 2048]
    plans, Ws, ys = [], [], []
    for i in range(len(dims) - 1):
        K, N = dims[i], dims[i + 1]
        t = generate(Projection(M, N, K, "bf16", seed=50 + i))
        Ws.append(to_dev(t.W))
        plans.append(skg.Plan(M, N, K, "bf16"))
        ys.append(torch.empty(M, N, dtype=torch.bfloat16, device="cuda"))
    x0 = to_dev(generate(Projection(M, dims[1], dims[0], "bf16", seed=49)).x)
    try:
        ref = _chain_run(plans, Ws, x0, ys, pdl=False, serialize=True)
        for a in ref:
            assert not np.any((a & 0x7FFF) > 0x7F80), "NaN in the serialised chain"
        check_chain(x0, Ws, ref, f"M={M} serialised chain")
        for _ in range(10):
            got = _chain_run(plans, Ws, x0, ys, pdl=True, serialize=False)
            for a, b in zip(got, ref):
                assert np.array_equal(a, b)
    finally:
        for p in plans:
            p.close()


@pytest.mark.parametrize("M", (1, 16))
def test_prefetch_beside_projection(M):
    cur = generate(Projection(M, 7168, 7168, "bf16", seed=60))
    nxt = generate(Projection(M, 12288, 7168, "bf16", seed=61))
    p_cur, p_next = skg.Plan(M, 7168, 7168, "bf16"), skg.Plan(M, 12288, 7168, "bf16")
    try:
        info = p_next.info()
        assert 0 < info["prefetch_bytes"] <= 2 * 12288 * 7168
        x, W, W2, x2 = to_dev(cur.x), to_dev(cur.W), to_dev(nxt.W), to_dev(nxt.x)
        y = torch.empty(M, 7168, dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty(M, 12288, dtype=torch.bfloat16, device="cuda")
        p_cur.run(x, W, None, y)
        p_next.run(x2, W2, None, y2)
        torch.cuda.synchronize()
        ref, ref2 = out_bits(y), out_bits(y2)
        want, want2 = Reference(x, W), Reference(x2, W2)
        side = torch.cuda.Stream()
        main = torch.cuda.current_stream()
        for joined in (True, False):
            for y_ in (y, y2):
                y_.view(torch.int16).fill_(0x7FC0)
            for _ in range(5):
                side.wait_stream(main)
                p_next.prefetch(W2, side)
                p_cur.run(x, W, None, y)
                if joined:                       # the next projection after its prefetch
                    main.wait_stream(side)
                p_next.run(x2, W2, None, y2)
            main.wait_stream(side)
            torch.cuda.synchronize()
            want.check(out_bits(y), f"M={M} beside the prefetch (joined={joined})")
            want2.check(out_bits(y2), f"M={M} after its prefetch (joined={joined})")
            assert np.array_equal(out_bits(y), ref) and np.array_equal(out_bits(y2), ref2)
        skg.skg_plan_set_prefetch_fraction(p_next.handle, 0.0)
        assert p_next.info()["prefetch_bytes"] == 0
        p_next.prefetch(W2, side)
        torch.cuda.synchronize()
        p_cur.check()
        p_next.check()
    finally:
        p_cur.close()
        p_next.close()


def test_graph_capture_of_a_chain():
    """skg_run allocates nothing, so a chain captures into one CUDA graph."""
    M = 8
    dims = [7168, 4096, 7168]
    plans, Ws, ys = [], [], []
    for i in range(2):
        t = generate(Projection(M, dims[i + 1], dims[i], "bf16", seed=70 + i))
        Ws.append(to_dev(t.W))
        plans.append(skg.Plan(M, dims[i + 1], dims[i], "bf16"))
        ys.append(torch.empty(M, dims[i + 1], dtype=torch.bfloat16, device="cuda"))
    x0 = to_dev(generate(Projection(M, 4096, 7168, "bf16", seed=69)).x)
    try:
        ref = _chain_run(plans, Ws, x0, ys, pdl=False, serialize=True)
        for p in plans:
            p.set_pdl(True)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            plans[0].run(x0, Ws[0], None, ys[0], s)
            plans[1].run(ys[0], Ws[1], None, ys[1], s)
        for y in ys:
            y.view(torch.int16).fill_(0x7FC0)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        got = [out_bits(y) for y in ys]
        check_chain(x0, Ws, got, "graph replay")
        for a, b in zip(got, ref):
            assert np.array_equal(a, b)
    finally:
        for p in plans:
            p.close()


@pytest.mark.parametrize("M", (1, 2, 3, 16, 64))
def test_next_weight_prefetch_inside_the_launch(M):
    """A plan told the next projection's weight asks the L2 for it from inside
    its own launch: the outputs of both projections keep their bits, and the
    setting is checked and can be turned off."""
    cur = generate(Projection(M, 7168, 7168, "bf16", seed=80))
    nxt = generate(Projection(M, 4096, 7168, "bf16_residual", seed=81))
    p_cur, p_next = skg.Plan(M, 7168, 7168, "bf16"), skg.Plan(M, 4096, 7168, "bf16_residual")
    try:
        x, W, x2, W2, r2 = to_dev(cur.x), to_dev(cur.W), to_dev(nxt.x), to_dev(nxt.W), to_dev(nxt.res)
        y = torch.empty(M, 7168, dtype=torch.bfloat16, device="cuda")
        y2 = torch.empty(M, 4096, dtype=torch.bfloat16, device="cuda")
        p_cur.run(x, W, None, y)
        p_next.run(x2, W2, r2, y2)
        torch.cuda.synchronize()
        ref, ref2 = out_bits(y), out_bits(y2)
        want, want2 = Reference(x, W), Reference(x2, W2, r2)
        for nbytes in (16, 1 << 20, 2 * 4096 * 7168, 1 << 40):   # capped at the L2 size
            p_cur.set_next_weight(W2, nbytes)
            p_next.set_next_weight(W, nbytes)
            for y_ in (y, y2):
                y_.view(torch.int16).fill_(0x7FC0)
            for _ in range(3):
                p_cur.run(x, W, None, y)
                p_next.run(x2, W2, r2, y2)
            torch.cuda.synchronize()
            want.check(out_bits(y), f"M={M} prefetching {nbytes} bytes of the next weight")
            want2.check(out_bits(y2), f"M={M} after the in-launch prefetch of {nbytes} bytes")
            assert np.array_equal(out_bits(y), ref) and np.array_equal(out_bits(y2), ref2), nbytes
        with pytest.raises(skg.SkgError) as e:
            p_cur.set_next_weight(W2.data_ptr() + 2, 1 << 20)
        assert e.value.status == skg.SKG_ERR_ALIGNMENT
        p_cur.set_next_weight(None, 1 << 20)
        p_cur.run(x, W, None, y)
        torch.cuda.synchronize()
        assert np.array_equal(out_bits(y), ref)
        p_cur.check()
        p_next.check()
    finally:
        p_cur.close()
        p_next.close()
