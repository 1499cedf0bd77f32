"""Helpers for the GPU tests: move seeded operands to the device, run one
projection through the C ABI, bring the output back as raw bits."""
from __future__ import annotations

import numpy as np
import torch

from projection_gemm_gb300 import skg
from projection_gemm_gb300.inputs import Projection, Tensors, bits, generate


def to_dev(t):
    return None if t is None else t.to("cuda", non_blocking=False).contiguous()


def out_tensor(M, N, epilogue):
    dt = torch.float32 if skg._epi(epilogue) == skg.SKG_EPI_FP32 else torch.bfloat16
    return torch.empty(M, N, dtype=dt, device="cuda")


def out_bits(y: torch.Tensor) -> np.ndarray:
    y = y.cpu()
    if y.dtype == torch.float32:
        return y.numpy().astype(np.float64)
    return bits(y)


class DeviceCase:
    """A projection's operands on the GPU plus its plan."""

    def __init__(self, p: Projection, tensors: Tensors | None = None):
        self.p = p
        self.t = tensors if tensors is not None else generate(p)
        self.x = to_dev(self.t.x)
        self.W = to_dev(self.t.W)
        self.res = to_dev(self.t.res)
        self.plan = skg.Plan(p.M, p.N, p.K, p.epilogue)

    def run(self, y=None, stream=None) -> torch.Tensor:
        if y is None:
            y = out_tensor(self.p.M, self.p.N, self.p.epilogue)
        self.plan.run(self.x, self.W, self.res, y, stream)
        return y

    def run_bits(self) -> np.ndarray:
        y = self.run()
        torch.cuda.synchronize()
        return out_bits(y)

    def host_bits(self):
        return (bits(self.t.x), bits(self.t.W), None if self.t.res is None else bits(self.t.res))

    def close(self):
        self.plan.close()
