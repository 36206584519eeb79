"""Helpers for the GPU parity tests: upload seeded inputs, run the C ABI, fetch results."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from synth import inputs as S

TOL = 1e-2   # max|gpu - oracle| / max|oracle| per floating-point tensor


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def lib_api():
    """The product binding; building it is part of the test setup (nvcc), never a fallback."""
    import top_softmax_router_gb300.build as B
    B.build()
    import top_softmax_router_gb300 as M
    return M


def bf16_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


def bf16_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bf16_as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DevInputs:
    def __init__(self, T: S.Tensors, dev="cuda"):
        self.X = bf16_dev(T.X, dev)
        self.Wr = torch.from_numpy(T.Wr).to(dev)
        self.bias = None if T.bias is None else torch.from_numpy(T.bias).to(dev)
        self.Wg = bf16_dev(T.Wg, dev)
        self.Wu = bf16_dev(T.Wu, dev)
        self.Wd = bf16_dev(T.Wd, dev)
        self.dY = bf16_dev(T.dY, dev)


def run_block(M, w: S.Workload, D: DevInputs, K_max=None, want_dgates=True):
    """route + forward + backward through the C ABI; returns host numpy results."""
    cfg = M.Config(**{**w.cfg(), **({} if K_max is None else {"K_max": K_max})})
    blk = M.MoEBlock(cfg)
    idx, g = blk.route(D.X, D.Wr, D.bias)
    Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
    grads = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY, want_dgates=want_dgates)
    blk.check()
    torch.cuda.synchronize()
    out = dict(topk_idx=idx.cpu().numpy(), gates=f32(g), Y=bf16_as_f64(Y), Y_bits=bf16_host(Y),
               dX=bf16_as_f64(grads["dX"]), dX_bits=bf16_host(grads["dX"]),
               dWr=f32(grads["dWr"]), dWg=f32(grads["dWg"]), dWu=f32(grads["dWu"]), dWd=f32(grads["dWd"]),
               stats=M.last_stats(), K=blk.K, c_eff=blk.c_eff)
    if want_dgates:
        out["dgates"] = f32(grads["dgates"])
    return out
