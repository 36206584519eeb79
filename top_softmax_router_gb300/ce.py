"""Python binding of the vocabulary-projection cross-entropy head (include/moe_ce.h).

"bounded-streaming operators" summary, Methodology 2 (Ring-DTP), eqs. (2)-(3): the logits are never
formed whole; the forward folds 256-class tiles straight from tensor memory by the online-softmax
recurrence, and the backward writes the gradient of one vocabulary strip at a time.  Argument
marshalling only: every step runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import CeConfig, CeStats, check

__all__ = ["CEConfig", "ce_workspace_bytes", "ce_forward", "ce_backward", "ce_last_stats", "VocabCE"]


@dataclasses.dataclass(frozen=True)
class CEConfig:
    N: int   # tokens
    H: int   # hidden size (multiple of 64)
    V: int   # classes
    P: int   # vocabulary strips of the backward pass

    def c_struct(self) -> CeConfig:
        return CeConfig(self.N, self.H, self.V, self.P)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype, shape, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dtype != dtype:
        raise TypeError(f"{name}: expected a {dtype} tensor")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _ws(ws):
    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA uint8 tensor")
    return ws.data_ptr(), ws.numel()


def ce_workspace_bytes(cfg: CEConfig) -> tuple[int, int]:
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    check(_lib.load().moe_ce_workspace_bytes(ctypes.byref(cfg.c_struct()), ctypes.byref(f), ctypes.byref(b)),
          "moe_ce_workspace_bytes")
    return f.value, b.value


def ce_forward(cfg: CEConfig, X, W, targets, loss, lse, loss_mean, ws, stream=None) -> None:
    w, n = _ws(ws)
    check(_lib.load().moe_ce_forward(
        ctypes.byref(cfg.c_struct()), _ptr(X, torch.bfloat16, (cfg.N, cfg.H), "X"),
        _ptr(W, torch.bfloat16, (cfg.V, cfg.H), "W"), _ptr(targets, torch.int32, (cfg.N,), "targets"),
        _ptr(loss, torch.float32, (cfg.N,), "loss"), _ptr(lse, torch.float32, (cfg.N,), "lse"),
        _ptr(loss_mean, torch.float32, (1,), "loss_mean"), w, n, _stream(stream)), "moe_ce_forward")


def ce_backward(cfg: CEConfig, X, W, targets, lse, dloss, dX, dW, ws, stream=None) -> None:
    w, n = _ws(ws)
    check(_lib.load().moe_ce_backward(
        ctypes.byref(cfg.c_struct()), _ptr(X, torch.bfloat16, (cfg.N, cfg.H), "X"),
        _ptr(W, torch.bfloat16, (cfg.V, cfg.H), "W"), _ptr(targets, torch.int32, (cfg.N,), "targets"),
        _ptr(lse, torch.float32, (cfg.N,), "lse"), _ptr(dloss, torch.float32, (cfg.N,), "dloss"),
        _ptr(dX, torch.bfloat16, (cfg.N, cfg.H), "dX"), _ptr(dW, torch.float32, (cfg.V, cfg.H), "dW"), w, n,
        _stream(stream)), "moe_ce_backward")


def ce_last_stats() -> dict:
    s = CeStats()
    check(_lib.load().moe_ce_last_stats(ctypes.byref(s)), "moe_ce_last_stats")
    return {name: getattr(s, name) for name, _ in CeStats._fields_}


class VocabCE:
    """Owns one workspace for a shape and runs the forward (per-token loss, lse, mean) and the backward."""

    def __init__(self, cfg: CEConfig, device="cuda"):
        self.cfg = cfg
        f, b = ce_workspace_bytes(cfg)
        self.ws = torch.zeros(max(f, b, 256), dtype=torch.uint8, device=device)

    def forward(self, X, W, targets, stream=None):
        c = self.cfg
        loss = torch.empty(c.N, dtype=torch.float32, device=X.device)
        lse = torch.empty(c.N, dtype=torch.float32, device=X.device)
        mean = torch.empty(1, dtype=torch.float32, device=X.device)
        ce_forward(c, X, W, targets, loss, lse, mean, self.ws, stream)
        return loss, lse, mean

    def backward(self, X, W, targets, lse, dloss, stream=None):
        c = self.cfg
        dX = torch.empty(c.N, c.H, dtype=torch.bfloat16, device=X.device)
        dW = torch.empty(c.V, c.H, dtype=torch.float32, device=X.device)
        ce_backward(c, X, W, targets, lse, dloss, dX, dW, self.ws, stream)
        return dX, dW

    def check(self, stream=None) -> None:
        from .api import check_status
        check(check_status(self.ws, stream), "device status")
