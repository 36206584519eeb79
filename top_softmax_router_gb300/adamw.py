"""Python binding of the offloaded optimizer step (include/moe_adamw.h).

"bounded-streaming operators" summary, Methodology 4 (OffloadStreamAdamW), eq. (5):
fp32 master weights and Adam moments stay in page-locked host memory; buckets of
``bucket`` parameters rotate through ``slots`` device staging slots while the
library's three streams copy in, update (fused AdamW + bf16 working-weight
refresh) and write back.  Argument marshalling only: the update runs in the
library's CUDA kernel.
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import AdamwHparams, check

__all__ = ["AdamWHparams", "adamw_staging_bytes", "adamw_offload_step", "adamw_step", "OffloadStreamAdamW"]


@dataclasses.dataclass(frozen=True)
class AdamWHparams:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0

    def c_struct(self, step: int) -> AdamwHparams:
        return AdamwHparams(self.lr, self.beta1, self.beta2, self.eps, self.weight_decay, step)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _flat(t: torch.Tensor, dtype, n: int, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous() or t.numel() != n:
        raise ValueError(f"{name}: expected a contiguous tensor of {n} elements")
    return t


def _host_state(t: torch.Tensor, n: int, name: str) -> int:
    _flat(t, torch.float32, n, name)
    if n > 0 and (t.is_cuda or not t.is_pinned()):
        raise ValueError(f"{name}: expected page-locked host memory (pin_memory)")
    return t.data_ptr()


def _grad(g: torch.Tensor, n: int) -> tuple[int, int]:
    if g.dtype == torch.float32:
        code = _lib.MOE_GRAD_F32
    elif g.dtype == torch.bfloat16:
        code = _lib.MOE_GRAD_BF16
    else:
        raise TypeError(f"grad: expected float32 or bfloat16, got {g.dtype}")
    _flat(g, g.dtype, n, "grad")
    if not g.is_cuda:
        raise ValueError("grad: expected a CUDA tensor")
    return g.data_ptr(), code


def _weight(w: torch.Tensor, n: int) -> int:
    _flat(w, torch.bfloat16, n, "weight")
    if not w.is_cuda:
        raise ValueError("weight: expected a CUDA tensor")
    return w.data_ptr()


def adamw_staging_bytes(bucket: int, slots: int) -> int:
    out = ctypes.c_size_t()
    check(_lib.load().moe_adamw_staging_bytes(bucket, slots, ctypes.byref(out)), "moe_adamw_staging_bytes")
    return out.value


def adamw_offload_step(hp: AdamWHparams, step: int, master, exp_avg, exp_avg_sq, grad, weight, staging,
                       bucket: int, slots: int, stream=None) -> None:
    """One offloaded step (eq. (5)); the host state is updated in place, asynchronously on ``stream``."""
    n = master.numel()
    g, code = _grad(grad, n)
    if staging.dtype != torch.uint8 or not staging.is_cuda or not staging.is_contiguous():
        raise ValueError("staging: expected a contiguous CUDA uint8 tensor")
    h = hp.c_struct(step)
    check(_lib.load().moe_adamw_offload_step(
        ctypes.byref(h), n, bucket, slots, _host_state(master, n, "master"), _host_state(exp_avg, n, "exp_avg"),
        _host_state(exp_avg_sq, n, "exp_avg_sq"), g, code, _weight(weight, n), staging.data_ptr(),
        staging.numel(), _stream(stream)), "moe_adamw_offload_step")


def adamw_step(hp: AdamWHparams, step: int, master, exp_avg, exp_avg_sq, grad, weight, stream=None) -> None:
    """The fused update in place on device-resident state, or on page-locked host state read and written
    directly across the host link."""
    n = master.numel()
    g, code = _grad(grad, n)
    ptrs = []
    for t, name in ((master, "master"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        _flat(t, torch.float32, n, name)
        if n > 0 and not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name}: expected a CUDA tensor or page-locked host memory")
        ptrs.append(t.data_ptr())
    h = hp.c_struct(step)
    check(_lib.load().moe_adamw_step(ctypes.byref(h), n, *ptrs, g, code, _weight(weight, n), _stream(stream)),
          "moe_adamw_step")


class OffloadStreamAdamW:
    """AdamW over one flat parameter vector whose fp32 state lives in page-locked host memory.

    ``master`` (a CPU float32 tensor) gives the initial master weights; the moments start at zero.  Each
    ``step(grad, weight)`` streams the state through ``slots`` device slots of ``bucket`` parameters,
    writes bf16(p) into ``weight`` and returns without synchronising the host (``master``, ``exp_avg`` and
    ``exp_avg_sq`` are valid once the stream has passed the step).  ``direct=True`` runs the single kernel
    that reads and writes the host state across the host link instead of the staged pipeline.
    """

    def __init__(self, master: torch.Tensor, bucket: int = 1 << 23, slots: int = 4, hp: AdamWHparams | None = None,
                 direct: bool = False, device=None):
        n = master.numel()
        self.n, self.bucket, self.slots, self.direct = n, int(bucket), int(slots), direct
        self.hp = hp or AdamWHparams()
        self.t = 0
        self.master = torch.empty(n, dtype=torch.float32, pin_memory=True)
        self.master.copy_(master.reshape(-1))
        self.exp_avg = torch.zeros(n, dtype=torch.float32, pin_memory=True)
        self.exp_avg_sq = torch.zeros(n, dtype=torch.float32, pin_memory=True)
        nbytes = adamw_staging_bytes(self.bucket, self.slots)
        self.staging = None if direct else torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")

    def step(self, grad: torch.Tensor, weight: torch.Tensor, stream=None) -> None:
        self.t += 1
        if self.direct:
            adamw_step(self.hp, self.t, self.master, self.exp_avg, self.exp_avg_sq, grad.view(-1),
                       weight.view(-1), stream)
        else:
            adamw_offload_step(self.hp, self.t, self.master, self.exp_avg, self.exp_avg_sq, grad.view(-1),
                               weight.view(-1), self.staging, self.bucket, self.slots, stream)
