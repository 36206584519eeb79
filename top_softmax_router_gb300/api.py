"""Python binding over the C ABI of libmoe.so (include/moe.h), for torch tensors.

Argument marshalling only: every step of the block runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  bf16 tensors are passed
as ``torch.bfloat16`` (their bit patterns are what the ABI calls bf16).
"""
from __future__ import annotations

import ctypes
import dataclasses

import torch

from . import _lib
from ._lib import MoeConfig, MoeStats, check

__all__ = ["Config", "workspace_bytes", "chunk_plan", "route", "plan", "forward", "backward", "check_status",
           "set_wait_limit_ns", "set_gemm_form", "set_launch_chaining", "set_dispatch", "last_stats", "profile_enable", "profile_reset", "profile_read",
           "diag_wait_timeout", "MoEBlock", "hop_rows_worst_case", "hops_workspace_bytes", "forward_hops",
           "backward_hops", "MoEHopBlock", "MoEStepGraph"]


@dataclasses.dataclass(frozen=True)
class Config:
    N: int
    H: int
    E: int
    k: int
    I: int
    c: int
    K_max: int

    def c_struct(self) -> MoeConfig:
        return MoeConfig(self.N, self.H, self.E, self.k, self.I, self.c, self.K_max)


def _cfg(cfg) -> ctypes.POINTER(MoeConfig):
    if isinstance(cfg, dict):
        cfg = Config(**cfg)
    return ctypes.byref(cfg.c_struct())


def _ptr(t: torch.Tensor | None, dtype: torch.dtype, shape=None, name: str = "") -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(cfg) -> tuple[int, int, int]:
    r, f, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    check(_lib.load().moe_workspace_bytes(_cfg(cfg), ctypes.byref(r), ctypes.byref(f), ctypes.byref(b)),
          "moe_workspace_bytes")
    return r.value, f.value, b.value


def chunk_plan(cfg) -> tuple[int, int]:
    K, c = ctypes.c_int32(), ctypes.c_int32()
    check(_lib.load().moe_chunk_plan(_cfg(cfg), ctypes.byref(K), ctypes.byref(c)), "moe_chunk_plan")
    return K.value, c.value


def _ws(ws: torch.Tensor) -> tuple[int, int]:
    if ws.dtype != torch.uint8 or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace: expected a contiguous CUDA uint8 tensor")
    return ws.data_ptr(), ws.numel()


def route(cfg, X, Wr, bias, topk_idx, gates, ws, stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    w, n = _ws(ws)
    check(_lib.load().moe_route(_cfg(c), _ptr(X, torch.bfloat16, (c.N, c.H), "X"),
                                _ptr(Wr, torch.float32, (c.E, c.H), "Wr"),
                                _ptr(bias, torch.float32, (c.E,), "bias"),
                                _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                                _ptr(gates, torch.float32, (c.N, c.k), "gates"), w, n, _stream(stream)),
          "moe_route")


def plan(cfg, topk_idx, row_route, row_of, expert_off, ws, stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    K, c_eff = chunk_plan(c)
    w, n = _ws(ws)
    check(_lib.load().moe_plan(_cfg(c), _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                               _ptr(row_route, torch.int32, (K, c.k * c_eff), "row_route"),
                               _ptr(row_of, torch.int32, (c.N, c.k), "row_of"),
                               _ptr(expert_off, torch.int32, (K, c.E + 1), "expert_off"), w, n, _stream(stream)),
          "moe_plan")


def forward(cfg, X, topk_idx, gates, Wg, Wu, Wd, Y, ws, stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    w, n = _ws(ws)
    check(_lib.load().moe_forward(_cfg(c), _ptr(X, torch.bfloat16, (c.N, c.H), "X"),
                                  _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                                  _ptr(gates, torch.float32, (c.N, c.k), "gates"),
                                  _ptr(Wg, torch.bfloat16, (c.E, c.I, c.H), "Wg"),
                                  _ptr(Wu, torch.bfloat16, (c.E, c.I, c.H), "Wu"),
                                  _ptr(Wd, torch.bfloat16, (c.E, c.H, c.I), "Wd"),
                                  _ptr(Y, torch.bfloat16, (c.N, c.H), "Y"), w, n, _stream(stream)),
          "moe_forward")


def backward(cfg, X, Wr, topk_idx, gates, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dgates, ws, stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    w, n = _ws(ws)
    check(_lib.load().moe_backward(_cfg(c), _ptr(X, torch.bfloat16, (c.N, c.H), "X"),
                                   _ptr(Wr, torch.float32, (c.E, c.H), "Wr"),
                                   _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                                   _ptr(gates, torch.float32, (c.N, c.k), "gates"),
                                   _ptr(Wg, torch.bfloat16, (c.E, c.I, c.H), "Wg"),
                                   _ptr(Wu, torch.bfloat16, (c.E, c.I, c.H), "Wu"),
                                   _ptr(Wd, torch.bfloat16, (c.E, c.H, c.I), "Wd"),
                                   _ptr(dY, torch.bfloat16, (c.N, c.H), "dY"),
                                   _ptr(dX, torch.bfloat16, (c.N, c.H), "dX"),
                                   _ptr(dWr, torch.float32, (c.E, c.H), "dWr"),
                                   _ptr(dWg, torch.float32, (c.E, c.I, c.H), "dWg"),
                                   _ptr(dWu, torch.float32, (c.E, c.I, c.H), "dWu"),
                                   _ptr(dWd, torch.float32, (c.E, c.H, c.I), "dWd"),
                                   _ptr(dgates, torch.float32, (c.N, c.k), "dgates"), w, n, _stream(stream)),
          "moe_backward")


def check_status(ws, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the workspace's device status code."""
    return _lib.load().moe_check_status(ws.data_ptr(), _stream(stream))


def set_gemm_form(form: str) -> None:
    """'auto' (default), 'single' (one CTA per 128-row tile) or 'pair' (CTA pairs, 2-SM MMA)."""
    code = {"auto": _lib.MOE_GEMM_AUTO, "single": _lib.MOE_GEMM_SINGLE, "pair": _lib.MOE_GEMM_PAIR}[form]
    check(_lib.load().moe_set_gemm_form(code), "moe_set_gemm_form")


def set_launch_chaining(mode: str) -> None:
    """'late' (default), 'early' (programmatic dependent launch, every kernel waits for its predecessor
    before touching memory) or 'none' (plain stream order).  The results are the same in every mode."""
    code = {"none": _lib.MOE_CHAIN_NONE, "early": _lib.MOE_CHAIN_EARLY, "late": _lib.MOE_CHAIN_LATE}[mode]
    check(_lib.load().moe_set_launch_chaining(code), "moe_set_launch_chaining")


def set_dispatch(mode: str) -> None:
    """'gather' (default: a gather kernel fills the permuted buffers Xp and dYp) or 'on_load' (the GEMMs
    gather their rows from X and dY with TMA, halving the routed working set).  The results are the same
    bit for bit; workspace sizes follow the mode, so create blocks after choosing it."""
    code = {"gather": _lib.MOE_DISPATCH_GATHER, "on_load": _lib.MOE_DISPATCH_ON_LOAD}[mode]
    check(_lib.load().moe_set_dispatch(code), "moe_set_dispatch")


def set_wait_limit_ns(ns: int) -> None:
    check(_lib.load().moe_set_wait_limit_ns(int(ns)), "moe_set_wait_limit_ns")


def last_stats() -> dict:
    s = MoeStats()
    check(_lib.load().moe_last_stats(ctypes.byref(s)), "moe_last_stats")
    return {f: getattr(s, f) for f, _ in MoeStats._fields_}


def profile_enable(on: bool = True) -> None:
    check(_lib.load().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def profile_reset() -> None:
    check(_lib.load().moe_profile_reset(), "moe_profile_reset")


def profile_read() -> dict:
    n = len(_lib.KERNEL_CLASSES)
    launches = (ctypes.c_int32 * n)()
    ms = (ctypes.c_double * n)()
    names = (ctypes.c_char_p * n)()
    check(_lib.load().moe_profile_read(launches, ms, names), "moe_profile_read")
    return {names[i].decode(): (launches[i], ms[i]) for i in range(n)}


def diag_wait_timeout(limit_ns: int, ws, stream=None) -> None:
    w, n = _ws(ws)
    check(_lib.load().moe_diag_wait_timeout(int(limit_ns), w, n, _stream(stream)), "moe_diag_wait_timeout")


def hop_rows_worst_case(cfg, P: int) -> int:
    r = ctypes.c_int32()
    check(_lib.load().moe_hop_rows_worst_case(_cfg(cfg), int(P), ctypes.byref(r)), "moe_hop_rows_worst_case")
    return r.value


def hops_workspace_bytes(cfg, P: int, max_hop_rows: int) -> tuple[int, int]:
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    check(_lib.load().moe_hops_workspace_bytes(_cfg(cfg), int(P), int(max_hop_rows), ctypes.byref(f),
                                                ctypes.byref(b)), "moe_hops_workspace_bytes")
    return f.value, b.value


def forward_hops(cfg, P, max_hop_rows, X, topk_idx, gates, Wg, Wu, Wd, Y, ws, stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    w, n = _ws(ws)
    check(_lib.load().moe_forward_hops(_cfg(c), int(P), int(max_hop_rows),
                                       _ptr(X, torch.bfloat16, (c.N, c.H), "X"),
                                       _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                                       _ptr(gates, torch.float32, (c.N, c.k), "gates"),
                                       _ptr(Wg, torch.bfloat16, (c.E, c.I, c.H), "Wg"),
                                       _ptr(Wu, torch.bfloat16, (c.E, c.I, c.H), "Wu"),
                                       _ptr(Wd, torch.bfloat16, (c.E, c.H, c.I), "Wd"),
                                       _ptr(Y, torch.bfloat16, (c.N, c.H), "Y"), w, n, _stream(stream)),
          "moe_forward_hops")


def backward_hops(cfg, P, max_hop_rows, X, Wr, topk_idx, gates, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dgates, ws,
                  stream=None) -> None:
    c = cfg if isinstance(cfg, Config) else Config(**cfg)
    w, n = _ws(ws)
    check(_lib.load().moe_backward_hops(_cfg(c), int(P), int(max_hop_rows),
                                        _ptr(X, torch.bfloat16, (c.N, c.H), "X"),
                                        _ptr(Wr, torch.float32, (c.E, c.H), "Wr"),
                                        _ptr(topk_idx, torch.int32, (c.N, c.k), "topk_idx"),
                                        _ptr(gates, torch.float32, (c.N, c.k), "gates"),
                                        _ptr(Wg, torch.bfloat16, (c.E, c.I, c.H), "Wg"),
                                        _ptr(Wu, torch.bfloat16, (c.E, c.I, c.H), "Wu"),
                                        _ptr(Wd, torch.bfloat16, (c.E, c.H, c.I), "Wd"),
                                        _ptr(dY, torch.bfloat16, (c.N, c.H), "dY"),
                                        _ptr(dX, torch.bfloat16, (c.N, c.H), "dX"),
                                        _ptr(dWr, torch.float32, (c.E, c.H), "dWr"),
                                        _ptr(dWg, torch.float32, (c.E, c.I, c.H), "dWg"),
                                        _ptr(dWu, torch.float32, (c.E, c.I, c.H), "dWu"),
                                        _ptr(dWd, torch.float32, (c.E, c.H, c.I), "dWd"),
                                        _ptr(dgates, torch.float32, (c.N, c.k), "dgates"), w, n, _stream(stream)),
          "moe_backward_hops")


class MoEBlock:
    """Owns a workspace (a torch uint8 buffer) for one shape and runs the three calls."""

    def __init__(self, cfg: Config, device="cuda"):
        self.cfg = cfg
        r, f, b = workspace_bytes(cfg)
        self.ws_bytes = max(r, f, b, 256)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.K, self.c_eff = chunk_plan(cfg)

    def route(self, X, Wr, bias=None, stream=None):
        c = self.cfg
        idx = torch.empty(c.N, c.k, dtype=torch.int32, device=X.device)
        g = torch.empty(c.N, c.k, dtype=torch.float32, device=X.device)
        route(c, X, Wr, bias, idx, g, self.ws, stream)
        return idx, g

    def forward(self, X, idx, gates, Wg, Wu, Wd, stream=None):
        Y = torch.empty_like(X)
        forward(self.cfg, X, idx, gates, Wg, Wu, Wd, Y, self.ws, stream)
        return Y

    def backward(self, X, Wr, idx, gates, Wg, Wu, Wd, dY, stream=None, want_dgates=True):
        c = self.cfg
        dX = torch.empty_like(X)
        dWr = torch.empty(c.E, c.H, dtype=torch.float32, device=X.device)
        dWg = torch.empty(c.E, c.I, c.H, dtype=torch.float32, device=X.device)
        dWu = torch.empty_like(dWg)
        dWd = torch.empty(c.E, c.H, c.I, dtype=torch.float32, device=X.device)
        dg = torch.empty(c.N, c.k, dtype=torch.float32, device=X.device) if want_dgates else None
        backward(c, X, Wr, idx, gates, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dg, self.ws, stream)
        return dict(dX=dX, dWr=dWr, dWg=dWg, dWu=dWu, dWd=dWd, dgates=dg)

    def check(self, stream=None) -> None:
        code = check_status(self.ws, stream)
        check(code, "device status")


class MoEHopBlock(MoEBlock):
    """The expert-partition schedule: P hops of experts, workspace sized for `max_hop_rows` routed rows per hop
    (default: the worst case for this shape, which always suffices)."""

    def __init__(self, cfg: Config, P: int, max_hop_rows: int | None = None, device="cuda"):
        self.cfg = cfg
        self.P = P
        self.cap = max_hop_rows if max_hop_rows is not None else hop_rows_worst_case(cfg, P)
        r, _, _ = workspace_bytes(cfg)
        f, b = hops_workspace_bytes(cfg, P, self.cap)
        self.ws_bytes = max(r, f, b, 256)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.K, self.c_eff = chunk_plan(cfg)

    def forward(self, X, idx, gates, Wg, Wu, Wd, stream=None):
        Y = torch.empty_like(X)
        forward_hops(self.cfg, self.P, self.cap, X, idx, gates, Wg, Wu, Wd, Y, self.ws, stream)
        return Y

    def backward(self, X, Wr, idx, gates, Wg, Wu, Wd, dY, stream=None, want_dgates=True):
        c = self.cfg
        dX = torch.empty_like(X)
        dWr = torch.empty(c.E, c.H, dtype=torch.float32, device=X.device)
        dWg = torch.empty(c.E, c.I, c.H, dtype=torch.float32, device=X.device)
        dWu = torch.empty_like(dWg)
        dWd = torch.empty(c.E, c.H, c.I, dtype=torch.float32, device=X.device)
        dg = torch.empty(c.N, c.k, dtype=torch.float32, device=X.device) if want_dgates else None
        backward_hops(c, self.P, self.cap, X, Wr, idx, gates, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dg, self.ws,
                      stream)
        return dict(dX=dX, dWr=dWr, dWg=dWg, dWu=dWu, dWd=dWd, dgates=dg)


class MoEStepGraph:
    """route + forward + backward of one block, captured once as a CUDA graph over fixed buffers and
    replayed per step.  An MoEBlock is captured with the chunk schedule, an MoEHopBlock with its
    expert-partition schedule.

    Every launch reads its tile and expert lists from device memory (nothing is read back to the
    host), so a replay after new contents were copied into X, dY or the weights routes and computes
    afresh; the results are bitwise those of the eager calls.  One eager step runs first so that
    per-device setup (kernel attributes, the library's side stream) happens outside the capture.
    """

    def __init__(self, blk: MoEBlock, X, Wr, bias, Wg, Wu, Wd, dY, stream=None):
        c = blk.cfg
        self.blk = blk
        self.args = (X, Wr, bias, Wg, Wu, Wd, dY)
        dev = X.device
        self.idx = torch.empty(c.N, c.k, dtype=torch.int32, device=dev)
        self.gates = torch.empty(c.N, c.k, dtype=torch.float32, device=dev)
        self.Y = torch.empty_like(X)
        self.dX = torch.empty_like(X)
        self.dWr = torch.empty(c.E, c.H, dtype=torch.float32, device=dev)
        self.dWg = torch.empty(c.E, c.I, c.H, dtype=torch.float32, device=dev)
        self.dWu = torch.empty_like(self.dWg)
        self.dWd = torch.empty(c.E, c.H, c.I, dtype=torch.float32, device=dev)
        self.dgates = torch.empty(c.N, c.k, dtype=torch.float32, device=dev)
        s = stream if stream is not None else torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            self._step()
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=s):
            self._step()

    def _step(self):
        c, ws = self.blk.cfg, self.blk.ws
        X, Wr, bias, Wg, Wu, Wd, dY = self.args
        route(c, X, Wr, bias, self.idx, self.gates, ws)
        if isinstance(self.blk, MoEHopBlock):   # the expert-partition schedule
            P, cap = self.blk.P, self.blk.cap
            forward_hops(c, P, cap, X, self.idx, self.gates, Wg, Wu, Wd, self.Y, ws)
            backward_hops(c, P, cap, X, Wr, self.idx, self.gates, Wg, Wu, Wd, dY, self.dX, self.dWr, self.dWg,
                          self.dWu, self.dWd, self.dgates, ws)
            return
        forward(c, X, self.idx, self.gates, Wg, Wu, Wd, self.Y, ws)
        backward(c, X, Wr, self.idx, self.gates, Wg, Wu, Wd, dY, self.dX, self.dWr, self.dWg, self.dWu, self.dWd,
                 self.dgates, ws)

    def replay(self) -> None:
        self.graph.replay()

    def grads(self) -> dict:
        return dict(dX=self.dX, dWr=self.dWr, dWg=self.dWg, dWu=self.dWu, dWd=self.dWd, dgates=self.dgates)
