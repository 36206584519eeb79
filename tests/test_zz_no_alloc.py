"""moe_route_noalloc: the router for callers that cannot allocate device memory.

It keeps the logits in a fixed array inside the library instead of a caller
workspace.  Checked through the C ABI against moe_route (the workspace
version) on two calls in a row, since every call reuses the same array.
Collected last so that a stop-at-first-failure run has already run the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import inputs as S
from gpu_util import DevInputs, need_gpu, lib_api

pytestmark = pytest.mark.gpu


def _noalloc(L, cfg, D, idx, g, stream):
    return L.moe_route_noalloc(ctypes.byref(cfg), D.X.data_ptr(), D.Wr.data_ptr(),
                               None if D.bias is None else D.bias.data_ptr(),
                               idx.data_ptr(), g.data_ptr(), stream)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_noalloc_matches_workspace_router_twice(name):
    need_gpu()
    M = lib_api()
    from top_softmax_router_gb300 import _lib
    L = _lib.load()
    w = S.WORKLOADS[name]
    D = DevInputs(S.make(w))
    cfg = _lib.MoeConfig(*[w.cfg()[n] for n in ("N", "H", "E", "k", "I", "c", "K_max")])
    stream = torch.cuda.current_stream().cuda_stream
    # the existing entry point, with a caller workspace
    r, _, _ = M.workspace_bytes(M.Config(**w.cfg()))
    ws = torch.zeros(max(r, 256), dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty(w.N, w.k, dtype=torch.int32, device="cuda")
    ref_g = torch.empty(w.N, w.k, dtype=torch.float32, device="cuda")
    M.route(M.Config(**w.cfg()), D.X, D.Wr, D.bias, ref_idx, ref_g, ws)
    torch.cuda.synchronize()
    for call in range(2):
        idx = torch.full((w.N, w.k), -7, dtype=torch.int32, device="cuda")
        g = torch.full((w.N, w.k), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(L, cfg, D, idx, g, stream) == 0, f"call {call}"
        torch.cuda.synchronize()
        # the same kernels on the same logits: the same bits
        assert torch.equal(idx, ref_idx), f"call {call}: expert ids differ"
        assert torch.equal(g, ref_g), f"call {call}: gates differ"


def test_noalloc_at_the_size_limit():
    """N * E exactly at the array's capacity (4096 tokens x 1024 experts): accepted, and bitwise equal to
    the workspace router on two calls in a row."""
    need_gpu()
    M = lib_api()
    from top_softmax_router_gb300 import _lib
    L = _lib.load()
    w = S.Workload("noalloc_limit", N=4096, H=128, E=1024, k=8, I=64, c=4096, K_max=1)
    assert w.N * w.E == 4 * 1024 * 1024
    D = DevInputs(S.make(w))
    cfg = _lib.MoeConfig(*[w.cfg()[n] for n in ("N", "H", "E", "k", "I", "c", "K_max")])
    stream = torch.cuda.current_stream().cuda_stream
    r, _, _ = M.workspace_bytes(M.Config(**w.cfg()))
    ws = torch.zeros(max(r, 256), dtype=torch.uint8, device="cuda")
    ref_idx = torch.empty(w.N, w.k, dtype=torch.int32, device="cuda")
    ref_g = torch.empty(w.N, w.k, dtype=torch.float32, device="cuda")
    M.route(M.Config(**w.cfg()), D.X, D.Wr, D.bias, ref_idx, ref_g, ws)
    for call in range(2):
        idx = torch.full((w.N, w.k), -7, dtype=torch.int32, device="cuda")
        g = torch.full((w.N, w.k), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(L, cfg, D, idx, g, stream) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx), f"call {call}: expert ids differ"
        assert torch.equal(g, ref_g), f"call {call}: gates differ"


def test_noalloc_rejects_too_many_logits():
    need_gpu()
    lib_api()
    from top_softmax_router_gb300 import _lib
    L = _lib.load()
    cap = 4 * 1024 * 1024
    E = 1024
    N = cap // E + 1
    cfg = _lib.MoeConfig(N, 64, E, 8, 64, 64, 1)
    p = ctypes.c_void_p(256)          # never dereferenced: the size check comes first
    assert L.moe_route_noalloc(ctypes.byref(cfg), p, p, None, p, p, None) == _lib.MOE_ERR_UNSUPPORTED_SHAPE
