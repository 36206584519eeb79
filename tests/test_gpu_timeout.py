"""Device-side waits are bounded: a wait on a barrier nothing signals ends with
MOE_ERR_TIMEOUT in the workspace status word, and the context stays usable.
(No trap, no fault: the kernel gives up after its limit and returns.)"""
import numpy as np
import pytest
import torch

from gpu_util import need_gpu, lib_api

pytestmark = pytest.mark.gpu


def test_wait_times_out_and_context_survives():
    need_gpu()
    M = lib_api()
    from top_softmax_router_gb300 import _lib
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    M.diag_wait_timeout(50_000_000, ws)          # 50 ms
    assert M.check_status(ws) == _lib.MOE_ERR_TIMEOUT
    assert M.check_status(ws) == 0               # cleared by the first check
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum()) == float(np.arange(1024).sum() * 2)


def test_bad_expert_id_is_reported_not_faulted():
    need_gpu()
    M = lib_api()
    from top_softmax_router_gb300 import _lib
    cfg = M.Config(N=64, H=64, E=4, k=2, I=64, c=64, K_max=1)
    K, c_eff = M.chunk_plan(cfg)
    ws = torch.zeros(max(M.workspace_bytes(cfg)), dtype=torch.uint8, device="cuda")
    idx = torch.zeros(64, 2, dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    idx[5, 1] = 9                                 # out of range: the plan kernel checks and reports
    rr = torch.empty(K, 2 * c_eff, dtype=torch.int32, device="cuda")
    ro = torch.empty(64, 2, dtype=torch.int32, device="cuda")
    off = torch.empty(K, 5, dtype=torch.int32, device="cuda")
    M.plan(cfg, idx, rr, ro, off, ws)
    assert M.check_status(ws) == _lib.MOE_ERR_DEVICE_CHECK
