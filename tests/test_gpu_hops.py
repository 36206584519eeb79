"""GPU parity of the expert-partition ("hop") schedule against the oracle and the chunk schedule.

RelayMoE summary, sections 3.1 and 3.3: hops over partitions of the experts.
The block's definition does not depend on the schedule, so the same oracle
and tolerance apply; Y and dX are summed in a different fp32 order than the
chunk schedule, so the two schedules agree to rounding, not bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as O
from synth import inputs as S
from gpu_util import TOL, DevInputs, bf16_as_f64, f32, need_gpu, lib_api, run_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    need_gpu()
    return lib_api()


def run_hops(M, w, D, P, cap=None):
    cfg = M.Config(**w.cfg())
    blk = M.MoEHopBlock(cfg, P, cap)
    idx, g = blk.route(D.X, D.Wr, D.bias)
    Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
    gr = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY)
    code = M.check_status(blk.ws)
    torch.cuda.synchronize()
    out = dict(topk_idx=idx.cpu().numpy(), gates=f32(g), Y=bf16_as_f64(Y), dX=bf16_as_f64(gr["dX"]),
               dgates=f32(gr["dgates"]), dWr=f32(gr["dWr"]), dWg=f32(gr["dWg"]), dWu=f32(gr["dWu"]),
               dWd=f32(gr["dWd"]), status=code, stats=M.last_stats())
    return out


def workload(name):
    if "/" in name:
        base, f = name.split("/")
        return S.WORKLOADS[base].scaled(int(f))
    return S.WORKLOADS[name]


@pytest.mark.parametrize("name,P", [("tiny", 1), ("tiny", 3), ("tiny", 8), ("mid/8", 8), ("extreme/8", 16),
                                    ("long/8", 4)])
def test_hops_vs_oracle_and_chunks(M, name, P):
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    got = run_hops(M, w, D, P)
    assert got["status"] == 0
    ref = O.block(T.X, T.Wr, T.bias, (T.Wg, T.Wu, T.Wd), T.dY, w.k)
    assert np.array_equal(got["topk_idx"], ref["topk_idx"])
    names = ("Y", "dX", "dgates", "dWr", "dWg", "dWu", "dWd")
    errs = {n: O.normalised_error(got[n], ref[n]) for n in names}
    assert all(v <= TOL for v in errs.values()), errs
    chunks = run_block(M, w, D)
    for n in names:
        assert O.normalised_error(got[n], chunks[n]) <= TOL, n


def test_hops_reproducible(M):
    w = workload("mid/8")
    D = DevInputs(S.make(w))
    a = run_hops(M, w, D, 8)
    b = run_hops(M, w, D, 8)
    for n in ("Y", "dX", "dgates", "dWr", "dWg", "dWu", "dWd"):
        assert np.array_equal(a[n], b[n]), n


def test_hop_overflow_is_reported(M):
    """A hop with more routed rows than the workspace holds is skipped and reported, never overrun."""
    from top_softmax_router_gb300 import _lib
    w = S.Workload("ovf", N=256, H=64, E=4, k=2, I=64, c=256, K_max=1)
    T = S.make(w)
    T.bias = np.array([30.0, 0.0, 0.0, 0.0], np.float32)    # every token picks expert 0
    got = run_hops(M, w, DevInputs(T), P=4, cap=64)
    assert got["status"] == _lib.MOE_ERR_DEVICE_CHECK


def test_hops_pair_and_single_forms_agree(M):
    w = workload("mid/8")
    D = DevInputs(S.make(w))
    try:
        M.set_gemm_form("single")
        one = run_hops(M, w, D, 4)
        M.set_gemm_form("pair")
        two = run_hops(M, w, D, 4)
    finally:
        M.set_gemm_form("auto")
    for n in ("Y", "dX", "dgates", "dWr", "dWg", "dWu", "dWd"):
        assert np.array_equal(one[n], two[n]), n


def test_hop_schedule_graph_replay_matches_eager(M):
    """The hop schedule captured as one CUDA graph (as bench.py times it) gives the eager calls' bits."""
    w = workload("mid/8")
    T = S.make(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())
    blk = M.MoEHopBlock(cfg, 8)
    N, H, E, k, I = w.N, w.H, w.E, w.k, w.I
    idx = torch.empty(N, k, dtype=torch.int32, device="cuda")
    g = torch.empty(N, k, device="cuda")
    Y = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty_like(Y)
    dWr = torch.empty(E, H, device="cuda")
    dWg = torch.empty(E, I, H, device="cuda")
    dWu = torch.empty_like(dWg)
    dWd = torch.empty(E, H, I, device="cuda")
    dg = torch.empty(N, k, device="cuda")

    def step(st):
        M.route(cfg, D.X, D.Wr, D.bias, idx, g, blk.ws, st)
        M.forward_hops(cfg, 8, blk.cap, D.X, idx, g, D.Wg, D.Wu, D.Wd, Y, blk.ws, st)
        M.backward_hops(cfg, 8, blk.cap, D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY, dX, dWr, dWg, dWu, dWd, dg,
                        blk.ws, st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (Y, dX, dWr, dWg, dWu, dWd, dg)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for t in (Y, dX, dWr, dWg, dWu, dWd, dg):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert M.check_status(blk.ws) == 0
    for a, b in zip(eager, (Y, dX, dWr, dWg, dWu, dWd, dg)):
        assert torch.equal(a, b)


def test_step_graph_of_a_hop_block_runs_the_hop_schedule(M):
    """MoEStepGraph over an MoEHopBlock captures the expert-partition calls: its replay gives the bits of
    the block's own eager forward/backward (which run the hop schedule)."""
    w = workload("mid/8")
    T = S.make(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())
    blk = M.MoEHopBlock(cfg, 8)
    idx, g = blk.route(D.X, D.Wr, D.bias)
    Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
    gr = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY)
    torch.cuda.synchronize()
    step = M.MoEStepGraph(blk, D.X, D.Wr, D.bias, D.Wg, D.Wu, D.Wd, D.dY)
    for t in (step.Y, step.dX, step.dWg):
        t.zero_()
    step.replay()
    torch.cuda.synchronize()
    blk.check()
    assert torch.equal(step.idx, idx)
    assert torch.equal(step.Y, Y)
    got = step.grads()
    for n in ("dX", "dWr", "dWg", "dWu", "dWd", "dgates"):
        assert torch.equal(got[n], gr[n]), n
