"""GPU parity of the whole block (route, permutation, forward, backward) against the oracle.

Every case calls the C ABI through the Python binding and compares with the
CPU oracle element by element: routing and permutation bit for bit, floating
point within max|gpu - oracle| / max|oracle| <= 1e-2.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import moe_ref as O
from synth import inputs as S
from gpu_util import TOL, DevInputs, bf16_dev, need_gpu, lib_api, run_block

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    need_gpu()
    return lib_api()


def oracle_block(T):
    return O.block(T.X, T.Wr, T.bias, (T.Wg, T.Wu, T.Wd), T.dY, T.w.k)


def compare(got, ref, names=("Y", "dX", "dgates", "dWr", "dWg", "dWu", "dWd")):
    assert np.array_equal(got["topk_idx"], ref["topk_idx"]), "routing differs from the oracle"
    assert O.normalised_error(got["gates"], ref["gates"]) < 1e-5
    errs = {n: O.normalised_error(got[n], ref[n]) for n in names if n in got}
    bad = {n: e for n, e in errs.items() if not e <= TOL}
    assert not bad, f"normalised errors above {TOL}: {bad} (all: {errs})"
    return errs


WORKLOADS = ["tiny", "mid/8", "long/8", "many/8", "many_zipf/8", "extreme/8"]


def workload(name):
    if "/" in name:
        base, f = name.split("/")
        return S.WORKLOADS[base].scaled(int(f))
    return S.WORKLOADS[name]


@pytest.mark.parametrize("name", WORKLOADS)
def test_block_vs_oracle(M, name):
    w = workload(name)
    T = S.make(w)
    got = run_block(M, w, DevInputs(T))
    ref = oracle_block(T)
    compare(got, ref)
    st = got["stats"]
    assert st["routed_bytes_peak"] == st["routed_bytes_bound"]   # two k c_eff H b buffers: the pages' bound


@pytest.mark.parametrize("name", ["tiny", "mid/8", "many_zipf/8", "extreme/8"])
def test_gather_on_load_matches_the_gather_kernel_bitwise(M, name):
    """The dispatch gather fused into the GEMMs' operand loads (TMA row gathers from X and dY, no Xp or dYp
    buffer) gives every output of the block bit for bit as the gather kernel does, for the chunk and the
    hop schedule, with half the routed working set; and it matches the oracle."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())

    def outputs(blk):
        idx, g = blk.route(D.X, D.Wr, D.bias)
        Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
        gr = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY)
        st = M.last_stats()
        blk.check()
        torch.cuda.synchronize()
        return [idx, g, Y] + [gr[n] for n in ("dX", "dWr", "dWg", "dWu", "dWd", "dgates")], st, blk.ws_bytes

    try:
        for form in ("auto", "pair") if name == "mid/8" else ("auto",):
            M.set_gemm_form(form)          # "pair": the CTA-pair kernels gather their rows on load too
            for make in (lambda: M.MoEBlock(cfg), lambda: M.MoEHopBlock(cfg, 4)):
                M.set_dispatch("gather")
                ref, st_ref, ws_ref = outputs(make())
                M.set_dispatch("on_load")
                got, st, ws = outputs(make())
                for a, b in zip(got, ref):
                    assert torch.equal(a, b), form
                assert 2 * st["routed_bytes_peak"] == st_ref["routed_bytes_peak"]
                assert ws < ws_ref
        M.set_gemm_form("auto")
        M.set_dispatch("on_load")
        compare(run_block(M, w, D), oracle_block(T))
    finally:
        M.set_dispatch("gather")
        M.set_gemm_form("auto")


@pytest.mark.parametrize("name", ["tiny", "mid/8", "extreme/8"])
def test_permutation_bit_exact(M, name):
    w = workload(name)
    T = S.make(w, weights=False)
    idx, _, _ = O.route(T.X, T.Wr, T.bias, w.k)
    cfg = M.Config(**w.cfg())
    K, c_eff = M.chunk_plan(cfg)
    assert (K, c_eff) == O.chunk_plan(w.N, w.c, w.K_max)
    ws = torch.zeros(max(M.workspace_bytes(cfg)), dtype=torch.uint8, device="cuda")
    d_idx = torch.from_numpy(idx).cuda()
    rr = torch.full((K, w.k * c_eff), -1, dtype=torch.int32, device="cuda")
    row_of = torch.empty(w.N, w.k, dtype=torch.int32, device="cuda")
    off = torch.empty(K, w.E + 1, dtype=torch.int32, device="cuda")
    M.plan(cfg, d_idx, rr, row_of, off, ws)
    assert M.check_status(ws) == 0
    rr, row_of, off = rr.cpu().numpy(), row_of.cpu().numpy(), off.cpu().numpy()
    for i in range(K):
        r_rr, r_off, r_row_of = O.permute_chunk(idx, K, i, w.E)
        n = len(r_rr)
        assert np.array_equal(rr[i, :n], r_rr)
        assert np.array_equal(off[i], r_off)
        toks = O.chunk_tokens(w.N, K, i)
        assert np.array_equal(row_of[toks], r_row_of)


@pytest.mark.parametrize("name", ["mid/8", "extreme/8", "many_zipf/8"])
def test_one_chunk_multiblock_plan_bit_exact(M, name):
    """K = 1 with at least 8,192 routes takes the multi-block plan (count, lists, scatter): the
    permutation matches the oracle bit for bit.  (The expert-partition schedule's global plan takes
    the same path; its tests compare every output with the oracle.)"""
    w = workload(name)
    w1 = dataclasses.replace(w, K_max=1)
    T = S.make(w1, weights=False)
    idx, _, _ = O.route(T.X, T.Wr, T.bias, w1.k)
    assert w1.N * w1.k >= 8192
    cfg = M.Config(**w1.cfg())
    K, c_eff = M.chunk_plan(cfg)
    assert K == 1
    ws = torch.zeros(max(M.workspace_bytes(cfg)), dtype=torch.uint8, device="cuda")
    rr = torch.full((1, w1.k * c_eff), -1, dtype=torch.int32, device="cuda")
    row_of = torch.empty(w1.N, w1.k, dtype=torch.int32, device="cuda")
    off = torch.empty(1, w1.E + 1, dtype=torch.int32, device="cuda")
    M.plan(cfg, torch.from_numpy(idx).cuda(), rr, row_of, off, ws)
    assert M.check_status(ws) == 0
    r_rr, r_off, r_row_of = O.permute_chunk(idx, 1, 0, w1.E)
    assert np.array_equal(rr.cpu().numpy()[0], r_rr)
    assert np.array_equal(off.cpu().numpy()[0], r_off)
    assert np.array_equal(row_of.cpu().numpy(), r_row_of)


@pytest.mark.parametrize("name", WORKLOADS)
def test_k_invariance_and_determinism(M, name):
    """Order only, exact results (bounded-streaming summary, "Core principle" and design requirements
    1-2): on every workload (tiny and the x8-scaled replicas of mid, long, many, many-Zipf and extreme,
    with their own E, k, K and skew), K = 1 and K = K_max give bitwise-identical per-token outputs
    (routing, gates, Y, dX, dgates); repeated runs are bitwise equal on every output; the weight
    gradients of the two chunkings agree within the tolerance (their fp32 sums over chunks differ in
    order only)."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    a = run_block(M, w, D)
    b = run_block(M, w, D)
    one = run_block(M, w, D, K_max=1)
    assert a["K"] > 1 and one["K"] == 1
    for n in ("topk_idx", "gates", "Y_bits", "dX_bits", "dgates", "dWr", "dWg", "dWu", "dWd"):
        assert np.array_equal(a[n], b[n]), f"{n} not reproducible run to run"
    for n in ("topk_idx", "gates", "Y_bits", "dX_bits", "dgates"):
        assert np.array_equal(a[n], one[n]), f"{n} differs between K={a['K']} and K=1"
    for n in ("dWr", "dWg", "dWu", "dWd"):
        assert O.normalised_error(a[n], one[n]) < TOL
    assert one["stats"]["routed_bytes_peak"] >= a["stats"]["routed_bytes_peak"]


@pytest.mark.parametrize("name", ["mid/8", "tiny", "long/8"])
def test_chained_launches_match_serialised_launches(M, name):
    """Neighbouring kernels of a call overlap (programmatic dependent launch; a few kernels wait for their
    predecessor only at their end).  With profiling on, an event is recorded between every two kernels,
    which serialises them; the outputs must be the same bits either way, for the chunk and the hop
    schedule."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())

    def both(blk):
        idx, g = blk.route(D.X, D.Wr, D.bias)
        Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
        gr = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY)
        blk.check()
        torch.cuda.synchronize()
        return [Y] + [gr[n] for n in ("dX", "dWr", "dWg", "dWu", "dWd", "dgates")]

    for blk in (M.MoEBlock(cfg), M.MoEHopBlock(cfg, 4)):
        chained = both(blk)
        M.profile_reset()
        M.profile_enable(True)
        try:
            serial = both(blk)
        finally:
            M.profile_enable(False)
        assert M.profile_read()["gemm_dw"][0] > 0      # the profiled pass did record every launch
        for a, b in zip(chained, serial):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["mid/8", "tiny"])
def test_launch_chaining_modes_give_the_same_bits(M, name):
    """moe_set_launch_chaining only changes how neighbouring kernels overlap: plain stream order,
    early-waiting programmatic launches and the default (some kernels wait at their end) give the same
    bits, for the chunk and the hop schedule."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())

    def outputs(blk):
        idx, g = blk.route(D.X, D.Wr, D.bias)
        Y = blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)
        gr = blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY)
        blk.check()
        torch.cuda.synchronize()
        return [idx, g, Y] + [gr[n] for n in ("dX", "dWr", "dWg", "dWu", "dWd", "dgates")]

    try:
        for blk in (M.MoEBlock(cfg), M.MoEHopBlock(cfg, 4)):
            runs = {}
            for mode in ("none", "early", "late"):
                M.set_launch_chaining(mode)
                runs[mode] = outputs(blk)
            for mode in ("none", "early"):
                for a, b in zip(runs[mode], runs["late"]):
                    assert torch.equal(a, b), mode
    finally:
        M.set_launch_chaining("late")


EDGE = {
    "ragged": S.Workload("ragged", N=1000, H=128, E=6, k=3, I=192, c=300, K_max=16),
    "single_token": S.Workload("single", N=1, H=64, E=4, k=2, I=64, c=16, K_max=4),
    "k1": S.Workload("k1", N=300, H=128, E=5, k=1, I=128, c=64, K_max=8),
    "k_eq_E": S.Workload("kE", N=200, H=128, E=4, k=4, I=128, c=64, K_max=8),
    "E1": S.Workload("E1", N=257, H=192, E=1, k=1, I=320, c=100, K_max=3),
    "wide_rows": S.Workload("wide", N=700, H=64, E=3, k=2, I=64, c=700, K_max=1),
    "top32": S.Workload("top32", N=96, H=64, E=40, k=32, I=64, c=50, K_max=2),
    "E_max": S.Workload("Emax", N=300, H=64, E=1024, k=8, I=64, c=100, K_max=4),
    "one_token_chunks": S.Workload("c1", N=40, H=64, E=8, k=2, I=64, c=1, K_max=64),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(M, name):
    w = EDGE[name]
    T = S.make(w)
    got = run_block(M, w, DevInputs(T))
    ref = oracle_block(T)
    compare(got, ref)
    if w.k == 1:
        assert np.all(got["gates"] == 1.0)


def test_router_ties_go_to_the_lower_expert(M):
    """Duplicated router rows give bitwise-equal logits (one fixed-order fp32 chain per logit); the
    selection must then order the tied experts by id, as the oracle does, and every output follows."""
    w = S.Workload("ties", N=256, H=128, E=12, k=4, I=128, c=64, K_max=8)
    T = S.make(w)
    T.Wr[7] = T.Wr[2]
    T.Wr[9] = T.Wr[2]
    T.Wr[11] = T.Wr[5]
    got = run_block(M, w, DevInputs(T))
    ref = oracle_block(T)
    both = (np.isin(ref["topk_idx"], [2, 7]).sum(axis=1) == 2)
    assert both.any(), "the seed gives no token with both tied experts selected"
    compare(got, ref)


def test_one_hot_expert_takes_every_token(M):
    """A bias that sends every token to expert 3 first: one segment of c_eff rows per chunk."""
    w = S.Workload("hot", N=600, H=128, E=8, k=2, I=128, c=150, K_max=8)
    T = S.make(w)
    T.bias = np.zeros(w.E, np.float32)
    T.bias[3] = 50.0
    got = run_block(M, w, DevInputs(T))
    ref = oracle_block(T)
    assert np.all(ref["topk_idx"][:, 0] == 3)
    compare(got, ref)


def test_empty_batch(M):
    cfg = M.Config(N=0, H=64, E=4, k=2, I=64, c=8, K_max=4)
    blk = M.MoEBlock(cfg)
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    Wr = torch.randn(4, 64, device="cuda")
    idx, g = blk.route(X, Wr)
    W = torch.randn(4, 64, 64, device="cuda").to(torch.bfloat16)
    Y = blk.forward(X, idx, g, W, W, W)
    gr = blk.backward(X, Wr, idx, g, W, W, W, X)
    blk.check()
    assert Y.shape == (0, 64)
    for n in ("dWr", "dWg", "dWu", "dWd"):
        assert torch.count_nonzero(gr[n]) == 0


def test_unused_experts_get_zero_gradients(M):
    w = S.Workload("few", N=64, H=64, E=16, k=1, I=64, c=64, K_max=1)
    T = S.make(w)
    T.bias = np.full(w.E, -40.0, np.float32)
    T.bias[[2, 5]] = 0.0
    got = run_block(M, w, DevInputs(T))
    used = set(np.unique(got["topk_idx"]).tolist())
    assert used <= {2, 5}
    for e in range(w.E):
        if e not in used:
            for n in ("dWr", "dWg", "dWu", "dWd"):
                assert not np.any(got[n][e]), (n, e)


@pytest.mark.parametrize("name", ["mid/8", "extreme/8", "tiny"])
def test_cta_pair_gemms_match_single_cta_bitwise(M, name):
    """The 2-SM (CTA-pair) row-tile GEMMs give the same bits as the one-CTA form, and match the oracle."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    try:
        M.set_gemm_form("single")
        one = run_block(M, w, D)
        M.set_gemm_form("pair")
        two = run_block(M, w, D)
    finally:
        M.set_gemm_form("auto")
    for n in ("Y_bits", "dX_bits", "dgates", "dWr", "dWg", "dWu", "dWd"):
        assert np.array_equal(one[n], two[n]), n
    compare(two, oracle_block(T))


@pytest.mark.parametrize("name", ["tiny", "mid/8", "mid"])
def test_cuda_graph_replay_matches_eager(M, name):
    """The whole step captured as a CUDA graph gives the eager calls' bits, and a replay after new input
    contents routes afresh (the launches read their tile lists from device memory)."""
    w = workload(name)
    T = S.make(w)
    D = DevInputs(T)
    G = M.MoEStepGraph(M.MoEBlock(M.Config(**w.cfg())), D.X, D.Wr, D.bias, D.Wg, D.Wu, D.Wd, D.dY)
    G.replay()
    torch.cuda.synchronize()
    eager = run_block(M, w, D)
    assert np.array_equal(G.idx.cpu().numpy(), eager["topk_idx"])
    assert np.array_equal(bf16_host_bits(G.Y), eager["Y_bits"])
    for n in ("dWr", "dWg", "dWu", "dWd", "dgates"):
        assert np.array_equal(G.grads()[n].cpu().numpy(), eager[n]), n
    # new contents in the same buffers: a different seed's tokens
    T2 = S.make(w, seed=7)
    D.X.copy_(bf16_dev(T2.X))
    D.dY.copy_(bf16_dev(T2.dY))
    G.replay()
    torch.cuda.synchronize()
    eager2 = run_block(M, w, D)
    assert not np.array_equal(eager2["topk_idx"], eager["topk_idx"])
    assert np.array_equal(G.idx.cpu().numpy(), eager2["topk_idx"])
    assert np.array_equal(bf16_host_bits(G.dX), eager2["dX_bits"])
    assert np.array_equal(G.dWg.cpu().numpy(), eager2["dWg"])


def bf16_host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "mid/8", "extreme/8"])
def test_forward_against_the_storage_mirror(M, name):
    """Diagnostic: against the oracle's mirror mode (bf16 rounding where the kernels store bf16), the GPU's
    Y is within 2 bf16 ulps nearly everywhere, i.e. its error is the storage rounding, nothing else."""
    w = workload(name)
    T = S.make(w)
    got = run_block(M, w, DevInputs(T))
    idx, g, _ = O.route(T.X, T.Wr, T.bias, w.k)
    Ym = O.forward(T.X, idx, g, (T.Wg, T.Wu, T.Wd), mirror=True)
    mbits = S.f32_to_bf16(Ym.astype(np.float32)).astype(np.int32)
    gbits = got["Y_bits"].astype(np.int32)
    same_sign = (mbits >> 15) == (gbits >> 15)
    ulps = np.where(same_sign, np.abs(mbits - gbits), 1 << 16)
    assert np.mean(ulps <= 2) > 0.999, np.bincount(np.minimum(ulps, 8).ravel())
    assert O.normalised_error(got["Y"], Ym) <= 2.0 ** -7     # two bf16 ulps of the largest element


def test_autograd_wrappers_match_the_direct_calls(M):
    """MoEFunction and VocabCEFunction: loss.backward() hands out the direct calls' gradients, in each
    parameter's dtype (bf16 weights get the fp32 gradients rounded to bf16)."""
    w = workload("mid/8")
    T = S.make(w)
    D = DevInputs(T)
    blk = M.MoEBlock(M.Config(**w.cfg()))
    X = D.X.clone().requires_grad_(True)
    Wr = D.Wr.clone().requires_grad_(True)
    Wg, Wu, Wd = (t.clone().requires_grad_(True) for t in (D.Wg, D.Wu, D.Wd))
    Y = M.moe_block(X, Wr, D.bias, Wg, Wu, Wd, blk)
    (Y.float() * D.dY.float()).sum().backward()
    ref = run_block(M, w, D)
    assert np.array_equal(bf16_host_bits(Y.detach()), ref["Y_bits"])
    assert np.array_equal(bf16_host_bits(X.grad), ref["dX_bits"])
    assert np.array_equal(Wr.grad.cpu().numpy(), ref["dWr"])
    for t, n in ((Wg, "dWg"), (Wu, "dWu"), (Wd, "dWd")):
        want = torch.from_numpy(ref[n]).to(torch.bfloat16)
        assert torch.equal(t.grad.cpu(), want), n

    cw = S.CE_WORKLOADS["ce_small"]
    CT = S.ce_make(cw)
    ce = M.VocabCE(M.CEConfig(**cw.cfg()))
    Xc = bf16_dev(CT.X).requires_grad_(True)
    Wc = bf16_dev(CT.W).requires_grad_(True)
    tc = torch.from_numpy(CT.targets).cuda()
    loss = M.vocab_cross_entropy(Xc, Wc, tc, ce)
    (2.0 * loss).backward()
    _, lse, mean = ce.forward(Xc.detach(), Wc.detach(), tc)
    assert torch.equal(loss.detach(), mean[0])
    dX, dW = ce.backward(Xc.detach(), Wc.detach(), tc, lse, torch.full((cw.N,), 2.0 / cw.N, device="cuda"))
    assert torch.equal(Xc.grad, dX)
    assert torch.equal(Wc.grad, dW.to(torch.bfloat16))
