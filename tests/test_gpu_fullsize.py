"""Full-size parity: the five large workloads, in the launch configuration bench.py times.

The whole block runs on the GPU at full size through the C ABI.  Against the
oracle (computed from the same seeded inputs, never from GPU outputs):
  * routing of all N tokens and the permutation of every chunk: bit for bit;
  * Y, dX and dgates on a seeded sample of tokens (plus every token of the
    coldest expert and some of the hottest): max|gpu-oracle|/max|oracle| <= 1e-2;
  * weight-gradient slices of the hottest, median and coldest non-empty
    experts (columns of dWd, rows of dWg and dWu); the coldest expert's
    gradients and its dWr row in full;
  * experts that no token selects get exactly zero gradients;
  * every row of dWr, step-wise: formed in float64 from the oracle's gates and
    the GPU's dgates (themselves checked on the sample);
  * order only, exact results: the unchunked block (K = 1) gives bitwise the
    same routing, gates, Y, dX and dgates as the chunked one (K = K_max).
"""
import gc

import numpy as np
import pytest
import torch

from oracle import moe_ref as O
from synth import inputs as S
from gpu_util import TOL, DevInputs, need_gpu, lib_api

pytestmark = pytest.mark.gpu

_cache = {}


def inputs_for(w: S.Workload):
    key = (w.N, w.H, w.E, w.I)
    if key not in _cache:
        _cache.clear()
        gc.collect()
        _cache[key] = S.make(w)
    T = _cache[key]
    bias, _ = S.bias_for(w)
    return S.Tensors(w, T.X, T.Wr, bias, T.Wg, T.Wu, T.Wd, T.dY)


def err(gpu, ref):
    return O.normalised_error(np.asarray(gpu, np.float64), ref)


@pytest.mark.parametrize("name", ["mid", "long", "many", "many_zipf", "extreme"])
def test_full_size(name):
    need_gpu()
    M = lib_api()
    w = S.WORKLOADS[name]
    T = inputs_for(w)
    N, H, E, k, I = w.N, w.H, w.E, w.k, w.I
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())
    blk = M.MoEBlock(cfg)
    idx_d, g_d = blk.route(D.X, D.Wr, D.bias)
    Y_d = blk.forward(D.X, idx_d, g_d, D.Wg, D.Wu, D.Wd)
    gr = blk.backward(D.X, D.Wr, idx_d, g_d, D.Wg, D.Wu, D.Wd, D.dY)
    blk.check()
    st = M.last_stats()
    assert st["routed_bytes_peak"] <= st["routed_bytes_bound"]

    # ---- routing, all tokens, bit for bit
    idx, g, _ = O.route(T.X, T.Wr, T.bias, k)
    gidx = idx_d.cpu().numpy()
    assert np.array_equal(gidx, idx), f"{int((gidx != idx).sum())} routing entries differ"
    assert err(g_d.cpu().numpy(), g) < 1e-5

    # ---- permutation of every chunk, bit for bit
    K, c_eff = M.chunk_plan(cfg)
    rr = torch.empty(K, k * c_eff, dtype=torch.int32, device="cuda")
    ro = torch.empty(N, k, dtype=torch.int32, device="cuda")
    off = torch.empty(K, E + 1, dtype=torch.int32, device="cuda")
    M.plan(cfg, idx_d, rr, ro, off, blk.ws)
    assert M.check_status(blk.ws) == 0
    rr, ro, off = rr.cpu().numpy(), ro.cpu().numpy(), off.cpu().numpy()
    for i in range(K):
        r_rr, r_off, r_ro = O.permute_chunk(idx, K, i, E)
        assert np.array_equal(rr[i, :len(r_rr)], r_rr), f"chunk {i}: row order differs"
        assert np.array_equal(off[i], r_off), f"chunk {i}: expert offsets differ"
        assert np.array_equal(ro[O.chunk_tokens(N, K, i)], r_ro), f"chunk {i}: row_of differs"

    # ---- per-token outputs on a sample
    counts = np.bincount(idx.reshape(-1), minlength=E)
    used = np.flatnonzero(counts)
    hot = int(used[np.argmax(counts[used])])
    cold = int(used[np.argmin(counts[used])])
    med = int(used[np.argsort(counts[used])[len(used) // 2]])
    rng = np.random.default_rng(1234)
    tok_cold = np.unique(np.nonzero(idx == cold)[0])[:64]
    tok_hot = np.unique(np.nonzero(idx == hot)[0])
    tok_hot = rng.choice(tok_hot, size=min(32, len(tok_hot)), replace=False)
    sel = np.unique(np.concatenate([rng.choice(N, size=min(192, N), replace=False), tok_cold, tok_hot]))
    W = (T.Wg, T.Wu, T.Wd)
    Y_ref = O.forward(T.X[sel], idx[sel], g[sel], W)
    b_ref = O.backward(T.X[sel], T.Wr, idx[sel], g[sel], W, T.dY[sel], want_weight_grads=False)
    sel_d = torch.from_numpy(sel).cuda()
    errs = {"Y": err(Y_d[sel_d].float().cpu().numpy(), Y_ref),
            "dX": err(gr["dX"][sel_d].float().cpu().numpy(), b_ref["dX"]),
            "dgates": err(gr["dgates"][sel_d].cpu().numpy(), b_ref["dgates"])}

    # ---- weight-gradient slices
    cols = np.sort(rng.choice(I, size=4, replace=False))
    rows = np.sort(rng.choice(I, size=4, replace=False))
    for tag, e in (("hot", hot), ("median", med), ("cold", cold)):
        t, j = np.nonzero(idx == e)
        ce = np.arange(I) if tag == "cold" else cols
        re_ = np.arange(I) if tag == "cold" else rows
        dWd_c, dWg_r, dWu_r = O.expert_grad_slices(T.X[t], g[t, j], T.dY[t], (T.Wg[e], T.Wu[e], T.Wd[e]), ce, re_)
        ce_d, re_d = torch.from_numpy(ce).cuda(), torch.from_numpy(re_).cuda()
        errs[f"dWd[{tag}]"] = err(gr["dWd"][e][:, ce_d].cpu().numpy(), dWd_c)
        errs[f"dWg[{tag}]"] = err(gr["dWg"][e][re_d].cpu().numpy(), dWg_r)
        errs[f"dWu[{tag}]"] = err(gr["dWu"][e][re_d].cpu().numpy(), dWu_r)
    # the coldest expert's router-weight row: needs dlogit of every token that routes to it
    tc = np.unique(np.nonzero(idx == cold)[0])
    bc = O.backward(T.X[tc], T.Wr, idx[tc], g[tc], W, T.dY[tc], want_weight_grads=False)
    errs["dWr[cold]"] = err(gr["dWr"][cold].cpu().numpy(), bc["dWr"][cold])
    bad = {n: v for n, v in errs.items() if not v <= TOL}
    assert not bad, f"{name}: above {TOL}: {bad} (all {errs})"

    # ---- experts nobody selected: exactly zero gradients
    unused = np.flatnonzero(counts == 0)[:4]
    for e in unused:
        for n in ("dWr", "dWg", "dWu", "dWd"):
            assert torch.count_nonzero(gr[n][int(e)]) == 0, (n, int(e))

    # ---- the whole router-weight gradient, step-wise: dWr[e] = sum over the routes (t, j) to e of
    # dlogit[t, j] X[t], with dlogit = g_j (dg_j - sum_i g_i dg_i) formed in float64 from the oracle's
    # gates and the GPU's dgates (checked on the sample above): every row, the hottest expert's included
    dg_gpu = gr["dgates"].cpu().numpy().astype(np.float64)
    dl = g * (dg_gpu - np.sum(g * dg_gpu, axis=1, keepdims=True))
    dWr_ref = router_weight_grad(idx, dl, T.X, E)
    dWr_gpu = gr["dWr"].cpu().numpy()
    for tag, e in (("hot", hot), ("median", med), ("cold", cold)):
        errs[f"dWr_stepwise[{tag}]"] = err(dWr_gpu[e], dWr_ref[e])
    errs["dWr_stepwise[all]"] = err(dWr_gpu, dWr_ref)
    bad = {n: v for n, v in errs.items() if not v <= TOL}
    assert not bad, f"{name}: above {TOL}: {bad} (all {errs})"

    # ---- order only, exact results: the unchunked block (K = 1) gives the same per-token bits
    keep = {n: gr[n] for n in ("dX", "dgates")}
    del gr
    torch.cuda.empty_cache()
    cfg1 = M.Config(**{**w.cfg(), "K_max": 1})
    blk1 = M.MoEBlock(cfg1)
    assert blk1.K == 1 < blk.K
    del blk
    torch.cuda.empty_cache()
    idx1, g1 = blk1.route(D.X, D.Wr, D.bias)
    Y1 = blk1.forward(D.X, idx1, g1, D.Wg, D.Wu, D.Wd)
    gr1 = blk1.backward(D.X, D.Wr, idx1, g1, D.Wg, D.Wu, D.Wd, D.dY)
    blk1.check()
    assert torch.equal(idx1, idx_d) and torch.equal(g1, g_d), f"{name}: routing differs between K and 1"
    assert torch.equal(Y1, Y_d), f"{name}: Y differs between K={K} and K=1"
    for n in ("dX", "dgates"):
        assert torch.equal(gr1[n], keep[n]), f"{name}: {n} differs between K={K} and K=1"
    del D, blk1, gr1, keep
    torch.cuda.empty_cache()


def router_weight_grad(idx: np.ndarray, dlogit: np.ndarray, X_bf16: np.ndarray, E: int) -> np.ndarray:
    """dWr [E, H] float64 = sum over routes (t, j) of dlogit[t, j] * X[t] into row idx[t, j]: the plain
    gradient of the logits X . Wr^T with respect to Wr, restricted to the selected slots (one sparse
    E x N matrix of dlogit times X, exact bf16 inputs widened to float64)."""
    import scipy.sparse as sp
    N, k = idx.shape
    A = sp.csr_matrix((dlogit.reshape(-1), (idx.reshape(-1).astype(np.int64), np.repeat(np.arange(N), k))),
                      shape=(E, N))
    out = np.empty((E, X_bf16.shape[1]))
    for c0 in range(0, X_bf16.shape[1], 1024):        # column slabs keep the float64 copy of X small
        out[:, c0:c0 + 1024] = A @ O.bf16_to_f64(X_bf16[:, c0:c0 + 1024])
    return out


def dev_err(a: torch.Tensor, b: torch.Tensor) -> float:
    """max|a - b| / max|b| on the device, a slab at a time (the full-size gradients are tens of GB)."""
    num = den = 0.0
    for x, y in zip(a.reshape(a.shape[0], -1).split(64), b.reshape(b.shape[0], -1).split(64)):
        x, y = x.float(), y.float()
        num = max(num, float((x - y).abs().max()))
        den = max(den, float(y.abs().max()))
    return num / den if den > 0 else num


@pytest.mark.parametrize("name,P,chain", [("mid", 8, None), ("extreme", 8, None), ("many_zipf", 8, "none"),
                                          ("many_zipf", 8, None)])
def test_full_size_hop_schedule(name, P, chain):
    """The expert-partition schedule at full size (CTA-pair GEMMs): every output against the chunk
    schedule (itself checked against the oracle above), compared on the device, and sampled tokens
    against the oracle.  `chain` selects the launch chaining of the run (None: the library's default;
    "none": plain stream order, no kernel overlaps another)."""
    need_gpu()
    M = lib_api()
    if chain is not None:
        M.set_launch_chaining(chain)
    try:
        _hop_schedule_vs_chunk_schedule(M, name, P)
    finally:
        M.set_launch_chaining("late")


def _hop_schedule_vs_chunk_schedule(M, name, P):
    w = S.WORKLOADS[name]
    T = inputs_for(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())
    blk = M.MoEBlock(cfg)
    idx, g = blk.route(D.X, D.Wr, D.bias)
    ref = {"Y": blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)}
    ref.update(blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY))
    blk.check()
    del blk
    torch.cuda.empty_cache()
    hb = M.MoEHopBlock(cfg, P)
    got = {"Y": hb.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)}
    got.update(hb.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY))
    assert M.check_status(hb.ws) == 0
    errs = {n: dev_err(got[n], ref[n]) for n in ("Y", "dX", "dgates", "dWr", "dWg", "dWu", "dWd")}
    rng = np.random.default_rng(99)
    sel = np.sort(rng.choice(w.N, size=128, replace=False))
    oi, og, _ = O.route(T.X[sel], T.Wr, T.bias, w.k)
    assert np.array_equal(oi, idx.cpu().numpy()[sel])
    sel_d = torch.from_numpy(sel).cuda()
    errs["Y_vs_oracle"] = err(got["Y"][sel_d].float().cpu().numpy(), O.forward(T.X[sel], oi, og, (T.Wg, T.Wu, T.Wd)))
    bad = {n: v for n, v in errs.items() if not v <= TOL}
    assert not bad, f"{name}: {bad} (all {errs})"
    del D, hb, got, ref
    torch.cuda.empty_cache()


def test_full_size_gather_on_load_matches_the_gather_kernel():
    """mid at full size: the dispatch gather fused into the GEMMs (TMA row gathers from X and dY) gives every
    output of the chunk schedule bit for bit as the gather kernel does, with half the routed working set."""
    need_gpu()
    M = lib_api()
    w = S.WORKLOADS["mid"]
    T = inputs_for(w)
    D = DevInputs(T)
    cfg = M.Config(**w.cfg())

    def run():
        blk = M.MoEBlock(cfg)
        idx, g = blk.route(D.X, D.Wr, D.bias)
        out = {"idx": idx, "g": g, "Y": blk.forward(D.X, idx, g, D.Wg, D.Wu, D.Wd)}
        out.update(blk.backward(D.X, D.Wr, idx, g, D.Wg, D.Wu, D.Wd, D.dY))
        st = M.last_stats()
        blk.check()
        return out, st

    ref, st_ref = run()
    try:
        M.set_dispatch("on_load")
        got, st = run()
    finally:
        M.set_dispatch("gather")
    for n in ref:
        assert torch.equal(got[n], ref[n]), n
    assert 2 * st["routed_bytes_peak"] == st_ref["routed_bytes_peak"] == st_ref["routed_bytes_bound"]
    del D, got, ref
    torch.cuda.empty_cache()
