"""GPU parity of the vocabulary-projection cross-entropy head (Ring-DTP's single-device form,
"bounded-streaming operators" summary, Methodology 2, eqs. (2)-(3)) against the float64 oracle,
through the C ABI of include/moe_ce.h.

  * loss and lse within 2e-3 absolute (fp32 logits, fp32 online fold);
  * dX and dW within max|gpu - oracle| / max|oracle| <= 1e-2 (d is stored in bf16);
  * forward outputs and dW do not depend on the strip count P (bit for bit), dX within tolerance;
  * repeated runs are bitwise equal; edge cases (ragged N and V, one token, one class, targets on
    tile edges, N = 0) and a bad class id reported through the status word;
  * the 16,384-token, H = 7,168, V = 200,000 head: sampled tokens' loss, lse and dX against the
    oracle one token at a time, and dW against a second strip count bit for bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import TOL, bf16_dev, bf16_host, need_gpu, lib_api
from oracle import ce_ref as C
from synth import inputs as S

pytestmark = pytest.mark.gpu

LOSS_ATOL = 2e-3


@pytest.fixture(scope="module")
def M():
    need_gpu()
    return lib_api()


def widen(bits):
    return S.bf16_to_f32(bits).astype(np.float64)


def run(M, w, T, P=None, dloss=None):
    cfg = M.CEConfig(w.N, w.H, w.V, P or w.P)
    ce = M.VocabCE(cfg)
    X, W = bf16_dev(T.X), bf16_dev(T.W)
    t = torch.from_numpy(T.targets).cuda()
    loss, lse, mean = ce.forward(X, W, t)
    g = torch.full((w.N,), 1.0 / max(w.N, 1), device="cuda") if dloss is None else torch.from_numpy(dloss).cuda()
    dX, dW = ce.backward(X, W, t, lse, g)
    ce.check()
    st = M.ce_last_stats()
    return dict(loss=loss.cpu().numpy(), lse=lse.cpu().numpy(), mean=float(mean.cpu()), dX=bf16_host(dX),
                dW=dW.cpu().numpy(), stats=st)


def check_vs_oracle(w, T, got, g):
    Xf, Wf = widen(T.X), widen(T.W)
    loss, lse = C.forward(Xf, Wf, T.targets)
    dX, dW = C.backward(Xf, Wf, T.targets, g)
    assert np.max(np.abs(got["loss"] - loss)) < LOSS_ATOL
    assert np.max(np.abs(got["lse"] - lse)) < LOSS_ATOL
    assert abs(got["mean"] - loss.mean()) < LOSS_ATOL
    errs = {"dX": C_err(widen(got["dX"]), dX), "dW": C_err(got["dW"], dW)}
    assert all(e <= TOL for e in errs.values()), errs
    return errs


def C_err(a, ref):
    return float(np.max(np.abs(np.asarray(a, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-300))


@pytest.mark.parametrize("name", ["ce_tiny", "ce_small", "ce_mid"])
def test_ce_vs_oracle(M, name):
    w = S.CE_WORKLOADS[name]
    T = S.ce_make(w)
    got = run(M, w, T)
    check_vs_oracle(w, T, got, np.full(w.N, 1.0 / w.N))
    st = got["stats"]
    assert st["strip_bytes"] == w.N * st["strip_classes"] * 2
    assert st["strip_bytes"] <= st["strip_bound_bytes"] + w.N * 255 * 2


def test_per_token_upstream_gradients(M):
    w = S.CE_WORKLOADS["ce_small"]
    T = S.ce_make(w, seed=4)
    g = np.random.default_rng(0).normal(size=w.N).astype(np.float32)
    check_vs_oracle(w, T, run(M, w, T, dloss=g), g.astype(np.float64))


def test_strip_count_changes_no_result(M):
    w = S.CE_WORKLOADS["ce_small"]
    T = S.ce_make(w, seed=2)
    runs = {P: run(M, w, T, P=P) for P in (1, 4, 7, 19)}
    base = runs[1]
    for P, r in runs.items():
        for n in ("loss", "lse", "dW"):
            assert np.array_equal(r[n].view(np.uint32), base[n].view(np.uint32)), (P, n)
        assert C_err(widen(r["dX"]), widen(base["dX"])) < 1e-2
    again = run(M, w, T, P=7)
    for n in ("loss", "lse", "dX", "dW"):
        assert np.array_equal(again[n], runs[7][n]), n


@pytest.mark.parametrize("shape", [(1, 64, 300, 1), (257, 64, 1, 1), (129, 192, 513, 2), (64, 128, 256, 256)])
def test_edge_shapes(M, shape):
    N, H, V, P = shape
    w = S.CeWorkload("edge", N=N, H=H, V=V, P=P)
    T = S.ce_make(w, seed=N + V)
    # targets on tile and strip edges where the vocabulary has them
    edges = np.array([0, V - 1, min(255, V - 1), min(256, V - 1)], np.int32)
    T.targets[: min(N, 4)] = edges[: min(N, 4)]
    got = run(M, w, T)
    check_vs_oracle(w, T, got, np.full(N, 1.0 / N))
    if V == 1:
        assert np.all(np.abs(got["loss"]) < 1e-6)


def test_empty_batch(M):
    cfg = M.CEConfig(0, 64, 100, 2)
    ce = M.VocabCE(cfg)
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.randn(100, 64, device="cuda").to(torch.bfloat16)
    t = torch.empty(0, dtype=torch.int32, device="cuda")
    loss, lse, mean = ce.forward(X, W, t)
    dX, dW = ce.backward(X, W, t, lse, torch.empty(0, device="cuda"))
    ce.check()
    assert float(mean.cpu()) == 0.0 and torch.count_nonzero(dW) == 0


def test_bad_class_is_reported(M):
    from top_softmax_router_gb300._lib import MoeError
    w = S.CeWorkload("bad", N=40, H=64, V=300, P=2)
    T = S.ce_make(w)
    T.targets[5] = 300
    cfg = M.CEConfig(w.N, w.H, w.V, w.P)
    ce = M.VocabCE(cfg)
    ce.forward(bf16_dev(T.X), bf16_dev(T.W), torch.from_numpy(T.targets).cuda())
    with pytest.raises(MoeError) as e:
        ce.check()
    assert e.value.code == -6


def test_full_size_ring_dtp_shape(M):
    """N = 16,384, H = 7,168, V = 200,000, P = 8: sampled tokens against the oracle, one token at a
    time (loss, lse, dX row); dW bit for bit against P = 5 (the strips only reorder independent work)."""
    w = S.CE_WORKLOADS["ce_full"]
    T = S.ce_make(w)
    cfg = M.CEConfig(w.N, w.H, w.V, w.P)
    ce = M.VocabCE(cfg)
    X, W = bf16_dev(T.X), bf16_dev(T.W)
    t = torch.from_numpy(T.targets).cuda()
    loss, lse, mean = ce.forward(X, W, t)
    g = torch.full((w.N,), 1.0 / w.N, device="cuda")
    dX, dW = ce.backward(X, W, t, lse, g)
    ce.check()
    st = M.ce_last_stats()
    assert st["strips"] == 8 and st["strip_bytes"] <= 2 * w.N * 25_088
    sel = [0, 1, 127, 128, w.N - 1] + list(np.random.default_rng(3).choice(w.N, size=3, replace=False))
    Wf = S.bf16_to_f32(T.W)
    loss_h, lse_h, dX_h = loss.cpu().numpy(), lse.cpu().numpy(), bf16_host(dX)
    l, s, dx = C.rows_forward_backward(widen(T.X[sel]), Wf, T.targets[sel], np.full(len(sel), 1.0 / w.N))
    for i, n in enumerate(sel):
        assert abs(loss_h[n] - l[i]) < LOSS_ATOL and abs(lse_h[n] - s[i]) < LOSS_ATOL, n
        assert C_err(widen(dX_h[n]), dx[i]) <= TOL, n
    dW5 = torch.empty_like(dW)
    ce5 = M.VocabCE(M.CEConfig(w.N, w.H, w.V, 5))
    dX5 = torch.empty_like(dX)
    M.ce_backward(ce5.cfg, X, W, t, lse, g, dX5, dW5, ce5.ws)
    ce5.check()
    assert torch.equal(dW.view(torch.int32), dW5.view(torch.int32))
