"""Pins for the oracle's permutation, forward and backward (CPU only).

Forward: a dense-masked torch float64 formulation (every expert on every token,
masked by the gates), the E = 1, k = 1 textbook SwiGLU FFN, and the k = E
dense softmax mixture.  Backward: torch float64 autograd of the dense-masked
block (router included) and float64 central finite differences.
Permutation: a library stable sort and the inverse-map / stability invariants.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as O
from synth import inputs as S


# --------------------------------------------------------------------------- #
# permutation
# --------------------------------------------------------------------------- #
def check_permutation(idx, K, E):
    N, k = idx.shape
    total = 0
    for i in range(K):
        toks = O.chunk_tokens(N, K, i)
        rr, off, row_of = O.permute_chunk(idx, K, i, E)
        n = len(toks)
        counts = np.bincount(idx[toks].reshape(-1), minlength=E)
        assert np.array_equal(np.diff(off), counts)
        assert off[0] == 0 and off[-1] == n * k
        # same rows as a library stable sort of the chunk's routes by expert
        q = (toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)
        order = np.argsort(idx[toks].reshape(-1), kind="stable")
        assert np.array_equal(rr, q[order].astype(np.int32))
        # inverse maps
        for l, t in enumerate(toks):
            for j in range(k):
                assert rr[row_of[l, j]] == t * k + j
        # rows of one expert ascend by token (stability)
        for e in range(E):
            seg = rr[off[e]:off[e + 1]]
            assert np.all(np.diff(seg // k) > 0)
            assert np.all(idx.reshape(-1)[seg] == e)
        total += off[-1]
    assert total == N * k


@pytest.mark.parametrize("N,E,k,K", [(512, 8, 2, 4), (101, 7, 3, 5), (64, 16, 16, 2), (9, 3, 1, 9), (50, 40, 4, 1)])
def test_permutation(N, E, k, K):
    rng = np.random.default_rng(N + E)
    skew = rng.dirichlet(np.full(E, 0.3))
    idx = np.stack([rng.choice(E, size=k, replace=False, p=skew) for _ in range(N)]).astype(np.int32)
    check_permutation(idx, K, E)


# --------------------------------------------------------------------------- #
# forward
# --------------------------------------------------------------------------- #
def t64(a):
    return torch.from_numpy(O.bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, np.float64))


def dense_masked_forward(X, Wg, Wu, Wd, mask):
    """torch float64: Y = sum_e mask[:, e] * (silu(X Wg_e^T) * (X Wu_e^T)) Wd_e^T over ALL experts."""
    x = t64(X)
    Y = torch.zeros_like(x)
    for e in range(mask.shape[1]):
        h = torch.nn.functional.silu(x @ t64(Wg[e]).T) * (x @ t64(Wu[e]).T)
        Y = Y + mask[:, e:e + 1] * (h @ t64(Wd[e]).T)
    return Y


def mask_of(idx, g, E):
    m = torch.zeros(idx.shape[0], E, dtype=torch.float64)
    m.scatter_(1, torch.from_numpy(idx.astype(np.int64)), torch.from_numpy(np.asarray(g, np.float64)))
    return m


def test_forward_vs_dense_masked(tiny):
    w, T = tiny
    idx, g, _ = O.route(T.X, T.Wr, T.bias, w.k)
    Y = O.forward(T.X, idx, g, (T.Wg, T.Wu, T.Wd))
    Yd = dense_masked_forward(T.X, T.Wg, T.Wu, T.Wd, mask_of(idx, g, w.E)).numpy()
    np.testing.assert_allclose(Y, Yd, rtol=1e-10, atol=1e-12)


def test_forward_single_expert_is_swiglu():
    N, H, I = 64, 128, 192
    X = S.normal_bf16(7, 0, (N, H), 1.0)
    Wg = S.normal_bf16(7, 2, (1, I, H), H ** -0.5)
    Wu = S.normal_bf16(7, 3, (1, I, H), H ** -0.5)
    Wd = S.normal_bf16(7, 4, (1, H, I), I ** -0.5)
    Wr = S.normal_f32(7, 1, (1, H), H ** -0.5)
    idx, g, _ = O.route(X, Wr, None, 1)
    assert np.all(idx == 0) and np.all(g == 1.0)
    Y = O.forward(X, idx, g, (Wg, Wu, Wd))
    x = t64(X)
    ref = torch.nn.functional.silu(x @ t64(Wg[0]).T) * (x @ t64(Wu[0]).T) @ t64(Wd[0]).T
    np.testing.assert_allclose(Y, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_forward_k_equals_E_is_softmax_mixture():
    N, H, I, E = 32, 64, 64, 4
    X = S.normal_bf16(8, 0, (N, H), 1.0)
    Wr = S.normal_f32(8, 1, (E, H), H ** -0.5)
    Wg = S.normal_bf16(8, 2, (E, I, H), H ** -0.5)
    Wu = S.normal_bf16(8, 3, (E, I, H), H ** -0.5)
    Wd = S.normal_bf16(8, 4, (E, H, I), I ** -0.5)
    idx, g, L = O.route(X, Wr, None, E)
    Y = O.forward(X, idx, g, (Wg, Wu, Wd))
    p = torch.softmax(torch.from_numpy(L.astype(np.float64)), dim=1)      # full softmax, natural expert order
    x = t64(X)
    ref = sum(p[:, e:e + 1] * ((torch.nn.functional.silu(x @ t64(Wg[e]).T) * (x @ t64(Wu[e]).T)) @ t64(Wd[e]).T)
              for e in range(E))
    np.testing.assert_allclose(Y, ref.numpy(), rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------- #
# backward
# --------------------------------------------------------------------------- #
def autograd_block(X, Wr, bias, Wg, Wu, Wd, dY, idx):
    """torch float64 autograd of the dense-masked block; gates from float64 logits, selection fixed."""
    x = t64(X).requires_grad_(True)
    wr = t64(Wr).requires_grad_(True)
    wg = t64(Wg).requires_grad_(True)
    wu = t64(Wu).requires_grad_(True)
    wd = t64(Wd).requires_grad_(True)
    logits = x @ wr.T + (0 if bias is None else t64(bias))
    sel = torch.from_numpy(idx.astype(np.int64))
    g = torch.softmax(torch.gather(logits, 1, sel), dim=1)
    g.retain_grad()
    E = Wr.shape[0]
    mask = torch.zeros(x.shape[0], E, dtype=torch.float64).scatter(1, sel, g)
    Y = torch.zeros_like(x)
    for e in range(E):
        h = torch.nn.functional.silu(x @ wg[e].T) * (x @ wu[e].T)
        Y = Y + mask[:, e:e + 1] * (h @ wd[e].T)
    (Y * t64(dY)).sum().backward()
    return dict(Y=Y.detach().numpy(), g=g.detach().numpy(), dX=x.grad.numpy(), dWr=wr.grad.numpy(),
                dWg=wg.grad.numpy(), dWu=wu.grad.numpy(), dWd=wd.grad.numpy(), dgates=g.grad.numpy())


def test_backward_vs_torch_autograd(tiny):
    w, T = tiny
    n = 96
    X, dY = T.X[:n], T.dY[:n]
    idx, g, _ = O.route(X, T.Wr, T.bias, w.k)
    ref = autograd_block(X, T.Wr, T.bias, T.Wg, T.Wu, T.Wd, dY, idx)
    # The oracle's gates come from fp32 logits, torch's from float64 ones: same to ~1e-7.
    np.testing.assert_allclose(g, ref["g"], rtol=1e-5, atol=1e-7)
    got = O.backward(X, T.Wr, idx, ref["g"], (T.Wg, T.Wu, T.Wd), dY)
    for name in ("dX", "dWr", "dWg", "dWu", "dWd", "dgates"):
        err = O.normalised_error(got[name], ref[name])
        assert err < 1e-10, (name, err)


def fd_loss(X64, Wr64, bias, W64, dY, idx):
    logits = X64 @ Wr64.T + (0 if bias is None else bias.astype(np.float64))
    lsel = np.take_along_axis(logits, idx.astype(np.int64), axis=1)
    e = np.exp(lsel - lsel.max(axis=1, keepdims=True))
    g = e / e.sum(axis=1, keepdims=True)
    Y = O.forward(X64, idx, g, W64)
    return float(np.sum(Y * O.bf16_to_f64(dY))), g


def test_backward_vs_finite_differences():
    N, H, I, E, k = 24, 64, 64, 5, 2
    rng = np.random.default_rng(11)
    X64 = O.bf16_to_f64(S.normal_bf16(11, 0, (N, H), 1.0))
    Wr64 = S.normal_f32(11, 1, (E, H), H ** -0.5).astype(np.float64)
    bias = S.normal_f32(11, 5, (E,), 0.3)
    W64 = [O.bf16_to_f64(S.normal_bf16(11, 2 + s, shp, sd)) for s, (shp, sd) in
           enumerate((((E, I, H), H ** -0.5), ((E, I, H), H ** -0.5), ((E, H, I), I ** -0.5)))]
    dY = S.normal_bf16(11, 6, (N, H), 1.0)
    L = X64 @ Wr64.T + bias
    idx = np.argsort(-L, axis=1, kind="stable")[:, :k].astype(np.int32)
    _, g = fd_loss(X64, Wr64, bias, W64, dY, idx)
    got = O.backward(X64, Wr64, idx, g, tuple(W64), dY)
    eps = 1e-5
    params = {"dX": X64, "dWr": Wr64, "dWg": W64[0], "dWu": W64[1], "dWd": W64[2]}
    for name, P in params.items():
        for _ in range(12):
            pos = tuple(int(rng.integers(s)) for s in P.shape)
            if name in ("dWg", "dWu", "dWd"):
                pos = (int(idx[rng.integers(N), 0]),) + pos[1:]        # an expert that is in use
            old = P[pos]
            P[pos] = old + eps
            lp, _ = fd_loss(X64, Wr64, bias, W64, dY, idx)
            P[pos] = old - eps
            lm, _ = fd_loss(X64, Wr64, bias, W64, dY, idx)
            P[pos] = old
            fd = (lp - lm) / (2 * eps)
            an = got[name][pos]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, pos, fd, an)


def test_expert_grad_slices_match_full_backward(tiny):
    """The per-expert slice helper used at full size agrees with the full backward."""
    w, T = tiny
    idx, g, _ = O.route(T.X, T.Wr, T.bias, w.k)
    full = O.backward(T.X, T.Wr, idx, g, (T.Wg, T.Wu, T.Wd), T.dY)
    for e in range(w.E):
        t, j = np.nonzero(idx == e)
        if len(t) == 0:
            continue
        cols = [0, 7, w.I - 1]
        rows = [3, w.I // 2]
        dWd_c, dWg_r, dWu_r = O.expert_grad_slices(T.X[t], g[t, j], T.dY[t], (T.Wg[e], T.Wu[e], T.Wd[e]),
                                                    cols, rows)
        np.testing.assert_allclose(dWd_c, full["dWd"][e][:, cols], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dWg_r, full["dWg"][e][rows, :], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dWu_r, full["dWu"][e][rows, :], rtol=1e-10, atol=1e-12)


def test_mirror_mode_rounds_like_bf16_storage():
    """The diagnostic mirror mode: mirror=False is the definition; mirror=True differs from it only by the
    bf16 rounding of stored intermediates (within a few bf16 ulps), and its own rounding is exact RNE."""
    from oracle import moe_ref as O
    from synth import inputs as S
    r = O._bf16_round(np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0]))
    assert np.array_equal(r, [1.0, 1.0, 1.0 + 2 ** -7, -2.5, 0.0])     # ties to even, exact values kept
    w = S.WORKLOADS["tiny"]
    T = S.make(w)
    idx, g, _ = O.route(T.X, T.Wr, T.bias, w.k)
    Y = O.forward(T.X, idx, g, (T.Wg, T.Wu, T.Wd))
    Ym = O.forward(T.X, idx, g, (T.Wg, T.Wu, T.Wd), mirror=True)
    assert np.array_equal(O._bf16_round(Ym), Ym)
    err = O.normalised_error(Ym, Y)
    assert 1e-4 < err < 1e-2
