"""Pins for the cross-entropy oracle (CPU only): torch's float64 cross_entropy and autograd, closed forms,
the online recurrence of eq. (3), and planted mistakes."""
import numpy as np
import pytest
import torch

from oracle import ce_ref as C


def _case(N=7, H=5, V=11, seed=0, scale=1.0):
    r = np.random.default_rng(seed)
    return (r.normal(size=(N, H)) * scale, r.normal(size=(V, H)) * scale, r.integers(0, V, size=N),
            r.normal(size=N))


def test_forward_matches_torch_cross_entropy():
    X, W, t, _ = _case()
    loss, lse = C.forward(X, W, t)
    y = torch.tensor(X) @ torch.tensor(W).T
    ref = torch.nn.functional.cross_entropy(y, torch.tensor(t), reduction="none")
    np.testing.assert_allclose(loss, ref.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, torch.logsumexp(y, dim=1).numpy(), rtol=1e-13, atol=1e-13)


def test_backward_matches_autograd():
    X, W, t, g = _case(N=9, H=6, V=13, seed=3)
    tX = torch.tensor(X, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(tX @ tW.T, torch.tensor(t), reduction="none")
    (loss * torch.tensor(g)).sum().backward()
    dX, dW = C.backward(X, W, t, g)
    np.testing.assert_allclose(dX, tX.grad.numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dW, tW.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_uniform_logits_give_log_v():
    """W = 0: every logit is 0, loss = log V, and dX = 0 (the softmax is uniform, the gradient rows of W are 0)."""
    N, H, V = 4, 3, 37
    X = np.ones((N, H))
    W = np.zeros((V, H))
    t = np.arange(N) % V
    loss, lse = C.forward(X, W, t)
    np.testing.assert_allclose(loss, np.log(V), rtol=1e-15)
    dX, dW = C.backward(X, W, t, np.ones(N))
    assert np.all(dX == 0)
    # dW[v] = sum_n (1/V - [v = t_n]) X[n]
    expect = np.full((V, H), N / V)
    for n in range(N):
        expect[t[n]] -= 1.0
    np.testing.assert_allclose(dW, expect, rtol=1e-13, atol=1e-15)


def test_single_class_and_gradient_invariants():
    X, W, t, g = _case(V=1)
    loss, _ = C.forward(X, W, t)
    np.testing.assert_allclose(loss, 0.0, atol=1e-15)
    X, W, t, g = _case(N=6, V=9, seed=5)
    dX, dW = C.backward(X, W, t, g)
    # each token's d row sums to zero, so the rows of dW sum to zero
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-12)


def test_large_logits_do_not_overflow():
    X, W, t, _ = _case(scale=30.0)
    loss, lse = C.forward(X, W, t)
    assert np.all(np.isfinite(loss)) and np.all(loss >= -1e-9)


def test_row_form_matches_the_full_form():
    X, W, t, g = _case(N=5, H=4, V=50, seed=8)
    loss, lse = C.forward(X, W, t)
    dX, _ = C.backward(X, W, t, g)
    sel = [0, 2, 4]
    l, s, dx = C.rows_forward_backward(X[sel], W, t[sel], g[sel], block=7)
    np.testing.assert_allclose(l, loss[sel], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s, lse[sel], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dx, dX[sel], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("splits", [[50], [1, 49], [7, 7, 7, 29], [25, 25]])
def test_online_fold_equals_logsumexp(splits):
    """eq. (3) over any strip partition gives the plain log-sum-exp."""
    y = np.random.default_rng(1).normal(size=50) * 10
    strips = np.split(y, np.cumsum(splits)[:-1])
    m, z = C.online_fold(strips)
    assert abs((m + np.log(z)) - C.logsumexp_rows(y[None])[0]) < 1e-12


def test_planted_mistakes_are_caught():
    """A dropped max shift overflows; a sign error or a missing one-hot breaks the autograd pin."""
    X, W, t, g = _case(N=6, H=5, V=8, seed=11)
    tX = torch.tensor(X, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(tX @ torch.tensor(W).T, torch.tensor(t), reduction="none")
    (loss * torch.tensor(g)).sum().backward()
    y = X @ W.T
    lse = C.logsumexp_rows(y)
    d = np.exp(y - lse[:, None]) * g[:, None]          # one-hot term dropped
    assert not np.allclose(d @ W, tX.grad.numpy(), atol=1e-6)
    d2 = np.exp(y - lse[:, None])
    d2[np.arange(6), t] += 1.0                         # wrong sign on the one-hot
    assert not np.allclose((d2 * g[:, None]) @ W, tX.grad.numpy(), atol=1e-6)
    with np.errstate(over="ignore"):
        naive = np.log(np.exp(y * 1000).sum(axis=1))   # no shift
    assert not np.all(np.isfinite(naive)) and np.all(np.isfinite(C.logsumexp_rows(y * 1000)))


def test_strip_bound():
    assert C.strip_bound_bytes(16384, 200_000, 8) == 16384 * 25_000 * 2
