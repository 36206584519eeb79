"""Pins for the AdamW oracle (CPU only): torch.optim.AdamW in float64 and closed forms."""
import numpy as np
import pytest
import torch

from oracle import adamw_ref as A


@pytest.mark.parametrize("wd,steps", [(0.0, 1), (0.1, 3), (0.01, 5)])
def test_matches_torch_adamw(wd, steps):
    rng = np.random.default_rng(0)
    n = 1000
    p0 = rng.normal(size=n)
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=wd)
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=kw["lr"], betas=(kw["beta1"], kw["beta2"]), eps=kw["eps"], weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, steps + 1):
        g = rng.normal(size=n)
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = A.adamw_step(p, m, v, g, step=t, **kw)
        st = opt.state[tp]
        np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(m, st["exp_avg"].numpy(), rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=1e-15)


def test_first_step_is_sign_like():
    """At t = 1 with zero moments and eps -> 0, the update is lr * sign(g) (Adam's first step)."""
    g = np.array([3.0, -0.5, 1e-3, -7.0])
    p, m, v = A.adamw_step(np.zeros(4), np.zeros(4), np.zeros(4), g, lr=0.1, beta1=0.9, beta2=0.999, eps=0.0,
                           weight_decay=0.0, step=1)
    np.testing.assert_allclose(p, -0.1 * np.sign(g), rtol=1e-12)


def test_zero_gradient_only_decays():
    p0 = np.array([1.0, -2.0, 0.5])
    p, m, v = A.adamw_step(p0, np.zeros(3), np.zeros(3), np.zeros(3), lr=0.01, beta1=0.9, beta2=0.99, eps=1e-8,
                           weight_decay=0.5, step=1)
    np.testing.assert_allclose(p, p0 * (1 - 0.01 * 0.5), rtol=1e-15)
    assert np.all(m == 0) and np.all(v == 0)


def test_floor_bytes():
    assert A.stream_floor_bytes(1000) == 12000
