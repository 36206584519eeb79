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


def _fp32_adamw(st, hp, step, plant=None):
    """An fp32 restatement of the update, standing in for the device path in checks of the comparison
    itself; `plant` inserts one plausible mistake."""
    f = np.float32
    b1, b2 = f(hp["beta1"]), f(hp["beta2"])
    bc1 = 1 - hp["beta1"] ** step
    bc2 = 1 - hp["beta2"] ** step
    p = st.p * f(1 - hp["lr"] * hp["weight_decay"])
    m = b1 * st.m + f(1 - hp["beta1"]) * st.g
    v = b2 * st.v + f(1 - hp["beta2"]) * st.g * st.g
    if plant == "no_bias_correction_v":
        bc2 = 1.0
    if plant == "decay_after":
        p = st.p
    upd = f(hp["lr"] / bc1) * m / (np.sqrt(v) * f(1 / np.sqrt(bc2)) + f(hp["eps"]))
    if plant == "sign":
        upd = -upd
    p = p - upd
    if plant == "decay_after":
        p = p * f(1 - hp["lr"] * hp["weight_decay"])
    return p.astype(np.float32), m.astype(np.float32), v.astype(np.float32)


HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _check(plant, step=3):
    from synth import inputs as S
    from synth.inputs import f32_to_bf16
    import adam_check as C
    st = S.adam_state(20000, seed=5)
    p, m, v = _fp32_adamw(st, HP, step, plant)
    ref = A.adamw_step(st.p, st.m, st.v, st.g, step=step, **HP)
    tol = C.bounds(st.p, st.m, st.v, st.g, step=step, **HP)
    return C.compare((p, m, v, f32_to_bf16(p)), ref, tol)


def test_comparison_accepts_an_fp32_restatement():
    assert _check(None) == {}


@pytest.mark.parametrize("plant", ["no_bias_correction_v", "decay_after", "sign"])
def test_comparison_catches_planted_mistakes(plant):
    assert _check(plant)
