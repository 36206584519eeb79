"""Pins for the oracle's router: fp32 logits, top-k and gates (CPU only).

* The fp32 fused-multiply-add chain is checked bit for bit against an exact
  rational re-execution of the same chain (each step rounded to fp32 by hand),
  and against the exactly rounded dot product within the chain's error bound.
* Top-k is checked against k rounds of brute-force argmax with the tie rule.
* Gates reduce to closed forms: k = 1 gives 1; k = E gives the full softmax
  (scipy); they always sum to 1.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.special

from oracle import moe_ref as O
from synth import inputs as S


def rn_fp32(x: Fraction) -> float:
    """Round an exact rational to the nearest fp32 value, ties to even (normal range)."""
    if x == 0:
        return 0.0
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = float(Fraction(sign * n) * ulp)
    assert float(np.float32(v)) == v
    return v


def exact_chain(x_bf16: np.ndarray, w: np.ndarray, bias: float | None) -> float:
    xs = S.bf16_to_f32(x_bf16).astype(np.float64)
    acc = Fraction(0)
    for xv, wv in zip(xs.tolist(), np.asarray(w, np.float32).astype(np.float64).tolist()):
        acc = Fraction(rn_fp32(Fraction(xv) * Fraction(wv) + acc))
    if bias is not None:
        acc = Fraction(rn_fp32(acc + Fraction(float(np.float32(bias)))))
    return float(acc)


@pytest.mark.parametrize("seed", [0, 1])
def test_logits_bit_exact_vs_rational_chain(seed):
    rows, H, E = 5, 48, 4
    X = S.normal_bf16(seed, 100, (rows, H), 1.0)
    Wr = S.normal_f32(seed, 101, (E, H), 1.0 / math.sqrt(H))
    bias = S.normal_f32(seed, 102, (E,), 0.5)
    L = O.router_logits(X, Wr, bias)
    for r in range(rows):
        for e in range(E):
            ref = exact_chain(X[r], Wr[e], float(bias[e]))
            assert np.float32(L[r, e]).tobytes() == np.float32(ref).tobytes(), (r, e, L[r, e], ref)


def test_logits_bit_exact_cancellation():
    """Inputs with large cancellation make any other summation order round differently."""
    H, E = 40, 3
    xs = np.array([(1.0 if h % 2 == 0 else -1.0) * (1 + h / 64) for h in range(H)], np.float32)
    X = S.f32_to_bf16(xs)[None, :]
    Wr = np.stack([np.full(H, 1e4, np.float32) + np.arange(H, dtype=np.float32) * 1e-3 * (e + 1)
                   for e in range(E)]).astype(np.float32)
    L = O.router_logits(X, Wr, None)
    for e in range(E):
        assert np.float32(L[0, e]).tobytes() == np.float32(exact_chain(X[0], Wr[e], None)).tobytes()


def test_logits_within_dot_bound():
    """|chain - exact dot| <= gamma_H * sum|x w| + |bias rounding| (recursive summation bound)."""
    w = S.WORKLOADS["tiny"]
    X = S.normal_bf16(3, 0, (16, w.H), 1.0)
    Wr = S.normal_f32(3, 1, (w.E, w.H), 1.0 / math.sqrt(w.H))
    L = O.router_logits(X, Wr, None).astype(np.float64)
    x64 = S.bf16_to_f32(X).astype(np.float64)
    u = 2.0 ** -24
    gam = w.H * u / (1 - w.H * u)
    for r in range(16):
        for e in range(w.E):
            prods = (x64[r] * Wr[e].astype(np.float64)).tolist()   # exact: 8-bit x 24-bit significands
            exact = math.fsum(prods)
            assert abs(L[r, e] - exact) <= gam * math.fsum(abs(p) for p in prods) + 1e-30


def brute_topk(row: np.ndarray, k: int) -> list[int]:
    taken = []
    for _ in range(k):
        best = None
        for e, v in enumerate(row.tolist()):
            if e in taken:
                continue
            if best is None or v > row[best]:   # strict '>' keeps the lower id on ties
                best = e
        taken.append(best)
    return taken


@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_topk_brute_force(tiny, k):
    w, T = tiny
    L = O.router_logits(T.X[:64], T.Wr, T.bias)
    idx = O.topk(L, k)
    for r in range(64):
        assert idx[r].tolist() == brute_topk(L[r], k)


def test_topk_ties_go_to_lower_id():
    H, E = 64, 6
    X = S.normal_bf16(5, 0, (32, H), 1.0)
    Wr = S.normal_f32(5, 1, (E, H), 0.1)
    Wr[4] = Wr[1]          # experts 1 and 4 always tie
    Wr[5] = Wr[2]          # and 2 and 5
    L = O.router_logits(X, Wr, None)
    assert np.all(L[:, 4] == L[:, 1])
    idx = O.topk(L, 4)
    for r in range(32):
        assert idx[r].tolist() == brute_topk(L[r], 4)
        pos = {e: p for p, e in enumerate(idx[r].tolist())}
        for lo, hi in ((1, 4), (2, 5)):
            if lo in pos and hi in pos:
                assert pos[lo] < pos[hi]
            if hi in pos:
                assert lo in pos


def test_gates_k1_is_one(tiny):
    w, T = tiny
    L = O.router_logits(T.X, T.Wr, T.bias)
    g = O.gates_of(L, O.topk(L, 1))
    assert np.all(g == 1.0)


def test_gates_k_equals_E_is_softmax(tiny):
    w, T = tiny
    L = O.router_logits(T.X, T.Wr, T.bias)
    idx = O.topk(L, w.E)
    g = O.gates_of(L, idx)
    sm = scipy.special.softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(g, np.take_along_axis(sm, idx.astype(np.int64), axis=1), rtol=1e-12, atol=0)


def test_gates_sum_to_one_and_order(tiny):
    w, T = tiny
    L = O.router_logits(T.X, T.Wr, T.bias)
    idx = O.topk(L, w.k)
    g = O.gates_of(L, idx)
    np.testing.assert_allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(g, axis=1) <= 0)          # slot order follows the logits
    # ratio of two gates is exp(l_i - l_j), whatever the other experts do
    lsel = np.take_along_axis(L.astype(np.float64), idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(g[:, 0] / g[:, 1], np.exp(lsel[:, 0] - lsel[:, 1]), rtol=1e-12)
