"""The pins catch plausible oracle mistakes (CPU only).

Each case plants one mistake in the oracle (monkeypatched, on the CPU, for the
duration of the test) and checks that at least one pin then fails.
"""
import numpy as np
import pytest

from oracle import moe_ref as O
import test_oracle_block as B
import test_oracle_plan as P
import test_oracle_router as R


def _fails(fn, *a):
    try:
        fn(*a)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


def test_mutation_silu_grad_dropped_term(monkeypatch, tiny):
    monkeypatch.setattr(O, "silu_grad", lambda z: 1.0 / (1.0 + np.exp(-z)))
    assert _fails(B.test_backward_vs_torch_autograd, tiny)


def test_mutation_wrong_activation(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda z: z / (1.0 + np.exp(z)))
    assert _fails(B.test_forward_single_expert_is_swiglu)


def test_mutation_gates_not_renormalised(monkeypatch, tiny):
    def bad(logits, idx):
        l = logits.astype(np.float64)
        p = np.exp(l - l.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        return np.take_along_axis(p, idx.astype(np.int64), axis=1)
    monkeypatch.setattr(O, "gates_of", bad)
    assert _fails(R.test_gates_sum_to_one_and_order, tiny)


def test_mutation_ties_to_higher_id(monkeypatch):
    def bad(logits, k):
        E = logits.shape[1]
        order = np.argsort(-logits[:, ::-1], axis=1, kind="stable")
        return (E - 1 - order[:, :k]).astype(np.int32)
    monkeypatch.setattr(O, "topk", bad)
    assert _fails(R.test_topk_ties_go_to_lower_id)


def test_mutation_consecutive_chunks(monkeypatch):
    def bad(N, K, i):
        c = -(-N // K)
        return np.arange(i * c, min(N, (i + 1) * c), dtype=np.int64)
    monkeypatch.setattr(O, "chunk_tokens", bad)
    assert _fails(P.test_strided_membership, 512, 4)


def test_mutation_router_gradient_sign(monkeypatch, tiny):
    real = O.backward

    def bad(*a, **kw):
        out = real(*a, **kw)
        X = a[0]
        x64 = O.bf16_to_f64(X) if X.dtype == np.uint16 else X
        idx = a[2].astype(np.int64)
        Wr64 = np.asarray(a[1], np.float64)
        out["dX"] = out["dX"] - 2 * np.einsum("tj,tjh->th", out["dlogit"], Wr64[idx])
        return out
    monkeypatch.setattr(O, "backward", bad)
    assert _fails(B.test_backward_vs_torch_autograd, tiny)


def test_mutation_unstable_permutation(monkeypatch):
    real = O.permute_chunk

    def bad(idx, K, i, E):
        rr, off, row_of = real(idx, K, i, E)
        rr = rr.copy()
        for e in range(E):
            rr[off[e]:off[e + 1]] = rr[off[e]:off[e + 1]][::-1]
        return rr, off, row_of
    monkeypatch.setattr(O, "permute_chunk", bad)
    assert _fails(B.test_permutation, 101, 7, 3, 5)


def test_mutation_down_projection_transposed(monkeypatch, tiny):
    real = O._weights_getter

    def bad(W):
        get = real(W)
        return lambda e: (lambda g, u, d: (g, u, d.reshape(d.shape[1], d.shape[0])))(*get(e))
    monkeypatch.setattr(O, "_weights_getter", bad)
    assert _fails(B.test_forward_vs_dense_masked, tiny)
