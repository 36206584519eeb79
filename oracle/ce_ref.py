"""CPU oracle of the vocabulary-projection cross-entropy head.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import or run
it.  It shares no code with the CUDA path.

Sources (page title, then section / equation):
  * "bounded-streaming operators" summary, Methodology 2 (Ring-DTP): exact vocabulary projection;
    each round forms only a logit strip X W_r (V/P columns), folds its partial normaliser into a
    running per-token state (max, sum, target logit) and releases the strip; eq. (2) bounds the peak
    logit memory by O(N V b / P); eq. (3) is the online-softmax recurrence
        m' = max(m, max_v y_v),   z' = exp(m - m') z + sum_v exp(y_v - m').
  * "Training Trillion-Parameter MoE ..." blog, section 3.5 (vocabulary-axis chunking): softmax and
    cross-entropy in vocabulary shards by a two-pass scan (global max and sum-exp first, then each
    shard's loss and gradients), numerically equivalent to the standard implementation.

Both describe the same exact result, so the oracle is the plain definition, in float64:
    y[n, v]  = X[n] . W[v]                    (bf16 inputs widened exactly)
    lse[n]   = log sum_v exp(y[n, v])
    loss[n]  = lse[n] - y[n, t_n]
and, for an upstream gradient g[n] of loss[n] (g = 1/N for the mean loss),
    d[n, v]  = g[n] (exp(y[n, v] - lse[n]) - [v = t_n])
    dX[n]    = sum_v d[n, v] W[v],     dW[v] = sum_n d[n, v] X[n].
``online_fold`` restates eq. (3) for the tests that pin it to the plain log-sum-exp.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def logits(X, W) -> np.ndarray:
    """y = X W^T in float64 (X [N, H], W [V, H] as exact float values)."""
    return _f64(X) @ _f64(W).T


def logsumexp_rows(y: np.ndarray) -> np.ndarray:
    """log sum_v exp(y[n, v]), shifted by the row maximum so no term overflows."""
    m = y.max(axis=1)
    return m + np.log(np.exp(y - m[:, None]).sum(axis=1))


def forward(X, W, targets):
    """Per-token loss and log-sum-exp: (loss [N], lse [N])."""
    y = logits(X, W)
    lse = logsumexp_rows(y)
    t = np.asarray(targets, dtype=np.int64)
    loss = lse - y[np.arange(len(t)), t]
    return loss, lse


def backward(X, W, targets, g):
    """Gradients of sum_n g[n] loss[n]: (dX [N, H], dW [V, H]), float64."""
    y = logits(X, W)
    lse = logsumexp_rows(y)
    t = np.asarray(targets, dtype=np.int64)
    d = np.exp(y - lse[:, None])
    d[np.arange(len(t)), t] -= 1.0
    d *= _f64(g)[:, None]
    return d @ _f64(W), d.T @ _f64(X)


def rows_forward_backward(Xs, W, ts, gs, block: int = 8192):
    """Some tokens' (loss, lse, dX rows), with W streamed in blocks of vocabulary rows, for checks at sizes
    where the full logit matrix does not fit: the logits of the chosen tokens only, then the plain
    formulas row by row."""
    Xs = np.atleast_2d(_f64(Xs))
    ts = np.atleast_1d(np.asarray(ts, dtype=np.int64))
    gs = np.atleast_1d(_f64(gs))
    V = W.shape[0]
    y = np.concatenate([Xs @ _f64(W[v0:v0 + block]).T for v0 in range(0, V, block)], axis=1)
    lse = logsumexp_rows(y)
    d = np.exp(y - lse[:, None])
    d[np.arange(len(ts)), ts] -= 1.0
    d *= gs[:, None]
    dx = np.zeros_like(Xs)
    for v0 in range(0, V, block):
        dx += d[:, v0:v0 + block] @ _f64(W[v0:v0 + block])
    return lse - y[np.arange(len(ts)), ts], lse, dx


def online_fold(strips):
    """eq. (3): fold the logit strips of one token, in order, into (m, z); log-sum-exp = m + log z."""
    m, z = -np.inf, 0.0
    for y in strips:
        y = _f64(y)
        m_new = max(m, float(y.max()))
        z = np.exp(m - m_new) * z + float(np.exp(y - m_new).sum())
        m = m_new
    return m, z


def strip_bound_bytes(N: int, V: int, P: int, b: int = 2) -> int:
    """eq. (2) without its constant: one strip of N x ceil(V/P) logits of b bytes."""
    return N * -(-V // P) * b
