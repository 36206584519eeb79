"""CPU oracle for the chunk-bounded, top-k-softmax-routed MoE block.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or run anything under ``oracle/``.
It shares no code with the CUDA path (no kernels, headers, helpers or
constants); the only module both sides use is the seeded input generator in
``synth/``, which holds none of the block's arithmetic.

What it computes is the plain definition of the block, in float64 unless a
step below says otherwise.  The chunked method claims results identical to the
unchunked block (bounded-streaming summary: "Core principle" and design
requirements 1-2), so apart from the chunk plan and the per-chunk permutation,
which are checked bit for bit as outputs in their own right, the oracle does
not chunk at all.

Sources (page title, then section / equation):
  * "bounded-streaming operators" summary, Methodology 1 (PipelinedLLEP),
    eq. (1): K = min(ceil(N/c), K_max), c_eff = ceil(N/K); strided chunk
    membership (chunk i holds positions i, i+K, i+2K, ...); the buffer bound
    2 E_p k c H b.
  * RelayMoE summary, section 2.1: tokens select their top-k experts; the
    dispatcher expands and permutes tokens to experts, then returns and
    recombines their outputs; sections 1 and 3.1: dropless, padding-free
    expert compute.
  * Workload text: softmax then top-k with the gates renormalised over the
    top-k; SwiGLU expert FFN of width I; logits = X.W_r + bias.

Readings taken where the pages are silent (each one is listed with its reason
in the design notes):
  * top-k is decided on the fp32 logits of ``router_ref.c`` (the one place the
    oracle computes in fp32): descending logit, equal logits to the lower
    expert id; slot j is the rank.
  * gates: p = softmax over all E experts, g_j = p[idx_j] / sum_j p[idx_j].
  * SwiGLU: act = silu(x Wg_e^T) * (x Wu_e^T), o = act Wd_e^T,
    silu(z) = z / (1 + exp(-z)); Y[t] = sum_j g_j o_j.
  * backward: the plain gradient of sum(Y * dY) with respect to X, Wr, Wg,
    Wu, Wd and the gates, holding the selected set fixed; the bias gets none.
  * per-chunk permutation: within a chunk, routes are visited in (local token,
    slot) order and appended to their expert's bucket; buckets are laid out in
    expert order.  Rows therefore ascend by token within an expert.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_router.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile router_ref.c with plain gcc (no contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "router_ref.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_router_logits.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
            lib.oracle_router_logits.restype = None
            _lib = lib
    return _lib


# --------------------------------------------------------------------------- #
# bf16 helpers (the inputs arrive as bf16 bit patterns in uint16 arrays)
# --------------------------------------------------------------------------- #
def bf16_to_f64(a: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns, as float64."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- #
# Chunk plan -- bounded-streaming summary, Methodology 1, eq. (1)
# --------------------------------------------------------------------------- #
def chunk_plan(N: int, c: int, K_max: int) -> tuple[int, int]:
    """K = min(ceil(N / c), K_max) and c_eff = ceil(N / K)  (eq. 1)."""
    if N <= 0:
        return 0, 0
    K = min(-(-N // c), K_max)
    c_eff = -(-N // K)
    return K, c_eff


def chunk_tokens(N: int, K: int, i: int) -> np.ndarray:
    """Strided membership: chunk i holds positions i, i+K, i+2K, ... (Methodology 1)."""
    return np.arange(i, N, K, dtype=np.int64)


def routed_bound_bytes(k: int, c_eff: int, H: int, b: int = 2, E_p: int = 1) -> int:
    """Dispatch-buffer bound 2 E_p k c H b (Methodology 1, 'Memory bound'); E_p = 1 on one device."""
    return 2 * E_p * k * c_eff * H * b


# --------------------------------------------------------------------------- #
# Router -- RelayMoE summary 2.1; workload text (softmax, top-k, renormalise)
# --------------------------------------------------------------------------- #
def router_logits(X_rows: np.ndarray, Wr: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """fp32 logits [rows, E]: one fmaf chain per (t, e) over h ascending, then + bias (router_ref.c)."""
    X_rows = np.ascontiguousarray(X_rows, dtype=np.uint16)
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    rows, H = X_rows.shape
    E = Wr.shape[0]
    assert Wr.shape[1] == H
    out = np.empty((rows, E), dtype=np.float32)
    b = None
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float32)
        assert b.shape == (E,)
    _L().oracle_router_logits(X_rows.ctypes.data, Wr.ctypes.data,
                              None if b is None else b.ctypes.data, rows, H, E, out.ctypes.data)
    return out


def topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert ids [rows, k] int32: descending fp32 logit, ties to the lower id."""
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def gates_of(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Gates [rows, k] float64: softmax over all experts, renormalised over the chosen k."""
    l = logits.astype(np.float64)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    p = e / e.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def route(X: np.ndarray, Wr: np.ndarray, bias: np.ndarray | None, k: int):
    """(topk_idx [N,k] int32, gates [N,k] float64, logits [N,E] fp32)."""
    logits = router_logits(X, Wr, bias)
    idx = topk(logits, k)
    return idx, gates_of(logits, idx), logits


# --------------------------------------------------------------------------- #
# Per-chunk permutation (counting sort by expert) -- RelayMoE summary 2.1;
# "Training Trillion-Parameter MoE ..." blog, 3.3 (permute / unpermute)
# --------------------------------------------------------------------------- #
def permute_chunk(topk_idx: np.ndarray, K: int, i: int, E: int):
    """Expand and permute chunk i's routes by expert.

    Returns (row_route, expert_off, row_of):
      row_route [n_i * k] int32 : global route id t*k + j of each permuted row
      expert_off [E + 1] int32  : rows of expert e are expert_off[e]:expert_off[e+1]
      row_of [n_i, k] int32     : permuted row of (local token l, slot j)
    """
    N, k = topk_idx.shape
    toks = chunk_tokens(N, K, i)
    buckets = [[] for _ in range(E)]
    for l, t in enumerate(toks.tolist()):
        for j in range(k):
            buckets[int(topk_idx[t, j])].append((l, j, t * k + j))
    row_route = np.empty(len(toks) * k, dtype=np.int32)
    row_of = np.empty((len(toks), k), dtype=np.int32)
    expert_off = np.zeros(E + 1, dtype=np.int32)
    r = 0
    for e in range(E):
        expert_off[e] = r
        for (l, j, q) in buckets[e]:
            row_route[r] = q
            row_of[l, j] = r
            r += 1
    expert_off[E] = r
    return row_route, expert_off, row_of


# --------------------------------------------------------------------------- #
# Expert FFN (SwiGLU) and the block, forward and backward, float64
# --------------------------------------------------------------------------- #
def silu(z):
    return z / (1.0 + np.exp(-z))


def silu_grad(z):
    """d silu / dz = s (1 + z (1 - s)) with s = sigmoid(z)."""
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def _weights_getter(W):
    """Accept (Wg, Wu, Wd) arrays [E,...] or a callable e -> (Wg_e, Wu_e, Wd_e); yield float64."""
    if callable(W):
        return lambda e: tuple(bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, np.float64)
                               for a in W(e))
    Wg, Wu, Wd = W

    def get(e):
        return tuple(bf16_to_f64(a[e]) if a.dtype == np.uint16 else np.asarray(a[e], np.float64)
                     for a in (Wg, Wu, Wd))
    return get


def _routes_by_expert(topk_idx: np.ndarray):
    """{e: (token ids, slot ids)} over all routes, tokens ascending."""
    n, k = topk_idx.shape
    flat = topk_idx.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    es = flat[order]
    out = {}
    bounds = np.flatnonzero(np.diff(es)) + 1
    for seg in np.split(np.arange(len(order)), bounds):
        if len(seg) == 0:
            continue
        e = int(es[seg[0]])
        q = order[seg]
        out[e] = (q // k, q % k)
    return out


def _bf16_round(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (through fp32, both round-to-nearest-even), back as float64."""
    u = np.asarray(a, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def forward(X: np.ndarray, topk_idx: np.ndarray, gates: np.ndarray, W, mirror: bool = False) -> np.ndarray:
    """Y [n, H] float64 = sum_j g[t,j] * FFN_{idx[t,j]}(X[t])  (RelayMoE 2.1; SwiGLU FFN).

    mirror=True is the diagnostic mode: the expert activation and the expert output are rounded to
    bf16 where a bf16 device implementation stores them between its GEMMs, and Y is rounded to bf16
    at the end; the arithmetic is still float64.  The checked definition is mirror=False."""
    x64 = bf16_to_f64(X) if X.dtype == np.uint16 else np.asarray(X, np.float64)
    get = _weights_getter(W)
    Y = np.zeros_like(x64)
    g = np.asarray(gates, np.float64)
    rnd = _bf16_round if mirror else (lambda a: a)
    for e, (t, j) in _routes_by_expert(topk_idx).items():
        Wg, Wu, Wd = get(e)
        x = x64[t]
        act = rnd(silu(x @ Wg.T) * (x @ Wu.T))
        o = rnd(act @ Wd.T)
        np.add.at(Y, t, g[t, j][:, None] * o)
    return rnd(Y)


def backward(X, Wr, topk_idx, gates, W, dY, want_weight_grads: bool = True):
    """Plain gradient of sum(Y * dY) (selected set held fixed).

    Returns dict with dX [n,H], dgates [n,k], dlogit [n,k] (on the selected
    slots), dWr [E,H] and, if requested, dWg [E,I,H], dWu [E,I,H], dWd [E,H,I].
    """
    x64 = bf16_to_f64(X) if X.dtype == np.uint16 else np.asarray(X, np.float64)
    dy = bf16_to_f64(dY) if dY.dtype == np.uint16 else np.asarray(dY, np.float64)
    Wr64 = np.asarray(Wr, np.float64)
    E, H = Wr64.shape
    n, k = topk_idx.shape
    g = np.asarray(gates, np.float64)
    get = _weights_getter(W)
    dX = np.zeros_like(x64)
    dg = np.zeros((n, k))
    grads = {}
    for e, (t, j) in _routes_by_expert(topk_idx).items():
        Wg, Wu, Wd = get(e)
        x = x64[t]
        z_g = x @ Wg.T
        z_u = x @ Wu.T
        act = silu(z_g) * z_u
        o = act @ Wd.T
        dg[t, j] = np.einsum("rh,rh->r", dy[t], o)
        dO = g[t, j][:, None] * dy[t]                 # d(loss)/d(o) for this route
        dAct = dO @ Wd                                # [R, I]
        dZg = dAct * z_u * silu_grad(z_g)
        dZu = dAct * silu(z_g)
        np.add.at(dX, t, dZg @ Wg + dZu @ Wu)
        if want_weight_grads:
            grads[e] = (dZg.T @ x, dZu.T @ x, dO.T @ act)
    # gates g_j = exp(l_j) / sum_{i in S} exp(l_i)  =>  dl_i = g_i (dg_i - sum_j g_j dg_j)
    dlogit = g * (dg - np.sum(g * dg, axis=1, keepdims=True))
    sel = topk_idx.astype(np.int64)
    dX += np.einsum("tj,tjh->th", dlogit, Wr64[sel])
    dWr = np.zeros((E, H))
    np.add.at(dWr, sel.reshape(-1), dlogit.reshape(-1)[:, None] * np.repeat(x64, k, axis=0))
    out = dict(dX=dX, dgates=dg, dlogit=dlogit, dWr=dWr)
    if want_weight_grads:
        I = get(0)[0].shape[0]
        dWg = np.zeros((E, I, H))
        dWu = np.zeros((E, I, H))
        dWd = np.zeros((E, H, I))
        for e, (a, b, c) in grads.items():
            dWg[e], dWu[e], dWd[e] = a, b, c
        out.update(dWg=dWg, dWu=dWu, dWd=dWd)
    return out


def expert_grad_slices(X_rows, g_rows, dY_rows, We, cols_d, rows_gu):
    """Slices of one expert's weight gradients, from the routes that reach it.

    The same chain rule as ``backward`` restricted to one expert e: for each
    route r to e (token row x_r, gate g_r, output gradient dY_r),
      dWd_e[:, i] = sum_r (g_r dY_r) * act_r[i]
      dWg_e[i, :] = sum_r dAct_r[i] * up_r[i] * silu'(gate_r[i]) * x_r
      dWu_e[i, :] = sum_r dAct_r[i] * silu(gate_r[i]) * x_r
    with gate_r = x_r Wg_e^T, up_r = x_r Wu_e^T, act = silu(gate) * up and
    dAct_r = (g_r dY_r) Wd_e.  Only the requested columns i of dWd_e and rows i
    of dWg_e / dWu_e are formed, so the cost per route is O(H) per slice.
    Returns (dWd_e[:, cols_d] [H, len], dWg_e[rows_gu, :], dWu_e[rows_gu, :]).
    """
    x = bf16_to_f64(X_rows) if X_rows.dtype == np.uint16 else np.asarray(X_rows, np.float64)
    dy = bf16_to_f64(dY_rows) if dY_rows.dtype == np.uint16 else np.asarray(dY_rows, np.float64)
    Wg, Wu, Wd = (bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, np.float64) for a in We)
    dO = np.asarray(g_rows, np.float64)[:, None] * dy
    cols_d = np.asarray(cols_d, np.int64)
    rows_gu = np.asarray(rows_gu, np.int64)
    z_g = x @ Wg[cols_d].T
    z_u = x @ Wu[cols_d].T
    dWd_cols = dO.T @ (silu(z_g) * z_u)
    z_g2 = x @ Wg[rows_gu].T
    z_u2 = x @ Wu[rows_gu].T
    dAct = dO @ Wd[:, rows_gu]
    dWg_rows = (dAct * z_u2 * silu_grad(z_g2)).T @ x
    dWu_rows = (dAct * silu(z_g2)).T @ x
    return dWd_cols, dWg_rows, dWu_rows


def block(X, Wr, bias, W, dY, k):
    """Route, forward and backward of the whole block (all float64 except the fp32 logits)."""
    idx, g, logits = route(X, Wr, bias, k)
    Y = forward(X, idx, g, W)
    grads = backward(X, Wr, idx, g, W, dY)
    return dict(topk_idx=idx, gates=g, logits=logits, Y=Y, **grads)


def normalised_error(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max|gpu - ref| / max|ref| (the parity metric for floating-point outputs)."""
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(np.asarray(gpu, np.float64) - ref))) if ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den
