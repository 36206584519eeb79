"""Seeded synthetic workloads for the chunk-bounded MoE block.

Test and benchmark infrastructure shared by the CPU oracle and the CUDA path.
It holds none of the block's arithmetic: it names the workload shapes and draws
the input tensors.  Every element is a pure function of (seed, tensor stream,
element index) -- see ``gen.c`` -- so a slice (one expert's weights, a few token
rows) can be drawn on its own and matches the same slice of the full tensor.

Workload shapes follow the configurations named for this block (tiny, mid,
long, many, many_zipf, extreme); the pages' production models are not
available, so these seeded tensors stand in for them:

* X ~ N(0, 1) bf16 [N, H];  dY ~ N(0, 1) bf16 [N, H]
* Wr ~ N(0, 1/H) fp32 [E, H] (nn.Linear layout of the H x E router matrix)
* Wg, Wu ~ N(0, 1/H) bf16 [E, I, H];  Wd ~ N(0, 1/I) bf16 [E, H, I]
* bias fp32 [E]: none, Zipf(s) popularity, or one hot expert + Zipf(1.0).

Bias construction (a reading; the source pages give none): target route shares
q_e proportional to rank_e^-s, ranks a seeded permutation of 1..E; shares are
capped at 0.9/k because one expert can take at most one route per token; the
bias is then fitted by 60 damped probit-space steps
b += 0.5 * (probit(k q) - probit(k achieved)), where "achieved" is measured on a
Monte Carlo model of the logits (iid N(0,1) per expert, which is the
distribution of X.Wr^T for these X and Wr), not on the workload's own tensors.
For the "long" workload the hot expert's share is read as 30% of tokens
(0.30/k of routes), since one expert can never take more than 1/k of routes.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

# Tensor streams.  Fixed ids so that a tensor's values never depend on the
# sizes of the others.
STREAM_X, STREAM_WR, STREAM_WG, STREAM_WU, STREAM_WD, STREAM_RANKS, STREAM_DY, STREAM_CALIB = range(8)


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libsynth.so (plain gcc + OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    src = os.path.join(_HERE, "gen.c")
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
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            for name in ("synth_normal_bf16", "synth_normal_f32"):
                getattr(lib, name).argtypes = [u64, u64, u64, i64, dbl, vp]
                getattr(lib, name).restype = None
            lib.synth_uniform_f64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_u64.argtypes = [u64, u64, u64, i64, vp]
            lib.synth_bf16_to_f32.argtypes = [vp, i64, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal_bf16(seed, stream, shape, std, offset=0, out=None) -> np.ndarray:
    """bf16 bit patterns (uint16) of std * N(0,1)."""
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == n
    _L().synth_normal_bf16(seed, stream, offset, n, float(std), _ptr(out))
    return out


def normal_f32(seed, stream, shape, std, offset=0, out=None) -> np.ndarray:
    n = int(np.prod(shape))
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.size == n
    _L().synth_normal_f32(seed, stream, offset, n, float(std), _ptr(out))
    return out


def uniform_f64(seed, stream, n, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().synth_uniform_f64(seed, stream, offset, n, _ptr(out))
    return out


def u64(seed, stream, n, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _L().synth_u64(seed, stream, offset, n, _ptr(out))
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp32."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# --------------------------------------------------------------------------- #
# Workloads
# --------------------------------------------------------------------------- #
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    H: int
    E: int
    k: int
    I: int
    c: int
    K_max: int
    bias: str = "none"          # "none" | "zipf" | "hot+zipf"
    zipf_s: float = 0.0
    hot_token_share: float = 0.0

    def cfg(self):
        return dict(N=self.N, H=self.H, E=self.E, k=self.k, I=self.I, c=self.c, K_max=self.K_max)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def scaled(self, factor: int = 8) -> "Workload":
        """Same E, k, K and skew; N, H, I cut by `factor` (H, I rounded up to 64)."""
        def r64(v):
            return max(64, ((v // factor + 63) // 64) * 64)
        N = max(self.N // factor, 1)
        c = max(self.c // factor, 1)
        return dataclasses.replace(self, name=self.name + f"/{factor}", N=N, H=r64(self.H),
                                   I=r64(self.I), c=c)


WORKLOADS = {
    "tiny": Workload("tiny", N=512, H=256, E=8, k=2, I=512, c=128, K_max=4),
    "mid": Workload("mid", N=16384, H=2048, E=64, k=8, I=1408, c=2048, K_max=8,
                    bias="zipf", zipf_s=1.1),
    "long": Workload("long", N=65536, H=4096, E=128, k=8, I=1536, c=4096, K_max=16,
                     bias="hot+zipf", zipf_s=1.0, hot_token_share=0.30),
    "many": Workload("many", N=32768, H=7168, E=384, k=8, I=2048, c=2048, K_max=16),
    "many_zipf": Workload("many_zipf", N=32768, H=7168, E=384, k=8, I=2048, c=2048, K_max=16,
                          bias="zipf", zipf_s=1.2),
    "extreme": Workload("extreme", N=16384, H=4096, E=896, k=16, I=1024, c=1024, K_max=16,
                        bias="zipf", zipf_s=1.3),
}


def target_shares(w: Workload, seed: int) -> np.ndarray:
    """Target route share per expert (sums to 1), before calibration."""
    E, k = w.E, w.k
    ranks = np.argsort(u64(seed, STREAM_RANKS, E), kind="stable").argsort() + 1  # a permutation of 1..E
    ranks = ranks.astype(np.float64)
    if w.bias == "zipf":
        q = ranks ** (-w.zipf_s)
        q /= q.sum()
    elif w.bias == "hot+zipf":
        hot = w.hot_token_share / k          # token share -> route share
        rest = ranks ** (-w.zipf_s)
        rest[ranks == 1] = 0.0
        rest = rest / rest.sum() * (1.0 - hot)
        q = rest
        q[ranks == 1] = hot
    else:
        return np.full(E, 1.0 / E)
    cap = 0.9 / k
    for _ in range(64):
        over = q > cap
        if not over.any():
            break
        excess = (q[over] - cap).sum()
        q[over] = cap
        free = ~over & (q < cap)
        q[free] += excess * q[free] / q[free].sum()
    return q


def bias_for(w: Workload, seed: int = 0, samples: int = 4096, iters: int = 60):
    """fp32 router bias [E] (or None) and the Monte Carlo route shares it reaches."""
    if w.bias == "none":
        return None, None
    from scipy.special import ndtri
    q = target_shares(w, seed)
    E, k = w.E, w.k
    Z = normal_f32(seed, STREAM_CALIB, (samples, E), 1.0).astype(np.float64)
    lo, hi = 0.5 / samples, 1.0 - 0.5 / samples
    p_target = np.clip(k * q, lo, hi)            # probability that a token picks e
    b = ndtri(p_target)
    achieved = None
    for _ in range(iters):
        L = Z + b
        sel = np.argpartition(-L, k - 1, axis=1)[:, :k]
        achieved = np.bincount(sel.ravel(), minlength=E) / (samples * k)
        b = b + 0.5 * (ndtri(p_target) - ndtri(np.clip(k * achieved, lo, hi)))
        b = b - b.mean()
    return b.astype(np.float32), achieved


@dataclasses.dataclass
class Tensors:
    """Host tensors of one workload.  bf16 tensors are uint16 bit patterns."""
    w: Workload
    X: np.ndarray
    Wr: np.ndarray
    bias: np.ndarray | None
    Wg: np.ndarray
    Wu: np.ndarray
    Wd: np.ndarray
    dY: np.ndarray


def make(w: Workload, seed: int = 0, weights: bool = True) -> Tensors:
    """Draw every input tensor of workload `w` on the host."""
    N, H, E, I = w.N, w.H, w.E, w.I
    X = normal_bf16(seed, STREAM_X, (N, H), 1.0)
    Wr = normal_f32(seed, STREAM_WR, (E, H), 1.0 / np.sqrt(H))
    bias, _ = bias_for(w, seed)
    if weights:
        Wg = normal_bf16(seed, STREAM_WG, (E, I, H), 1.0 / np.sqrt(H))
        Wu = normal_bf16(seed, STREAM_WU, (E, I, H), 1.0 / np.sqrt(H))
        Wd = normal_bf16(seed, STREAM_WD, (E, H, I), 1.0 / np.sqrt(I))
    else:
        Wg = Wu = Wd = None
    dY = normal_bf16(seed, STREAM_DY, (N, H), 1.0)
    return Tensors(w, X, Wr, bias, Wg, Wu, Wd, dY)


def expert_weights(w: Workload, e: int, seed: int = 0):
    """One expert's (Wg_e [I,H], Wu_e [I,H], Wd_e [H,I]) bf16, drawn on its own."""
    H, I = w.H, w.I
    off = e * I * H
    Wg = normal_bf16(seed, STREAM_WG, (I, H), 1.0 / np.sqrt(H), offset=off)
    Wu = normal_bf16(seed, STREAM_WU, (I, H), 1.0 / np.sqrt(H), offset=off)
    Wd = normal_bf16(seed, STREAM_WD, (H, I), 1.0 / np.sqrt(I), offset=off)
    return Wg, Wu, Wd


def token_rows(w: Workload, stream: int, rows: np.ndarray, seed: int = 0) -> np.ndarray:
    """bf16 rows `rows` of X (stream STREAM_X) or dY (STREAM_DY), drawn on their own."""
    out = np.empty((len(rows), w.H), dtype=np.uint16)
    for n, t in enumerate(np.asarray(rows, dtype=np.int64)):
        normal_bf16(seed, stream, (w.H,), 1.0, offset=int(t) * w.H, out=out[n])
    return out


# --------------------------------------------------------------------------- #
# Optimizer state (the offloaded AdamW step)
# --------------------------------------------------------------------------- #
STREAM_ADAM_P, STREAM_ADAM_M, STREAM_ADAM_V, STREAM_ADAM_G = 101, 102, 103, 104


@dataclasses.dataclass
class AdamState:
    """fp32 master weights, moments and gradient of n parameters starting at `offset`."""
    p: np.ndarray
    m: np.ndarray
    v: np.ndarray
    g: np.ndarray


def adam_state(n: int, seed: int = 0, offset: int = 0, fresh: bool = False, out: AdamState | None = None) -> AdamState:
    """Seeded state of a flat parameter vector, as mid-training: p ~ N(0, 0.02^2) (a typical weight
    init scale), g ~ N(0, 1e-3^2), m ~ N(0, 1e-3^2), v = (N(0, 1e-3^2))^2, so sqrt(v) is on the scale of |g|.
    `fresh` gives zero moments (the state before step 1).  Element i is a pure function of
    (seed, stream, offset + i), so any window can be drawn on its own.  `out` (float32 arrays of n
    elements, e.g. views of page-locked buffers) receives the state in place."""
    o = out or AdamState(*(np.empty(n, np.float32) for _ in range(4)))
    normal_f32(seed, STREAM_ADAM_P, (n,), 0.02, offset, out=o.p)
    normal_f32(seed, STREAM_ADAM_G, (n,), 1e-3, offset, out=o.g)
    if fresh:
        o.m[...] = 0.0
        o.v[...] = 0.0
    else:
        normal_f32(seed, STREAM_ADAM_M, (n,), 1e-3, offset, out=o.m)
        normal_f32(seed, STREAM_ADAM_V, (n,), 1e-3, offset, out=o.v)
        np.square(o.v, out=o.v)
    return o


def block_parameter_count(w: Workload) -> int:
    """Parameters of one block: router Wr [E,H] plus the expert weights Wg, Wu [E,I,H] and Wd [E,H,I]."""
    return w.E * w.H + 3 * w.E * w.I * w.H


# --------------------------------------------------------------------------- #
# Vocabulary-projection cross-entropy head
# --------------------------------------------------------------------------- #
STREAM_CE_X, STREAM_CE_W, STREAM_CE_T = 110, 111, 112


@dataclasses.dataclass(frozen=True)
class CeWorkload:
    """N tokens of hidden size H against V classes, the backward in P vocabulary strips."""
    name: str
    N: int
    H: int
    V: int
    P: int

    def cfg(self) -> dict:
        return dict(N=self.N, H=self.H, V=self.V, P=self.P)


# ce_full: H = 7168, V = 200,000 and P = 8 are the Ring-DTP benchmark's (bounded-streaming summary,
# isolated component benchmarks); N = 16,384 tokens is a reading (the page gives none).
CE_WORKLOADS = {
    "ce_tiny": CeWorkload("ce_tiny", N=300, H=128, V=1000, P=3),
    "ce_small": CeWorkload("ce_small", N=1000, H=256, V=5000, P=4),
    "ce_mid": CeWorkload("ce_mid", N=2048, H=1024, V=32000, P=8),
    "ce_full": CeWorkload("ce_full", N=16384, H=7168, V=200_000, P=8),
    # a profiling case: operands above the 129 MB L2, a few GB on the device in all
    "ce_4k": CeWorkload("ce_4k", N=4096, H=4096, V=32768, P=8),
}


@dataclasses.dataclass
class CeTensors:
    X: np.ndarray        # [N, H] bf16 bits
    W: np.ndarray        # [V, H] bf16 bits
    targets: np.ndarray  # [N] int32


def ce_make(w: CeWorkload, seed: int = 0, weights: bool = True) -> CeTensors:
    """X ~ N(0, 1) bf16 (hidden states), W ~ N(0, 1/H) bf16 (so logits are about N(0, 1), an untrained
    head), targets uniform over the V classes."""
    X = normal_bf16(seed, STREAM_CE_X, (w.N, w.H), 1.0)
    W = normal_bf16(seed, STREAM_CE_W, (w.V, w.H), 1.0 / np.sqrt(w.H)) if weights else None
    t = (u64(seed, STREAM_CE_T, w.N) % np.uint64(w.V)).astype(np.int32)
    return CeTensors(X, W, t)


def ce_rows(w: CeWorkload, rows, seed: int = 0) -> np.ndarray:
    """bf16 rows `rows` of X, drawn on their own."""
    out = np.empty((len(rows), w.H), dtype=np.uint16)
    for i, n in enumerate(np.asarray(rows, dtype=np.int64)):
        normal_bf16(seed, STREAM_CE_X, (w.H,), 1.0, offset=int(n) * w.H, out=out[i])
    return out
