"""Element-wise comparison of an fp32 AdamW result with the float64 oracle.

Error model (fp32 arithmetic, unit roundoff u = 2^-24): each of m, v and p is formed with at most
four roundings, plus the fp32 rounding of the per-step constants (beta, 1 - beta, lr / (1 - beta1^t),
1 / sqrt(1 - beta2^t), 1 - lr * wd), each at most u relative.  So, with the float64 terms of the update,
  |dm| <= 8u (beta1 |m0| + (1 - beta1) |g|)
  |dv| <= 8u (beta2 v0 + (1 - beta2) g^2)
  |dp| <= 8u (|p0 (1 - lr wd)| + |s|) + (lr / bc1) |dm| / denom,   s = (lr / bc1) m / denom
m may cancel (beta1 m0 against (1 - beta1) g), hence bounds on the terms, not on the result.
The bf16 working weight is a decision taken on fp32 p: where the oracle's p lies farther than the p
tolerance from a bf16 rounding midpoint, the weight must be exactly round-to-nearest-even(p_oracle);
elsewhere it must be the rounding of some value within the p tolerance (rounding is monotone, so
that is every bf16 value between the roundings of the interval's two ends).
"""
from __future__ import annotations

import numpy as np

from synth.inputs import bf16_to_f32, f32_to_bf16

U = 2.0 ** -24


def bounds(p0, m0, v0, g, *, lr, beta1, beta2, eps, weight_decay, step):
    p0, m0, v0, g = (np.asarray(a, np.float64) for a in (p0, m0, v0, g))
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    tm = 8 * U * (beta1 * np.abs(m0) + (1 - beta1) * np.abs(g))
    tv = 8 * U * (beta2 * v0 + (1 - beta2) * g * g)
    m1 = beta1 * m0 + (1 - beta1) * g
    v1 = beta2 * v0 + (1 - beta2) * g * g
    denom = np.sqrt(v1) / np.sqrt(bc2) + eps
    s = lr / bc1 * np.abs(m1) / denom
    tp = 8 * U * (np.abs(p0) * abs(1 - lr * weight_decay) + s) + lr / bc1 * tm / denom
    return tp, tm, tv


def compare(got, ref, tol):
    """got = (p, m, v, w_bf16_bits) from the fp32 path; ref = (p, m, v) float64; tol = (tp, tm, tv).
    Returns a dict of failures (empty when every element is within its bound)."""
    bad = {}
    for name, a, r, t in zip(("p", "m", "v"), got[:3], ref, tol):
        d = np.abs(np.asarray(a, np.float64) - r)
        over = d > t
        if over.any():
            i = int(np.argmax(d - t))
            bad[name] = f"{int(over.sum())} elements; worst i={i} got={a[i]!r} ref={r[i]!r} tol={t[i]:.3g}"
    p_ref, tp = ref[0], tol[0]
    lo = f32_to_bf16((p_ref - tp).astype(np.float32))
    hi = f32_to_bf16((p_ref + tp).astype(np.float32))
    w = np.asarray(got[3], np.uint16)
    wf = bf16_to_f32(w)
    wrong = (wf < bf16_to_f32(lo)) | (wf > bf16_to_f32(hi)) | ((lo == hi) & (w != lo))
    if wrong.any():
        i = int(np.flatnonzero(wrong)[0])
        bad["w"] = f"{int(wrong.sum())} elements; first i={i} got={w[i]:#06x} expected {lo[i]:#06x}/{hi[i]:#06x}"
    return bad
