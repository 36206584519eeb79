"""CPU oracle of the offloaded optimizer step (OffloadStreamAdamW).  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import or run
it.  It shares no code with the CUDA path.

"bounded-streaming operators" summary, Methodology 4 (OffloadStreamAdamW), eq. (5): the fp32
optimizer state lives on the host; buckets of at most beta parameters are copied to the device,
updated by a fused AdamW step that also refreshes the bf16 working weights, and copied back.
The bucketing changes only the order of independent elementwise updates, so the oracle is the
plain AdamW step over the whole parameter vector, in float64.

Reading (the pages name AdamW but print no formula): AdamW with decoupled weight decay
(Loshchilov and Hutter, "Decoupled Weight Decay Regularization", 2019), in the form
  p <- p (1 - lr wd)
  m <- b1 m + (1 - b1) g ;  v <- b2 v + (1 - b2) g^2
  p <- p - (lr / (1 - b1^t)) m / (sqrt(v) / sqrt(1 - b2^t) + eps)
with step count t >= 1, and the bf16 working weight = round-to-nearest-even(p).
"""
from __future__ import annotations

import numpy as np


def adamw_step(p, m, v, g, *, lr, beta1, beta2, eps, weight_decay, step):
    """One AdamW step in float64; returns new (p, m, v)."""
    p = np.asarray(p, np.float64)
    m = np.asarray(m, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    p = p * (1.0 - lr * weight_decay)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    p = p - (lr / bc1) * m / (np.sqrt(v) / np.sqrt(bc2) + eps)
    return p, m, v


def stream_floor_bytes(n_params: int) -> int:
    """Host-link round trip of the fp32 state: master, m and v, 12 bytes per parameter each way."""
    return 12 * n_params
