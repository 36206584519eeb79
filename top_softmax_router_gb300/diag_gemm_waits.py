"""Where the expert GEMMs wait: a diagnostic run of one workload's step on the wait-accounting build.

    python -m top_softmax_router_gb300.diag_gemm_waits mid [auto|single|pair]

Builds ``_build_wait_stats/libmoe.so`` (the library with -DMOE_GEMM_WAIT_STATS) when it is missing, runs three
route + forward + backward steps of the named synthetic workload (after three warm-up steps) through it,
and prints, per GEMM class, the shares of the MMA warp's lifetime spent waiting for operands and for a free
accumulator, the share of it the producer spent waiting for a free stage, and the cycles per 64-deep K
block.  The counters slow the kernels down, so the table attributes waits; it does not time anything.
"""
from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

CLASS_NAMES = {0: "gate/up + SwiGLU", 1: "gate/up recompute", 2: "down", 3: "dX", 4: "dActU (+ epilogue)"}
WEIGHT_GRAD = 8          # epilogue 4 (weight gradients) * 2
FIELDS = 8


def _class_name(c: int) -> str:
    form, rest = divmod(c, 16)
    epi, two_phase = divmod(rest, 2)
    if rest == WEIGHT_GRAD:
        name = "weight gradients"
    else:
        name = {0: CLASS_NAMES[0], 1: CLASS_NAMES[1], 2: CLASS_NAMES[3] if two_phase else CLASS_NAMES[2],
                3: CLASS_NAMES[4]}.get(epi, f"epilogue {epi}")
    return f"{'CTA pair' if form else 'one CTA':8s} {name}"


def main(argv: list[str]) -> None:
    name = argv[0] if argv else "mid"
    form = argv[1] if len(argv) > 1 else "auto"
    from . import build as B
    from . import _lib
    if not os.path.exists(B.WAIT_STATS_LIB):
        B.build(wait_stats=True)
    _lib.LIB_PATH = B.WAIT_STATS_LIB
    import torch
    from . import api as M
    from synth import inputs as S

    w = S.WORKLOADS[name]
    T = S.make(w)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    X, dY, Wg, Wu, Wd = dev(T.X), dev(T.dY), dev(T.Wg), dev(T.Wu), dev(T.Wd)
    Wr = torch.from_numpy(T.Wr).cuda()
    bias = None if T.bias is None else torch.from_numpy(T.bias).cuda()
    M.set_gemm_form(form)
    try:
        blk = M.MoEBlock(M.Config(**w.cfg()))

        def step():
            idx, g = blk.route(X, Wr, bias)
            blk.forward(X, idx, g, Wg, Wu, Wd)
            blk.backward(X, Wr, idx, g, Wg, Wu, Wd, dY)

        lib = _lib.load()
        counters = (ctypes.c_uint64 * (_lib.MOE_GEMM_WAIT_CLASSES * FIELDS))()
        for _ in range(3):
            step()
        M.check(lib.moe_diag_gemm_wait_stats(None, 1), "moe_diag_gemm_wait_stats")   # enable and zero
        steps = 3
        for _ in range(steps):
            step()
        M.check(lib.moe_diag_gemm_wait_stats(counters, 1), "moe_diag_gemm_wait_stats")
        blk.check()
    finally:
        M.set_gemm_form("auto")
    a = np.array(counters[:], dtype=np.float64).reshape(-1, FIELDS)
    print(f"{name}, GEMM form {form}: {steps} steps; shares of the MMA warp's lifetime (SM cycles)")
    print(f"  {'class':28s} {'CTAs':>7s} {'life/CTA us':>11s} {'MMA: operands':>13s} {'accumulator':>11s} "
          f"{'producer: stage':>15s} {'cycles/K block':>14s}")
    for c in range(a.shape[0]):
        n, life, opnd, accu, stage, kb = a[c, :6]
        if n == 0 or life == 0:
            continue
        print(f"  {_class_name(c):28s} {int(n):7d} {life / n / 2.07e3:11.1f} {100 * opnd / life:12.1f}% "
              f"{100 * accu / life:10.1f}% {100 * stage / life:14.1f}% {life / max(kb, 1):14.0f}")


if __name__ == "__main__":
    main(sys.argv[1:])
