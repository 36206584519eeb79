"""The GEMM wait accounting of the diagnostic build (-DMOE_GEMM_WAIT_STATS).

A child process runs the block through the diagnostic library with the counters enabled; its outputs
must be bitwise those of the library, and its counters must describe the GEMMs that ran (CTAs,
lifetimes, waits no longer than the lifetimes, K blocks).
"""
import hashlib
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from synth import inputs as S
from gpu_util import DevInputs, lib_api, need_gpu, run_block

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUTPUTS = ("topk_idx", "gates", "Y_bits", "dX_bits", "dWr", "dWg", "dWu", "dWd", "dgates")

CHILD = r"""
import ctypes, hashlib, json, sys
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import top_softmax_router_gb300.build as B
from top_softmax_router_gb300 import _lib
B.build(wait_stats=True)
_lib.LIB_PATH = B.WAIT_STATS_LIB
from synth import inputs as S
from gpu_util import DevInputs, lib_api, run_block
M = lib_api()
L = _lib.load()
n = _lib.MOE_GEMM_WAIT_CLASSES * _lib.MOE_GEMM_WAIT_FIELDS
buf = (ctypes.c_uint64 * n)()
assert L.moe_diag_gemm_wait_stats(None, 1) == 0
w = S.WORKLOADS["tiny"]
got = run_block(M, w, DevInputs(S.make(w)))
assert L.moe_diag_gemm_wait_stats(buf, 1) == 0
print(json.dumps({"digests": {k: hashlib.sha256(got[k].tobytes()).hexdigest() for k in sys.argv[2:]},
                  "counters": list(buf)}))
"""


def test_wait_accounting_counts_without_changing_results():
    need_gpu()
    M = lib_api()
    w = S.WORKLOADS["tiny"]
    ref = run_block(M, w, DevInputs(S.make(w)))
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, *OUTPUTS], capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    child = json.loads(r.stdout.strip().splitlines()[-1])
    for k in OUTPUTS:
        assert child["digests"][k] == hashlib.sha256(ref[k].tobytes()).hexdigest(), k
    from top_softmax_router_gb300 import _lib
    c = np.array(child["counters"], dtype=np.float64).reshape(_lib.MOE_GEMM_WAIT_CLASSES, _lib.MOE_GEMM_WAIT_FIELDS)
    ctas, life, operands, accum, stage, kblocks = (c[:, i] for i in range(6))
    # one-CTA classes of the tiny block: gate/up + SwiGLU (0), recompute (2), down (4), dX (5), dActU (6),
    # weight gradients (8)
    for cls in (0, 2, 4, 5, 6, 8):
        assert ctas[cls] > 0 and life[cls] > 0 and kblocks[cls] > 0, cls
    assert np.all(operands <= life) and np.all(accum <= life)
    assert np.all((ctas > 0) | (life == 0))
