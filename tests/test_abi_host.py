"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/*.h declares, validates arguments and sizes its workspace
from the shape alone."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import top_softmax_router_gb300.build as B
    B.build()
    from top_softmax_router_gb300 import _lib
    return _lib


def declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    L = lib.load()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing
    assert sorted(lib.EXPORTS) == names


def test_workspace_depends_on_shape_only(lib):
    import top_softmax_router_gb300 as M
    a = M.workspace_bytes(M.Config(16384, 2048, 64, 8, 1408, 2048, 8))
    b = M.workspace_bytes(M.Config(16384, 2048, 64, 8, 1408, 2048, 8))
    assert a == b and min(a) > 0
    # the routed H-wide buffers fit the 2 k c_eff H b bound
    r, f, bw = a
    K, c_eff = M.chunk_plan(M.Config(16384, 2048, 64, 8, 1408, 2048, 8))
    assert (K, c_eff) == (8, 2048)
    bound = 2 * 8 * c_eff * 2048 * 2
    inter = 3 * 8 * c_eff * 1408 * 2
    assert bw <= bound + inter + 64 * 1024 * 1024


def test_chunk_plan_matches_oracle_golden(lib):
    import json
    import top_softmax_router_gb300 as M
    from oracle import moe_ref as O
    cases = json.load(open(os.path.join(ROOT, "tests", "golden", "chunk_plan.json")))["cases"]
    for c in cases:
        got = M.chunk_plan(M.Config(c["N"], 64, 4, 2, 64, c["c"], c["K_max"]))
        assert got == (c["K"], c["c_eff"]) == O.chunk_plan(c["N"], c["c"], c["K_max"])


@pytest.mark.parametrize("cfg,code", [
    ((16, 65, 4, 2, 64, 8, 2), -2),      # H not a multiple of 64
    ((16, 64, 4, 2, 96, 8, 2), -2),      # I not a multiple of 64
    ((16, 64, 4, 5, 64, 8, 2), -2),      # k > E
    ((16, 64, 2048, 2, 64, 8, 2), -2),   # E > 1024
    ((16, 64, 64, 33, 64, 8, 2), -2),    # k > 32
    ((-1, 64, 4, 2, 64, 8, 2), -1),      # negative N
    ((16, 64, 4, 2, 64, 0, 2), -1),      # c = 0
    ((16, 64, 4, 2, 64, 8, 0), -1),      # K_max = 0
])
def test_shape_validation(lib, cfg, code):
    import ctypes
    L = lib.load()
    c = lib.MoeConfig(*cfg)
    r = ctypes.c_size_t()
    assert L.moe_workspace_bytes(ctypes.byref(c), ctypes.byref(r), None, None) == code
    assert L.moe_strerror(code)


def test_null_and_small_workspace_rejected_before_any_launch(lib):
    import ctypes
    L = lib.load()
    c = lib.MoeConfig(16, 64, 4, 2, 64, 8, 2)
    fake = ctypes.c_void_p(4096)          # never dereferenced: the checks fail first
    assert L.moe_forward(ctypes.byref(c), None, None, None, None, None, None, None, fake, 1 << 20, None) == -1
    assert L.moe_forward(ctypes.byref(c), fake, fake, fake, fake, fake, fake, fake, fake, 16, None) == -3
    assert L.moe_route(ctypes.byref(c), fake, fake, None, fake, fake, None, 1 << 20, None) == -1
    mis = ctypes.c_void_p(4096 + 4)       # misaligned
    assert L.moe_route(ctypes.byref(c), mis, fake, None, fake, fake, fake, 1 << 20, None) == -1
    assert L.moe_diag_wait_timeout(0, fake, 4096, None) == -1


def test_wait_accounting_is_absent_from_the_library(lib):
    """The GEMMs' wait accounting exists only in the diagnostic build: the library reports it as not built,
    without touching the device."""
    import ctypes
    L = lib.load()
    buf = (ctypes.c_uint64 * (lib.MOE_GEMM_WAIT_CLASSES * lib.MOE_GEMM_WAIT_FIELDS))()
    assert L.moe_diag_gemm_wait_stats(buf, 1) == lib.MOE_ERR_NOT_BUILT
    assert b"built without" in L.moe_strerror(lib.MOE_ERR_NOT_BUILT)


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    from top_softmax_router_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def test_binding_imports_no_oracle():
    """The product package never imports the oracle."""
    import subprocess
    import sys
    code = ("import sys, top_softmax_router_gb300, top_softmax_router_gb300.api, top_softmax_router_gb300.build;"
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, check=True)
    assert out.stdout.strip() == "False"


def test_adamw_staging_bytes(lib):
    """Staging of the offloaded optimizer step: slots x 3 fp32 arrays of `bucket` parameters, each rounded
    up to 256 bytes (eq. (5), M_stage = O(s beta)); bad bucket or slot counts are argument errors."""
    import top_softmax_router_gb300 as M
    assert M.adamw_staging_bytes(1 << 23, 4) == 4 * 3 * (1 << 25)
    assert M.adamw_staging_bytes(4, 1) == 3 * 256
    assert M.adamw_staging_bytes(100, 16) == 16 * 3 * 512
    for bucket, slots in [(0, 1), (6, 1), (2, 1), (64, 0), (64, 17), (-4, 2)]:
        with pytest.raises(lib.MoeError) as e:
            M.adamw_staging_bytes(bucket, slots)
        assert e.value.code == lib.MOE_ERR_INVALID_ARG


def test_ce_workspace_and_argument_checks(lib):
    """Vocabulary head (no GPU work): workspace sizes follow the shape (the backward's strip of d is
    N x ceil(ceil(V/P)/256)*256 bf16), bad shapes and arguments are rejected before any launch."""
    import ctypes
    import top_softmax_router_gb300 as M
    f, b = M.ce_workspace_bytes(M.CEConfig(16384, 7168, 200_000, 8))
    strip = 16384 * 25_088 * 2
    assert strip <= b <= strip + 16384 * 7168 * 4 + (1 << 20)   # d strip + fp32 dX accumulator + lists
    pairs = 16384 * 782 * 8
    assert pairs <= f <= pairs + (1 << 20)
    for cfg in [(16, 65, 100, 2), (16, 64, 0, 1), (16, 64, 10, 11), (16, 64, 10, 0)]:
        with pytest.raises(lib.MoeError) as e:
            M.ce_workspace_bytes(M.CEConfig(*cfg))
        assert e.value.code == lib.MOE_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(lib.MoeError) as e:
        M.ce_workspace_bytes(M.CEConfig(-1, 64, 10, 1))
    assert e.value.code == lib.MOE_ERR_INVALID_ARG
    L = lib.load()
    c = lib.CeConfig(16, 64, 100, 2)
    assert L.moe_ce_forward(ctypes.byref(c), None, None, None, None, None, None, None, 0, None) == \
        lib.MOE_ERR_INVALID_ARG
    assert L.moe_ce_backward(ctypes.byref(c), None, None, None, None, None, None, None, None, 0, None) == \
        lib.MOE_ERR_INVALID_ARG


def test_adamw_hparam_checks(lib):
    """Bad hyper-parameters are rejected before any CUDA call."""
    import ctypes
    L = lib.load()
    for hp in [dict(step=0), dict(beta1=1.0), dict(beta2=-0.1), dict(eps=-1.0), dict(lr=float("nan"))]:
        base = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1)
        base.update(hp)
        h = lib.AdamwHparams(base["lr"], base["beta1"], base["beta2"], base["eps"], base["weight_decay"],
                             base["step"])
        assert L.moe_adamw_step(ctypes.byref(h), 16, None, None, None, None, 0, None, None) == \
            lib.MOE_ERR_INVALID_ARG, hp


def test_launch_chaining_modes(lib):
    L = lib.load()
    for mode in (lib.MOE_CHAIN_NONE, lib.MOE_CHAIN_EARLY, lib.MOE_CHAIN_LATE):
        assert L.moe_set_launch_chaining(mode) == 0
    assert L.moe_set_launch_chaining(3) == -1
    assert L.moe_set_launch_chaining(-1) == -1
    assert L.moe_set_launch_chaining(lib.MOE_CHAIN_LATE) == 0   # leave the default in place


@pytest.mark.parametrize("shape", [(16384, 2048, 64, 8, 1408, 2048, 8), (32768, 7168, 384, 8, 2048, 2048, 16),
                                   (16384, 4096, 896, 16, 1024, 1024, 16), (100, 64, 10, 3, 64, 10, 4)])
def test_hop_worst_case_rows_and_workspace(lib, shape):
    """A hop of the expert-partition schedule holds at most ceil(E/P) experts, so at most
    N * min(k, ceil(E/P)) routes (one per token and expert); the workspace grows with the hop capacity."""
    import top_softmax_router_gb300 as M
    cfg = M.Config(*shape)
    N, _, E, k = shape[:4]
    for P in (1, 2, 3, 8, E):
        if P > E:
            continue
        rows = M.hop_rows_worst_case(cfg, P)
        assert rows == N * min(k, -(-E // P)), P
        f1, b1 = M.hops_workspace_bytes(cfg, P, max(1, rows // 2))
        f2, b2 = M.hops_workspace_bytes(cfg, P, rows)
        assert 0 < f1 <= f2 and 0 < b1 <= b2


def test_hop_argument_checks(lib):
    import top_softmax_router_gb300 as M
    from top_softmax_router_gb300._lib import MoeError
    cfg = M.Config(1000, 64, 8, 2, 64, 100, 4)
    for P in (0, 9):
        with pytest.raises(MoeError):
            M.hop_rows_worst_case(cfg, P)
    with pytest.raises(MoeError):
        M.hops_workspace_bytes(cfg, 4, 1000 * 2 + 1)     # more rows than N * k routes exist
    with pytest.raises(MoeError):
        M.hops_workspace_bytes(cfg, 4, 0)


def test_dispatch_mode_sets_the_workspace_layout(lib):
    """moe_set_dispatch: the gather dispatch keeps Xp and dYp (two k c_eff H bf16 buffers per pass), the
    gather-on-load dispatch drops them; the workspace sizes follow the mode, by exactly one k c_eff H b
    buffer in each pass (two in the hop schedule's backward: Xp and dYp); other values are rejected."""
    import top_softmax_router_gb300 as M
    L = lib.load()
    cfg = M.Config(16384, 2048, 64, 8, 1408, 2048, 8)
    K, c_eff = M.chunk_plan(cfg)
    buf = 8 * c_eff * 2048 * 2
    try:
        M.set_dispatch("gather")
        r0, f0, b0 = M.workspace_bytes(cfg)
        hf0, hb0 = M.hops_workspace_bytes(cfg, 8, 30000)
        M.set_dispatch("on_load")
        r1, f1, b1 = M.workspace_bytes(cfg)
        hf1, hb1 = M.hops_workspace_bytes(cfg, 8, 30000)
    finally:
        M.set_dispatch("gather")
    assert r1 == r0
    assert f0 - f1 == buf and b0 - b1 == buf
    assert hf0 - hf1 == 30000 * 2048 * 2 and hb0 - hb1 == 30000 * 2048 * 2
    for bad in (-1, 2, 7):
        assert L.moe_set_dispatch(bad) == lib.MOE_ERR_INVALID_ARG
