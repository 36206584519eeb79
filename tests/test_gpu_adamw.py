"""GPU parity of the offloaded AdamW step (OffloadStreamAdamW, "bounded-streaming operators" summary,
Methodology 4, eq. (5)) against the float64 oracle, through the C ABI of include/moe_adamw.h.

  * every element of p, m, v within the fp32 error bound of tests/adam_check.py, and every bf16
    working weight equal to the rounding of the oracle's p where that rounding is unambiguous;
  * every (bucket, slots) choice, the host-direct kernel and the device-resident kernel give the same
    bits (the bucketing only reorders independent elementwise updates);
  * edge cases (n = 0, n < 4, ragged tails, bucket > n, one slot, bf16 gradients) and argument errors.
"""
import numpy as np
import pytest
import torch

import adam_check as C
from gpu_util import bf16_host, need_gpu, lib_api
from oracle import adamw_ref as A
from synth import inputs as S

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


@pytest.fixture(scope="module")
def M():
    need_gpu()
    return lib_api()


def hparams(M):
    return M.AdamWHparams(**HP)


def pinned(a: np.ndarray) -> torch.Tensor:
    t = torch.empty(a.size, dtype=torch.float32, pin_memory=True)
    t.copy_(torch.from_numpy(np.ascontiguousarray(a, np.float32)))
    return t


def grad_dev(g: np.ndarray, dtype=torch.float32) -> torch.Tensor:
    return torch.from_numpy(g).to("cuda").to(dtype)


def run_offload(M, st, step, bucket, slots, grad_dtype=torch.float32):
    n = st.p.size
    P, Mm, V = pinned(st.p), pinned(st.m), pinned(st.v)
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    staging = torch.empty(M.adamw_staging_bytes(bucket, slots), dtype=torch.uint8, device="cuda")
    M.adamw_offload_step(hparams(M), step, P, Mm, V, grad_dev(st.g, grad_dtype), W, staging, bucket, slots)
    torch.cuda.synchronize()
    return P.numpy().copy(), Mm.numpy().copy(), V.numpy().copy(), bf16_host(W)


def run_resident(M, st, step, host=False, grad_dtype=torch.float32):
    n = st.p.size
    if host:
        P, Mm, V = pinned(st.p), pinned(st.m), pinned(st.v)
    else:
        P, Mm, V = (torch.from_numpy(a).cuda() for a in (st.p, st.m, st.v))
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    M.adamw_step(hparams(M), step, P, Mm, V, grad_dev(st.g, grad_dtype), W)
    torch.cuda.synchronize()
    return P.cpu().numpy(), Mm.cpu().numpy(), V.cpu().numpy(), bf16_host(W)


def oracle_check(st, got, step, g=None):
    g = st.g if g is None else g
    ref = A.adamw_step(st.p, st.m, st.v, g, step=step, **HP)
    tol = C.bounds(st.p, st.m, st.v, g, step=step, **HP)
    bad = C.compare(got, ref, tol)
    assert not bad, bad


@pytest.mark.parametrize("n,bucket,slots,step", [
    (1_000_003, 65_536, 3, 7),     # 16 buckets, ragged last bucket, n mod 4 = 3
    (262_144, 65_536, 4, 1),       # exact buckets, slots = buckets
    (100_001, 4_096, 1, 2),        # one slot: copy, update and write-back serialised
    (5_000, 1 << 20, 2, 3),        # bucket larger than n
])
def test_offload_step_matches_oracle(M, n, bucket, slots, step):
    st = S.adam_state(n, seed=n)
    oracle_check(st, run_offload(M, st, step, bucket, slots), step)


def test_fresh_state_first_step(M):
    st = S.adam_state(50_000, seed=3, fresh=True)
    oracle_check(st, run_offload(M, st, 1, 8_192, 3), 1)


def test_bf16_gradients(M):
    st = S.adam_state(300_007, seed=11)
    g16 = S.bf16_to_f32(S.f32_to_bf16(st.g))      # the gradient the kernel sees, widened exactly
    got = run_offload(M, st, 4, 32_768, 3, grad_dtype=torch.bfloat16)
    oracle_check(st, got, 4, g=g16)


def test_every_schedule_gives_the_same_bits(M):
    st = S.adam_state(100_003, seed=21)
    base = run_resident(M, st, 5)
    oracle_check(st, base, 5)
    runs = {"host_direct": run_resident(M, st, 5, host=True)}
    for bucket, slots in [(4_096, 1), (4_096, 2), (65_536, 4), (12_500, 16), (1 << 20, 3)]:
        runs[f"offload_{bucket}x{slots}"] = run_offload(M, st, 5, bucket, slots)
    for name, got in runs.items():
        for a, b, what in zip(got, base, ("p", "m", "v", "w")):
            assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  b.view(np.uint32) if b.dtype == np.float32 else b), (name, what)


def test_tiny_buckets(M):
    st = S.adam_state(1_001, seed=8)
    oracle_check(st, run_offload(M, st, 2, 8, 3), 2)


@pytest.mark.parametrize("n", [1, 3, 4, 5, 7])
def test_small_and_ragged_sizes(M, n):
    st = S.adam_state(n, seed=40 + n)
    oracle_check(st, run_offload(M, st, 3, 4, 2), 3)
    oracle_check(st, run_resident(M, st, 3), 3)


def test_empty_is_a_no_op(M):
    e = torch.empty(0, dtype=torch.float32, pin_memory=True)
    W = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    g = torch.empty(0, dtype=torch.float32, device="cuda")
    staging = torch.empty(M.adamw_staging_bytes(64, 2), dtype=torch.uint8, device="cuda")
    M.adamw_offload_step(hparams(M), 1, e, e, e, g, W, staging, 64, 2)
    M.adamw_step(hparams(M), 1, e, e, e, g, W)
    torch.cuda.synchronize()


def test_three_steps_through_the_optimizer_object(M):
    """State carried across steps in host memory; each step's gradient drawn from its own seed."""
    n = 200_003
    st = S.adam_state(n, seed=2, fresh=True)
    opt = M.OffloadStreamAdamW(torch.from_numpy(st.p), bucket=16_384, slots=3, hp=hparams(M))
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    p, m, v = st.p.astype(np.float64), np.zeros(n), np.zeros(n)
    for t in (1, 2, 3):
        g = S.adam_state(n, seed=100 + t).g
        prev = (opt.master.numpy().copy(), opt.exp_avg.numpy().copy(), opt.exp_avg_sq.numpy().copy())
        opt.step(grad_dev(g), W)
        torch.cuda.synchronize()
        got = (opt.master.numpy(), opt.exp_avg.numpy(), opt.exp_avg_sq.numpy(), bf16_host(W))
        # this step against the oracle, from the state the previous step left
        ref = A.adamw_step(*prev, g, step=t, **HP)
        bad = C.compare(got, ref, C.bounds(*prev, g, step=t, **HP))
        assert not bad, (t, bad)
        p, m, v = A.adamw_step(p, m, v, g, step=t, **HP)
    # and the three steps end close to three float64 steps from the start
    assert np.max(np.abs(opt.master.numpy() - p)) <= 1e-6 * np.max(np.abs(p))


def test_argument_errors(M):
    import ctypes
    from top_softmax_router_gb300 import _lib
    n = 1024
    st = S.adam_state(n, seed=1)
    P, Mm, V = pinned(st.p), pinned(st.m), pinned(st.v)
    G = grad_dev(st.g)
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    staging = torch.empty(M.adamw_staging_bytes(256, 2), dtype=torch.uint8, device="cuda")
    hp = hparams(M)
    L = _lib.load()
    h = hp.c_struct(1)

    def raw(p=P, m=Mm, v=V, g=G, w=W, bucket=256, slots=2, sbytes=None, step=1, n_=n):
        hh = hp.c_struct(step)
        return L.moe_adamw_offload_step(ctypes.byref(hh), n_, bucket, slots, p.data_ptr(), m.data_ptr(),
                                        v.data_ptr(), g.data_ptr(), 0, w.data_ptr(), staging.data_ptr(),
                                        staging.numel() if sbytes is None else sbytes, None)

    assert raw() == 0
    torch.cuda.synchronize()
    pageable = torch.from_numpy(st.p.copy())
    assert raw(p=pageable) == -1                       # pageable host state
    assert raw(p=torch.from_numpy(st.p).cuda()) == -1  # device memory passed as host state
    assert raw(bucket=254) == -1                       # bucket not a multiple of 4
    assert raw(slots=0) == -1 and raw(slots=17) == -1
    assert raw(sbytes=staging.numel() - 1) == -3       # staging too small
    assert raw(step=0) == -1
    assert L.moe_adamw_offload_step(ctypes.byref(h), n - 1, 256, 2, P.data_ptr() + 4, Mm.data_ptr(),
                                    V.data_ptr(), G.data_ptr(), 0, W.data_ptr(), staging.data_ptr(),
                                    staging.numel(), None) == -1   # misaligned master
    assert L.moe_adamw_step(ctypes.byref(h), n, pageable.data_ptr(), Mm.data_ptr(), V.data_ptr(),
                            G.data_ptr(), 0, W.data_ptr(), None) == -1
    assert L.moe_adamw_step(ctypes.byref(h), n, P.data_ptr(), Mm.data_ptr(), V.data_ptr(),
                            G.data_ptr(), 7, W.data_ptr(), None) == -1   # bad grad dtype
    bad_hp = M.AdamWHparams(lr=1e-3, beta1=1.0).c_struct(1)
    assert L.moe_adamw_step(ctypes.byref(bad_hp), n, P.data_ptr(), Mm.data_ptr(), V.data_ptr(),
                            G.data_ptr(), 0, W.data_ptr(), None) == -1
    with pytest.raises(ValueError):
        M.adamw_offload_step(hp, 1, pageable, Mm, V, G, W, staging, 256, 2)
    torch.cuda.synchronize()


def test_full_size_block_parameters(M):
    """The optimizer step over every parameter of the 16,384-token, H = 2,048, E = 64, I = 1,408 block
    (553,779,200 parameters) with the schedule the benchmark times: sampled windows against the oracle
    (bucket edges, the tail, random places) and every element bitwise against the device-resident kernel."""
    w = S.WORKLOADS["mid"]
    n = S.block_parameter_count(w)
    bucket, slots = 1 << 23, 4
    st = S.adam_state(n, seed=77)
    P, Mm, V = pinned(st.p), pinned(st.m), pinned(st.v)
    Pd, Md, Vd = (torch.from_numpy(a).cuda() for a in (st.p, st.m, st.v))
    G = grad_dev(st.g)
    del st
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    staging = torch.empty(M.adamw_staging_bytes(bucket, slots), dtype=torch.uint8, device="cuda")
    M.adamw_offload_step(hparams(M), 9, P, Mm, V, G, W, staging, bucket, slots)
    torch.cuda.synchronize()
    Wh = bf16_host(W)
    rng = np.random.default_rng(5)
    starts = [0, n - 4099] + [b * bucket - 7 for b in range(1, (n + bucket - 1) // bucket)] + \
        list(rng.integers(0, n - 4096, size=32))
    for s0 in starts:
        s0 = int(max(0, min(s0, n - 4096)))
        win = S.adam_state(4096, seed=77, offset=s0)
        sl = slice(s0, s0 + 4096)
        got = (P.numpy()[sl], Mm.numpy()[sl], V.numpy()[sl], Wh[sl])
        oracle_check(win, got, 9)
    # bitwise against the device-resident kernel on the same inputs
    Wd = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    M.adamw_step(hparams(M), 9, Pd, Md, Vd, G, Wd)
    torch.cuda.synchronize()
    for host, dev in ((P, Pd), (Mm, Md), (V, Vd)):
        assert torch.equal(host.view(torch.int32), dev.cpu().view(torch.int32))
    assert torch.equal(W.view(torch.int16), Wd.view(torch.int16))
