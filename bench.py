"""Benchmark of the chunk-bounded MoE block: route + forward + backward per step.

Default workload (the largest single-GPU configuration): N=32768 tokens,
H=7168, E=384 experts, top-8, SwiGLU width I=2048, token budget c=2048,
K_max=16 (K=16 chunks of 2048 tokens), near-uniform router (no bias), seed 0
-- synthetic bf16 data on one GPU.

Metric: routed token*k pairs per second through route + forward + backward.
Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a deliberately slow baseline, not the target).

Timing: W untimed warm-up steps, then K steps between CUDA events on the
launching stream, bracketed by a barrier and torch.cuda.synchronize().  The
expert weights (33.8 GB for the default workload) exceed the 129 MB L2, so
every step streams them from HBM; no extra L2 flush is done.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import inputs as S  # noqa: E402

# fp32 SIMT peak for the router's fused multiply-add chains: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz
# (the maximum SM clock); the kernels the driver measures peaks for are copies and bf16 GEMMs.
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
METRIC = "routed token*k pairs/s fwd+bwd"
UNIT = "pairs/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="many", choices=sorted(S.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time the plain calls instead of a CUDA-graph replay")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-route-tokens", type=int, default=2048,
                    help="tokens of the CPU baseline's routing sample")
    ap.add_argument("--cpu-max-tokens", type=int, default=256,
                    help="most tokens of the CPU baseline's forward+backward sample")
    ap.add_argument("--cpu-weight-budget", type=float, default=4e9,
                    help="bytes of float64 expert weights the CPU baseline widens once per run")
    ap.add_argument("--no-hops", action="store_true", help="skip the expert-partition schedule measurement")
    ap.add_argument("--hops", type=int, default=8, help="expert partitions of the alternative schedule")
    ap.add_argument("--hops-workload", default="mid", choices=sorted(S.WORKLOADS),
                    help="workload of the expert-partition schedule measurement (with the chunk schedule "
                         "timed beside it on the same inputs)")
    ap.add_argument("--no-runs", action="store_true", help="skip the table over every workload")
    ap.add_argument("--runs-steps", type=int, default=5, help="timed steps per workload of that table")
    ap.add_argument("--no-adamw", action="store_true", help="skip the offloaded optimizer step measurement")
    ap.add_argument("--no-unchunked", action="store_true", help="skip the K = 1 comparison of the same block")
    ap.add_argument("--adamw-only", action="store_true",
                    help="run only the offloaded optimizer step measurement and print its JSON object")
    ap.add_argument("--no-ce", action="store_true", help="skip the vocabulary cross-entropy head measurement")
    ap.add_argument("--ce-only", action="store_true",
                    help="run only the vocabulary cross-entropy head measurement and print its JSON object")
    ap.add_argument("--ce-workload", default="ce_full", help="cross-entropy head shape (synth CE_WORKLOADS)")
    ap.add_argument("--adamw-params", type=int, default=0,
                    help="parameters of the optimizer step (default: every parameter of the mid block, "
                         "553.8 M; the largest blocks would need hundreds of GB of page-locked state)")
    return ap.parse_args()


def workload_desc(w: S.Workload) -> str:
    bias = {"none": "no router bias", "zipf": f"router bias with Zipf({w.zipf_s}) popularity",
            "hot+zipf": f"hot expert ({w.hot_token_share:.0%} of tokens) + Zipf({w.zipf_s})"}[w.bias]
    return (f"{w.name}: N={w.N}, H={w.H}, E={w.E}, k={w.k}, I={w.I}, c={w.c}, K_max={w.K_max}, {bias}; "
            f"X,dY~N(0,1) bf16, Wr~N(0,1/H) fp32, Wg,Wu~N(0,1/H), Wd~N(0,1/I) bf16")


# Kernel sources whose ncu DRAM counters (profiles/*.json) stay valid only while these files are unchanged.
PROFILED_SOURCES = ["top_softmax_router_gb300/csrc/gemm_kernel.cuh", "top_softmax_router_gb300/csrc/gemm_dw.cu",
                    "top_softmax_router_gb300/csrc/gemm_fwd.cu", "top_softmax_router_gb300/csrc/gemm_bwd.cu",
                    "top_softmax_router_gb300/csrc/gemm_launch.cuh", "top_softmax_router_gb300/csrc/common.cuh",
                    "top_softmax_router_gb300/csrc/tma.cu"]


def sources_hash(files=None) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files or PROFILED_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from a committed ncu capture, if the kernel is unchanged since
    (the capture names the source files it depends on; the default list is the GEMM sources)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    if not os.path.exists(p):
        return None, None
    d = json.load(open(p))
    if d.get("sources_sha256_16") != sources_hash(d.get("sources")):
        return None, d
    return d.get("dram_bytes_per_launch"), d


def max_over_ranks(ms: float, dist, device) -> float:
    """Slowest rank's time: the whole job is done only when every replica is."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: int, world: int, steps: int, ms: float) -> float:
    """Whole-job units per second: every rank processes its own units (replicas, weak scaling)."""
    return world * units_per_rank_step * steps / (ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# --------------------------------------------------------------------------- #
# algorithmic bytes / flops per kernel class (from the chunk histograms)
# --------------------------------------------------------------------------- #
def algorithmic(w: S.Workload, topk_idx: np.ndarray, K: int, on_load: bool = False):
    """Algorithmic bytes and flops per kernel class for one step.  on_load: the dispatch gather fused into
    the GEMMs (MOE_DISPATCH_ON_LOAD): no gather kernel, and a gathering GEMM reads the chunk's n token rows
    of X or dY once from HBM (their k - 1 further uses hit L2) instead of the R rows of Xp or dYp."""
    H, I, E, k = w.H, w.I, w.E, w.k
    b = 2
    n_dact = 2 * -(-I // 256)          # dgate partial sums per row (two per 256-column tile)
    by = {}
    fl = {}

    def add(name, nbytes, nflops=0.0):
        by[name] = by.get(name, 0.0) + nbytes
        fl[name] = fl.get(name, 0.0) + nflops

    seen = np.zeros(E, dtype=bool)
    for i in range(K - 1, -1, -1):           # backward order decides first touch
        tok = topk_idx[i::K]
        n = tok.shape[0]
        R = n * k
        counts = np.bincount(tok.reshape(-1), minlength=E)
        act = counts > 0
        A = int(act.sum())
        first = act & ~seen
        seen |= act
        nf, nr = int(first.sum()), int((act & ~first).sum())
        rows = n if on_load else R               # rows of X / dY a GEMM reads per use of the operand
        # forward
        if not on_load:
            add("gather", n * H * b + R * H * b)
        add("gemm_gateup", rows * H * b + A * 2 * I * H * b + R * I * b, 4.0 * R * H * I)
        add("gemm_down", R * I * b + A * H * I * b + R * H * b, 2.0 * R * H * I)
        add("combine", R * H * b + n * H * b + R * 8)
        # backward
        if not on_load:
            add("gather", 2 * (n * H * b + R * H * b))
        add("gemm_gateup", rows * H * b + A * 2 * I * H * b + 2 * R * I * b, 4.0 * R * H * I)
        add("gemm_dact", rows * H * b + A * H * I * b + 5 * R * I * b + R * n_dact * 4, 2.0 * R * H * I)
        w_rmw = nf * 4 + nr * 8                 # fp32 weight-gradient bytes per element
        add("gemm_dw", (2 * n if on_load else 3 * R) * H * b + 3 * R * I * b + 3 * H * I * w_rmw, 6.0 * R * H * I)
        # dX adds each row's router-path term dl Wr[e] in its epilogue (one Wr row per active expert)
        add("gemm_dx", 2 * R * I * b + A * 2 * I * H * b + R * H * b + A * H * 4 + R * 4, 4.0 * R * H * I)
        # route grad (dActU partials, gates -> dgates, dlogit, dl per row), then the unpermute sum
        add("route_grad", R * n_dact * 4 + R * 20)
        add("unpermute", R * H * b + n * H * b)
        add("router_dw", n * H * b + A * H * 4 * (1 if nf == A else 2))
    add("router_logits", w.N * H * b + E * H * 4 + w.N * E * 4, 2.0 * w.N * H * E)
    add("router_topk", w.N * E * 4 + w.N * k * 8)
    add("plan", 2 * (w.N * k * 4 * 4))
    add("zero", 3 * H * I * 4 * int((~seen).sum()))
    return by, fl


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# the CPU oracle as a baseline (host cores)
# --------------------------------------------------------------------------- #
class CpuSample:
    """The CPU baseline's seeded samples of one workload, fixed per run, so every timing of the oracle
    (the GPU arm's leg and each step of the reference arm) measures the same work.

    * routing: the first `route_tokens` tokens of a seeded permutation.  Every token's logits are E
      fp32 chains of H fused multiply-adds, so the routing cost per token is fixed.
    * forward + backward: the first tokens of the same permutation, taken in order while the experts
      they select still fit `weight_budget` bytes of float64 weights (at most `max_tokens` tokens).
      Those experts' weights are widened to float64 once, here, outside every timed call; the oracle
      reads them through its callable-weights form.  Without this, each timed call would widen every
      expert it touches, a cost per expert and not per routed pair.
    """

    def __init__(self, w: S.Workload, T: S.Tensors, route_tokens: int, max_tokens: int, weight_budget: float):
        from oracle import moe_ref as O
        self.O, self.w, self.T = O, w, T
        rng = np.random.default_rng(0)
        perm = rng.permutation(w.N)
        self.route_sel = np.sort(perm[:min(route_tokens, w.N)])
        idx, _, _ = O.route(T.X[perm[:min(max_tokens, w.N)]], T.Wr, T.bias, w.k)
        per_expert = 3 * w.H * w.I * 8
        experts, n = {0}, 0          # the oracle's backward reads expert 0's weights for the shape of dW
        for row in idx:
            grown = experts | set(int(e) for e in row)
            if n > 0 and len(grown) * per_expert > weight_budget:
                break
            experts, n = grown, n + 1
        self.fb_sel = np.sort(perm[:n])
        self.fb_idx, self.fb_g, _ = O.route(T.X[self.fb_sel], T.Wr, T.bias, w.k)
        self.experts = sorted(experts)
        self.wide = {e: tuple(O.bf16_to_f64(a[e]) for a in (T.Wg, T.Wu, T.Wd)) for e in self.experts}
        self.cores = len(os.sched_getaffinity(0))

    def time(self):
        """One timing of the oracle on both samples; pairs/s = 1 / (route s/pair + fwd+bwd s/pair)."""
        O, w, T = self.O, self.w, self.T
        t0 = time.perf_counter()
        O.route(T.X[self.route_sel], T.Wr, T.bias, w.k)
        t_route = time.perf_counter() - t0
        sel, idx, g = self.fb_sel, self.fb_idx, self.fb_g
        W = self.wide.__getitem__
        t0 = time.perf_counter()
        O.forward(T.X[sel], idx, g, W)
        O.backward(T.X[sel], T.Wr, idx, g, W, T.dY[sel])
        t_fb = time.perf_counter() - t0
        per_pair = t_route / (len(self.route_sel) * w.k) + t_fb / (len(sel) * w.k)
        return {"value": 1.0 / per_pair, "unit": UNIT, "cores": self.cores, "kind": "oracle",
                "sample": (f"routing of {len(self.route_sel)} seeded tokens ({t_route:.2f} s) + float64 "
                           f"forward+backward of {len(sel)} seeded tokens ({len(sel) * w.k} pairs over "
                           f"{len(self.experts)} experts, {t_fb:.2f} s; their float64 weights widened once "
                           f"per run, outside the timing); pairs/s = 1 / (route s/pair + fwd+bwd s/pair)"),
                "route_s_per_pair": t_route / (len(self.route_sel) * w.k),
                "fwd_bwd_s_per_pair": t_fb / (len(sel) * w.k)}


def cpu_baseline(w: S.Workload, T: S.Tensors, args):
    """Oracle pairs/s on the host cores (one timing of the fixed samples; see CpuSample)."""
    return CpuSample(w, T, args.cpu_route_tokens, args.cpu_max_tokens, args.cpu_weight_budget).time()


def offload_adamw(M, torch, w: S.Workload, peaks, stream, n_params: int = 0):
    """The offloaded AdamW step (OffloadStreamAdamW, eq. (5) of the bounded-streaming summary) over
    n_params parameters (by default every parameter of the mid block, 553.8 M; the larger blocks' fp32
    state would need hundreds of GB of page-locked host memory): fp32 state in page-locked host memory,
    fp32 gradients and bf16 working weights in HBM.  Reports the staged pipeline over a small (bucket, slots) sweep, the single kernel that reads
    the host state directly, the update kernel on HBM-resident state (its HBM roofline), the host-link
    floor measured with plain copies, and the oracle and torch's CPU AdamW on a sample of the host cores."""
    from oracle import adamw_ref as A
    n = n_params or S.block_parameter_count(S.WORKLOADS["mid"])
    hp_d = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    hp = M.AdamWHparams(**hp_d)
    out = {"params": n, "state_bytes_each_way": 12 * n, "grad": "fp32 in HBM", "hparams": hp_d}

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=5, warm=2, trials=1):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        res = []
        for _ in range(trials):
            a, b = ev(), ev()
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            res.append(a.elapsed_time(b) / reps)
        return res

    t = {"step": 0}

    def nxt():
        t["step"] += 1
        return t["step"]

    # ---- seeded state, drawn straight into page-locked buffers
    Ph = torch.empty(n, dtype=torch.float32, pin_memory=True)
    Mh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    Vh = torch.empty(n, dtype=torch.float32, pin_memory=True)
    gh = np.empty(n, np.float32)
    S.adam_state(n, seed=7, out=S.AdamState(Ph.numpy(), Mh.numpy(), Vh.numpy(), gh))
    G = torch.from_numpy(gh).cuda()
    del gh
    W = torch.empty(n, dtype=torch.bfloat16, device="cuda")

    # ---- the update kernel alone on HBM-resident state (first, so a profiler can take its first launch)
    Pd, Md, Vd = Ph.cuda(), Mh.cuda(), Vh.cuda()
    ms = min(timed(lambda: M.adamw_step(hp, nxt(), Pd, Md, Vd, G, W, stream), reps=10, warm=3, trials=3))
    byts = 30 * n
    tr_cap, cap = measured_traffic("adamw_update", "64M")
    out["device_resident"] = {"ms_per_step": ms, "algorithmic_bytes": byts,
                              "achieved_gbs": byts / (ms / 1e3) / 1e9, "peak_gbs": peaks["hbm_gbs"],
                              "frac": byts / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                              "traffic": None if tr_cap is None else tr_cap * n / cap["params"],
                              "traffic_note": None if cap is None else cap.get("note"),
                              "bytes_note": "p, m, v, fp32 g read (16 B) + p, m, v, bf16 w written (14 B) per parameter"}
    del Pd, Md, Vd

    # ---- the host link, measured with plain copies of up to 1 GiB (one way alone, then both ways at once)
    nb = min(n, 1 << 28)
    da, db = torch.empty(nb, device="cuda"), torch.empty(nb, device="cuda")
    hb = torch.empty(nb, dtype=torch.float32, pin_memory=True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def copies(h2d: bool, d2h: bool, reps=3):
        best = None
        for _ in range(reps):
            a, b1, b2 = ev(), ev(), ev()
            torch.cuda.synchronize()
            a.record(stream)
            s1.wait_stream(stream)
            s2.wait_stream(stream)
            if h2d:
                with torch.cuda.stream(s1):
                    da.copy_(Ph[:nb], non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    hb.copy_(db, non_blocking=True)
            b1.record(s1)
            b2.record(s2)
            torch.cuda.synchronize()
            tt = max(a.elapsed_time(b1) if h2d else 0.0, a.elapsed_time(b2) if d2h else 0.0)
            best = tt if best is None else min(best, tt)
        return nb * 4 / (best / 1e3) / 1e9

    h2d, d2h, both = copies(True, False), copies(False, True), copies(True, True)
    out["link"] = {"h2d_gbs": h2d, "d2h_gbs": d2h, "both_ways_gbs_each": both,
                   "method": f"cudaMemcpyAsync of {nb * 4 >> 20} MiB page-locked <-> HBM; best of 3"}
    floor_ms = 12 * n / (both * 1e9) * 1e3
    out["floor_ms"] = floor_ms
    del da, db, hb

    # ---- the staged pipeline of eq. (5) over a (bucket, slots) sweep, then the direct kernel
    sweep = []
    for bucket, slots in [(1 << 20, 2), (1 << 21, 3), (1 << 22, 4), (1 << 23, 4), (1 << 24, 3)]:
        staging = torch.empty(M.adamw_staging_bytes(bucket, slots), dtype=torch.uint8, device="cuda")
        tr = timed(lambda: M.adamw_offload_step(hp, nxt(), Ph, Mh, Vh, G, W, staging, bucket, slots, stream),
                   reps=3, warm=2, trials=3)
        sweep.append({"bucket": bucket, "slots": slots, "ms": statistics.median(tr), "trials_ms": tr,
                      "staging_bytes": staging.numel()})
        del staging
    best = min(sweep, key=lambda r: r["ms"])
    staging = torch.empty(best["staging_bytes"], dtype=torch.uint8, device="cuda")
    M.profile_reset()
    M.profile_enable(True)
    timed(lambda: M.adamw_offload_step(hp, nxt(), Ph, Mh, Vh, G, W, staging, best["bucket"], best["slots"],
                                       stream), reps=2, warm=0)
    M.profile_enable(False)
    upd_n, upd_ms = M.profile_read()["adamw"]
    del staging
    ms = best["ms"]
    out["pipeline"] = {"bucket": best["bucket"], "slots": best["slots"], "ms_per_step": ms,
                       "params_per_s": n / (ms / 1e3), "frac_of_floor": floor_ms / ms,
                       "staging_bytes": best["staging_bytes"],
                       "update_kernel_ms_per_step": upd_ms / 2, "update_launches_per_step": upd_n / 2}
    out["sweep"] = sweep
    tr = timed(lambda: M.adamw_step(hp, nxt(), Ph, Mh, Vh, G, W, stream), reps=3, warm=2, trials=3)
    ms = statistics.median(tr)
    out["host_direct"] = {"ms_per_step": ms, "trials_ms": tr, "params_per_s": n / (ms / 1e3),
                          "frac_of_floor": floor_ms / ms,
                          "note": "one kernel reads and writes the page-locked state across the host link"}
    del G, W

    # ---- host cores: the oracle (float64 numpy) and torch's CPU AdamW (fp32), on a sample
    ns = 1 << 22
    st = S.adam_state(ns, seed=7)
    t0 = time.perf_counter()
    A.adamw_step(st.p, st.m, st.v, st.g, step=3, **hp_d)
    t_or = time.perf_counter() - t0
    prm = torch.nn.Parameter(torch.from_numpy(st.p.copy()))
    opt = torch.optim.AdamW([prm], lr=hp_d["lr"], betas=(hp_d["beta1"], hp_d["beta2"]), eps=hp_d["eps"],
                            weight_decay=hp_d["weight_decay"])
    prm.grad = torch.from_numpy(st.g.copy())
    opt.step()
    t0 = time.perf_counter()
    for _ in range(3):
        opt.step()
    t_tc = (time.perf_counter() - t0) / 3
    out["cpu_baseline"] = {"value": ns / t_or, "unit": "params/s", "cores": 1, "kind": "oracle",
                           "sample": f"float64 numpy AdamW step over {ns} seeded parameters ({t_or:.2f} s)"}
    out["cpu_torch_adamw"] = {"value": ns / t_tc, "unit": "params/s", "cores": torch.get_num_threads(),
                              "sample": f"torch.optim.AdamW fp32 step on the host over {ns} parameters",
                              "step_ms_at_full_size": n / (ns / t_tc) * 1e3}
    return out


def vocab_ce(M, torch, peaks, stream, name: str = "ce_full", steps: int = 3, warmup: int = 2):
    """The vocabulary-projection cross-entropy head (Ring-DTP's single-device form, eqs. (2)-(3) of the
    bounded-streaming summary): one forward + backward step, timed with CUDA events, its kernels timed
    by the library's profiler, against the bf16 tensor peak; the oracle on a few tokens for scale."""
    from oracle import ce_ref as C
    w = S.CE_WORKLOADS[name]
    N, H, V, P = w.N, w.H, w.V, w.P
    cfg = M.CEConfig(N, H, V, P)
    ce = M.VocabCE(cfg)
    # the synth recipe's distributions, drawn on the device by torch's seeded generator (the values do
    # not change the work; the parity tests use the counter-based host generator)
    gen = torch.Generator(device="cuda").manual_seed(11)
    X = torch.randn(N, H, device="cuda", generator=gen).to(torch.bfloat16)
    W = (torch.randn(V, H, device="cuda", generator=gen) / H ** 0.5).to(torch.bfloat16)
    t = torch.randint(0, V, (N,), device="cuda", generator=gen, dtype=torch.int32)
    g = torch.full((N,), 1.0 / N, device="cuda")
    loss = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    mean = torch.empty(1, device="cuda")
    dX = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, H, device="cuda")

    def step():
        M.ce_forward(cfg, X, W, t, loss, lse, mean, ce.ws, stream)
        n = M.ce_last_stats()["kernel_launches"]
        M.ce_backward(cfg, X, W, t, lse, g, dX, dW, ce.ws, stream)
        st = M.ce_last_stats()
        return n + st["kernel_launches"], st

    for _ in range(warmup):
        step()
    ce.check(stream)
    # the step time without the profiler (whose events between kernels would serialise them) ...
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    launches = 0
    for _ in range(steps):
        n, st = step()
        launches += n
    b.record(stream)
    torch.cuda.synchronize()
    ce.check(stream)
    ms = a.elapsed_time(b) / steps
    # ... and the split by kernel class from a second, profiled pass
    M.profile_reset()
    M.profile_enable(True)
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    M.profile_enable(False)
    prof = M.profile_read()
    ce.check(stream)
    flops = 8.0 * N * H * V      # forward logits, backward recompute, dX, dW: 2 N H V each
    peak = peaks["bf16_tflops_sustained"]
    kern = {}
    for k, per in (("ce_logits", 2.0), ("ce_dlogit", 2.0), ("ce_dx", 2.0), ("ce_dw", 2.0), ("ce_merge", 0.0)):
        n_l, tot = prof.get(k, (0, 0.0))
        if n_l:
            tf = per * N * H * V * steps / (tot / 1e3) / 1e12 if per else None
            kern[k] = {"launches_per_step": n_l / steps, "ms_per_step": tot / steps, "tflops": tf,
                       "frac_of_bf16_peak": None if tf is None else tf / peak}
    # the oracle on the host cores: two tokens' loss, lse and dX row
    t0 = time.perf_counter()
    Wh = W[:, :].float().cpu().numpy()
    Xh = X[:2].float().cpu().numpy()
    t_copy = time.perf_counter() - t0
    t0 = time.perf_counter()
    C.rows_forward_backward(Xh, Wh, t[:2].cpu().numpy(), np.full(2, 1.0 / N))
    t_or = time.perf_counter() - t0
    return {
        "source": "bounded-streaming summary, Methodology 2 (Ring-DTP), eqs. (2)-(3), on one device",
        "workload": f"{name}: N={N} tokens, H={H}, V={V}, P={P} strips; X ~ N(0,1), W ~ N(0,1/H) bf16, "
                    "uniform targets",
        "ms_per_step": ms, "tokens_per_s": N / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
        "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / peak, "peak_tflops": peak,
        "peak_source": f"{peaks['source']} bf16 sustained", "flops_per_step": flops,
        "kernels": kern, "gpu_launches_per_step": launches / steps,
        "strip_bytes": st["strip_bytes"], "strip_bound_bytes_NVb_over_P": st["strip_bound_bytes"],
        "full_logits_bytes_fp32": N * V * 4,
        "cpu_baseline": {"value": 2 / t_or, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                         "kind": "oracle", "sample": f"float64 loss, lse and dX row of 2 tokens against all "
                                                     f"{V} classes ({t_or:.2f} s; W copy {t_copy:.1f} s not counted)"},
    }


class DeviceInputs:
    """The synth recipe's distributions for workload `w`, drawn on the device by torch's seeded generator:
    X, dY ~ N(0,1) bf16, Wr ~ N(0,1/H) fp32, Wg, Wu ~ N(0,1/H) and Wd ~ N(0,1/I) bf16, and the recipe's
    router bias (fitted on the host).  Used by the timing-only companion runs; the headline run and every
    parity test use the host counter-based generator."""

    def __init__(self, torch, w: S.Workload, seed: int = 0):
        gen = torch.Generator(device="cuda").manual_seed(1000 + seed)

        def normal(shape, std, dtype):
            out = torch.empty(shape, dtype=dtype, device="cuda")
            flat = out.view(-1)
            step = 1 << 28
            for i in range(0, flat.numel(), step):
                n = min(step, flat.numel() - i)
                flat[i:i + n].copy_(torch.randn(n, device="cuda", generator=gen) * std)
            return out

        N, H, E, I = w.N, w.H, w.E, w.I
        self.X = normal((N, H), 1.0, torch.bfloat16)
        self.Wr = normal((E, H), 1.0 / H ** 0.5, torch.float32)
        self.Wg = normal((E, I, H), 1.0 / H ** 0.5, torch.bfloat16)
        self.Wu = normal((E, I, H), 1.0 / H ** 0.5, torch.bfloat16)
        self.Wd = normal((E, H, I), 1.0 / I ** 0.5, torch.bfloat16)
        self.dY = normal((N, H), 1.0, torch.bfloat16)
        b, _ = S.bias_for(w, seed)
        self.bias = None if b is None else torch.from_numpy(b).cuda()


def schedule_run(M, torch, w: S.Workload, D, steps: int, warmup: int, P: int | None = None) -> dict:
    """route + forward + backward of `w` on device inputs D, as one CUDA graph per step (the product's
    MoEStepGraph), replayed `warmup` times untimed and `steps` times between CUDA events.  The chunk
    schedule, or with P the expert-partition schedule over P hops."""
    cfg = M.Config(**w.cfg())
    blk = M.MoEBlock(cfg) if P is None else M.MoEHopBlock(cfg, P)
    G = M.MoEStepGraph(blk, D.X, D.Wr, D.bias, D.Wg, D.Wu, D.Wd, D.dY)
    stats = M.last_stats()
    for _ in range(warmup):
        G.replay()
    torch.cuda.synchronize()
    blk.check()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        G.replay()
    b.record()
    torch.cuda.synchronize()
    blk.check()
    ms = a.elapsed_time(b) / steps
    idx = G.idx.cpu().numpy()
    out = {"ms_per_step": ms, "pairs_per_s": w.N * w.k / (ms / 1e3), "K": blk.K, "idx": idx,
           "stats": stats, "workspace_bytes": blk.ws_bytes}
    if P is not None:
        out["cap"] = blk.cap
    del G, blk
    torch.cuda.empty_cache()
    return out


RUN_ORDER = ("tiny", "mid", "long", "many", "many_zipf", "extreme")


def all_runs(M, torch, args, peaks, done: dict) -> dict:
    """The chunk schedule on every workload (six runs: many once near-uniform, once Zipf 1.2): ms/step,
    pairs/s, the step's fraction of the HBM roofline (algorithmic bytes from the measured per-chunk
    histograms) and of the bf16 peak, and the routed peak against 2 k c_eff H b.  Runs already measured
    (the headline) are passed in `done`; the others draw their inputs on the device."""
    out = {}
    for name in RUN_ORDER:
        if name in done:
            out[name] = done[name]
            continue
        rw = S.WORKLOADS[name]
        D = DeviceInputs(torch, rw)
        r = schedule_run(M, torch, rw, D, args.runs_steps, args.warmup)
        del D
        torch.cuda.empty_cache()
        by, fl = algorithmic(rw, r["idx"], r["K"])
        t = r["ms_per_step"] / 1e3
        pairs = rw.N * rw.k
        out[name] = {"ms_per_step": r["ms_per_step"], "pairs_per_s": r["pairs_per_s"], "K": r["K"],
                     "step_hbm_frac": sum(by.values()) / t / (peaks["hbm_gbs"] * 1e9),
                     "pct_bf16_peak": 22.0 * rw.H * rw.I * pairs / t / (peaks["bf16_tflops_sustained"] * 1e12),
                     "routed_bytes_peak": r["stats"]["routed_bytes_peak"],
                     "routed_bytes_bound_2kcHb": r["stats"]["routed_bytes_bound"],
                     "inputs": "device generator (torch, seeded)", "steps": args.runs_steps}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = S.WORKLOADS[args.workload]
    T = S.make(w)
    samp = CpuSample(w, T, args.cpu_route_tokens, args.cpu_max_tokens, args.cpu_weight_budget)
    vals = []
    for _ in range(args.warmup):
        samp.time()
    for _ in range(args.steps):
        vals.append(samp.time())
    v = statistics.median(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w)}, "cpu_baseline": cb,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# the GPU arm
# --------------------------------------------------------------------------- #
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    from top_softmax_router_gb300 import build as B
    B.build()                                   # no-op when the in-tree library is current
    import top_softmax_router_gb300 as M

    if args.ce_only:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        if int(os.environ.get("RANK", "0")) == 0:
            res = vocab_ce(M, torch, load_peaks(), torch.cuda.current_stream(), args.ce_workload)
            print(json.dumps({"vocab_ce": res}), flush=True)
        return

    if args.adamw_only:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        if int(os.environ.get("RANK", "0")) == 0:
            res = offload_adamw(M, torch, S.WORKLOADS[args.workload], load_peaks(), torch.cuda.current_stream(),
                                args.adamw_params)
            print(json.dumps({"offload_adamw": res}), flush=True)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    w = S.WORKLOADS[args.workload]
    seed = rank
    T = S.make(w, seed=seed)

    def dev_bf16(a):
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)

    X, dY = dev_bf16(T.X), dev_bf16(T.dY)
    Wg, Wu, Wd = dev_bf16(T.Wg), dev_bf16(T.Wu), dev_bf16(T.Wd)
    Wr = torch.from_numpy(T.Wr).cuda()
    bias = None if T.bias is None else torch.from_numpy(T.bias).cuda()
    cfg = M.Config(**w.cfg())
    N, H, E, k, I = w.N, w.H, w.E, w.k, w.I
    idx = torch.empty(N, k, dtype=torch.int32, device="cuda")
    g = torch.empty(N, k, dtype=torch.float32, device="cuda")
    Y = torch.empty_like(X)
    dX = torch.empty_like(X)
    dWr = torch.empty(E, H, device="cuda")
    dWg = torch.empty(E, I, H, device="cuda")
    dWu = torch.empty_like(dWg)
    dWd = torch.empty(E, H, I, device="cuda")
    dg = torch.empty(N, k, device="cuda")
    stream = torch.cuda.current_stream()
    launches = {"n": 0}

    def working_set(cfg_):
        """Device high-water mark, above the inputs and outputs, of creating a block's workspace and
        running one route + forward + backward into the outputs above (the library itself allocates
        nothing, so this is the workspace plus anything a call might allocate)."""
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        b_ = M.MoEBlock(cfg_)
        M.route(cfg_, X, Wr, bias, idx, g, b_.ws, stream)
        st1 = M.last_stats()
        M.forward(cfg_, X, idx, g, Wg, Wu, Wd, Y, b_.ws, stream)
        st2 = M.last_stats()
        M.backward(cfg_, X, Wr, idx, g, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dg, b_.ws, stream)
        st3 = M.last_stats()
        torch.cuda.synchronize()
        b_.check(stream)
        peak = torch.cuda.max_memory_allocated() - base
        routed = max(x["routed_bytes_peak"] for x in (st1, st2, st3))
        inter = max(x["inter_bytes_peak"] for x in (st1, st2, st3))
        c_eff = st3["c_eff"]
        closed = 2 * k * c_eff * H * 2 + 3 * k * c_eff * I * 2
        return b_, {"K": st3["K"], "c_eff": c_eff, "measured_peak_bytes": peak, "workspace_bytes": b_.ws_bytes,
                    "routed_bytes_peak": routed, "routed_bytes_bound_2kcHb": 2 * k * c_eff * H * 2,
                    "inter_bytes_peak": inter, "inter_bytes_bound_3kcIb": 3 * k * c_eff * I * 2,
                    "closed_form_2kcHb_plus_3kcIb": closed,
                    "metadata_bytes": peak - closed}

    blk, ws_kmax = working_set(cfg)

    def step(Xs=X, dYs=dY, st=None):
        st = stream if st is None else st
        M.route(cfg, Xs, Wr, bias, idx, g, blk.ws, st)
        n = M.last_stats()["kernel_launches"]
        M.forward(cfg, Xs, idx, g, Wg, Wu, Wd, Y, blk.ws, st)
        n += M.last_stats()["kernel_launches"]
        M.backward(cfg, Xs, Wr, idx, g, Wg, Wu, Wd, dYs, dX, dWr, dWg, dWu, dWd, dg, blk.ws, st)
        n += M.last_stats()["kernel_launches"]
        launches["n"] += n

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    launches["n"] = 0
    for _ in range(args.warmup):
        step()
    blk.check(stream)
    stats = M.last_stats()
    launches_per_step = launches["n"] // max(args.warmup, 1)
    # the library allocates no device memory: torch's peak allocation does not move across a step
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    mem0 = torch.cuda.max_memory_allocated()
    step()
    torch.cuda.synchronize()
    alloc_delta = torch.cuda.max_memory_allocated() - mem0
    launches["n"] -= launches_per_step
    # One step's launches captured as a CUDA graph (the kernels read their tile lists from device
    # memory, so each replay routes and computes afresh); --eager times the plain calls instead.
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            step(st=cap)
        stream.wait_stream(cap)
        graph.replay()
        barrier()

    # ---- timed region (inputs resident in HBM)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    blk.check(stream)
    ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    ms_per_step = ms / args.steps
    pairs = N * k
    value = job_throughput(pairs, world, args.steps, ms)
    n_launch = launches_per_step * args.steps
    # ---- the same steps again with every launch bracketed by CUDA events on its own stream (the
    # per-kernel durations of the roofline; kept out of the region above so the events cost nothing there)
    M.profile_reset()
    M.profile_enable(True)
    barrier()
    for _ in range(args.steps):
        step()
    barrier()
    M.profile_enable(False)
    prof = M.profile_read()
    blk.check(stream)

    # ---- end to end through host buffers (pinned), copies inside the timed region
    e2e = None
    e2e_graphs = None
    if not args.no_e2e:
        # Each step copies its X and dY in from page-locked host memory and its Y and dX back out.
        # The copies run on their own streams, double-buffered, so step s+1's inputs travel while
        # step s computes and step s's outputs travel while step s+1 computes; every copy of every
        # timed step is inside the timed region.
        hX = torch.from_numpy(T.X.view(np.int16)).view(torch.bfloat16).pin_memory()
        hdY = torch.from_numpy(T.dY.view(np.int16)).view(torch.bfloat16).pin_memory()
        hY = torch.empty_like(hX).pin_memory()
        hdX = torch.empty_like(hX).pin_memory()
        ins = [(torch.empty_like(X), torch.empty_like(dY)) for _ in range(2)]
        outs = [(torch.empty_like(X), torch.empty_like(X)) for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

        def h2d(s_, b):
            with torch.cuda.stream(h2d_s):
                if s_ >= 2:
                    h2d_s.wait_event(comp_done[b])       # step s-2 has finished reading this buffer
                ins[b][0].copy_(hX, non_blocking=True)
                ins[b][1].copy_(hdY, non_blocking=True)
                h2d_done[b].record(h2d_s)

        def compute(b, st):
            Xs, dYs = ins[b]
            Ys, dXo = outs[b]
            M.route(cfg, Xs, Wr, bias, idx, g, blk.ws, st)
            M.forward(cfg, Xs, idx, g, Wg, Wu, Wd, Ys, blk.ws, st)
            M.backward(cfg, Xs, Wr, idx, g, Wg, Wu, Wd, dYs, dXo, dWr, dWg, dWu, dWd, dg, blk.ws, st)

        graphs = None

        def run_steps(n):
            h2d(0, 0)
            for s_ in range(n):
                b = s_ % 2
                if s_ + 1 < n:
                    h2d(s_ + 1, 1 - b)
                stream.wait_event(h2d_done[b])
                if s_ >= 2:
                    stream.wait_event(d2h_done[b])       # step s-2's outputs have left this buffer
                Xs, dYs = ins[b]
                Ys, dXo = outs[b]
                if graphs is not None:
                    graphs[b].replay()
                else:
                    compute(b, stream)
                comp_done[b].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(comp_done[b])
                    hY.copy_(Ys, non_blocking=True)
                    hdX.copy_(dXo, non_blocking=True)
                    d2h_done[b].record(d2h_s)
            stream.wait_stream(d2h_s)

        run_steps(2)
        barrier()
        graphs = None
        if not args.eager:
            # one graph per buffer set, as for the resident-input timing
            graphs = []
            for b in range(2):
                cap = torch.cuda.Stream()
                cap.wait_stream(stream)
                gr_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr_, stream=cap):
                    compute(b, cap)
                stream.wait_stream(cap)
                graphs.append(gr_)
            barrier()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d_s.wait_stream(stream)
        d2h_s.wait_stream(stream)
        run_steps(args.steps)
        b_.record(stream)
        barrier()
        ems = max_over_ranks(a.elapsed_time(b_), dist, "cuda")
        e2e_graphs = graphs
        del ins, outs, graphs
        e2e = {"value": job_throughput(pairs, world, args.steps, ems), "unit": UNIT,
               "h2d_bytes_per_step": 2 * N * H * 2, "d2h_bytes_per_step": 2 * N * H * 2,
               "copies": "double-buffered on two copy streams, overlapping the neighbouring steps' compute",
               "launch": "eager calls" if args.eager else "one CUDA graph per buffer set, replayed"}

    # ---- the expert-partition ("hop") schedule beside the chunk schedule, on one workload's inputs
    hops = None
    on_load = None
    if not args.no_hops and world == 1:
        hw = S.WORKLOADS[args.hops_workload]
        P = max(1, min(hw.E, args.hops))
        HD = DeviceInputs(torch, hw)
        ch = schedule_run(M, torch, hw, HD, args.steps, args.warmup)
        hr = schedule_run(M, torch, hw, HD, args.steps, args.warmup, P=P)
        hidx = hr.pop("idx")
        ch.pop("idx")
        per_hop = [int(np.isin(hidx, np.arange(h * hw.E // P, (h + 1) * hw.E // P)).sum()) for h in range(P)]
        hops = {"schedule": f"expert partitions: P={P} hops of {hw.E // P} experts (RelayMoE-style, one device)",
                "workload": workload_desc(hw) + " (inputs drawn on the device, torch seeded generator)",
                "ms_per_step": hr["ms_per_step"], "value": hr["pairs_per_s"], "unit": UNIT,
                "chunk_schedule_ms_per_step": ch["ms_per_step"], "chunk_schedule_K": ch["K"],
                "speedup_over_chunk_schedule": ch["ms_per_step"] / hr["ms_per_step"],
                "routed_rows_largest_hop": max(per_hop), "routed_rows_per_hop": per_hop,
                "routed_bytes_largest_hop": 2 * max(per_hop) * hw.H * 2,
                "routed_bytes_workspace": 2 * hr["cap"] * hw.H * 2,
                "chunk_schedule_bound_2kcHb": ch["stats"]["routed_bytes_bound"],
                "launch": "one CUDA graph per step, replayed"}
        # the dispatch gather fused into the GEMMs (MOE_DISPATCH_ON_LOAD) on the same inputs
        M.set_dispatch("on_load")
        try:
            ol = schedule_run(M, torch, hw, HD, args.steps, args.warmup)
        finally:
            M.set_dispatch("gather")
        ol.pop("idx")
        on_load = {"workload": hops["workload"], "ms_per_step": ol["ms_per_step"], "value": ol["pairs_per_s"],
                   "unit": UNIT, "gather_kernel_ms_per_step": ch["ms_per_step"],
                   "routed_bytes_peak": ol["stats"]["routed_bytes_peak"],
                   "gather_kernel_routed_bytes_peak": ch["stats"]["routed_bytes_peak"],
                   "routed_bytes_bound_2kcHb": ol["stats"]["routed_bytes_bound"],
                   "workspace_bytes": ol["workspace_bytes"], "gather_kernel_workspace_bytes": ch["workspace_bytes"],
                   "launch": "one CUDA graph per step, replayed"}
        del HD
        torch.cuda.empty_cache()

    # ---- the same block unchunked (K = 1): the working set the chunking bounds, and what the bound costs
    unchunked = None
    peaks_early = load_peaks()
    ws_k1 = None
    if not args.no_unchunked and w.K_max > 1:
        cfg1 = M.Config(**{**w.cfg(), "K_max": 1})
        blk1, ws_k1 = working_set(cfg1)

        def ustep(st=None):
            st = stream if st is None else st
            M.route(cfg1, X, Wr, bias, idx, g, blk1.ws, st)
            M.forward(cfg1, X, idx, g, Wg, Wu, Wd, Y, blk1.ws, st)
            M.backward(cfg1, X, Wr, idx, g, Wg, Wu, Wd, dY, dX, dWr, dWg, dWu, dWd, dg, blk1.ws, st)

        for _ in range(args.warmup):
            ustep()
        barrier()
        ust = M.last_stats()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            ustep()
        b.record(stream)
        barrier()
        blk1.check(stream)
        ums = max_over_ranks(a.elapsed_time(b), dist, "cuda") / args.steps
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        barrier()
        cms = max_over_ranks(a.elapsed_time(b), dist, "cuda") / args.steps
        # per-class GEMM rates of the unchunked step (profiled pass): one segment per expert, so the
        # tiles are full and each expert's weights stream once
        M.profile_reset()
        M.profile_enable(True)
        for _ in range(args.steps):
            ustep()
        barrier()
        M.profile_enable(False)
        uprof = M.profile_read()
        ugemm = {}
        for name, per_pair in (("gemm_gateup", 8.0), ("gemm_down", 2.0), ("gemm_dact", 2.0), ("gemm_dx", 4.0),
                               ("gemm_dw", 6.0)):
            n_l, tot = uprof.get(name, (0, 0.0))
            if n_l:
                tf = per_pair * H * I * N * k * args.steps / (tot / 1e3) / 1e12
                ugemm[name] = {"ms_per_step": tot / args.steps, "tflops": tf,
                               "frac_of_bf16_sustained": tf / peaks_early["bf16_tflops_sustained"]}
        unchunked = {"chunked_eager_ms_per_step": cms, "time_ratio_chunked_over_unchunked": cms / ums,
                     "gemm_classes": ugemm,"K": 1, "ms_per_step_eager": ums, "routed_bytes_peak": ust["routed_bytes_peak"],
                     "inter_bytes_peak": ust["inter_bytes_peak"], "workspace_bytes": ust["workspace_bytes"],
                     "routed_peak_cut_by_chunking": 1.0 - stats["routed_bytes_peak"] / ust["routed_bytes_peak"],
                     "note": "both timed as eager calls"}
        del blk1

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel class
    peaks = load_peaks()
    adamw = None
    if not args.no_adamw and world == 1:
        del dWg, dWu, dWd
        torch.cuda.empty_cache()
        adamw = offload_adamw(M, torch, w, peaks, stream, args.adamw_params)
    ce_res = None
    if not args.no_ce and world == 1:
        torch.cuda.empty_cache()
        ce_res = vocab_ce(M, torch, peaks, stream, args.ce_workload)
    K = blk.K
    idx_host = idx.cpu().numpy()
    by, fl = algorithmic(w, idx_host, K)
    per_class = {}
    for name, (n_l, tot_ms) in prof.items():
        if n_l == 0:
            continue
        per_launch_s = tot_ms / n_l / 1e3
        bytes_l = by.get(name, 0.0) / (n_l / args.steps)
        flops_l = fl.get(name, 0.0) / (n_l / args.steps)
        t_hbm = bytes_l / (peaks["hbm_gbs"] * 1e9)
        t_tc = flops_l / (peaks["bf16_tflops_sustained"] * 1e12)
        bound = "tensor" if t_tc > t_hbm else "hbm"
        if name == "router_logits":
            # fp32 fused multiply-add chains on the SIMT units, not the tensor cores
            t_alu = flops_l / (ALU_FP32_TFLOPS * 1e12)
            bound, t_tc = ("alu", t_alu) if t_alu > t_hbm else (bound, t_tc)
        per_class[name] = dict(launches_per_step=n_l / args.steps, ms_per_launch=tot_ms / n_l,
                               ms_per_step=tot_ms / args.steps, bound=bound,
                               gbs=bytes_l / per_launch_s / 1e9, tflops=flops_l / per_launch_s / 1e12,
                               frac=(t_tc if bound in ("tensor", "alu") else t_hbm) / per_launch_s)
    dom = max(per_class, key=lambda n: per_class[n]["ms_per_step"])
    d = per_class[dom]
    traffic, traffic_src = measured_traffic(dom, args.workload)
    if d["bound"] == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": d["tflops"], "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": d["tflops"] / peaks["bf16_tflops_sustained"], "traffic": traffic,
                "peak_source": f"{peaks['source']} bf16 sustained"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": d["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": d["gbs"] / peaks["hbm_gbs"], "traffic": traffic, "peak_source": f"{peaks['source']} HBM copy"}
    if traffic is not None:
        roof["traffic_note"] = traffic_src.get("note", "")
        roof["traffic_algorithmic_same_launches"] = traffic_src.get("algorithmic_bytes_per_launch")
    step_bytes = sum(by.values())
    step_flops = sum(fl.values())
    flops22 = 22.0 * H * I * pairs
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w), "K": K, "c_eff": blk.c_eff, "pairs_per_step": pairs,
                   "l2": "no flush: expert weights (%.2f GB) exceed the 129 MB L2 and are streamed every step"
                         % (3 * E * H * I * 2 / 1e9),
                   "parallelism": f"replicas x{world} (no collective on the data path)",
                   "launch": "eager calls" if args.eager else
                             "route + forward + backward captured once as a CUDA graph, replayed each step"},
        "pct_bf16_peak": flops22 / (ms_per_step / 1e3) / (peaks["bf16_tflops_sustained"] * 1e12),
        "pct_bf16_peak_note": "22 H I flop per pair (forward 6, backward 12, recompute 4); "
                              "model flops 18 H I: %.4f" % (18.0 * H * I * pairs / (ms_per_step / 1e3) /
                                                           (peaks["bf16_tflops_sustained"] * 1e12)),
        "step_roofline": {"algorithmic_bytes": step_bytes, "flops": step_flops,
                          "hbm_frac": step_bytes / (ms_per_step / 1e3) / (peaks["hbm_gbs"] * 1e9),
                          "tensor_frac": step_flops / (ms_per_step / 1e3) / (peaks["bf16_tflops_sustained"] * 1e12)},
        "peak_bytes_vs_bound": {"routed_bytes_peak": stats["routed_bytes_peak"],
                                "routed_bytes_bound_2kcHb": stats["routed_bytes_bound"],
                                "inter_bytes_peak": stats["inter_bytes_peak"],
                                "inter_bytes_bound_3kcIb": stats["inter_bytes_bound"],
                                "workspace_bytes": stats["workspace_bytes"],
                                "torch_peak_alloc_delta_over_a_step": alloc_delta,
                                "measured_K_max": ws_kmax, "measured_K_1": ws_k1,
                                "note": "measured_*: torch.cuda.max_memory_allocated() from before the "
                                        "workspace is allocated through one route + forward + backward, "
                                        "above the block's inputs and outputs"},
        "roofline": roof,
        "kernels": {n: {kk: (round(v, 4) if isinstance(v, float) else v) for kk, v in c.items()}
                    for n, c in per_class.items()},
        "gpu_launches": n_launch,
        "clocks": clk,
        "e2e": e2e,
        "alt_schedule": hops,
        "dispatch_on_load": on_load,
        "unchunked": unchunked,
        "offload_adamw": adamw,
        "vocab_ce": ce_res,
    }
    if not args.no_runs and world == 1:
        main_row = {"ms_per_step": ms_per_step, "pairs_per_s": value, "K": K,
                    "step_hbm_frac": line["step_roofline"]["hbm_frac"], "pct_bf16_peak": line["pct_bf16_peak"],
                    "routed_bytes_peak": stats["routed_bytes_peak"],
                    "routed_bytes_bound_2kcHb": stats["routed_bytes_bound"], "inputs": "host generator (headline)"}
        del X, dY, Wg, Wu, Wd, Y, dX, dWr, dg, blk, graph
        if args.no_adamw:
            del dWg, dWu, dWd
        if e2e_graphs is not None:
            del e2e_graphs
        torch.cuda.empty_cache()
        line["runs"] = all_runs(M, torch, args, peaks, {args.workload: main_row})
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, T, args)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
