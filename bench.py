#!/usr/bin/env python
"""Benchmark of NSA selected attention (forward + backward) on one GB300 per rank.

One step = one pass of the whole hot path over one synthetic batch: index build
(histogram, scan, scatter), forward main + merge, backward preprocess, main, dQ
and dK/dV reductions, all through the C ABI.  Workload: 64K tokens, 4 KV heads,
d = 128, B_K = 64, T = 16, GQA group g (default 4), distance-weighted selection;
inputs (q, k, v, dO ~ N(0, 1), bf16) are larger than L2.

Metric (useful work): forward FLOPs = 4 * d * sum over query heads and tokens of
the keys attended; backward = 2.5x forward.  Prints one JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--g G] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selected-attn fwd/bwd ms & useful TFLOP/s (% BF16 tensor peak) at 64K, B_K=64, T=16"
DOMINANT = ("fwd_main", "bwd_main")

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the dominant
# kernels on the 64K workload, from one ncu capture of the kernel sources whose
# SHA-256 is given (profiles/dram_traffic_fwd64k_g4.md).  Reported only while the
# sources are unchanged; otherwise the roofline's traffic is null.
TRAFFIC = {"sources_sha256": "a3fded1d5a79fbe509a33ae2e9196e6d9f2b75e216b583d0eceebc1681db37a4",
           "bytes": {"fwd_main": {"4": 925600000 + 4403003392},
                     "bwd_main": {"4": 2803539200 + 4798355456}}}


def kernel_sources_hash() -> str:
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_sparse_attention_nsa_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()


def captured_traffic(kernel: str, g: int):
    if not TRAFFIC["sources_sha256"] or TRAFFIC["sources_sha256"] != kernel_sources_hash():
        return None
    return TRAFFIC["bytes"].get(kernel, {}).get(str(g))


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--g", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="skip the g = 1, 2, 4, 8 sweep")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--extended", action="store_true",
                    help="also time g = 16, 32K tokens, and (B_K, T) = (128, 8) at d = 64")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", 0)), \
            float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, 6800.0, "fallback"


def useful_fwd_flops(cfg):
    from workloads import keys_attended
    n_t = keys_attended(cfg.seqlens, cfg.block, cfg.topk)
    return 4.0 * cfg.d * cfg.h_q * float(n_t.sum())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
class Runner:
    def __init__(self, cfg, seed, device):
        import torch
        import block_sparse_attention_nsa_gb300 as nsa
        from workloads import make_inputs
        self.torch, self.nsa, self.cfg = torch, nsa, cfg
        self.host = make_inputs(cfg, seed=seed, with_dout=True)
        h = self.host
        self.q, self.k, self.v, self.dout = (h[x].to(device) for x in ("q", "k", "v", "dout"))
        self.sel = torch.from_numpy(h["sel_idx"]).to(device)
        self.cu = torch.from_numpy(h["cu_seqlens"]).to(device)
        self.dims = nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d, cfg.block,
                                  cfg.topk, self.q.dtype)
        self.ws = nsa.alloc_workspace(self.dims, device)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((cfg.h_q, cfg.n), dtype=torch.float32, device=device)
        self.dq, self.dk, self.dv = (torch.empty_like(x) for x in (self.q, self.k, self.v))
        self.resident_bytes = sum(x.numel() * x.element_size() for x in
                                  (self.q, self.k, self.v, self.dout, self.sel))

    def fwd(self):
        c = self.cfg
        self.nsa.fwd(self.q, self.k, self.v, self.sel, self.cu, c.block, c.scale,
                     workspace=self.ws, out=self.out, lse=self.lse)

    def bwd(self):
        c = self.cfg
        self.nsa.bwd(self.q, self.k, self.v, self.sel, self.cu, c.block, c.scale, self.out,
                     self.lse, self.dout, workspace=self.ws, index_ready=True, dq=self.dq,
                     dk=self.dk, dv=self.dv)

    def bwd_rebuild(self):
        c = self.cfg
        self.nsa.bwd(self.q, self.k, self.v, self.sel, self.cu, c.block, c.scale, self.out,
                     self.lse, self.dout, workspace=self.ws, index_ready=False, dq=self.dq,
                     dk=self.dk, dv=self.dv)

    def step(self):
        self.fwd()
        self.bwd()

    def check_status(self):
        code, bits = self.nsa.get_status(self.dims, self.ws)
        if code != 0:
            raise RuntimeError(f"device status {code} (bits {bits})")


def time_reps(torch, fn, reps):
    """Per-call device times (ms) of `reps` back-to-back calls, CUDA events on the
    current stream, synchronised before and after."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    torch.cuda.synchronize()
    evs[0].record()
    for i in range(reps):
        fn()
        evs[i + 1].record()
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(reps)]


def dist(ms_list):
    a = np.asarray(ms_list, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "reps": int(a.size)}


def e2e_measure(r: Runner, iters: int):
    """Same step through nsa_sel_attn_step_host: pinned host inputs -> device -> host outputs."""
    torch, nsa = r.torch, r.nsa
    h = r.host
    pin = lambda t: t.contiguous().pin_memory()
    host = {"q": pin(h["q"]), "k": pin(h["k"]), "v": pin(h["v"]), "dout": pin(h["dout"]),
            "sel_idx": pin(torch.from_numpy(h["sel_idx"])),
            "cu_seqlens": pin(torch.from_numpy(h["cu_seqlens"]))}
    for name, like in (("out", "q"), ("dq", "q"), ("dk", "k"), ("dv", "v")):
        host[name] = torch.empty_like(host[like]).pin_memory()
    host["lse"] = torch.empty((r.cfg.h_q, r.cfg.n), dtype=torch.float32).pin_memory()
    staging = torch.empty(nsa.staging_size(r.dims), dtype=torch.uint8, device="cuda")
    h2d = sum(host[x].numel() * host[x].element_size()
              for x in ("q", "k", "v", "dout", "sel_idx", "cu_seqlens"))
    d2h = sum(host[x].numel() * host[x].element_size() for x in ("out", "lse", "dq", "dk", "dv"))
    nsa.step_host(r.dims, host, r.cfg.scale, staging, r.ws)     # warm-up
    torch.cuda.synchronize()
    times = []
    for _ in range(iters):
        t0 = time.perf_counter()
        nsa.step_host(r.dims, host, r.cfg.scale, staging, r.ws)  # returns after the D2H copies
        times.append(time.perf_counter() - t0)
    dt = float(np.median(times))
    del staging
    return dt, h2d, d2h


def cpu_baseline(cfg, host, seconds, useful_rate_scale=1.0):
    """The oracle, as it stands, on sampled (token, query head) forward rows."""
    import oracle
    from workloads import keys_attended
    n_t = keys_attended(cfg.seqlens, cfg.block, cfg.topk)
    rng = np.random.default_rng(123)
    threads = oracle.max_threads()
    batch, done_rows, flops, t_used = 256, 0, 0.0, 0.0
    q64 = host["q"].float().numpy().astype(np.float64)
    k64 = host["k"].float().numpy().astype(np.float64)
    v64 = host["v"].float().numpy().astype(np.float64)
    while t_used < seconds:
        rows = np.stack([rng.integers(0, cfg.n, batch), rng.integers(0, cfg.h_q, batch)], axis=1)
        t0 = time.perf_counter()
        oracle.fwd_rows(host["cu_seqlens"], cfg.block, host["sel_idx"], q64, k64, v64, cfg.scale,
                        rows)
        t_used += time.perf_counter() - t0
        done_rows += batch
        flops += 4.0 * cfg.d * float(n_t[rows[:, 0]].sum())
        batch = min(batch * 2, 8192)
    return {"value": flops / t_used / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle forward on {done_rows} random (token, query head) rows of the "
                      f"same workload, {t_used:.1f} s; useful forward FLOPs of those rows / time "
                      f"(the oracle backward has no row-sampled form)"}


def run_ours(args, rank, world):
    import torch
    import block_sparse_attention_nsa_gb300 as nsa
    from workloads import CONFIGS

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    nsa.load()
    cfg = CONFIGS["fwd64k"].with_g(args.g)
    r = Runner(cfg, cfg.seed + rank, dev)
    fwd_flops = useful_fwd_flops(cfg)
    step_flops = 3.5 * fwd_flops
    for _ in range(max(3, args.warmup)):
        r.step()
    torch.cuda.synchronize()
    r.check_status()

    # ---- headline: exactly K steps, the library's event profiler off ----
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(dev.index) as clk:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        step_ms = time_reps(torch, r.step, args.steps)
        if world > 1:
            torch.distributed.barrier()
    ms = float(np.sum(step_ms)) / args.steps
    r.check_status()
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # ---- per-kernel split: a separate pass with the event profiler on ----
    prof_steps = 3
    nsa.profile_enable(True)
    for _ in range(prof_steps):
        r.step()
    torch.cuda.synchronize()
    nsa.profile_enable(False)
    kern = nsa.profile_collect()
    r.check_status()

    # ---- forward / backward alone (outside the headline region) ----
    reps = max(50, args.steps)
    fwd_d = dist(time_reps(torch, r.fwd, reps))
    bwd_d = dist(time_reps(torch, r.bwd, reps))
    bwd0_d = dist(time_reps(torch, r.bwd_rebuild, max(10, reps // 5)))
    fwd_ms, bwd_ms = fwd_d["median"], bwd_d["median"]

    pk_burst, pk_sust, hbm, pk_kind = peaks()
    launches = int(round(sum(n for n, _ in kern.values()) / prof_steps))
    dom = max(DOMINANT, key=lambda name: kern.get(name, (0, 0.0))[1])
    n_l, tot = kern[dom]
    per_launch_ms = tot / max(1, n_l)
    dom_flops = fwd_flops if dom == "fwd_main" else 2.5 * fwd_flops
    achieved = dom_flops / (per_launch_ms * 1e-3) / 1e12
    step_tot = sum(t for _, t in kern.values())
    result = {
        "metric": METRIC,
        "value": world * step_flops / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"fwd64k g={cfg.g}: N=65536, h_k=4, h_q={cfg.h_q}, d=128, "
                               f"B_K=64, T=16, distance-weighted selection, fwd+bwd step",
                   "global_batch": world, "seq_len": cfg.n, "g": cfg.g,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({r.resident_bytes / 1e6:.0f} MB resident per "
                         f"rank), no flush"},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": 2.5 * fwd_flops / (bwd_ms * 1e-3) / 1e12,
        "pct_bf16_peak_step": 100.0 * (step_flops / (ms * 1e-3) / 1e12) / pk_burst,
        "step_ms_dist": dist(step_ms),
        "fwd_ms_dist": fwd_d, "bwd_ms_dist": bwd_d,
        "bwd_rebuild_index_ms_dist": bwd0_d,
        "kernels_ms_per_step": {k: t / prof_steps for k, (n, t) in kern.items() if n},
        "kernels_sum_ms_per_step": step_tot / prof_steps,
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": pk_burst,
                     "unit": "TFLOP/s", "frac": achieved / pk_burst,
                     "traffic": captured_traffic(dom, cfg.g),
                     "peak_kind": f"{pk_kind} bf16 burst",
                     "share_of_step": tot / step_tot if step_tot else None,
                     "algorithmic_flops_per_launch": dom_flops},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if world == 1 and not args.no_e2e:
        dt, h2d, d2h = e2e_measure(r, 5)
        result["e2e"] = {"value": step_flops / dt / 1e12, "unit": "TFLOP/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": dt * 1e3}
    if world == 1 and not args.no_sweep:
        sweep = {}
        for g in (1, 2, 4, 8):
            c = CONFIGS["fwd64k"].with_g(g)
            rr = r if g == cfg.g else Runner(c, c.seed, dev)
            ff = useful_fwd_flops(c)
            rr.step()
            f_ms = dist(time_reps(torch, rr.fwd, 20))["median"]
            b_ms = dist(time_reps(torch, rr.bwd, 20))["median"]
            sweep[f"g{g}"] = {"fwd_ms": f_ms, "bwd_ms": b_ms,
                              "fwd_tflops": ff / (f_ms * 1e-3) / 1e12,
                              "bwd_tflops": 2.5 * ff / (b_ms * 1e-3) / 1e12,
                              "fwd_pct_peak": 100 * ff / (f_ms * 1e-3) / 1e12 / pk_burst}
            if rr is not r:
                del rr
                torch.cuda.empty_cache()
        result["sweep"] = sweep
    if world == 1 and args.extended:
        result["extended"] = extended_sweep(torch, dev, pk_burst)
    if rank == 0 and world == 1 and not args.no_cpu and args.cpu_seconds > 0:
        result["cpu_baseline"] = cpu_baseline(cfg, r.host, args.cpu_seconds)
    return result


def extended_sweep(torch, dev, pk_burst):
    """Forward and backward times beyond the headline sweep: g = 16 at 64K tokens,
    32K-token sequences, and the pages' (B_K, T) = (128, 8) pair (at d = 64: the
    library does not offer d = 128 with B_K = 128)."""
    import dataclasses
    from workloads import CONFIGS
    base = CONFIGS["fwd64k"]
    cases = {
        "64k_g16": base.with_g(16),
        "32k_g1": dataclasses.replace(base.with_g(1), seqlens=(32768,), name="fwd32k_g1"),
        "32k_g4": dataclasses.replace(base.with_g(4), seqlens=(32768,), name="fwd32k_g4"),
        "32k_g16": dataclasses.replace(base.with_g(16), seqlens=(32768,), name="fwd32k_g16"),
        "64k_d64_b128_t8_g4": dataclasses.replace(base.with_g(4), d=64, block=128, topk=8,
                                                  name="fwd64k_d64_b128_t8_g4"),
    }
    outd = {}
    for key, c in cases.items():
        rr = Runner(c, c.seed, dev)
        ff = useful_fwd_flops(c)
        rr.step()
        torch.cuda.synchronize()
        rr.check_status()
        f_ms = dist(time_reps(torch, rr.fwd, 20))["median"]
        b_ms = dist(time_reps(torch, rr.bwd, 20))["median"]
        outd[key] = {"n": c.n, "g": c.g, "d": c.d, "B_K": c.block, "T": c.topk,
                     "fwd_ms": f_ms, "bwd_ms": b_ms,
                     "fwd_tflops": ff / (f_ms * 1e-3) / 1e12,
                     "bwd_tflops": 2.5 * ff / (b_ms * 1e-3) / 1e12,
                     "fwd_pct_peak": 100 * ff / (f_ms * 1e-3) / 1e12 / pk_burst}
        del rr
        torch.cuda.empty_cache()
    outd.update(decode_sweep(torch, dev))
    outd.update(window_sweep(torch, dev, pk_burst))
    outd.update(cmp_sweep(torch, dev, pk_burst))
    return outd


def window_sweep(torch, dev, pk_burst):
    """Sliding-window branch (window 512) on the 64K workload's shape, g = 4, and the
    gated combination of three branch outputs of that shape."""
    import dataclasses
    import block_sparse_attention_nsa_gb300 as nsa
    from workloads import CONFIGS, make_inputs
    W, blk = 512, 64
    topk = (W - 1 + blk - 1) // blk + 1
    c = dataclasses.replace(CONFIGS["fwd64k"].with_g(4), topk=topk, name="window64k_g4")
    inp = make_inputs(c, with_dout=True)
    q, k, v, do = (inp[x].to(dev) for x in ("q", "k", "v", "dout"))
    cu = torch.from_numpy(inp["cu_seqlens"]).to(dev)
    sel = nsa.window_select(cu, c.n, c.h_k, blk, topk, W)
    ws = nsa.alloc_workspace(nsa.make_dims(1, c.n, c.h_q, c.h_k, c.d, blk, topk, q.dtype), dev)
    state = {}

    def fwd():
        state["o"] = nsa.fwd_window(q, k, v, sel, cu, blk, c.scale, W, workspace=ws)

    def bwd():
        o, l = state["o"]
        nsa.bwd_window(q, k, v, sel, cu, blk, c.scale, W, o, l, do, workspace=ws,
                       index_ready=True)
    fwd()
    bwd()
    torch.cuda.synchronize()
    f_ms = dist(time_reps(torch, fwd, 20))["median"]
    fwd()
    b_ms = dist(time_reps(torch, bwd, 20))["median"]
    keys = float(np.minimum(np.arange(c.n) + 1, W).sum())          # one 64K sequence
    ff = 4.0 * c.d * c.h_q * keys
    outd = {"window64k_w512_g4": {"fwd_ms": f_ms, "bwd_ms": b_ms,
                                  "fwd_tflops": ff / (f_ms * 1e-3) / 1e12,
                                  "bwd_tflops": 2.5 * ff / (b_ms * 1e-3) / 1e12,
                                  "fwd_pct_peak": 100 * ff / (f_ms * 1e-3) / 1e12 / pk_burst}}
    o = state["o"][0]
    branches = [o, o.clone(), o.clone()]
    gates = torch.rand(c.n, c.h_q, 3, device=dev)
    comb = lambda: nsa.gate_combine(branches, gates)
    comb()
    ms = dist(time_reps(torch, comb, 20))["median"]
    nbytes = 4 * o.numel() * o.element_size() + gates.numel() * 4
    outd["gate_combine_3x64k_g4"] = {"us": ms * 1e3, "GB/s": nbytes / (ms * 1e-3) / 1e9,
                                     "frac_of_measured_hbm": nbytes / (ms * 1e-3) / 1e9 /
                                     peaks()[2]}
    del ws, q, k, v, do
    torch.cuda.empty_cache()
    return outd


def cmp_sweep(torch, dev, pk_burst):
    """The step before selected attention on the 64K workload's shape (h_k = 4, d = 128,
    g = 1 and 4): compression (kernel_size 32, stride 16), then compressed attention
    with block importance and top-16 selection (B_K = 64, 1 init and 2 local blocks).
    Useful FLOPs are QK^T and PV over the visible compressed tokens; the kernel also
    recomputes QK^T once to form the exact probabilities for the importance."""
    import block_sparse_attention_nsa_gb300 as nsa
    from workloads import CONFIGS, make_inputs
    outd = {}
    for g in (1, 4):
        c = CONFIGS["fwd64k"].with_g(g)
        inp = make_inputs(c)
        q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
        cu = torch.from_numpy(inp["cu_seqlens"]).to(dev)
        state = {}

        def comp():
            state["c"] = nsa.compress_kv(k, v, cu, 32, 16)

        dims = nsa.make_dims(1, c.n, c.h_q, c.h_k, c.d, 64, 16, q.dtype)
        need = nsa.cmp_workspace_size(dims, 32, 16, c.n)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

        def sel():
            kc, vc, cc = state["c"]
            nsa.cmp_attn_select(q, kc, vc, cu, cc, 32, 16, c.n, c.scale, 64, 16, 1, 2,
                                workspace=ws)
        comp()
        sel()
        torch.cuda.synchronize()
        c_ms = dist(time_reps(torch, comp, 20))["median"]
        s_ms = dist(time_reps(torch, sel, 10))["median"]
        tau = np.arange(c.n)
        nv = float(np.where(tau >= 31, (tau - 31) // 16 + 1, 0).sum())
        ff = 4.0 * c.d * c.h_q * nv
        outd[f"cmp_select_64k_g{g}"] = {
            "compress_ms": c_ms, "attn_select_ms": s_ms,
            "useful_tflops": ff / (s_ms * 1e-3) / 1e12,
            "issued_tflops": 1.5 * ff / (s_ms * 1e-3) / 1e12,
            "pct_peak_issued": 100 * 1.5 * ff / (s_ms * 1e-3) / 1e12 / pk_burst}
        del q, k, v, state, ws
        torch.cuda.empty_cache()
    return outd


def decode_sweep(torch, dev):
    """One-step decode: 64 sequences with 8192-token caches, 4 KV heads, d = 128,
    B_K = 64, T = 16, distance-weighted selection of the last token.  HBM-bound: the
    algorithmic bytes are the kept K/V blocks (plus q and out)."""
    import block_sparse_attention_nsa_gb300 as nsa
    from workloads import make_decode_inputs
    outd = {}
    B, L, h_k, d, blk, T = 64, 8192, 4, 128, 64, 16
    for g in (4, 16):
        inp = make_decode_inputs([L] * B, h_k, g, d, blk, T, "distance", "bf16", seed=2000 + g)
        q, k, v = (inp[x].to(dev) for x in ("q", "k", "v"))
        sel = torch.from_numpy(inp["sel_idx"]).to(dev)
        cu = torch.from_numpy(inp["cu_seqlens"]).to(dev)
        out = torch.empty_like(q)
        lse = torch.empty((h_k * g, B), dtype=torch.float32, device=dev)
        run = lambda: nsa.decode(q, k, v, sel, cu, blk, inp["scale"], out=out, lse=lse)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        ms = dist(time_reps(torch, run, 50))["median"]
        kept = int((inp["sel_idx"] >= 0).sum())                 # one (head, block) per kept slot
        kv_bytes = kept * blk * d * 2 * 2
        io_bytes = 2 * q.numel() * q.element_size() + lse.numel() * 4
        gbs = (kv_bytes + io_bytes) / (ms * 1e-3) / 1e9
        outd[f"decode_b{B}_{L // 1024}k_g{g}"] = {
            "us": ms * 1e3, "algorithmic_bytes": kv_bytes + io_bytes, "GB/s": gbs,
            "frac_of_measured_hbm": gbs / peaks()[2],
            "useful_tflops": 4.0 * d * g * kept * blk / (ms * 1e-3) / 1e12}
        del q, k, v, out
        torch.cuda.empty_cache()
    return outd


def run_reference(args, rank, world):
    """The fp64 oracle, as it stands, on the host cores (bounded samples of the workload)."""
    from workloads import CONFIGS, make_inputs
    cfg = CONFIGS["fwd64k"].with_g(args.g)
    host = make_inputs(cfg)
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(cfg, host, per_step / 4)
    vals, t0 = [], time.perf_counter()
    cb = None
    for _ in range(args.steps):
        cb = cpu_baseline(cfg, host, per_step)
        vals.append(cb["value"])
    wall = time.perf_counter() - t0
    value = float(np.median(vals))
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": f"fwd64k g={cfg.g}: N=65536, h_k=4, h_q={cfg.h_q}, d=128, "
                                   f"B_K=64, T=16", "global_batch": 1, "seq_len": cfg.n,
                       "g": cfg.g, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        result = run_ours(args, rank, world)
        if rank == 0:
            result["impl"] = "ours"
            print(json.dumps(result), flush=True)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
