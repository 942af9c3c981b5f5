"""Throughput of the credit-assignment scans on one or more GPUs.

Workload: GAE + discounted returns + TD(lambda), float32, 4096 environments x
128 steps, env-major [E, T]; rewards and values N(0, 1), termination 1%,
truncation 0.5% with N(0, 1) continuation values, N(0, 1) bootstrap values,
gamma = 0.99, lambda = 0.95 (the "thousands of environments, short
rollouts" regime of rl-triton, arXiv:2608.17641, §6-§7).

One step = one call of each of the three estimators on one batch (three
kernel launches).  The metric is env-steps per second per estimator:
3 * E * T * steps / time.  Inputs stay resident in HBM; the timed steps
rotate over enough replicas of the batch that their footprint exceeds
three times the L2 cache, so every step reads from DRAM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import csv
import ctypes as C
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

E, T = 4096, 128
GAMMA, LAMBDA = 0.99, 0.95
P_TERM, P_TRUNC = 0.01, 0.005
N_EST = 3
METRIC = "env-steps/s per estimator at 4096 envs x 128 steps"
WORKLOAD = "gae+discounted_return+td_lambda f32 4096x128 env-major"
FALLBACK_HBM_GBS = 6800.0


def _workload_config(extra=None):
    cfg = {"workload": WORKLOAD, "E": E, "T": T, "layout": "env-major [E,T]",
           "estimators": ["gae(adv+ret)", "discounted_return", "td_lambda"],
           "gamma": GAMMA, "lambda": LAMBDA, "p_terminated": P_TERM, "p_truncated": P_TRUNC,
           "parallelism": "replicas (env-sharded, no collective)"}
    if extra:
        cfg.update(extra)
    return cfg


def _batch_cpu():
    from first_order_linear_gb300 import synth
    return synth.value_rollout(E, T, seed=synth.config_seed("4096x128"), p_term=P_TERM, p_trunc=P_TRUNC,
                               with_trunc=True, device="cpu")


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------------
# CPU oracle (the reported baseline and the reference arm)
# --------------------------------------------------------------------------

def _oracle_step(ref, n):
    ref.gae(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
            gamma=GAMMA, lam=LAMBDA)
    ref.discounted_return(n["rewards"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
                          gamma=GAMMA)
    ref.td_lambda(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
                  gamma=GAMMA, lam=LAMBDA)


def _oracle_rows(d, rows):
    from first_order_linear_gb300 import synth
    n = synth.numpy(d)
    return {k: (v[:rows] if isinstance(v, type(n["rewards"])) else v) for k, v in n.items()}


def cpu_baseline(d, budget_s=8.0):
    """The oracle as it stands, on the host, over repeated full batches."""
    from oracle import rlca_ref as ref
    n = _oracle_rows(d, E)
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(ref, n)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 1000:
            break
    return {"value": N_EST * E * T * reps / el, "unit": "env-steps/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} full {E}x{T} batches (GAE, discounted return, TD(lambda)) in float64 NumPy, "
                      f"{el:.1f} s on one host thread"}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    d = _batch_cpu()
    from oracle import rlca_ref as ref
    n = _oracle_rows(d, E)
    t0 = time.perf_counter()
    _oracle_step(ref, n)
    t_full = time.perf_counter() - t0
    # bound the whole run to about a minute of CPU work
    rows = E if (args.steps + args.warmup) * t_full <= 60.0 else max(
        32, int(E * 60.0 / ((args.steps + args.warmup) * t_full)))
    sub = _oracle_rows(d, rows)
    for _ in range(args.warmup):
        _oracle_step(ref, sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(ref, sub)
    el = time.perf_counter() - t0
    units = N_EST * rows * T * args.steps
    value = units / el
    sample = f"first {rows} of {E} envs x {T} steps per step, GAE + discounted return + TD(lambda), float64 NumPy"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "env-steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _workload_config({"rows_per_step": rows}),
            "cpu_baseline": {"value": value, "unit": "env-steps/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "env-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, path=None):
        self.index = index
        self.proc = None
        self.path = path
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        if self.path:
            with open(self.path, "w") as f:
                f.write(out)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "first_order_linear_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _recorded_traffic():
    """DRAM bytes per GAE launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "gae_4096x128_traffic.txt")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != _kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def run_ours(args):
    import torch

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from first_order_linear_gb300 import _lib, build
    build.build()
    lib = _lib.load()
    d_cpu = _batch_cpu()
    d = {k: (v.to(dev) if v is not None else None) for k, v in d_cpu.items()}

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    in_bytes = sum(v.numel() * v.element_size() for v in d.values() if v is not None)
    out_bytes = 4 * E * T * 4
    nb = max(2, math.ceil(3 * l2 / (in_bytes + out_bytes)))
    reps = []
    for i in range(nb):
        x = {k: (v.clone() if v is not None else None) for k, v in d.items()}
        x["adv"] = torch.empty(E, T, device=dev)
        x["ret"] = torch.empty(E, T, device=dev)
        x["disc"] = torch.empty(E, T, device=dev)
        x["td"] = torch.empty(E, T, device=dev)
        reps.append(x)
    footprint = nb * (in_bytes + out_bytes)

    P = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = torch.cuda.Stream(dev)
    sptr = C.c_void_p(stream.cuda_stream)

    def launch(x):
        st = lib.rlca_gae(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                          P(x["trunc_value"]), P(x["bootstrap"]), P(x["adv"]), P(x["ret"]), E, T, GAMMA, LAMBDA,
                          0, None, 0, sptr)
        st |= lib.rlca_discounted_return(P(x["rewards"]), P(x["terminated"]), P(x["truncated"]),
                                         P(x["trunc_value"]), P(x["bootstrap"]), P(x["disc"]), E, T, GAMMA, 0,
                                         None, 0, sptr)
        st |= lib.rlca_td_lambda(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                 P(x["trunc_value"]), P(x["bootstrap"]), P(x["td"]), E, T, GAMMA, LAMBDA, 0,
                                 None, 0, sptr)
        if st != 0:
            raise RuntimeError(f"launch failed with status {st}")

    # one CUDA graph per replica: [e0] gae [e1] discounted [e2] td(lambda) [e3]
    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        mk()
        timed_in_graph = True
    except TypeError:
        timed_in_graph = False
    graphs, evs = [], []
    with torch.cuda.stream(stream):
        for x in reps:  # warm the launch path outside capture
            launch(x)
    stream.synchronize()
    for x in reps:
        g = torch.cuda.CUDAGraph()
        ev = [mk() for _ in range(4)] if timed_in_graph else None
        with torch.cuda.graph(g, stream=stream):
            if ev:
                ev[0].record()
            st = lib.rlca_gae(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                              P(x["trunc_value"]), P(x["bootstrap"]), P(x["adv"]), P(x["ret"]), E, T, GAMMA,
                              LAMBDA, 0, None, 0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
            if ev:
                ev[1].record()
            st |= lib.rlca_discounted_return(P(x["rewards"]), P(x["terminated"]), P(x["truncated"]),
                                             P(x["trunc_value"]), P(x["bootstrap"]), P(x["disc"]), E, T, GAMMA,
                                             0, None, 0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
            if ev:
                ev[2].record()
            st |= lib.rlca_td_lambda(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                     P(x["trunc_value"]), P(x["bootstrap"]), P(x["td"]), E, T, GAMMA, LAMBDA,
                                     0, None, 0, C.c_void_p(torch.cuda.current_stream().cuda_stream))
            if ev:
                ev[3].record()
        if st != 0:
            raise RuntimeError(f"capture failed with status {st}")
        graphs.append(g)
        evs.append(ev)

    sampler = ClockSampler(dev.index, os.path.join(ROOT, "gpurun_out", "clocks.csv")
                           if os.path.isdir(os.path.join(ROOT, "gpurun_out")) else None)
    sampler.start()
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            graphs[k % nb].replay()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        t_start.record()
        for k in range(args.steps):
            graphs[k % nb].replay()
        t_end.record()
    stream.synchronize()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = t_start.elapsed_time(t_end)
    if world > 1:
        tt = torch.tensor([ms], device=dev, dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    ms_per_step = ms / args.steps
    value = world * N_EST * E * T * args.steps / (ms / 1e3)

    # per-kernel durations: the last replay of each replica's graph (all inside the timed region)
    per = None
    if timed_in_graph and args.steps >= 1:
        used = range(min(nb, args.steps))
        dur = [[evs[i][j].elapsed_time(evs[i][j + 1]) for i in used] for j in range(3)]
        per = [sum(x) / len(x) for x in dur]
    else:
        per = _graph_kernel_times(lib, reps, P, stream)
    n_trunc = int(d_cpu["truncated"].sum())
    gae_bytes = E * T * (4 + 4 + 1 + 1 + 4 + 4) + 32 * n_trunc + 4 * E
    peak, peak_kind = _peaks()
    achieved = gae_bytes / (per[0] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "em_scan_kernel<GaeEst<true>,32> (rlca_gae)", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                "traffic": _recorded_traffic(), "algorithmic_bytes_per_launch": gae_bytes,
                "avg_launch_us": per[0] * 1e3,
                "timing": "CUDA events recorded inside each replica's graph around the launch"
                if timed_in_graph else "CUDA events around replays of a graph of this kernel's launches"}
    per_est = {name: {"us_per_launch": t * 1e3, "env_steps_per_s": E * T / (t / 1e3)}
               for name, t in zip(("gae", "discounted_return", "td_lambda"), per)}

    e2e = None if args.skip_e2e else run_e2e(args, d_cpu, dev)
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        cpu = cpu_baseline(d_cpu)
    line = {"metric": METRIC, "value": value, "unit": "env-steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": _workload_config({
                "global_batch": world * E, "seq_len": T,
                "l2": f"inputs rotated over {nb} replicas ({footprint / 2**20:.0f} MiB > 3 x L2 "
                      f"{l2 / 2**20:.0f} MiB); no flush",
                "launch": "one CUDA graph per replica (3 kernels), replayed back to back"}),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": N_EST * args.steps, "per_estimator": per_est,
            "wall_s_timed_region": wall}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _graph_kernel_times(lib, reps, P, stream, replays=20):
    """Per-launch time of each estimator from a graph holding only that
    estimator's launches (one per replica), replayed between two events."""
    import torch
    E_, T_ = E, T
    calls = [
        lambda x, s: lib.rlca_gae(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                  P(x["trunc_value"]), P(x["bootstrap"]), P(x["adv"]), P(x["ret"]), E_, T_,
                                  GAMMA, LAMBDA, 0, None, 0, s),
        lambda x, s: lib.rlca_discounted_return(P(x["rewards"]), P(x["terminated"]), P(x["truncated"]),
                                                P(x["trunc_value"]), P(x["bootstrap"]), P(x["disc"]), E_, T_,
                                                GAMMA, 0, None, 0, s),
        lambda x, s: lib.rlca_td_lambda(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                        P(x["trunc_value"]), P(x["bootstrap"]), P(x["td"]), E_, T_, GAMMA,
                                        LAMBDA, 0, None, 0, s),
    ]
    out = []
    for call in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
            for x in reps:
                call(x, s)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            a.record()
            for _ in range(replays):
                g.replay()
            b.record()
        stream.synchronize()
        out.append(a.elapsed_time(b) / (replays * len(reps)))
    return out


def run_e2e(args, d_cpu, dev):
    """Same metric through the public Python API with host buffers: every
    step copies its inputs from pinned host memory to the device, runs the
    three estimators and copies their four outputs back."""
    import torch
    from first_order_linear_gb300 import rlca

    host = {k: (v.pin_memory() if v is not None else None) for k, v in d_cpu.items()}
    devb = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in d_cpu.items()}
    outs = [torch.empty(E, T, device=dev) for _ in range(4)]
    back = [torch.empty(E, T, pin_memory=True) for _ in range(4)]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sum(b.numel() * b.element_size() for b in back)
    steps = max(10, min(args.steps, 2000))

    def step():
        for k, v in host.items():
            if v is not None:
                devb[k].copy_(v, non_blocking=True)
        rlca.rlca_gae(devb["rewards"], devb["values"], devb["terminated"], devb["truncated"],
                      devb["trunc_value"], devb["bootstrap"], gamma=GAMMA, lambda_=LAMBDA,
                      advantages=outs[0], returns=outs[1])
        rlca.rlca_discounted_return(devb["rewards"], devb["terminated"], devb["truncated"], devb["trunc_value"],
                                    devb["bootstrap"], gamma=GAMMA, out=outs[2])
        rlca.rlca_td_lambda(devb["rewards"], devb["values"], devb["terminated"], devb["truncated"],
                            devb["trunc_value"], devb["bootstrap"], gamma=GAMMA, lambda_=LAMBDA, out=outs[3])
        for o, b in zip(outs, back):
            b.copy_(o, non_blocking=True)

    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        for _ in range(3):
            step()
        s.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            step()
        b.record()
    s.synchronize()
    ms = a.elapsed_time(b)
    return {"value": N_EST * E * T * steps / (ms / 1e3), "unit": "env-steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
