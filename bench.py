"""Throughput of the credit-assignment scans on one or more GPUs.

Workload: GAE + discounted returns + TD(lambda), float32, 4096 environments x
128 steps, env-major [E, T]; rewards and values N(0, 1), termination 1%,
truncation 0.5% with N(0, 1) continuation values, N(0, 1) bootstrap values,
gamma = 0.99, lambda = 0.95 (the "thousands of environments, short
rollouts" regime of rl-triton, arXiv:2608.17641, §6-§7).

One step = GAE, discounted returns and TD(lambda) of one batch, computed by
one fused launch (rlca_value_targets) that writes advantages, returns
(which are the TD(lambda) returns, bit for bit) and discounted returns; the
three separate entry points are timed as well.  The metric is env-steps per
second per estimator: E * T * steps / time (each step evaluates all three
estimators over the same E * T env-steps).  Inputs stay resident in HBM;
the timed steps rotate over enough replicas of the batch that their
footprint exceeds three times the L2 cache, so every step reads from DRAM.
The K timed launches are one CUDA graph whose first and last nodes are the
two timing events, so the time is the device's from the first launch to
the last, whatever K is.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle (the C reference, over all host cores) on the same workload instead.
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
# longest timed region captured as a single graph bracketed by its own events
MAX_GRAPH_STEPS = 50000


def _workload_config(extra=None):
    cfg = {"workload": WORKLOAD, "E": E, "T": T, "layout": "env-major [E,T]",
           "estimators": ["gae(adv+ret)", "discounted_return", "td_lambda"],
           "gamma": GAMMA, "lambda": LAMBDA, "p_terminated": P_TERM, "p_truncated": P_TRUNC,
           "parallelism": "replicas (env-sharded, no collective)"}
    if extra:
        cfg.update(extra)
    return cfg


def _batch_cpu(rank=0):
    """This rank's shard of the job: environments [rank * E, (rank + 1) * E)
    of a world * E environment batch, each shard from its own seed."""
    from first_order_linear_gb300 import synth
    name = "4096x128" if rank == 0 else f"4096x128-shard{rank}"
    return synth.value_rollout(E, T, seed=synth.config_seed(name), p_term=P_TERM, p_trunc=P_TRUNC,
                               with_trunc=True, device="cpu")


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _max_over_ranks(x, device):
    """The largest x of all ranks (the job's time is its slowest rank's);
    x itself when no process group is up."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(world, ms, steps):
    """Whole-job throughput per estimator: every rank processed its own
    E x T shard per step (for each of the N_EST estimators), in the slowest
    rank's time."""
    return world * E * T * steps / (ms / 1e3)


# --------------------------------------------------------------------------
# CPU oracle (the reported baseline and the reference arm)
# --------------------------------------------------------------------------

def _oracle_inputs(d, rows):
    """The first ``rows`` environments of a batch as float64 / uint8 NumPy
    arrays (converted once, outside any timing)."""
    import numpy as np
    from first_order_linear_gb300 import synth
    n = synth.numpy(d)
    out = {}
    for k, v in n.items():
        if isinstance(v, np.ndarray):
            v = v[:rows]
            v = np.ascontiguousarray(v.astype(np.uint8) if v.dtype == np.bool_ or v.dtype == np.uint8
                                     else v.astype(np.float64))
        out[k] = v
    return out


def _oracle_step(ref, n):
    """GAE, discounted return and TD(lambda) of one batch with one oracle
    module (the NumPy one or the C one: same signatures)."""
    ref.gae(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
            gamma=GAMMA, lam=LAMBDA)
    ref.discounted_return(n["rewards"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
                          gamma=GAMMA)
    ref.td_lambda(n["rewards"], n["values"], n["terminated"], n["truncated"], n["trunc_value"], n["bootstrap"],
                  gamma=GAMMA, lam=LAMBDA)


def _row_slices(n, parts):
    """``n`` split into ``parts`` contiguous row ranges (the oracle's rows
    are independent)."""
    rows = n["rewards"].shape[0]
    cuts = [rows * i // parts for i in range(parts + 1)]
    out = []
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        if hi > lo:
            out.append({k: (v[lo:hi] if getattr(v, "ndim", 0) >= 1 else v) for k, v in n.items()})
    return out


class OracleRunner:
    """The C oracle (oracle/rlca_ref.c, float64 loops over one row at a
    time) run over a batch by ``threads`` host threads, each on its own
    contiguous block of environments.  ctypes releases the interpreter lock
    during the C loops, so the threads run in parallel."""

    def __init__(self, threads):
        import concurrent.futures as cf
        from oracle import ref_c
        ref_c.load()
        self.ref = ref_c
        self.threads = threads
        self.pool = cf.ThreadPoolExecutor(max_workers=threads) if threads > 1 else None

    def step(self, n):
        if self.pool is None:
            _oracle_step(self.ref, n)
            return
        for f in [self.pool.submit(_oracle_step, self.ref, part) for part in _row_slices(n, self.threads)]:
            f.result()

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _time_oracle(step, n, budget_s):
    """Repeats ``step(n)`` for about ``budget_s`` seconds; (repeats, seconds)."""
    step(n)  # first call: library load, page faults
    reps, t0 = 0, time.perf_counter()
    while True:
        step(n)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 2000:
            return reps, el


def cpu_baseline(d, budget_s=6.0):
    """The oracle as it stands, on the host: the C reference over all host
    cores (the reported value), and single-threaded figures of the C and
    the NumPy references beside it."""
    from oracle import rlca_ref
    n = _oracle_inputs(d, E)
    cores = _host_cores()
    runner = OracleRunner(cores)
    try:
        reps, el = _time_oracle(runner.step, n, budget_s)
    finally:
        runner.close()
    one = OracleRunner(1)
    reps1, el1 = _time_oracle(one.step, n, budget_s / 2)
    nrows = max(64, E // 8)
    sub = _oracle_inputs(d, nrows)
    repsn, eln = _time_oracle(lambda x: _oracle_step(rlca_ref, x), sub, budget_s / 2)
    return {"value": E * T * reps / el, "unit": "env-steps/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} full {E}x{T} batches (GAE, discounted return, TD(lambda) each) through the C "
                      f"float64 oracle, rows split over {cores} host threads, {el:.1f} s",
            "c_oracle_1_thread": {"value": E * T * reps1 / el1, "cores": 1,
                                  "sample": f"{reps1} full batches, {el1:.1f} s"},
            "numpy_oracle_1_thread": {"value": nrows * T * repsn / eln, "cores": 1,
                                      "sample": f"{repsn} batches of the first {nrows} envs, {eln:.1f} s"}}


ORACLE_CONFIGS = [("gae 8x16", 8, 16), ("gae+disc+td 4096x128", 4096, 128), ("vtrace 4096x256", 4096, 256),
                  ("retrace 1024x2048", 1024, 2048)]


def run_oracle_configs(args):
    """The C oracle on each named configuration, one host thread and all of
    them (rows split across threads): env-steps per second per estimator,
    one JSON line per configuration.  Timed for about --oracle-seconds each."""
    import numpy as np
    from first_order_linear_gb300 import synth
    cores = _host_cores()
    budget = args.oracle_seconds
    for name, E_, T_ in ORACLE_CONFIGS:
        seed = synth.config_seed(name)
        if name.startswith("gae"):
            d = synth.value_rollout(E_, T_, seed, p_term=0.05 if E_ == 8 else P_TERM,
                                    p_trunc=0.02 if E_ == 8 else P_TRUNC, with_trunc=True)
            fns = ["gae"] if E_ == 8 else ["gae", "discounted_return", "td_lambda"]
        elif name.startswith("vtrace"):
            d = synth.vtrace_rollout(E_, T_, seed, p_term=0.01)
            fns = ["vtrace"]
        else:
            d = synth.retrace_rollout(E_, T_, seed, p_term=0.002)
            fns = ["retrace"]
        n = _oracle_inputs(d, E_)

        def one(x, fns=fns):
            from oracle import ref_c
            for f in fns:
                if f == "gae":
                    ref_c.gae(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                              x["bootstrap"], gamma=GAMMA, lam=LAMBDA)
                elif f == "discounted_return":
                    ref_c.discounted_return(x["rewards"], x["terminated"], x["truncated"], x["trunc_value"],
                                            x["bootstrap"], gamma=GAMMA)
                elif f == "td_lambda":
                    ref_c.td_lambda(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                                    x["bootstrap"], gamma=GAMMA, lam=LAMBDA)
                elif f == "vtrace":
                    ref_c.vtrace(x["rewards"], x["values"], x["logp_target"], x["logp_behaviour"],
                                 x["terminated"], x.get("truncated"), x.get("trunc_value"), x["bootstrap"],
                                 gamma=GAMMA)
                else:
                    ref_c.retrace(x["q"], x["pi"], x["mu_a"], x["actions"], x["rewards"], x["terminated"],
                                  x.get("truncated"), x.get("trunc_value"), x["bootstrap"], gamma=GAMMA,
                                  lam=LAMBDA)
        line = {"oracle_config": name, "E": E_, "T": T_, "estimators": fns, "unit": "env-steps/s per estimator"}
        for threads in (1, cores):
            pool = None
            if threads > 1:
                import concurrent.futures as cf
                pool = cf.ThreadPoolExecutor(max_workers=threads)
                parts = _row_slices(n, threads)

                def step(x, pool=pool, parts=parts):
                    for f in [pool.submit(one, p) for p in parts]:
                        f.result()
            else:
                step = one
            reps, el = _time_oracle(step, n, budget)
            if pool is not None:
                pool.shutdown()
            line[f"threads_{threads}"] = {"value": E_ * T_ * reps / el, "reps": reps, "seconds": round(el, 2)}
        print(json.dumps(line), flush=True)
    return 0


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    d = _batch_cpu()
    cores = _host_cores()
    runner = OracleRunner(cores)
    n = _oracle_inputs(d, E)
    t0 = time.perf_counter()
    runner.step(n)
    t_full = time.perf_counter() - t0
    # bound the whole run to about a minute of CPU work
    rows = E if (args.steps + args.warmup) * t_full <= 60.0 else max(
        cores, int(E * 60.0 / ((args.steps + args.warmup) * t_full)))
    sub = _oracle_inputs(d, rows)
    for _ in range(args.warmup):
        runner.step(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runner.step(sub)
    el = time.perf_counter() - t0
    runner.close()
    value = rows * T * args.steps / el
    sample = (f"first {rows} of {E} envs x {T} steps per step, GAE + discounted return + TD(lambda), C float64 "
              f"oracle, rows split over {cores} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "env-steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _workload_config({"rows_per_step": rows}),
            "cpu_baseline": {"value": value, "unit": "env-steps/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "env-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi polling the GPU's clocks and throttle reasons every 100 ms
    on a reader thread.  Started well before a timed region and waited for
    (``wait_first``): nvidia-smi's start-up, overlapping a short timed region,
    measured a few microseconds slower on it."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, path=None):
        self.index = index
        self.proc = None
        self.path = path
        self.lines = []
        self.thread = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def wait_first(self, timeout=10.0):
        """Block until the first sample is in (or the timeout passes)."""
        t0 = time.perf_counter()
        while self.proc is not None and not self.lines and self.proc.poll() is None \
                and time.perf_counter() - t0 < timeout:
            time.sleep(0.01)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        out = "".join(self.lines)
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
    """DRAM bytes per fused value-target launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "value_targets_4096x128_traffic.txt")
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


def _calls(lib, P):
    """The C-ABI calls of one step's estimators on a replica x and stream s."""
    def fused(x, s, flags=0x10, td=None):  # RLCA_INPUTS_READY: each step's inputs are resident before the timed region
        # the returns written to ret are the TD(lambda) returns, bit for bit:
        # the step writes them once (td=None), not a second identical copy
        return lib.rlca_value_targets(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                      P(x["trunc_value"]), P(x["bootstrap"]), P(x["adv"]), P(x["ret"]), P(x["disc"]),
                                      P(td), E, T, GAMMA, LAMBDA, flags, None, 0, s)

    def fused_serial(x, s):
        return fused(x, s, flags=0)

    def fused_td_copy(x, s):
        return fused(x, s, td=x["td"])

    def gae(x, s):
        return lib.rlca_gae(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                            P(x["trunc_value"]), P(x["bootstrap"]), P(x["adv"]), P(x["ret"]), E, T, GAMMA, LAMBDA,
                            0, None, 0, s)

    def disc(x, s):
        return lib.rlca_discounted_return(P(x["rewards"]), P(x["terminated"]), P(x["truncated"]),
                                          P(x["trunc_value"]), P(x["bootstrap"]), P(x["disc"]), E, T, GAMMA, 0,
                                          None, 0, s)

    def td(x, s):
        return lib.rlca_td_lambda(P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                                  P(x["trunc_value"]), P(x["bootstrap"]), P(x["td"]), E, T, GAMMA, LAMBDA, 0, None,
                                  0, s)
    return fused, fused_serial, fused_td_copy, gae, disc, td


def _capture(reps, fns, stream):
    """One CUDA graph holding, for each replica in order, the given calls."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        for x in reps:
            for f in fns:
                st = f(x, s)
                if st != 0:
                    raise RuntimeError(f"capture failed with status {st}")
    return g


def _timed_graph(reps, fn, stream, steps, first=0):
    """One CUDA graph of ``steps`` launches of ``fn`` on consecutive replicas
    (starting at replica ``first``), with a timing event recorded as the
    graph's first node and another as its last: the events time the device
    from the first launch to the end of the last, without the host's graph
    submission.  Returns (graph, start event, end event), or None when this
    PyTorch cannot record events inside a capture."""
    import torch
    try:
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        s = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        a.record()
        for i in range(steps):
            st = fn(reps[(first + i) % len(reps)], s)
            if st != 0:
                raise RuntimeError(f"capture failed with status {st}")
        b.record()
    return g, a, b


def _upload(g, stream):
    """cudaGraphUpload of a captured graph on ``stream``: a graph's first
    replay otherwise uploads its launch work node by node as it runs
    (measured here at 0.3-0.5 us per launch node), a one-time cost of the
    graph, not of the steps it holds.  Returns True when the upload ran."""
    import torch
    try:
        handle = g.raw_cuda_graph_exec()
        rt = C.CDLL("libcudart.so.13")
        rt.cudaGraphUpload.argtypes = [C.c_void_p, C.c_void_p]
        rt.cudaGraphUpload.restype = C.c_int
        ok = rt.cudaGraphUpload(C.c_void_p(handle), C.c_void_p(stream.cuda_stream)) == 0
    except (AttributeError, OSError, RuntimeError, TypeError):
        return False
    stream.synchronize()
    torch.cuda.synchronize()
    return ok


def _graph_us(g, launches, stream, replays=20):
    """Average time per launch of a graph replayed back to back."""
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        a.record()
        for _ in range(replays):
            g.replay()
        b.record()
    stream.synchronize()
    return a.elapsed_time(b) * 1e3 / (replays * launches)


def _full_call_us(fn, items, stream, n=200):
    """Host wall time per call of ``fn(item)`` issued back to back in plain
    stream order (argument checks, marshalling and launch included, one
    synchronisation at each end): the full-call time, as a caller sees it."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(min(5, n)):
            fn(items[i % len(items)])
        stream.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            fn(items[i % len(items)])
        stream.synchronize()
    return (time.perf_counter() - t0) / n * 1e6


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
    d_cpu = _batch_cpu(rank)
    d = {k: (v.to(dev) if v is not None else None) for k, v in d_cpu.items()}

    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    in_bytes = sum(v.numel() * v.element_size() for v in d.values() if v is not None)
    out_bytes = 4 * E * T * 4
    nb = max(2, math.ceil(3 * l2 / (in_bytes + out_bytes)))
    reps = []
    for i in range(nb):
        x = {k: (v.clone() if v is not None else None) for k, v in d.items()}
        for k in ("adv", "ret", "disc", "td"):
            x[k] = torch.empty(E, T, device=dev)
        reps.append(x)
    footprint = nb * (in_bytes + out_bytes)

    P = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    fused, fused_serial, fused_td_copy, gae, disc, td = _calls(lib, P)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):  # first calls (device attribute cache) outside capture
        for x in reps:
            for f in (fused, fused_serial, gae, disc, td):
                if f(x, C.c_void_p(stream.cuda_stream)) != 0:
                    raise RuntimeError("launch failed")
    stream.synchronize()

    # the timed region: one fused launch per step, consecutive steps on
    # consecutive replicas.  The warm-up steps are a graph of their own; the
    # K timed steps are one graph bracketed by its own timing events (for K
    # up to MAX_GRAPH_STEPS), so a short run measures the same steady state
    # as a long one.  Beyond that: graphs of one rotation, replayed back to
    # back, every one of them replayed once before the timed region.
    warm = _capture([reps[i % nb] for i in range(args.warmup)], [fused], stream)
    timed = _timed_graph(reps, fused, stream, args.steps, first=args.warmup) \
        if args.steps <= MAX_GRAPH_STEPS else None
    full = rem = None
    uploaded = False
    if timed is not None:
        uploaded = _upload(timed[0], stream)
    if timed is None:
        full = _capture(reps, [fused], stream)
        rem_n = args.steps % nb
        rem = _capture(reps[:rem_n], [fused], stream) if rem_n else None
        with torch.cuda.stream(stream):
            full.replay()
            if rem is not None:
                rem.replay()
        stream.synchronize()

    sampler = ClockSampler(dev.index, args.clock_log or None)
    sampler.start()
    sampler.wait_first()
    if timed is not None:
        # one untimed replay of the timed graph: a graph's first replay has
        # measured up to ~3 us slower than later ones even after the upload,
        # a one-time cost of the graph.  Its replicas then leave L2 through
        # a write of 2 x L2 before the warm-up steps run on other replicas.
        with torch.cuda.stream(stream):
            timed[0].replay()
            torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)
    with torch.cuda.stream(stream):
        warm.replay()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    if timed is not None:
        g_timed, t_start, t_end = timed
        with torch.cuda.stream(stream):
            g_timed.replay()
        timing_how = ("one CUDA graph of the K launches whose first and last nodes are the two CUDA events "
                      "(device time from the first launch to the end of the last)"
                      + ("; the graph uploaded (cudaGraphUpload) and replayed once, untimed, before the warm-up "
                         "steps, then L2 overwritten (2 x L2)" if uploaded else
                         "; graph not uploaded beforehand; replayed once, untimed, before the warm-up steps, "
                         "then L2 overwritten (2 x L2)"))
    else:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t_start.record()
            for _ in range(args.steps // nb):
                full.replay()
            if rem is not None:
                rem.replay()
            t_end.record()
        timing_how = ("CUDA events on the launching stream around back-to-back replays of graphs of one "
                      "rotation (each replayed once before)")
    stream.synchronize()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = t_start.elapsed_time(t_end)
    ms = _max_over_ranks(ms, dev)
    ms_per_step = ms / args.steps
    value = _job_value(world, ms, args.steps)
    del warm, full, rem, timed

    # per-kernel figures, each from a graph of one rotation of that launch
    kern = {}
    for name, fns in (("value_targets_fused", [fused]), ("value_targets_fused_without_inputs_ready", [fused_serial]),
                      ("value_targets_fused_with_separate_td_copy", [fused_td_copy]),
                      ("gae", [gae]), ("discounted_return", [disc]), ("td_lambda", [td]),
                      ("unfused_step_gae_disc_td", [gae, disc, td])):
        g = _capture(reps, fns, stream)
        us = _graph_us(g, nb, stream)
        kern[name] = {"us_per_launch" if len(fns) == 1 else "us_per_step": us,
                      "env_steps_per_s_per_estimator": E * T / (us / 1e6)}
        del g
    # the public Python call (rlca.rlca_value_targets), launches in plain
    # stream order without graphs: host wall time per call
    from first_order_linear_gb300 import rlca

    def api_call(x):
        rlca.rlca_value_targets(x["rewards"], x["values"], x["terminated"], x["truncated"], x["trunc_value"],
                                x["bootstrap"], gamma=GAMMA, lambda_=LAMBDA, advantages=x["adv"], returns=x["ret"],
                                disc_returns=x["disc"], td_lambda_returns=x["td"], inputs_ready=True, stream=stream)
    kern["value_targets_full_call"] = {"us_per_call": _full_call_us(api_call, reps, stream),
                                       "timing": "host wall clock over 200 back-to-back public-API calls"}
    n_trunc = int(d_cpu["truncated"].sum())
    # read r, V (4 B), two flag bytes; write adv, ret (= TD(lambda)), disc
    # (4 B); the truncation values at one 32-byte sector per truncated step;
    # the bootstrap vector
    fused_bytes = E * T * (4 + 4 + 1 + 1 + 3 * 4) + 32 * n_trunc + 4 * E
    peak, peak_kind = _peaks()
    # context, not the path: a plain torch device copy moving the same bytes
    # per launch (half read, half written), captured and replayed the same
    # way over replicas larger than 3 x L2 -- what one launch of this size
    # reaches on this machine
    n_copy = fused_bytes // 8
    srcs = [torch.zeros(n_copy, device=dev) for _ in range(nb)]
    dsts = [torch.empty(n_copy, device=dev) for _ in range(nb)]
    with torch.cuda.stream(stream):
        for a_, b_ in zip(srcs, dsts):
            b_.copy_(a_)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for a_, b_ in zip(srcs, dsts):
            b_.copy_(a_)
    us_copy = _graph_us(g, nb, stream)
    kern["torch_copy_same_bytes"] = {"us_per_launch": us_copy, "bytes_per_launch": 8 * n_copy,
                                     "frac_of_peak": 8 * n_copy / (us_copy / 1e6) / 1e9 / peak}
    del g, srcs, dsts
    avg_us = ms_per_step * 1e3
    achieved = fused_bytes / (avg_us / 1e6) / 1e9
    roofline = {"bound": "hbm", "kernel": "em_fast_kernel<ValueTargetsEst<true>,32,4> (rlca_value_targets)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} hbm_gbs", "traffic": _recorded_traffic(),
                "algorithmic_bytes_per_launch": fused_bytes,
                "algorithmic_bytes_note": "22 B per env-step (r, V, 2 flags in; adv, ret = TD(lambda), disc out) "
                                          "+ 32 B per truncated step + 4 B per env; a separate TD(lambda) copy "
                                          "(bit-identical to ret) is not written and not counted",
                "avg_launch_us": avg_us, "timing": "timed region / steps: " + timing_how}

    e2e = None if args.skip_e2e else run_e2e(args, d_cpu, dev)
    if e2e is not None and world > 1:
        # whole job: every rank's shard through its own host link, in the
        # slowest rank's time
        e2e_ms = _max_over_ranks(e2e["ms_per_step"], dev)
        e2e.update(ms_per_step=e2e_ms, value=world * E * T / (e2e_ms / 1e3),
                   h2d_bytes_per_step=world * e2e["h2d_bytes_per_step"],
                   d2h_bytes_per_step=world * e2e["d2h_bytes_per_step"], ranks=world)
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
                "launch": "one fused rlca_value_targets launch per step with RLCA_INPUTS_READY (inputs resident "
                          "before the timed region, so consecutive steps overlap through programmatic dependent "
                          "launch), writing advantages, returns (= TD(lambda) returns) and discounted returns; "
                          + timing_how}),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": args.steps, "kernels": kern, "wall_s_timed_region": wall}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_e2e(args, d_cpu, dev):
    """Same metric end to end through the C ABI with host buffers: every step
    copies its inputs from pinned host memory to the device, runs the fused
    value-target call (rlca_value_targets) and copies its three outputs back
    to pinned host memory.  Steps are pipelined as a data loader would: the
    copy in on one stream, the call on a second, the copy out on a third,
    over two device buffer sets, so step k's inputs arrive while step k-1
    computes and step k-2's outputs leave.  A step's inputs sit packed in one
    pinned block and its outputs in one [3, E, T] block: one copy each way.
    The pipeline of STEPS_PER_GRAPH steps is captured once as a CUDA graph
    (copies, calls and the streams' event dependencies) and replayed, so the
    host issues one launch per STEPS_PER_GRAPH steps.  The same graph without
    the calls gives the host link's ceiling for this step."""
    import torch
    from first_order_linear_gb300 import _lib

    lib = _lib.load()
    names = [k for k, v in d_cpu.items() if v is not None]
    offs, size = {}, 0
    for k in names:  # every tensor starts on a 256-byte boundary
        offs[k] = size
        size += -(-d_cpu[k].numel() * d_cpu[k].element_size() // 256) * 256

    def views(block):
        return {k: (block[offs[k]:offs[k] + d_cpu[k].numel() * d_cpu[k].element_size()].view(d_cpu[k].dtype)
                    .view(d_cpu[k].shape) if k in offs else None) for k in d_cpu}

    host_block = torch.empty(size, dtype=torch.uint8, pin_memory=True)
    for k, v in views(host_block).items():
        if v is not None:
            v.copy_(d_cpu[k])
    NB = args.e2e_buffers
    LANES = args.e2e_lanes
    dev_blocks = [torch.empty(size, dtype=torch.uint8, device=dev) for _ in range(NB)]
    devb = [views(blk) for blk in dev_blocks]
    outs = [torch.empty(3, E, T, device=dev) for _ in range(NB)]
    back = [torch.empty(3, E, T, pin_memory=True) for _ in range(NB)]

    def pieces(n):
        """LANES contiguous [lo, hi) ranges of n elements (each copy engine one)."""
        cuts = [n * i // LANES for i in range(LANES + 1)]
        return list(zip(cuts[:-1], cuts[1:]))
    in_pieces = pieces(size)
    out_pieces = pieces(back[0].numel())
    h2d = sum(d_cpu[k].numel() * d_cpu[k].element_size() for k in names)
    d2h = back[0].numel() * back[0].element_size()
    STEPS_PER_GRAPH = 20
    P = lambda t: C.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    s_main = torch.cuda.Stream(dev)
    s_ins = [torch.cuda.Stream(dev) for _ in range(LANES)]
    s_outs = [torch.cuda.Stream(dev) for _ in range(LANES)]
    s_run = torch.cuda.Stream(dev)

    def capture(call):
        """One graph of STEPS_PER_GRAPH pipelined steps (fork from the
        capture stream onto the three pipeline streams, join at the end)."""
        ev_in = [[torch.cuda.Event() for _ in range(LANES)] for _ in range(NB)]
        ev_run = [torch.cuda.Event() for _ in range(NB)]
        ev_out = [[torch.cuda.Event() for _ in range(LANES)] for _ in range(NB)]
        started = [False] * NB
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s_main):
            for st in s_ins + s_outs + [s_run]:
                st.wait_stream(s_main)
            for i in range(STEPS_PER_GRAPH):
                j = i % NB
                x, o = devb[j], outs[j]
                for lane, (lo, hi) in enumerate(in_pieces):  # the copy in, one piece per copy stream
                    with torch.cuda.stream(s_ins[lane]):
                        if started[j]:
                            s_ins[lane].wait_event(ev_run[j])  # this buffer set's previous call has read its inputs
                        dev_blocks[j][lo:hi].copy_(host_block[lo:hi], non_blocking=True)
                        ev_in[j][lane].record(s_ins[lane])
                with torch.cuda.stream(s_run):
                    for e in ev_in[j]:
                        s_run.wait_event(e)
                    if started[j]:
                        for e in ev_out[j]:
                            s_run.wait_event(e)  # its previous outputs have left
                    if call:
                        st = lib.rlca_value_targets(
                            P(x["rewards"]), P(x["values"]), P(x["terminated"]), P(x["truncated"]),
                            P(x["trunc_value"]), P(x["bootstrap"]), P(o[0]), P(o[1]), P(o[2]), None, E, T, GAMMA,
                            LAMBDA, 0, None, 0, C.c_void_p(s_run.cuda_stream))
                        if st != 0:
                            raise RuntimeError(f"rlca_value_targets failed with status {st}")
                    ev_run[j].record(s_run)
                for lane, (lo, hi) in enumerate(out_pieces):  # the copy out, likewise
                    with torch.cuda.stream(s_outs[lane]):
                        s_outs[lane].wait_event(ev_run[j])
                        back[j].view(-1)[lo:hi].copy_(o.view(-1)[lo:hi], non_blocking=True)
                        ev_out[j][lane].record(s_outs[lane])
                started[j] = True
            for st in s_ins + s_outs + [s_run]:
                s_main.wait_stream(st)
        _upload(g, s_main)
        return g

    def timed(g, reps):
        with torch.cuda.stream(s_main):
            g.replay()  # warm-up replay
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_main):
            a.record()
            for _ in range(reps):
                g.replay()
            b.record()
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b), reps * STEPS_PER_GRAPH

    reps = max(1, min(args.steps, 2000) // STEPS_PER_GRAPH)
    g_call = capture(True)
    ms, steps = timed(g_call, reps)
    del g_call
    g_link = capture(False)
    ms_link, _ = timed(g_link, reps)
    del g_link
    # the results of the last step reached the host: check them against the
    # device outputs (the copies are part of the step, not a formality)
    torch.cuda.synchronize(dev)
    last = (steps - 1) % NB
    if not torch.equal(back[last], outs[last].cpu()):
        raise RuntimeError("e2e: host copy of the outputs differs from the device outputs")
    return {"value": E * T * steps / (ms / 1e3), "unit": "env-steps/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "host_link_ceiling": {"value": E * T * steps / (ms_link / 1e3), "ms_per_step": ms_link / steps,
                                  "GBps_in_plus_out": (h2d + d2h) * steps / (ms_link / 1e3) / 1e9,
                                  "how": "the same pipelined pinned copies in and out, without the call"},
            "frac_of_host_link_ceiling": ms_link / ms,
            "pipeline": f"per step the packed pinned-host inputs copied in as {LANES} pieces on {LANES} streams, "
                        f"the C-ABI call on its own stream, the packed outputs copied out as {LANES} pieces on {LANES} "
                        f"more, over {NB} device buffer sets; {STEPS_PER_GRAPH} steps per CUDA graph, replayed"}


# --------------------------------------------------------------------------
# --sweep: device throughput of every estimator on the benchmark shapes
# --------------------------------------------------------------------------

SWEEP_KINDS = ("gae", "disc", "td", "vt", "vtrace", "retrace", "elig", "psum")
# (E, T, time_major, truncation): the named configurations, then the E x T grid in both layouts
SWEEP_SHAPES = [(4096, 128, False, True), (4096, 256, False, False), (1024, 2048, False, False)]
SWEEP_SHAPES += [(E, T, tm, tr) for E in (256, 1024, 4096, 16384) for T in (32, 128, 512, 2048)
                 for tm in (False, True) for tr in (False, True)]


def _sweep_case(kind, E, T, trunc, dev, bf16=False):
    """Seeded inputs (env-major), the algorithmic bytes of one call, and the
    output buffers' shapes and dtypes.  bf16: the float arrays are bfloat16
    (RLCA_BF16), 2 bytes per element."""
    import torch
    from first_order_linear_gb300 import synth
    seed = synth.config_seed(f"bench-{kind}-{E}-{T}-{trunc}")
    A = synth.NUM_ACTIONS
    fdt = torch.bfloat16 if bf16 else torch.float32
    fe = 2 if bf16 else 4
    if kind in ("gae", "disc", "td", "vt"):
        d = synth.value_rollout(E, T, seed, p_term=P_TERM, p_trunc=P_TRUNC, with_trunc=trunc, device=dev)
        reads = {"gae": 2, "disc": 1, "td": 2, "vt": 2}[kind] * fe + 1
        outs = {"gae": 2, "disc": 1, "td": 1, "vt": 3}[kind]  # vt: adv, ret (= TD(lambda)), disc
        spec = [((E, T), fdt)] * outs
    elif kind == "vtrace":
        d = synth.vtrace_rollout(E, T, seed, p_term=0.01, p_trunc=P_TRUNC if trunc else 0.0, with_trunc=trunc,
                                 device=dev)
        reads, spec = 4 * fe + 1, [((E, T), fdt)] * 2
    elif kind == "retrace":
        d = synth.retrace_rollout(E, T, seed, p_term=0.002, p_trunc=P_TRUNC if trunc else 0.0, with_trunc=trunc,
                                  device=dev)
        reads, spec = 2 * A * fe + fe + 4 + fe + 1, [((E, T), fdt)]
    else:
        d = synth.forward_rollout(E, T, seed, p_term=0.01, p_trunc=P_TRUNC, with_trunc=trunc, device=dev)
        reads, spec = fe + 1, [((E, T), fdt if kind == "elig" else torch.int32)]
    if bf16:
        d = {k: (v.to(torch.bfloat16) if isinstance(v, torch.Tensor) and v.dtype == torch.float32 else v)
             for k, v in d.items()}
    n_trunc = int(d["truncated"].sum()) if d.get("truncated") is not None else 0
    per_step = reads + (1 if d.get("truncated") is not None else 0) + sum(
        torch.empty(0, dtype=dt).element_size() for _, dt in spec)
    tv_bytes = 32 * n_trunc if kind in ("gae", "disc", "td", "vt", "vtrace", "retrace") else 0
    return d, per_step * E * T + tv_bytes, spec


def _sweep_call(kind, x, o, tm, ready=False):
    from first_order_linear_gb300 import rlca
    kw = dict(time_major=tm, inputs_ready=ready)
    b = (x.get("terminated"), x.get("truncated"), x.get("trunc_value"), x.get("bootstrap"))
    if kind == "gae":
        rlca.rlca_gae(x["rewards"], x["values"], *b, gamma=GAMMA, lambda_=LAMBDA, advantages=o[0], returns=o[1], **kw)
    elif kind == "disc":
        rlca.rlca_discounted_return(x["rewards"], *b, gamma=GAMMA, out=o[0], **kw)
    elif kind == "td":
        rlca.rlca_td_lambda(x["rewards"], x["values"], *b, gamma=GAMMA, lambda_=LAMBDA, out=o[0], **kw)
    elif kind == "vt":
        rlca.rlca_value_targets(x["rewards"], x["values"], *b, gamma=GAMMA, lambda_=LAMBDA, advantages=o[0],
                                returns=o[1], disc_returns=o[2], outputs=("advantages", "returns", "disc_returns"),
                                **kw)
    elif kind == "vtrace":
        rlca.rlca_vtrace(x["rewards"], x["values"], x["logp_target"], x["logp_behaviour"], *b, gamma=GAMMA, vs=o[0],
                         pg_advantages=o[1], **kw)
    elif kind == "retrace":
        rlca.rlca_retrace(x["q"], x["pi"], x["mu_a"], x["actions"], x["rewards"], *b, gamma=GAMMA, lambda_=LAMBDA,
                          out=o[0], **kw)
    elif kind == "elig":
        rlca.rlca_elig_trace(x["x_f32"], x["terminated"], x["truncated"], gamma=GAMMA, lambda_=LAMBDA, out=o[0], **kw)
    else:
        rlca.rlca_episodic_prefix_sum(x["x_i32"], x["terminated"], x["truncated"], out=o[0], **kw)


def run_sweep(args):
    """One JSON line per (estimator, E, T, layout, truncation): device time per
    call from CUDA graphs of back-to-back calls on replicas whose footprint
    exceeds 3 x L2, algorithmic bytes, achieved GB/s and fraction of peak;
    once in plain stream order and once with RLCA_INPUTS_READY (consecutive
    calls on independent replicas overlap)."""
    import torch
    from first_order_linear_gb300 import build, synth
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    peak, peak_kind = _peaks()
    kinds = args.sweep_kinds.split(",") if args.sweep_kinds else SWEEP_KINDS
    if args.sweep_dtype == "bf16":  # int32 prefix sums keep their storage
        kinds = [k for k in kinds if k != "psum"]
    shapes = SWEEP_SHAPES
    stream = torch.cuda.Stream(dev)
    for kind in kinds:
        for E, T, tm, trunc in shapes:
            d, nbytes, spec = _sweep_case(kind, E, T, trunc, dev, bf16=args.sweep_dtype == "bf16")
            foot = sum(v.numel() * v.element_size() for v in d.values() if isinstance(v, torch.Tensor))
            foot += sum(E * T * torch.empty(0, dtype=dt).element_size() for _, dt in spec)
            nb = max(2, min(64, math.ceil(3 * l2 / foot)))
            src = {k: (synth.to_time_major(v) if tm and isinstance(v, torch.Tensor) else v) for k, v in d.items()}
            reps = []
            for i in range(nb):
                x = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in src.items()}
                o = [torch.empty(sh if not tm else (sh[1], sh[0]), dtype=dt, device=dev) for sh, dt in spec]
                reps.append((x, o))
            del src
            with torch.cuda.stream(stream):
                for x, o in reps:
                    _sweep_call(kind, x, o, tm)
            stream.synchronize()
            times = {}
            for ready in (False, True):
                with torch.cuda.stream(stream):
                    _sweep_call(kind, reps[0][0], reps[0][1], tm, ready)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for x, o in reps:
                        _sweep_call(kind, x, o, tm, ready)
                us_first = _graph_us(g, nb, stream, replays=2)
                replays = max(3, min(200, int(20000 / max(1e-3, us_first * nb))))
                times[ready] = _graph_us(g, nb, stream, replays=replays)
                del g
            us, us_ready = times[False], times[True]
            gbps = nbytes / (us / 1e6) / 1e9
            gbps_ready = nbytes / (us_ready / 1e6) / 1e9
            print(json.dumps({"kind": kind, "E": E, "T": T, "layout": "time-major" if tm else "env-major",
                              "trunc": trunc, "dtype": args.sweep_dtype, "us_per_call": round(us, 3), "algorithmic_bytes": nbytes,
                              "GBps": round(gbps, 1), "frac_of_peak": round(gbps / peak, 4),
                              "us_per_call_inputs_ready": round(us_ready, 3),
                              "frac_of_peak_inputs_ready": round(gbps_ready / peak, 4),
                              "peak": f"{peak} GB/s {peak_kind}", "env_steps_per_s": E * T / (us / 1e6),
                              "replicas": nb}), flush=True)
            del reps, d
            torch.cuda.empty_cache()
    return 0


# ---------------------------------------------------------------------------
# The vectorised PyTorch doubling-scan baseline: the form of comparison the
# paper quotes its speed-ups against (rl-triton (arXiv:2608.17641) §6
# Benchmarking Methodology, baseline design; §7 Results): each estimator's
# (alpha, beta) built with whole-tensor torch ops, then log2(T)
# recursive-doubling passes of affine map composition over the whole
# [E, T] tensor (suffix passes for the backward estimators, prefix passes
# for the forward ones).  Env-major, float32 (int32 for the prefix sum).  A
# measurement baseline only: the library never runs it.
# ---------------------------------------------------------------------------

def torch_doubling_scan(alpha, beta, reverse=True):
    """A_t = alpha_t + beta_t * A_{t+1} (reverse) or A_{t-1} (forward) along
    the last dim, carry 0.  After the pass of stride s, (A_t, B_t) is the
    composition of the 2s maps from step t on (reverse) or back to it; maps
    past the row's end count as the identity."""
    import torch
    A, B = alpha, beta
    T = A.shape[-1]
    s = 1
    while s < T:
        if reverse:
            A = torch.cat([A[..., :-s] + B[..., :-s] * A[..., s:], A[..., -s:]], -1)
            B = torch.cat([B[..., :-s] * B[..., s:], B[..., -s:]], -1)
        else:
            A = torch.cat([A[..., :s], A[..., s:] + B[..., s:] * A[..., :-s]], -1)
            B = torch.cat([B[..., :s], B[..., s:] * B[..., :-s]], -1)
        s *= 2
    return A


def _torch_edges(x, term, trunc):
    """Per-step masks of the boundary rules: truncated (and not terminated),
    continues into t+1 inside the window, ends the window unflagged."""
    import torch
    T = x.shape[-1]
    tm = term.bool() if term is not None else torch.zeros_like(x, dtype=torch.bool)
    tr = (trunc.bool() & ~tm) if trunc is not None else torch.zeros_like(tm)
    inner = torch.arange(T, device=x.device) < T - 1
    free = ~tm & ~tr
    return tr, free & inner, free & ~inner


def _torch_next(x, last):
    import torch
    return torch.cat([x[..., 1:], last[..., None]], -1)


def torch_doubling(kind, x, gamma=GAMMA, lam=LAMBDA, rho_bar=1.0, c_bar=1.0, vtrace_lam=1.0):
    """One estimator call of the baseline on env-major inputs (the input
    dicts of the sweep); returns its outputs as a tuple."""
    import torch
    r = x.get("rewards")
    ref = r if r is not None else x.get("x_f32")
    E = ref.shape[0]
    zero_e = torch.zeros(E, dtype=torch.float32, device=ref.device)
    boot = x.get("bootstrap") if x.get("bootstrap") is not None else zero_e
    tv = x.get("trunc_value")
    if kind in ("elig", "psum"):
        xs = x["x_f32"] if kind == "elig" else x["x_i32"]
        tm, tr = x.get("terminated"), x.get("truncated")
        d = tm.bool() if tm is not None else torch.zeros_like(xs, dtype=torch.bool)
        if tr is not None:
            d = d | tr.bool()
        first = torch.ones_like(d[..., :1])
        keep = ~torch.cat([first, d[..., :-1]], -1)  # no edge just before t
        beta = keep.to(xs.dtype) * (gamma * lam if kind == "elig" else 1)
        return (torch_doubling_scan(xs, beta, reverse=False),)
    tr, cont, end = _torch_edges(r, x.get("terminated"), x.get("truncated"))
    tvt = torch.where(tr, tv, torch.zeros_like(r)) if tv is not None else torch.zeros_like(r)
    bend = end * boot[:, None]
    if kind == "retrace":
        q, pi = x["q"], x["pi"]
        ev = (pi * q).sum(-1)
        a = x["actions"].long()[..., None]
        qa = torch.gather(q, -1, a)[..., 0]
        c = lam * torch.clamp(torch.gather(pi, -1, a)[..., 0] / x["mu_a"], max=1.0)
        ev_n, qa_n, c_n = (_torch_next(t, zero_e) for t in (ev, qa, c))
        alpha = r + gamma * (tvt + bend + cont * (ev_n - c_n * qa_n))
        return (torch_doubling_scan(alpha, gamma * c_n * cont),)
    v = x["values"]
    v_n = _torch_next(v, zero_e)
    nv = tvt + bend + cont * v_n  # successor value (0 where terminated)
    if kind == "vtrace":
        ratio = torch.exp(x["logp_target"] - x["logp_behaviour"])
        rho = torch.clamp(ratio, max=rho_bar)
        c = vtrace_lam * torch.clamp(ratio, max=c_bar)
        dvs = torch_doubling_scan(rho * (r + gamma * nv - v), gamma * c * cont)
        vs = v + dvs
        nvs = tvt + bend + cont * _torch_next(vs, zero_e)
        return vs, rho * (r + gamma * nvs - v)
    outs = []
    if kind in ("gae", "vt"):
        adv = torch_doubling_scan(r + gamma * nv - v, gamma * lam * cont)
        outs += [adv, adv + v]
    if kind in ("disc", "vt"):
        outs.append(torch_doubling_scan(r + gamma * nv - gamma * cont * v_n, gamma * cont))
    if kind in ("td", "vt"):
        outs.append(torch_doubling_scan(r + gamma * (nv - lam * cont * v_n), gamma * lam * cont))
    return tuple(outs)


# the configurations of the paper's comparison this baseline is timed on:
# the fused value targets / single estimators at 4096 x 128 (with
# truncation), V-Trace at 4096 x 256, Retrace at 1024 x 2048 (A = 18)
TORCH_BASELINE_CASES = [("vt", 4096, 128, True), ("gae", 4096, 128, True), ("disc", 4096, 128, True),
                        ("td", 4096, 128, True), ("vtrace", 4096, 256, False), ("retrace", 1024, 2048, False),
                        ("elig", 4096, 128, True), ("psum", 4096, 128, True)]
TORCH_COMPILE_KINDS = tuple(c[0] for c in TORCH_BASELINE_CASES)


def run_torch_baseline(args):
    """One JSON line per case: device time per call of this library and of
    the PyTorch doubling-scan baseline (eager ops captured in a CUDA graph;
    torch.compile of the same function where it builds), on the same
    replicas (footprint > 3 x L2); the full-call (host wall) time per call of
    each in plain stream order; and the largest difference between the two
    results relative to (1 + |ours|)."""
    import torch
    from first_order_linear_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    stream = torch.cuda.Stream(dev)
    for kind, E, T, trunc in TORCH_BASELINE_CASES:
        d, nbytes, spec = _sweep_case(kind, E, T, trunc, dev)
        foot = sum(v.numel() * v.element_size() for v in d.values() if isinstance(v, torch.Tensor))
        nb = max(2, min(64, math.ceil(3 * l2 / foot)))
        reps = [({k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in d.items()},
                 [torch.empty(sh, dtype=dt, device=dev) for sh, dt in spec]) for _ in range(nb)]

        def timed(fn):
            with torch.cuda.stream(stream):
                for x, o in reps[:2]:
                    fn(x, o)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for x, o in reps:
                    fn(x, o)
            us = _graph_us(g, nb, stream, replays=max(3, min(50, int(20000 / max(1.0, _graph_us(g, nb, stream, 1) * nb)))))
            del g
            return us

        ours = timed(lambda x, o: _sweep_call(kind, x, o, False))
        eager = timed(lambda x, o: torch_doubling(kind, x))
        with torch.cuda.stream(stream):
            _sweep_call(kind, reps[0][0], reps[0][1], False)
            base = torch_doubling(kind, reps[0][0])
        stream.synchronize()
        diff = max(float(((b.double() - a.double()).abs() / (1 + a.double().abs())).max())
                   for a, b in zip(reps[0][1], base))
        full_ours = _full_call_us(lambda r: _sweep_call(kind, r[0], r[1], False), reps, stream)
        full_eager = _full_call_us(lambda r: torch_doubling(kind, r[0]), reps, stream)
        comp, comp_err, full_comp = None, None, None
        if kind in TORCH_COMPILE_KINDS and not args.skip_torch_compile:
            try:
                fn = torch.compile(lambda x: torch_doubling(kind, x), dynamic=False)
                comp = timed(lambda x, o: fn(x))
                full_comp = _full_call_us(lambda r: fn(r[0]), reps, stream)
            except Exception as exc:  # noqa: BLE001 - reported, not fatal
                comp_err = f"{type(exc).__name__}: {str(exc).splitlines()[0][:160] if str(exc) else ''}"
        line = {"torch_doubling": kind, "E": E, "T": T, "trunc": trunc, "layout": "env-major",
                "us_per_call_ours": round(ours, 3), "us_per_call_torch_eager": round(eager, 3),
                "speedup_vs_eager": round(eager / ours, 2),
                "us_per_call_torch_compile": None if comp is None else round(comp, 3),
                "speedup_vs_compile": None if comp is None else round(comp / ours, 2),
                "full_call_us_ours": round(full_ours, 2), "full_call_us_torch_eager": round(full_eager, 2),
                "full_call_us_torch_compile": None if full_comp is None else round(full_comp, 2),
                "full_call_speedup_vs_compile": None if full_comp is None else round(full_comp / full_ours, 2),
                "max_rel_diff": diff, "replicas": nb, "algorithmic_bytes": nbytes}
        if comp_err:
            line["torch_compile_error"] = comp_err
        print(json.dumps(line), flush=True)
        del reps, d
        torch.cuda.empty_cache()
    return 0


# the configurations the pages name, timed as the pages time them
PAGES_PROTOCOL_CASES = [("vt", 4096, 128, True), ("vtrace", 4096, 256, False), ("retrace", 1024, 2048, False)]


def run_pages_protocol(args):
    """The paper's timing protocol (rl-triton (arXiv:2608.17641) §6
    Benchmarking Methodology) on the named configurations: 20 untimed
    calls, then 5 trials of 50 calls, each call alone between two CUDA
    events on its stream; the figure is the smallest of the 5 per-trial
    medians.  Added here: L2 is flushed before each call, outside the
    events, by reading a buffer of twice the L2 size (a read leaves clean
    lines: a memset would leave that much dirty data to be written back
    during the timed call), so the figure is one isolated launch from a
    cold L2, nothing overlapped.  ``--pages-flush write`` flushes with a
    memset instead."""
    import torch
    from first_order_linear_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(dev)
    flush = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for kind, E, T, trunc in PAGES_PROTOCOL_CASES:
        d, nbytes, spec = _sweep_case(kind, E, T, trunc, dev)
        o = [torch.empty(sh, dtype=dt, device=dev) for sh, dt in spec]
        torch.cuda.synchronize()  # the inputs were written on the default stream
        with torch.cuda.stream(stream):
            for _ in range(20):
                _sweep_call(kind, d, o, False)
            stream.synchronize()
            medians = []
            for _ in range(5):
                ts = []
                for _ in range(50):
                    if args.pages_flush == "write":
                        flush.zero_()
                    else:
                        torch.sum(flush, dim=0, out=sink)
                    a.record(stream)
                    _sweep_call(kind, d, o, False)
                    b.record(stream)
                    b.synchronize()
                    ts.append(a.elapsed_time(b) * 1e3)
                medians.append(statistics.median(ts))
        us = min(medians)
        print(json.dumps({"pages_protocol": kind, "E": E, "T": T, "trunc": trunc, "layout": "env-major",
                          "us_per_call": round(us, 3), "trial_medians_us": [round(m, 3) for m in medians],
                          "algorithmic_bytes": nbytes, "frac_of_peak": round(nbytes / (us / 1e6) / 1e9 / peak, 4),
                          "peak": f"{peak} GB/s {peak_kind}", "env_steps_per_s": E * T / (us / 1e6),
                          "timing": f"cold L2 (2 x L2 {'memset' if args.pages_flush == 'write' else 'read'} "
                                    "before each call), one call between two events, "
                                    "min over 5 trials of the median of 50"}), flush=True)
        del d, o
        torch.cuda.empty_cache()
    return 0


def run_ncu_case(args):
    """Calls of one estimator and nothing else: the command lines ncu
    captures.  ``--ncu-case vt,4096,128,em`` makes four calls on one seeded
    batch (capture with ``-s 2 -c 1``).  With the option ``rot``
    (``vt,4096,128,em,rot``) the calls rotate over replicas whose footprint
    exceeds 3 x L2, 4 rotations in plain stream order, as the bench's timed
    region does; a capture with ``--cache-control none`` of a launch in the
    third rotation then sees the DRAM traffic of the steady state (reads of
    inputs no longer in L2, write-backs of outputs evicted from it).
    Option ``bf16``: bfloat16 storage."""
    import torch
    from first_order_linear_gb300 import build, synth
    parts = args.ncu_case.split(",")
    kind, E, T, lay = parts[:4]
    opts = set(parts[4:])
    bf16, rot = "bf16" in opts, "rot" in opts
    E, T, tm = int(E), int(T), lay == "tm"
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d, nbytes, spec = _sweep_case(kind, E, T, True, dev, bf16=bf16)
    x = {k: (synth.to_time_major(v) if tm and isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    nb = 1
    if rot:
        l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20)
        foot = sum(v.numel() * v.element_size() for v in x.values() if isinstance(v, torch.Tensor))
        foot += sum(E * T * torch.empty(0, dtype=dt).element_size() for _, dt in spec)
        nb = max(2, math.ceil(3 * l2 / foot))
    reps = []
    for i in range(nb):
        xi = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in x.items()} if rot else x
        reps.append((xi, [torch.empty(sh if not tm else (sh[1], sh[0]), dtype=dt, device=dev) for sh, dt in spec]))
    calls = 4 * nb if rot else 4
    torch.cuda.synchronize()
    for i in range(calls):
        xi, o = reps[i % nb]
        _sweep_call(kind, xi, o, tm)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_case": args.ncu_case, "algorithmic_bytes_per_call": nbytes, "calls": calls,
                      "replicas": nb}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--e2e-lanes", type=int, default=1, help="copy streams per direction in the e2e pipeline")
    ap.add_argument("--e2e-buffers", type=int, default=2, help="device buffer sets of the e2e pipeline")
    ap.add_argument("--sweep", action="store_true",
                    help="print one line per estimator and benchmark shape instead of the step metric")
    ap.add_argument("--sweep-kinds", default="", help="comma-separated subset of " + ",".join(SWEEP_KINDS))
    ap.add_argument("--clock-log", default="", help="also write the nvidia-smi clock samples of the timed region "
                                                    "to this CSV file")
    ap.add_argument("--sweep-dtype", choices=["f32", "bf16"], default="f32",
                    help="storage of the float arrays in --sweep (bf16: RLCA_BF16, float32 arithmetic)")
    ap.add_argument("--torch-baseline", action="store_true",
                    help="time the vectorised PyTorch doubling-scan baseline beside this library")
    ap.add_argument("--skip-torch-compile", action="store_true", help="with --torch-baseline: eager only")
    ap.add_argument("--pages-protocol", action="store_true",
                    help="time the named configurations with the paper's protocol (cold L2, isolated calls)")
    ap.add_argument("--oracle-configs", action="store_true",
                    help="time the C oracle on each named configuration, one thread and all host cores")
    ap.add_argument("--oracle-seconds", type=float, default=3.0)
    ap.add_argument("--pages-flush", choices=["read", "write"], default="read",
                    help="with --pages-protocol: flush L2 by reading (default) or by a memset of 2 x L2")
    ap.add_argument("--ncu-case", default="",
                    help="KIND,E,T,em|tm[,bf16]: four calls of one estimator on one batch (a case for ncu), no timing")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.ncu_case:
        return run_ncu_case(args)
    if args.sweep:
        return run_sweep(args)
    if args.torch_baseline:
        return run_torch_baseline(args)
    if args.pages_protocol:
        return run_pages_protocol(args)
    if args.oracle_configs:
        return run_oracle_configs(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
