"""Decode benchmark of the activation-sparse FFN on GB300.

Default workload: the OPT-30B-shaped 48-layer FFN stack (d = 7168,
n = 28672, r = 256 per layer, fp16 weights, residual adds, per-layer Zipf
activation profiles at 3-15 % density; about 39 GB of weights resident in
HBM), seeded and synthetic.  One step = one token decoded at batch 1
through all 48 layers (predictor, compaction, row-gather GEMV + ReLU,
row-axpy down projection, fixed-order reduction, residual add per layer):
one pi_decode_layers launch.  The stack exceeds the L2 cache hundreds of
times over, so every layer's weights come from HBM.

Single-layer workloads (--workload ...) run the same engine with rotating
weight replicas larger than L2.  Steps run as CUDA-graph replays; each
timed region is K steps bracketed by a barrier and device synchronisation,
timed with CUDA events on the launching stream, repeated and reported as
the median.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun (N > 1) every rank decodes its own token stream on its own
GPU (replicas only: each rank holds the whole model); rank 0 prints the
aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-FFN decode tokens/s at batch 1; achieved HBM GB/s vs peak (active bytes)"
DEFAULT_WORKLOAD = "opt30b_ffn_stack_48x_d7168_n28672_r256_f16"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ------------------------------------------------------------------ helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def aggregate(per_rank_ms, per_rank_units, n_gpus):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = max(per_rank_ms)
    return (sum(per_rank_units) / (t / 1e3)) if t > 0 else 0.0, t


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The largest of every rank's value (one all-reduce; the value itself
    when there is one rank).  device: where the reduction's tensor lives
    (the rank's GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "activation_sparse_decode_rank_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(d, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "pi.h"), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def stored_traffic(kernel_key):
    """The committed ncu figure for a kernel and workload, if it was taken on
    the current kernel source: (DRAM bytes per decode step, the algorithmic
    bytes per step of that capture); else None."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    try:
        j = json.load(open(PROFILE_TRAFFIC))
    except Exception:
        return None
    e = j.get(kernel_key)
    if not e or e.get("csrc_hash") != csrc_hash():
        return None
    if "dram_bytes_per_step" not in e:
        return None
    return float(e["dram_bytes_per_step"]), float(e.get("algorithmic_bytes_per_step", 0.0))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def timed_regions(torch, stream, fn, repeats, barrier):
    """Runs fn() (which enqueues one timed region of work on `stream`)
    `repeats` times, each bracketed by a barrier and device synchronisation
    and timed with CUDA events on the stream; returns the milliseconds of
    each region."""
    out = []
    for _ in range(repeats):
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn()
            e1.record(stream)
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


# ------------------------------------------------------------------ workload
def workload_spec(name):
    from synth.workloads import WORKLOADS
    w = dict(WORKLOADS[name])
    if "densities" in w:
        raise SystemExit(f"bench: workload {name} is not a batch-1 workload")
    return w


def hot_prefix_len(w):
    import synth
    c = synth.zipf_calibrate(w["n"], w["alpha"], w["density"])
    p = synth.zipf_probs(w["n"], w["alpha"], c)
    return int((p >= 0.5).sum())


def layer_config(w, args, hot, R, layer_bytes, step_bytes_est, l2):
    """The `config` of a single-layer line (shared by both arms)."""
    return {
        "workload": args.workload, "batch": 1, "weights": w["dtype"], "density": w["density"],
        "d": w["d"], "n": w["n"], "r": w["r"], "gated": bool(w["gated"]), "hot_prefix": hot,
        "layout": args.layout,
        "l2": (f"inputs larger than L2: {R} rotating weight replicas "
               f"({R * layer_bytes / 1e9:.1f} GB; each step reads its own copy)"
               if R * step_bytes_est >= 3 * l2 else
               f"L2-warm (not HBM-bound): {R} weight replica(s) of "
               f"{layer_bytes / 1e9:.2f} GB reused across steps"),
        "parallelism": "single GPU",
    }


def stack_config(w, L):
    """The `config` of a stack line (shared by both arms)."""
    d, n, r = w["d"], w["n"], w["r"]
    return {"workload": w["name"], "batch": 1, "layers": L, "weights": w["dtype"],
            "d": d, "n": n, "r": r, "gated": False, "layout": "packed",
            "hot_prefix": "per layer: neurons with p_i >= 0.5",
            "density": "per layer 3-15 % (Zipf alpha_l ~ U[0.7, 1.2])",
            "l2": f"inputs larger than L2: {L} distinct layers resident "
                  f"({L * (n * 2 * d * 2 + n * r * 2 + r * d * 2) / 1e9:.1f} GB)",
            "parallelism": "single GPU"}


def cpu_oracle_sample(w, budget_s, max_tokens, warm=3):
    """Times the fp64 oracle (predict + compact + sparse FFN) on the host
    cores over a bounded sample of the workload's decode steps: at most
    max_tokens steps, stopping once budget_s of oracle time is spent.  Input
    generation is outside the timed part."""
    import oracle
    import synth
    L = synth.make_layer(w["d"], w["n"], w["r"], w["dtype"], gated=w["gated"], alpha=w["alpha"],
                         density=w["density"], seed=w["seed"])
    for s in range(warm):
        oracle.layer_decode(L, synth.gen_x(w["seed"], s, 1, w["d"])[0])
    spent = 0.0
    done = 0
    for s in range(max_tokens):
        x = synth.gen_x(w["seed"], s, 1, w["d"])[0]
        t0 = time.perf_counter()
        oracle.layer_decode(L, x)
        spent += time.perf_counter() - t0
        done += 1
        if spent > budget_s:
            break
    return done, spent, oracle.get_threads()


# ------------------------------------------------------------------ the stack's layers
def build_stack(w, dev, L):
    """The first L layers of the residual stack, generated on the GPU and
    packed (one [W1 row | W2 row] record per neuron).  Returns descriptors,
    weight structs, the tensors that hold them and the predictor bytes."""
    import torch

    import activation_sparse_decode_rank_gb300 as pi
    import synth
    d, n, r = w["d"], w["n"], w["r"]
    alpha, rho, cz, scale = synth.stack_plan(w["seed"], w["layers"], n)
    descs, wts, keep, pred_bytes = [], [], [], 0
    for l in range(L):
        g = synth.make_layer_gpu(d, n, r, w["dtype"], alpha=float(alpha[l]), zipf_c=float(cz[l]),
                                 seed=w["seed"], layer=l, bias_scale=float(scale[l]), device=dev)
        p = synth.zipf_probs(n, float(alpha[l]), float(cz[l]))
        hot = int((p >= 0.5).sum())
        desc = pi.make_desc(d, n, r, w["dtype"], False, hot, packed=True)
        rec = torch.empty((n, 2 * d), dtype=torch.int16, device=dev)
        pi.check(pi.pi_pack_weights(desc, g["W1"], g["W2"], rec), "pi_pack_weights")
        torch.cuda.synchronize()
        del g["W1"], g["W2"]
        keep.append((g, rec))
        descs.append(desc)
        wts.append(pi.make_weights(g["A"], g["Bm"], g["b1"], rec, None, g["b2"]))
        pred_bytes += n * r * 2 + r * d * 2 + n * 4
    torch.cuda.empty_cache()
    return descs, wts, keep, pred_bytes


def host_layer(w, g, rec):
    """Host copy of one packed GPU layer in the oracle's split form."""
    import synth
    d = w["d"]
    cpu = lambda t: t.cpu().numpy()
    R = cpu(rec).view(np.uint16)
    return synth.Layer(d, w["n"], w["r"], w["dtype"], False, cpu(g["A"]).view(np.uint16),
                       cpu(g["Bm"]).view(np.uint16), cpu(g["b1"]),
                       np.ascontiguousarray(R[:, :d]), np.ascontiguousarray(R[:, d:]),
                       cpu(g["b2"]), {})


def stack_oracle_sample(w, keep, tokens, warm, budget_s, seed_off=0):
    """Times the fp64 oracle on the host cores through every layer of the
    stack, token by token: x_{l+1} = x_l + FFN_l(x_l) with predict, compact
    and the sparse FFN per layer, the residual stream kept in fp32.  Layers
    are visited one at a time (each copied to the host once, outside the
    timed part); `warm` untimed tokens go first.  If layer 0 shows that
    `tokens` would exceed budget_s of oracle time, the sample keeps the
    first tokens that fit.  Returns (timed tokens, seconds, threads)."""
    import oracle
    import synth
    d = w["d"]
    L = len(keep)
    xs = [synth.gen_x(w["seed"] + seed_off, s, 1, d)[0].astype(np.float32)
          for s in range(warm + tokens)]
    spent = [0.0] * (warm + tokens)
    keep_n = warm + tokens
    for l, (g, rec) in enumerate(keep):
        H = host_layer(w, g, rec)
        for t in range(keep_n):
            t0 = time.perf_counter()
            _, _, _, xn = oracle.layer_decode(H, xs[t], residual=True)
            spent[t] += time.perf_counter() - t0
            xs[t] = xn
        del H
        if l == 0 and tokens > 1:
            per_tok = sum(spent[warm:keep_n]) / tokens * L
            fit = max(1, int(budget_s / per_tok)) if per_tok > 0 else tokens
            keep_n = warm + min(tokens, fit)
    done = keep_n - warm
    return done, sum(spent[warm:keep_n]), oracle.get_threads()


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The oracle as the reference arm: the same workload, config, steps and
    warm-up as our arm, timed on the host cores (rank 0 only)."""
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    w = workload_spec(args.workload)
    w["name"] = args.workload
    budget = float(os.environ.get("PI_REF_BUDGET_S", "120"))
    if w.get("layers", 1) > 1:
        import torch
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        L = args.layers if args.layers > 0 else w["layers"]
        # the synthetic weights come from the GPU generator (input generation
        # only, untimed; the host generator would take minutes per layer)
        _, _, keep, _ = build_stack(w, dev, L)
        done, dt, cores = stack_oracle_sample(w, keep, args.steps, args.warmup, budget)
        config = stack_config(w, L)
        sample = (f"{done} of {args.steps} requested tokens (after {args.warmup} untimed) "
                  f"through all {L} layers of {args.workload}, fp64 oracle predict+compact+"
                  f"sparse FFN + residual per layer, on {cores} host threads")
    else:
        done, dt, cores = cpu_oracle_sample(w, budget_s=budget, max_tokens=args.steps,
                                            warm=args.warmup)
        hot = hot_prefix_len(w) if args.hot < 0 else args.hot
        config = layer_config(w, args, hot, 0, 0, 0, 1)
        config.pop("l2")
        sample = (f"{done} of {args.steps} requested decode steps of {args.workload} "
                  f"(time-bounded at {budget:.0f} s), fp64 oracle on {cores} host threads")
    v = done / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": done, "warmup": args.warmup, "ms_per_step": dt / done * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm: one layer
def run_ours(args):
    import torch

    import activation_sparse_decode_rank_gb300 as pi
    import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pi.build()
    w = workload_spec(args.workload)
    d, n, r = w["d"], w["n"], w["r"]
    gated = bool(w["gated"])
    m_rows = 3 if gated else 2
    hot = hot_prefix_len(w) if args.hot < 0 else args.hot

    L = synth.make_layer(d, n, r, w["dtype"], gated=gated, alpha=w["alpha"],
                         density=w["density"], seed=w["seed"])

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    # rotating weight replicas: every step reads a copy no other recent step touched
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20)
    pred_bytes = n * r * 2 + r * d * 2 + n * 4
    step_bytes_est = pred_bytes + w["density"] * n * m_rows * d * 2
    R = args.replicas if args.replicas > 0 else max(2, math.ceil(3 * l2 / step_bytes_est))
    R = min(R, 128)
    desc = pi.make_desc(d, n, r, w["dtype"], gated, hot, packed=args.layout == "packed")
    base = [up(L.A), up(L.Bm), up(L.b1), up(L.W1), up(L.W2), up(L.b2)]
    if args.layout == "packed":
        # offline step: one record per neuron ([W1 row(s) | W2 row])
        rec = torch.empty((n, m_rows * d), dtype=torch.int16, device=dev)
        pi.check(pi.pi_pack_weights(desc, base[3], base[4], rec), "pi_pack_weights")
        base = [base[0], base[1], base[2], rec, None, base[5]]
    reps = [base] + [[t.clone() if t is not None else None for t in base] for _ in range(R - 1)]
    layer_bytes = sum(t.numel() * t.element_size() for t in base if t is not None)
    wts = [pi.make_weights(*rp) for rp in reps]
    descs = [desc] * R

    K = args.steps
    # one pi_decode_layers launch decodes G steps (independent tokens, each
    # read only after the previous step is complete); K is a multiple of G
    G = min(K, args.graph_len)
    if K % G:
        raise SystemExit(f"bench: --steps must be a multiple of the steps per launch {G}")
    xs = torch.from_numpy(np.concatenate(
        [synth.gen_x(w["seed"] + 1000 * rank, s, 1, d) for s in range(G)])).to(dev)
    ys = torch.empty((G, d), dtype=torch.float32, device=dev)
    cseq = torch.zeros((G + 4,), dtype=torch.int32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = pi.workspace(desc, 1, dev)
    stream = torch.cuda.Stream(device=dev)

    def launch(J, xsrc, ydst, cnt):
        pi.check(pi.pi_decode_layers(descs, wts, J, xsrc, 0, ydst, cnt, None, st, ws,
                                     stream=stream), "pi_decode_layers")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                fn()
        return g

    with torch.cuda.stream(stream):
        launch(G, xs, ys, cseq)  # eager run first: attribute setup, sanity
        stream.synchronize()
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
    launches_per_region = K // G
    g_main = capture(lambda: [launch(G, xs, ys, cseq) for _ in range(launches_per_region)])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):  # warm-up (untimed): at least W steps
        for _ in range(max(1, math.ceil(args.warmup / K))):
            g_main.replay()
        stream.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    regions = timed_regions(torch, stream, g_main.replay, args.repeats, barrier)
    clocks = sampler.stop()
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
    ms = statistics.median(regions)

    # byte accounting from the run's own active counts
    cnt_host = cseq[:G].cpu().numpy().astype(np.float64)
    mean_cnt = float(cnt_host.mean())
    active_bytes = mean_cnt * m_rows * d * 2
    alg_bytes = pred_bytes + active_bytes

    value, t_max = aggregate([max_over_ranks(ms, world, dev)], [K * world], world)
    ms_per_step = t_max / K
    per_launch_s = ms / launches_per_region / 1e3
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes * G / per_launch_s / 1e9
    tr = stored_traffic(f"seq_kernel:{args.workload}")
    traffic = tr[0] * G if tr else None  # DRAM bytes of one launch of G steps

    # dense-FFN comparison point (same replicas, one launch per step)
    dense_steps = 200
    ws_d = pi.workspace(desc, 1, dev)
    y1 = torch.empty((1, d), dtype=torch.float32, device=dev)

    def dense_all():
        for s in range(dense_steps):
            pi.check(pi.pi_dense_ffn(desc, wts[s % R], xs[s % G], 1, y1, ws_d, stream=stream))

    with torch.cuda.stream(stream):
        for s in range(2):
            pi.check(pi.pi_dense_ffn(desc, wts[s % R], xs[s % G], 1, y1, ws_d, stream=stream))
    g_dense = capture(dense_all)
    with torch.cuda.stream(stream):
        g_dense.replay()
    dense_ms = statistics.median(timed_regions(torch, stream, g_dense.replay, 3,
                                               lambda: None)) / dense_steps
    dense_bytes = n * m_rows * d * 2 + n * 4

    # end to end through the C ABI with host buffers, per token: a pinned
    # host -> device copy of the token's x, one decode launch, a device ->
    # host copy of its y (the line's e2e); and the same amortised over the
    # G tokens of one launch (e2e_chunked)
    xh = torch.from_numpy(np.concatenate(
        [synth.gen_x(w["seed"] + 7 + 1000 * rank, s, 1, d) for s in range(G)])).pin_memory()
    yh = torch.empty((G, d), dtype=torch.float32).pin_memory()
    xin = torch.empty((G, d), dtype=torch.float32, device=dev)
    e2e_tokens = min(K, 200)

    def e2e_tok():
        for s in range(e2e_tokens):
            xin[s % G].copy_(xh[s % G], non_blocking=True)
            launch(1, xin[s % G], ys[s % G], None)
            yh[s % G].copy_(ys[s % G], non_blocking=True)

    def e2e_chunk():
        for _ in range(launches_per_region):
            xin.copy_(xh, non_blocking=True)
            launch(G, xin, ys, None)
            yh.copy_(ys, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_tok()
        e2e_chunk()
        stream.synchronize()
    g_e2e = capture(e2e_tok)
    g_e2c = capture(e2e_chunk)
    with torch.cuda.stream(stream):
        g_e2e.replay()
        g_e2c.replay()
    e2e_ms = statistics.median(timed_regions(torch, stream, g_e2e.replay, args.repeats, barrier))
    e2c_ms = statistics.median(timed_regions(torch, stream, g_e2c.replay, args.repeats, barrier))
    e2e_value, _ = aggregate([max_over_ranks(e2e_ms, world, dev)], [e2e_tokens * world], world)
    e2c_value, _ = aggregate([max_over_ranks(e2c_ms, world, dev)], [K * world], world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        budget = float(os.environ.get("PI_CPU_BUDGET_S", "15"))
        done, dt, cores = cpu_oracle_sample(w, budget_s=budget, max_tokens=100000)
        cpu = {"value": done / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"first {done} decode steps of {args.workload} (time-bounded at "
                         f"{budget:.0f} s), fp64 oracle predict+compact+sparse FFN"}

    config = layer_config(w, args, hot, R, layer_bytes, step_bytes_est, l2)
    config["steps_per_launch"] = G
    config["parallelism"] = "replicas" if world > 1 else "single GPU"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config,
        "repeats": args.repeats, "regions_ms": regions,
        "us_per_layer": ms_per_step * 1e3,
        "active_neurons_mean": mean_cnt,
        "bytes_per_step": {"predictor": pred_bytes, "active_rows": active_bytes,
                           "total": alg_bytes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth",
                     "kernel": f"seq_kernel (persistent, {G} decode steps per launch)",
                     "traffic_how": ("ncu dram__bytes_read.sum + dram__bytes_write.sum per step "
                                     f"(profiles/traffic.json) x {G} steps per launch"
                                     if tr else "null: no capture of the current kernel source")},
        "dense_ffn": {"us_per_step": dense_ms * 1e3, "tokens_per_s": 1e3 / dense_ms,
                      "achieved_gbs": dense_bytes / (dense_ms / 1e3) / 1e9,
                      "frac": dense_bytes / (dense_ms / 1e3) / 1e9 / peak},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": d * 4,
                "d2h_bytes_per_step": d * 4, "steps": e2e_tokens,
                "how": "per token: pinned H2D of its x, one pi_decode_layers launch (one step), "
                       "D2H of its y; CUDA-graph replay"},
        "e2e_chunked": {"value": e2c_value, "unit": "tokens/s", "h2d_bytes_per_step": d * 4,
                        "d2h_bytes_per_step": d * 4, "steps": K,
                        "how": f"per launch of {G} tokens: one pinned H2D of their x, one "
                               f"pi_decode_layers launch, one D2H of their y"},
        "gpu_launches": launches_per_region,
        "engine": "seq",
        "clocks": clocks,
        "cpu_baseline": cpu,
        "csrc_hash": csrc_hash(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ our arm: the stack
def run_stack(args):
    """One step = one token through every layer of the residual FFN stack
    (x_{l+1} = x_l + FFN_l(x_l)): one pi_decode_layers launch per token.
    The weights of all layers together exceed L2 hundreds of times over, so
    every layer's weights come from HBM."""
    import torch

    import activation_sparse_decode_rank_gb300 as pi
    import synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pi.build()
    w = workload_spec(args.workload)
    w["name"] = args.workload
    d, n, r = w["d"], w["n"], w["r"]
    L = args.layers if args.layers > 0 else w["layers"]
    descs, wts, keep, pred_bytes = build_stack(w, dev, L)
    K = args.steps
    xs = torch.from_numpy(np.concatenate(
        [synth.gen_x(w["seed"] + 1000 * rank, s, 1, d) for s in range(K)])).to(dev)
    ybuf = torch.empty((K, L, d), dtype=torch.float32, device=dev)
    cseq = torch.zeros((K, (L + 3) // 4 * 4), dtype=torch.int32, device=dev)  # 16-byte rows
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = pi.workspace(descs[0], 1, dev)
    stream = torch.cuda.Stream(device=dev)

    def token(s, xsrc, cnt=True):
        # the whole stack for one token in one persistent launch; y[l] = x_{l+1}
        pi.check(pi.pi_decode_layers(descs, wts, L, xsrc, 1, ybuf[s], cseq[s] if cnt else None,
                                     None, st, ws, stream=stream), "pi_decode_layers")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                fn()
        return g

    with torch.cuda.stream(stream):
        token(0, xs[0])
        stream.synchronize()
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
    g_main = capture(lambda: [token(s, xs[s]) for s in range(K)])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):  # warm-up (untimed): at least W tokens
        for _ in range(max(1, math.ceil(args.warmup / K))):
            g_main.replay()
        stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    regions = timed_regions(torch, stream, g_main.replay, args.repeats, barrier)
    clocks = sampler.stop()
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
    ms = statistics.median(regions)
    mean_cnt = cseq[:, :L].float().mean(dim=0).cpu().numpy()
    alg_bytes = pred_bytes + float(mean_cnt.sum()) * 2 * d * 2
    value, t_max = aggregate([max_over_ranks(ms, world, dev)], [K * world], world)
    ms_step = t_max / K
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (ms / K / 1e3) / 1e9
    tr = stored_traffic(f"seq_kernel:{args.workload}:{L}")
    traffic = tr[0] if tr else None  # one launch = one step (one token)

    # dense comparison point: pi_dense_ffn over every layer of the stack
    ws_d = pi.workspace(descs[0], 1, dev)
    yd = torch.empty((1, d), dtype=torch.float32, device=dev)

    def dense_token():
        for l in range(L):
            pi.check(pi.pi_dense_ffn(descs[l], wts[l], xs[0], 1, yd, ws_d, stream=stream))

    with torch.cuda.stream(stream):
        dense_token()
    g_dense = capture(dense_token)
    with torch.cuda.stream(stream):
        g_dense.replay()
    dense_ms = statistics.median(timed_regions(torch, stream, g_dense.replay, 3, lambda: None))
    dense_bytes = L * (n * 2 * d * 2 + n * 4)

    # end to end through the C ABI with host buffers, per token: a pinned
    # H2D copy of the token's x, one pi_decode_layers launch through all
    # layers, a D2H copy of its output x_L
    xh = torch.from_numpy(np.concatenate(
        [synth.gen_x(w["seed"] + 7 + 1000 * rank, s, 1, d) for s in range(K)])).pin_memory()
    yh = torch.empty((K, d), dtype=torch.float32).pin_memory()
    xin = torch.empty((K, d), dtype=torch.float32, device=dev)

    def e2e():
        for s in range(K):
            xin[s].copy_(xh[s], non_blocking=True)
            token(s, xin[s], cnt=False)
            yh[s].copy_(ybuf[s, L - 1], non_blocking=True)

    with torch.cuda.stream(stream):
        e2e()
        stream.synchronize()
    g_e2e = capture(e2e)
    with torch.cuda.stream(stream):
        g_e2e.replay()
    e2e_ms = statistics.median(timed_regions(torch, stream, g_e2e.replay, args.repeats, barrier))
    e2e_value, _ = aggregate([max_over_ranks(e2e_ms, world, dev)], [K * world], world)
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        budget = float(os.environ.get("PI_CPU_BUDGET_S", "15"))
        done, dt, cores = stack_oracle_sample(w, keep, 16, 1, budget, seed_off=13)
        cpu = {"value": done / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{done} tokens (after 1 untimed) through all {L} layers, fp64 oracle "
                         f"predict+compact+sparse FFN + residual per layer (layers visited one at "
                         f"a time; time-bounded at {budget:.0f} s)"}

    config = stack_config(w, L)
    config["parallelism"] = "replicas" if world > 1 else "single GPU"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config,
        "repeats": args.repeats, "regions_ms": regions,
        "us_per_token": ms_step * 1e3, "us_per_layer": ms_step * 1e3 / L,
        "density_per_layer": [float(v) / n for v in mean_cnt],
        "bytes_per_step": {"predictor": pred_bytes, "active_rows": alg_bytes - pred_bytes,
                           "total": alg_bytes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_kind": f"{peak_kind} copy bandwidth",
                     "kernel": f"seq_kernel (persistent, one token through {L} layers per launch)",
                     "traffic_how": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one "
                                     "launch (profiles/traffic.json)" if tr else
                                     "null: no capture of the current kernel source")},
        "dense_ffn": {"us_per_token": dense_ms * 1e3, "us_per_layer": dense_ms * 1e3 / L,
                      "tokens_per_s": 1e3 / dense_ms,
                      "achieved_gbs": dense_bytes / (dense_ms / 1e3) / 1e9,
                      "frac": dense_bytes / (dense_ms / 1e3) / 1e9 / peak},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": d * 4,
                "d2h_bytes_per_step": d * 4, "steps": K,
                "how": "per token: pinned H2D of its x, one pi_decode_layers launch through all "
                       "layers, D2H of its output; CUDA-graph replay"},
        "gpu_launches": K, "engine": "seq",
        "clocks": clocks, "cpu_baseline": cpu, "csrc_hash": csrc_hash(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_sweep(args):
    """Batched decode and density sweep (one JSON line, one entry per point):
    for each mean per-token density and batch B, one step = B tokens (each
    with its own x and its own predicted mask) through pi_layer_decode, the
    union of the tokens' active rows read once; the dense FFN at the same
    batch (pi_dense_ffn: every row read once for all B tokens) is the
    comparison point.  Two weight replicas alternate between steps."""
    import torch

    import activation_sparse_decode_rank_gb300 as pi
    import synth

    rank, world, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pi.build()
    from synth.workloads import WORKLOADS
    w = dict(WORKLOADS[args.workload])
    d, n, r = w["d"], w["n"], w["r"]
    K = max(20, min(args.steps, 400))
    G = 64
    pred_bytes = n * r * 2 + r * d * 2 + n * 4
    row_bytes = 2 * d * 2
    stream = torch.cuda.Stream(device=dev)
    points = []
    sampler = ClockSampler(local)
    sampler.start()
    for rho in w["densities"]:
        g = synth.make_layer_gpu(d, n, r, w["dtype"], alpha=w["alpha"], density=rho,
                                 seed=w["seed"], device=dev)
        pz = synth.zipf_probs(n, w["alpha"], synth.zipf_calibrate(n, w["alpha"], rho))
        hot = int((pz >= 0.5).sum()) if args.hot < 0 else args.hot
        desc = pi.make_desc(d, n, r, w["dtype"], False, hot, packed=True)
        rec = torch.empty((n, 2 * d), dtype=torch.int16, device=dev)
        pi.check(pi.pi_pack_weights(desc, g["W1"], g["W2"], rec), "pi_pack_weights")
        torch.cuda.synchronize()
        base = [g["A"], g["Bm"], g["b1"], rec, None, g["b2"]]
        reps = [base, [t.clone() if t is not None else None for t in base]]
        del g
        wts = [pi.make_weights(*rp) for rp in reps]
        for B in w["batches"]:
            xs = torch.from_numpy(np.stack(
                [synth.gen_x(w["seed"] + 100 * B, s, B, d) for s in range(G)])).to(dev)
            y = torch.empty((B, d), dtype=torch.float32, device=dev)
            st = torch.zeros(4, dtype=torch.int32, device=dev)
            ws = pi.workspace(desc, B, dev)
            cnt = torch.zeros((max(B, 4),), dtype=torch.int32, device=dev)

            def sp(s):
                pi.check(pi.pi_layer_decode(desc, wts[s % 2], xs[s % G], B, y, None, None, None,
                                            st, ws, stream=stream), "pi_layer_decode")

            def dn(s):
                pi.check(pi.pi_dense_ffn(desc, wts[s % 2], xs[s % G], B, y, ws, stream=stream),
                         "pi_dense_ffn")

            res = {}
            for name, fn in (("sparse", sp), ("dense", dn)):
                with torch.cuda.stream(stream):
                    for s in range(3):
                        fn(s)
                    stream.synchronize()
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=stream):
                        for s in range(K):
                            fn(s)
                    gr.replay()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    gr.replay()
                    e1.record(stream)
                    stream.synchronize()
                res[name] = e0.elapsed_time(e1) / K * 1e3  # us per step
                del gr
            if int(st[0]) != 0:
                raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
            # union sizes and per-token counts of the timed inputs (same kernels)
            logits = torch.empty((B, n), dtype=torch.float32, device=dev)
            idx = torch.empty((B, n), dtype=torch.int32, device=dev)
            uidx = torch.empty((n,), dtype=torch.int32, device=dev)
            ucnt = torch.zeros((4,), dtype=torch.int32, device=dev)
            tm = torch.empty((n,), dtype=torch.int32, device=dev)
            us, per_tok = [], []
            for s in range(0, G, 4):
                pi.check(pi.pi_predict(desc, reps[0][0], reps[0][1], reps[0][2], xs[s], B, logits,
                                       ws))
                pi.check(pi.pi_compact(logits, n, B, idx, cnt, n, uidx, ucnt, tm, st, ws))
                torch.cuda.synchronize()
                us.append(int(ucnt[0]))
                per_tok.append(float(cnt[:B].float().mean()))
            u_mean = float(np.mean(us))
            alg = pred_bytes + u_mean * row_bytes
            dense_alg = n * row_bytes + n * 4
            peak, _ = measured_peaks()
            points.append({
                "density": rho, "batch": B, "per_token_density": float(np.mean(per_tok)) / n,
                "union_density": u_mean / n,
                "sparse_us": res["sparse"], "dense_us": res["dense"],
                "sparse_tokens_per_s": B / res["sparse"] * 1e6,
                "dense_tokens_per_s": B / res["dense"] * 1e6,
                "speedup_vs_dense": res["dense"] / res["sparse"],
                "sparse_gbs": alg / res["sparse"] / 1e3, "sparse_frac": alg / res["sparse"] / 1e3 / peak,
                "dense_gbs": dense_alg / res["dense"] / 1e3,
                "dense_frac": dense_alg / res["dense"] / 1e3 / peak,
                "plan": sweep_plan(pi, desc, B, pz, res),
                "dispatched": sweep_dispatched(pi, torch, desc, wts[0], xs[0], B, pz, K, stream),
            })
            del xs, ws
        del reps, wts, base
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    cross = {}
    for B in w["batches"]:
        pts = sorted([p for p in points if p["batch"] == B], key=lambda p: p["density"])
        c = None
        for p0, p1 in zip(pts, pts[1:]):
            if p0["speedup_vs_dense"] >= 1.0 > p1["speedup_vs_dense"]:
                # log-linear interpolation of the speedup between the two densities
                a0, a1 = math.log(p0["speedup_vs_dense"]), math.log(p1["speedup_vs_dense"])
                c = p0["density"] + (p1["density"] - p0["density"]) * a0 / (a0 - a1)
        if c is None and pts and pts[-1]["speedup_vs_dense"] >= 1.0:
            c = f"> {pts[-1]['density']}"
        cross[str(B)] = c
    agree = [p["plan"]["agrees"] for p in points]
    peak, peak_kind = measured_peaks()
    print(json.dumps({
        "metric": "batched sparse-FFN decode: us per step and tokens/s vs the dense FFN",
        "workload": args.workload, "steps_per_point": K, "unit": "us",
        "config": {"d": d, "n": n, "r": r, "weights": w["dtype"], "layout": "packed",
                   "l2": "2 alternating weight replicas of 0.43 GB each"},
        "peak_gbs": peak, "peak_kind": peak_kind, "points": points,
        "crossover_density_per_batch": cross,
        "plan_agreement": {"points": len(agree), "agree": int(sum(agree)),
                           "how": "pi_plan_dispatch (built-in cost model, the generator's p_i, "
                                  "dense allowed) picks dense or the sparse path; agrees when "
                                  "the measured faster of the two is the same"},
        "clocks": clocks, "csrc_hash": csrc_hash(),
    }), flush=True)
    return 0


def sweep_dispatched(pi, torch, desc, w, x, B, pz, K, stream):
    """The step as a user runs it through the plan's executor: a pi_decoder
    (the generator's p_i as its profile, dense allowed) bound to fixed
    buffers, one graph launch per step; the path it chose and its measured
    microseconds per step."""
    d = desc.d
    dev = x.device
    xb = torch.zeros((32, d), dtype=torch.float32, device=dev)
    xb[:B].copy_(x)
    yb = torch.empty((32, d), dtype=torch.float32, device=dev)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    ws = pi.workspace(desc, 32, dev)
    rc, dec = pi.pi_decoder_create(desc, w, pz.astype(np.float32), 0.0, 1, None, xb, yb, None, st,
                                   ws)
    pi.check(rc, "pi_decoder_create")
    try:
        plan = pi.pi_plan()
        pi.check(pi.pi_decoder_plan(dec, B, plan))
        with torch.cuda.stream(stream):
            for _ in range(3):  # the first run captures the graph
                pi.check(pi.pi_decoder_run(dec, B, stream=stream))
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K):
                pi.check(pi.pi_decoder_run(dec, B, stream=stream))
            e1.record(stream)
            stream.synchronize()
        if int(st[0]) != 0:
            raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
        return {"path": pi.PATH_NAMES[plan.path], "us": e0.elapsed_time(e1) / K * 1e3,
                "how": "pi_decoder_run: one graph launch per step (one weight copy)"}
    finally:
        pi.pi_decoder_destroy(dec)


def sweep_plan(pi, desc, B, pz, res):
    """The dispatch plan of one sweep point against its measurement."""
    out = pi.pi_plan()
    pi.check(pi.pi_plan_dispatch(desc, B, pz.astype(np.float32), 0.0, 1, None, out),
             "pi_plan_dispatch")
    sp = pi.PI_PATH_FUSED if B == 1 else pi.PI_PATH_UNION
    plan_dense = out.est_us[pi.PI_PATH_DENSE] < out.est_us[sp]
    meas_dense = res["dense"] < res["sparse"]
    return {"path": pi.PATH_NAMES[out.path], "sparse_est_us": out.est_us[sp],
            "dense_est_us": out.est_us[pi.PI_PATH_DENSE],
            "per_token_est_us": out.est_us[pi.PI_PATH_PER_TOKEN],
            "union_rows_est": out.union_rows, "agrees": plan_dense == meas_dense}


def run_reorder(args):
    """Offline profiling and neuron placement, timed (one JSON line): the
    GPU predictor over sample tokens plus pi_profile_counts (per token),
    pi_hot_order, and pi_permute_neurons (bytes moved: every per-neuron
    tensor read and written once, against the HBM peak)."""
    import torch

    import activation_sparse_decode_rank_gb300 as pi
    import synth

    rank, world, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pi.build()
    w = workload_spec(args.workload)
    d, n, r = w["d"], w["n"], w["r"]
    gated = bool(w["gated"])
    if "alpha" in w:
        g = synth.make_layer_gpu(d, n, r, w["dtype"], gated=gated, alpha=w["alpha"],
                                 density=w["density"], seed=w["seed"], device=dev)
    else:  # a stack: its first layer
        alpha, _, cz, scale = synth.stack_plan(w["seed"], w["layers"], n)
        g = synth.make_layer_gpu(d, n, r, w["dtype"], gated=gated, alpha=float(alpha[0]),
                                 zipf_c=float(cz[0]), seed=w["seed"], layer=0,
                                 bias_scale=float(scale[0]), device=dev)
    torch.cuda.synchronize()
    desc = pi.make_desc(d, n, r, w["dtype"], gated, 0)
    src = pi.make_weights(g["A"], g["Bm"], g["b1"], g["W1"], g["W2"], g["b2"])
    B, T = 32, 256
    ws = pi.workspace(desc, B, dev)
    xs = torch.from_numpy(np.stack([synth.gen_x(w["seed"] + 77, s, B, d)
                                    for s in range(T // B)])).to(dev)
    lg = torch.empty((B, n), dtype=torch.float32, device=dev)
    counts = torch.zeros(n, dtype=torch.int32, device=dev)
    perm = torch.empty(n, dtype=torch.int32, device=dev)
    dst_t = [torch.empty_like(g["A"]), torch.empty_like(g["b1"]), torch.empty_like(g["W1"]),
             torch.empty_like(g["W2"])]
    dst = pi.make_weights(dst_t[0], g["Bm"], dst_t[1], dst_t[2], dst_t[3], g["b2"])
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            stream.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us

    def profile():
        for s in range(T // B):
            pi.check(pi.pi_predict(desc, g["A"], g["Bm"], g["b1"], xs[s], B, lg, ws, stream=stream))
            pi.check(pi.pi_profile_counts(lg, n, B, counts, stream=stream))

    us_prof = timed(profile, 5)
    us_rank = timed(lambda: pi.check(pi.pi_hot_order(counts, n, perm, stream=stream)), 5)
    us_perm = timed(lambda: pi.check(pi.pi_permute_neurons(desc, src, perm, dst, st,
                                                           stream=stream)), 10)
    if int(st[0]) != 0:
        raise SystemExit(f"bench: device status {pi.status_string(int(st[0]))}")
    moved = 2 * sum(t.numel() * t.element_size() for t in dst_t)
    peak, peak_kind = measured_peaks()
    print(json.dumps({
        "metric": "offline profiling and neuron placement", "workload": args.workload,
        "config": {"d": d, "n": n, "r": r, "weights": w["dtype"], "gated": gated,
                   "sample_tokens": T, "predictor_batch": B},
        "profile_us_per_token": us_prof / T, "hot_order_us": us_rank,
        "permute_us": us_perm, "permute_bytes": moved,
        "permute_gbs": moved / us_perm / 1e3, "permute_frac": moved / us_perm / 1e3 / peak,
        "peak_gbs": peak, "peak_kind": peak_kind, "csrc_hash": csrc_hash(),
    }), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="decode steps per timed region (default: 100 for the stack, 20000 "
                         "for one layer)")
    ap.add_argument("--warmup", type=int, default=None, help="untimed steps first (>= 3)")
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of --steps steps each; the median is reported")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0,
                    help="stack only: decode through its first LAYERS layers (0: all)")
    ap.add_argument("--replicas", type=int, default=0)
    ap.add_argument("--layout", default="packed", choices=["packed", "split"])
    ap.add_argument("--hot", type=int, default=-1, help="hot-prefix length (-1: p_i >= 0.5)")
    ap.add_argument("--graph-len", type=int, default=2000,
                    help="one layer: decode steps per pi_decode_layers launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reorder", action="store_true",
                    help="offline profiling + neuron placement timings for --workload")
    ap.add_argument("--sweep", action="store_true",
                    help="batched decode / density sweep (with --workload opt13b_ffn_batched_...)")
    args = ap.parse_args()
    from synth.workloads import WORKLOADS
    stack = WORKLOADS[args.workload].get("layers", 1) > 1
    if args.steps is None:
        args.steps = 100 if stack else 20000
    if args.warmup is None:
        args.warmup = 5 if stack else 2000
    if args.warmup < 3:
        raise SystemExit("bench: at least 3 warm-up steps")
    if args.repeats < 1:
        raise SystemExit("bench: at least one timed region")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.reorder:
        return run_reorder(args)
    if stack:
        return run_stack(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
