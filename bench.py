"""Benchmark of the MoE-layer forward on B300: one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config dsv3]
                    [--round off|nearest|up] [--impl ours|reference]

A step is one pass of the whole layer (route, permute or round, up-projection
+ SwiGLU, down-projection + gate weight, combine) over one batch of synthetic
tokens, launched through the C ABI stage by stage with CUDA events between the
stages (the same launches moe_forward makes), so the per-kernel durations come
from the timed region itself.  `value` is the active-expert TFLOP/s
(6*T*k*d*n useful FLOPs per step) summed over ranks; `tokens_per_s` and the
fraction of the measured bf16 peak ride along.  `e2e` is the same metric
through moe_forward with x copied from pinned host memory and y copied back
inside the timed region.

Multi-GPU: every rank runs its own replica on its own tokens (weak scaling, no
collective on the data path); timing is the max over ranks.

--impl reference times the fp64 CPU oracle (the checker the parity tests use)
on a bounded token sample on the host cores.

--backward measures the layer's backward pass instead (moe_backward through
the C ABI: routing, gathers and pre-activations recomputed, then the four
backward GEMMs and the router gradient); `value` counts 12*T*k*d*n FLOPs per
step (twice the forward's, recomputation not counted).

--graph adds a `graph` key: moe_forward captured once into a CUDA graph and
replayed per step.  --fp8 runs both expert GEMMs in e4m3.

With rounding off, and experts averaging at least 512 rows, the line also
carries `token_rounding`: the same layer with each expert's token count
rounded to the nearest multiple of the 256-row SM-pair tile, the method's
token rounding, timed the same way (--no-rounding-variant skips it).  It is
reported beside `value`, not in it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mixture_experts_layer_93_b300 import inputs as I  # noqa: E402

METRIC = "MoE fwd active TFLOPS & tokens/s on 1 B300; % bf16 tensor peak"
METRIC_BWD = "MoE bwd active TFLOPS & tokens/s on 1 B300; % bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# streams (and buffer sets) the forward e2e loop rotates over
E2E_STREAMS = 3
# token-rounding tile of the variant timed beside the plain layer: the
# 256-row M of an SM-pair tile
ROUND_TILE = 256

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# up-projection's main GEMM kernel, from an ncu capture of the current kernel,
# keyed by workload, A path and kernel revision; a kernel change bumps GEMM_REV
# and drops stale entries.  DeepSeek-V3-style layer: captured on the same layer
# with 32 of its 256 experts (T=2048, the same 512 rows per expert), 2.212 GB,
# scaled by the experts processed (x8).  The others at full size, on wide
# tiles: the 7B-class layer with the rows gathered in the operand load (A path
# 2), Mixtral-style and skewed layers on staged rows.
GEMM_REV = "wide-tiles-v15"
UP_TRAFFIC = {("dsv3", 0, GEMM_REV): 8 * 2211549440, ("mixtral", 0, GEMM_REV): 3741821696,
              ("b7", 2, GEMM_REV): 777297664, ("skew", 0, GEMM_REV): 5549915904}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- helpers
def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "ours") else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ oracle arm
class OracleLayerSampler:
    """Times the fp64 oracle (as it stands) on a bounded sample of the whole
    workload, the same way for the CPU baseline of our arm and for the
    reference arm.

    One sample is:
      1. the oracle's routing of every token (gate network, top-k, gate
         weights; token rounding when on): O.route;
      2. O.moe_forward over that routing for m seeded experts, i.e. each
         sampled expert's SwiGLU FFN over every row routed to it (its weights
         widened to fp64 inside the call, as the oracle does) and the
         gate-weighted sum into y.
    The oracle's time for the whole layer is estimated from the sample as
    t_route + (E / m) * t_experts (the m experts are a uniform random draw,
    so the scaled sum estimates all E).  m is fixed per workload from a
    one-expert probe so that a sample takes about `budget_s`."""

    def __init__(self, cfg, inp_host, round_mode, budget_s: float):
        from oracle import moe_oracle as O
        self.O, self.cfg, self.inp, self.mode = O, cfg, inp_host, round_mode
        self.rng = np.random.default_rng(1234)
        self._one(1)                        # the first call also pays one-time set-up
        t_route, t_exp, _ = self._one(1)
        per_expert = max(t_exp, 1e-3)
        self.m = int(min(cfg.E, max(1, round((budget_s - t_route) / per_expert))))

    def _one(self, m):
        O, cfg, inp = self.O, self.cfg, self.inp
        experts = np.sort(self.rng.choice(cfg.E, size=m, replace=False))
        c0 = time.process_time()
        t0 = time.perf_counter()
        routing = O.route(inp["x"], inp["Wr"], inp["bias"], cfg.k, cfg.tile, self.mode)
        t1 = time.perf_counter()
        O.moe_forward(inp["x"], inp["Wr"], inp["bias"], inp["W1"], inp["W3"], inp["W2"], k=cfg.k, tile=cfg.tile,
                      mode=self.mode, routing=routing, experts=experts)
        t2 = time.perf_counter()
        self.cpu = getattr(self, "cpu", 0.0) + time.process_time() - c0
        self.wall = getattr(self, "wall", 0.0) + t2 - t0
        return t1 - t0, t2 - t1, t2 - t0

    def sample(self):
        """One timed sample: (estimated whole-layer seconds, measured seconds)."""
        t_route, t_exp, t_all = self._one(self.m)
        return t_route + (self.cfg.E / self.m) * t_exp, t_all

    def threads(self):
        # threads actually used: process CPU time over wall time
        return max(1, int(round(self.cpu / self.wall))) if getattr(self, "wall", 0) > 0 else 1

    def describe(self, n_samples, measured_s):
        return (f"{n_samples} samples of the {self.cfg.name} workload, each the fp64 routing of all "
                f"{self.cfg.T} tokens plus the expert FFNs of {self.m} of {self.cfg.E} seeded experts over "
                f"all their rows (weights widened per call); whole-layer time estimated as "
                f"t_route + E/m * t_experts; {measured_s:.1f} s measured")


def oracle_baseline(cfg, inp_host, round_mode, budget_s: float, n_samples: int = 3):
    """The CPU-baseline object of our arm: the oracle's estimated whole-layer
    throughput from n_samples samples of about budget_s / n_samples each."""
    smp = OracleLayerSampler(cfg, inp_host, round_mode, budget_s / n_samples)
    est, meas = zip(*(smp.sample() for _ in range(n_samples)))
    t_layer = statistics.mean(est)
    return {"value": 6.0 * cfg.k * cfg.d * cfg.n * cfg.T / t_layer / 1e12, "unit": "TFLOP/s",
            "tokens_per_s": cfg.T / t_layer, "cores": smp.threads(), "host_cpus": os.cpu_count(),
            "kind": "oracle", "sample": smp.describe(n_samples, sum(meas))}


def bench_config(args):
    """The workload: the named config with --tokens, --experts and --tile applied."""
    from dataclasses import replace
    cfg = I.get_config(args.config)
    if getattr(args, "tokens", 0):
        cfg = cfg.with_tokens(args.tokens)
    if getattr(args, "experts", 0):
        cfg = replace(cfg, E=args.experts)
    if getattr(args, "tile", 0):
        cfg = replace(cfg, tile=args.tile)
    return cfg


def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = bench_config(args)
    inp = I.make_inputs(cfg, device="cpu", seed=0)
    if args.backward:
        inp["dy"] = torch.randn(cfg.T, cfg.d, generator=torch.Generator().manual_seed(1000)).to(torch.bfloat16)
        run_reference_backward(args, cfg, inp)
        return
    # each step is one sample; the warm-up steps are samples too
    budget = max(0.5, args.reference_seconds / max(args.steps, 1))
    smp = OracleLayerSampler(cfg, inp, args.round, budget)
    for _ in range(args.warmup):
        smp.sample()
    smp.cpu = smp.wall = 0.0
    est, meas = [], []
    for _ in range(args.steps):
        e, m = smp.sample()
        est.append(e)
        meas.append(m)
    t_layer = statistics.mean(est)
    value = 6.0 * cfg.k * cfg.d * cfg.n * cfg.T / t_layer / 1e12
    desc = smp.describe(args.steps, sum(meas))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(meas),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.description, "round": args.round, "sample": desc,
                   "value_from": "whole-layer oracle time estimated from each step's sample; ms_per_step is "
                                 "the sample's measured time"},
        "tokens_per_s": cfg.T / t_layer,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": smp.threads(), "kind": "oracle",
                         "sample": desc, "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_backward(args, cfg, inp):
    active_per_token = 12.0 * cfg.k * cfg.d * cfg.n
    for _ in range(args.warmup):
        oracle_backward_time(cfg, inp, 0.0, 0)   # one small call each
    times, toks, threads = [], 0, 1
    budget = max(1.0, args.reference_seconds / max(args.steps, 1))
    for i in range(args.steps):
        nt, dt, desc, th = oracle_backward_time(cfg, inp, budget, 100 + i)
        times.append(dt)
        toks += nt
        threads = max(threads, th)
    total = sum(times)
    tps = toks / total
    value = tps * active_per_token / 1e12
    line = {
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.description, "round": args.round, "tokens_per_step": toks // args.steps},
        "tokens_per_s": tps,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": desc, "host_cpus": os.cpu_count()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- backward
def oracle_backward_time(cfg, inp_host, budget_s: float, seed: int = 0):
    """Times the oracle's backward pass (as it stands) on token subsets of the
    workload until ~budget_s; returns (tokens, seconds, description, threads)."""
    from oracle import moe_oracle as O
    rng = np.random.default_rng(seed)
    n = 16
    total_tok, total_s, total_cpu = 0, 0.0, 0.0
    while True:
        toks = np.sort(rng.choice(cfg.T, size=min(n, cfg.T), replace=False))
        x = inp_host["x"][toks]
        dy = inp_host["dy"][toks]
        t0, c0 = time.perf_counter(), time.process_time()
        O.moe_backward(x, inp_host["Wr"], inp_host["bias"], inp_host["W1"], inp_host["W3"], inp_host["W2"], dy,
                       k=cfg.k)
        dt = time.perf_counter() - t0
        total_cpu += time.process_time() - c0
        total_tok += len(toks)
        total_s += dt
        if total_s >= budget_s:
            break
        if dt < budget_s / 4:
            n = min(cfg.T, n * 2)
    desc = (f"backward of {total_tok} sampled tokens of the {cfg.name} workload as token subsets (fp64), "
            f"{total_s:.1f} s")
    threads = max(1, int(round(total_cpu / total_s))) if total_s > 0 else 1
    return total_tok, total_s, desc, threads


def run_backward(args, world, rank, local):
    from mixture_experts_layer_93_b300 import binding as B
    import ctypes

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    cfg = bench_config(args)
    T, k, E, d, n = cfg.T, cfg.k, cfg.E, cfg.d, cfg.n
    shape = B.make_shape(T, d, n, E, k, cfg.tile, args.round, args.seed)
    inp = I.make_replica_inputs(cfg, rank, device=dev)
    g = torch.Generator(device=dev).manual_seed(1000 + rank)
    dy = torch.randn(T, d, generator=g, device=dev).to(torch.bfloat16)
    W13p, _ = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13i = B.moe_prepare_weights_bwd(inp["W1"], inp["W3"])
    W2 = inp["W2"]
    inp_host = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_host = {kk: (v.cpu() if isinstance(v, torch.Tensor) else v) for kk, v in inp.items()}
        inp_host["dy"] = dy.cpu()
    del inp["W1"], inp["W3"]
    torch.cuda.empty_cache()
    x, Wr, bias = inp["x"], inp["Wr"], inp["bias"]
    ws = B.Workspace(shape, dev, backward=True)
    out = {"dx": torch.empty(T, d, dtype=torch.float32, device=dev),
           "dWr": torch.empty(d, E, dtype=torch.float32, device=dev),
           "dbias": torch.empty(E, dtype=torch.float32, device=dev) if bias is not None else None,
           "dW1": torch.empty(E, d, n, dtype=torch.float32, device=dev),
           "dW3": torch.empty(E, d, n, dtype=torch.float32, device=dev),
           "dW2": torch.empty(E, n, d, dtype=torch.float32, device=dev)}
    L = B.lib()
    sp = ctypes.byref(shape)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = torch.cuda.current_stream(dev)

    def bwd(x_, dy_, dx_, ws_, st_):
        rc = L.moe_backward(sp, P(x_), P(Wr), P(bias), P(W13p), P(W13i), P(W2), P(dy_), P(dx_), P(out["dWr"]),
                            P(out["dbias"]), P(out["dW1"]), P(out["dW3"]), P(out["dW2"]), ws_.ptr, ws_.nbytes,
                            ctypes.c_void_p(st_.cuda_stream))
        if rc != 0:
            raise B.MoEError(rc, "moe_backward")

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        bwd(x, dy, out["dx"], ws, stream)
    torch.cuda.synchronize()
    B.moe_check_device_status(ws)
    clocks = ClockSampler(local)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(float(i))          # L2 flush between steps (not timed)
        ev[i][0].record(stream)
        bwd(x, dy, out["dx"], ws, stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    B.moe_check_device_status(ws)
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
    flops = 2.0 * cfg.active_flops()
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # e2e: x and dy in from pinned memory, dx back, every step; the weight
    # gradients stay on the device (an optimizer step would consume them there)
    x_host = torch.empty(T, d, dtype=torch.bfloat16, pin_memory=True)
    dy_host = torch.empty(T, d, dtype=torch.bfloat16, pin_memory=True)
    dx_host = torch.empty(T, d, dtype=torch.float32, pin_memory=True)
    x_host.copy_(x.cpu())
    dy_host.copy_(dy.cpu())
    x_dev, dy_dev, dx_dev = torch.empty_like(x), torch.empty_like(dy), torch.empty_like(out["dx"])

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        dy_dev.copy_(dy_host, non_blocking=True)
        bwd(x_dev, dy_dev, dx_dev, ws, stream)
        dx_host.copy_(dx_dev, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    B.moe_check_device_status(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    if rank != 0:
        return
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    # launches per moe_backward: route + permute (4, 5 or 6, as the forward;
    # with rounding route 3 + round 9, and no rows kernel), padded offsets and
    # rows (2), zero padding, two gathers, pre-activations, SwiGLU backward,
    # router backward, dW2, dW1/dW3, router transpose, dx rows (1, or 2 with
    # separate odd blocks), the rows' sum per token, dWr partial and final
    capp = T * k + (E * cfg.tile if args.round != "off" else 0) + 63 * E
    dx_launches = 1 if 128.0 * E <= 0.15 * capp else 2
    fused_route = 4 if (E <= 256 and k <= 8) else (5 if E <= 256 else 6)
    if args.round != "off":
        fused_route = 3 + 9 - 1
    launches = fused_route + 2 + 1 + 2 + 1 + 1 + 1 + 2 + 1 + dx_launches + 1 + 2
    line = {
        "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.description + ", backward pass", "T": T, "d": d, "n": n, "E": E, "k": k,
                   "round": args.round, "tile": cfg.tile if args.round != "off" else None,
                   "flops_per_step": flops, "outputs": "dx, dWr, dbias, dW1, dW3, dW2 in fp32",
                   "l2": "256 MiB buffer written between timed steps; expert weights also exceed L2",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": world * T * args.steps / (total_ms * 1e-3),
        "frac_of_bf16_peak": value / world / burst,
        "frac_of_bf16_sustained_peak": value / world / sustained,
        "peak_source": f"{peak_src} bf16_tflops (burst)",
        "e2e": {"value": world * flops * args.steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": 2 * T * d * 2, "d2h_bytes_per_step": T * d * 4,
                "how": "moe_backward per step with x and dy H2D from pinned memory and dx D2H; weight "
                       "gradients stay on the device"},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
    }
    if inp_host is not None:
        ntok, secs, desc, threads = oracle_backward_time(cfg, inp_host, budget_s=args.cpu_seconds)
        line["cpu_baseline"] = {"value": ntok * 12.0 * k * d * n / secs / 1e12, "unit": "TFLOP/s",
                                "tokens_per_s": ntok / secs, "cores": threads, "host_cpus": os.cpu_count(),
                                "kind": "oracle", "sample": desc}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    from mixture_experts_layer_93_b300 import binding as B

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    cfg = bench_config(args)
    mode = args.round
    shape = B.make_shape(cfg.T, cfg.d, cfg.n, cfg.E, cfg.k, cfg.tile, mode, args.seed)
    if args.gather < 0:  # the A path moe_forward takes (the e4m3 layer has its own quantising gather)
        args.gather = 0 if args.fp8 else B.moe_forward_a_path(shape)
    inp = I.make_replica_inputs(cfg, rank, device=dev)
    W13p, W2p = B.moe_prepare_weights(inp["W1"], inp["W3"], inp["W2"])
    W13q = sW13 = W2q = sW2 = None
    if args.fp8:
        # e4m3 GEMMs: codes with one scale per packed W1/W3 row and per packed W2 row
        W13q, sW13 = B.moe_quantize_rows_fp8(W13p)
        W2q, sW2 = B.moe_quantize_rows_fp8(W2p)
        del W13p, W2p
        W13p = W2p = None
    inp_host = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_host = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    del inp["W1"], inp["W3"], inp["W2"]
    torch.cuda.empty_cache()
    x, Wr, bias = inp["x"], inp["Wr"], inp["bias"]
    ws = B.Workspace(shape, dev, fp8=args.fp8)
    lay = B.moe_workspace_layout(shape)
    cap = B.moe_row_capacity(shape)
    T, k, E, d, n = cfg.T, cfg.k, cfg.E, cfg.d, cfg.n
    A = T * k

    def view(slot, dtype, numel):
        off = lay[slot]
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws.buf[off:off + numel * esz].view(dtype)

    logits = view("logits", torch.float32, T * E)
    idx = view("topk_idx", torch.int32, A)
    w = view("topk_w", torch.float32, A)
    counts = view("counts", torch.int32, E)
    offsets = view("offsets", torch.int32, E + 1)
    src = view("src", torch.int32, cap)
    dst = view("dst", torch.int32, A)
    row_token = view("row_token", torch.int32, cap)
    row_w = view("row_w", torch.float32, cap)
    tok_offsets = view("tok_offsets", torch.int32, T + 1)
    tok_rows = view("tok_rows", torch.int32, cap)
    h = view("h", torch.bfloat16, cap * n)
    ys = view("ys", torch.float16, cap * d)
    y = torch.empty(T, d, dtype=torch.float32, device=dev)
    L = B.lib()
    import ctypes
    sp = ctypes.byref(shape)
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    stream = torch.cuda.current_stream(dev)
    st = ctypes.c_void_p(stream.cuda_stream)
    # rounding off: route+permute fused (Wr split, router GEMM, fused top-k +
    # histogram, scan, scatter: 5 launches; 4 when k <= 8, where the router
    # GEMM's epilogue takes the top-k; 6 when E > 256); rounding: route
    # (Wr split, router GEMM, top-k: 3) then member, select, transpose, 2
    # offsets, sets + a 3-launch permutation (9).  up: row gather + SM-pair GEMM
    # + odd-block GEMM (A path 0) or one GEMM (paths 1, 2); down: SM-pair +
    # odd-block GEMMs; combine: 1
    stages = ["route_permute", "up", "down", "combine"] if mode == "off" else \
        ["route", "round", "up", "down", "combine"]
    # SM-pair GEMMs run an expert's odd last block in the same launch when
    # odd blocks are a small share (128 E <= 0.15 rows), else in a second one
    gemm_launches = 1 if 128.0 * E <= 0.15 * cap else 2
    up_launches = (1 + gemm_launches) if args.gather == 0 else (gemm_launches if d % 1 == 0 and n % 128 == 0 else 1)
    if args.fp8:
        up_launches = 2  # quantising gather + one SM-pair e4m3 GEMM
        gemm_launches = 2  # down: h quantisation + one SM-pair e4m3 GEMM
    fused_route = 4 if (E <= 256 and k <= 8) else (5 if E <= 256 else 6)
    # rounding: moe_route (weights prepared + router with the top-k where
    # k <= 8 and E <= 256, else + a top-k kernel) then the 9 rounding launches
    route_launches = fused_route if mode == "off" else (2 if (E <= 256 and k <= 8) else 3) + 9
    launches_per_step = route_launches + up_launches + gemm_launches + 1

    def check(rc, what):
        if rc != 0:
            raise B.MoEError(rc, what)

    def step(ev=None):
        marks = iter(ev) if ev else None

        def mark():
            if marks:
                next(marks).record(stream)

        mark()
        if mode == "off":
            check(L.moe_route_permute(sp, P(x), P(Wr), P(bias), P(logits), P(idx), P(w), P(counts), P(offsets),
                                      P(src), P(dst), P(row_token), P(row_w), ws.ptr, ws.nbytes, st), "route_permute")
            c_off, c_rows = None, dst
        else:
            check(L.moe_route(sp, P(x), P(Wr), P(bias), P(logits), P(idx), P(w), ws.ptr, st), "route")
            mark()
            check(L.moe_token_round(sp, P(logits), P(idx), P(counts), P(offsets), P(row_token), P(row_w),
                                    P(tok_offsets), P(tok_rows), ws.ptr, ws.nbytes, st), "round")
            c_off, c_rows = tok_offsets, tok_rows
        mark()
        if args.fp8:
            check(L.moe_expert_up_fp8(sp, P(x), P(W13q), P(sW13), P(counts), P(offsets), P(c_off), P(c_rows), P(h),
                                      ws.ptr, ws.nbytes, st), "up_fp8")
        else:
            check(L.moe_expert_up(sp, P(x), P(W13p), P(counts), P(offsets), P(row_token), P(c_off), P(c_rows),
                                  P(h), args.gather, ws.ptr, ws.nbytes, st), "up")
        mark()
        if args.fp8:
            check(L.moe_expert_down_fp8(sp, P(h), P(W2q), P(sW2), P(counts), P(offsets), P(row_w), P(ys), ws.ptr,
                                        ws.nbytes, st), "down_fp8")
        else:
            check(L.moe_expert_down(sp, P(h), P(W2p), P(counts), P(offsets), P(row_w), P(ys), ws.ptr, ws.nbytes,
                                    st), "down")
        mark()
        check(L.moe_combine(sp, P(ys), P(c_off), P(c_rows), P(y), st), "combine")
        mark()

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    B.moe_check_device_status(ws)

    clocks = ClockSampler(local)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(float(i))          # L2 flush between steps (not timed)
        step(events[i])
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    B.moe_check_device_status(ws)
    step_ms = [events[i][0].elapsed_time(events[i][-1]) for i in range(args.steps)]
    stage_ms = {s: [events[i][j].elapsed_time(events[i][j + 1]) for i in range(args.steps)]
                for j, s in enumerate(stages)}
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    R = int(offsets[E].item())
    active = cfg.active_flops()
    value = world * active * args.steps / (total_ms * 1e-3) / 1e12
    tokens_per_s = world * T * args.steps / (total_ms * 1e-3)

    # ------------------------------------------------ optional: the same layer replayed as one CUDA graph
    graph_line = None
    if args.graph:
        def forward_on(st_ptr):
            if args.fp8:
                check(L.moe_forward_fp8(sp, P(x), P(Wr), P(bias), P(W13q), P(sW13), P(W2q), P(sW2), P(y), ws.ptr,
                                        ws.nbytes, st_ptr), "forward_fp8")
            else:
                check(L.moe_forward(sp, P(x), P(Wr), P(bias), P(W13p), P(W2p), P(y), ws.ptr, ws.nbytes, st_ptr),
                      "forward")

        gstream = torch.cuda.Stream(dev)
        gstream.wait_stream(stream)
        forward_on(ctypes.c_void_p(gstream.cuda_stream))   # warm-up outside the capture
        stream.wait_stream(gstream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            forward_on(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            flush.fill_(float(i))
            gev[i][0].record(stream)
            graph.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        B.moe_check_device_status(ws)
        g_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in gev), world, dev)
        graph_line = {"value": world * cfg.active_flops() * args.steps / (g_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "ms_per_step": g_ms / args.steps,
                      "how": "moe_forward captured once into a CUDA graph, replayed per step (L2 flushed between)"}

    # ------------------------------------------------ the same layer with the pages' token rounding
    # Each expert's count rounded to the nearest multiple of the 256-row
    # SM-pair tile (MOE_ROUND_NEAREST): a variant of the method, reported
    # beside `value`, never in its place.  Rows come from the rounding of the
    # same logits, read outside the timed region.  Only where experts average
    # at least two tiles of rows: below that the rounding mostly drops rows.
    rounding_line = None
    if (args.round == "off" and not args.fp8 and not args.no_rounding_variant
            and T * k >= 2 * ROUND_TILE * E):
        rshape = B.make_shape(T, d, n, E, k, ROUND_TILE, "nearest", args.seed)
        rws = B.Workspace(rshape, dev)
        ry = torch.empty_like(y)
        rsp = ctypes.byref(rshape)

        def rforward():
            check(L.moe_forward(rsp, P(x), P(Wr), P(bias), P(W13p), P(W2p), P(ry), rws.ptr, rws.nbytes,
                                ctypes.c_void_p(stream.cuda_stream)), "forward (token rounding)")

        for _ in range(args.warmup):
            rforward()
        torch.cuda.synchronize()
        rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier(world)
        for i in range(args.steps):
            flush.fill_(float(i))
            rev[i][0].record(stream)
            rforward()
            rev[i][1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
        B.moe_check_device_status(rws)
        r_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in rev), world, dev)
        rlogits, ridx, _ = B.moe_route(x, Wr, bias, k, rws)
        R_round = int(B.moe_token_round(rshape, rlogits, ridx, rws)["offsets"][E].item())
        rounding_line = {"round": "nearest", "tile": ROUND_TILE,
                         "value": world * active * args.steps / (r_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                         "executed_tflops": world * 6.0 * R_round * d * n * args.steps / (r_ms * 1e-3) / 1e12,
                         "rows": R_round, "ms_per_step": r_ms / args.steps,
                         "how": "moe_forward on the same inputs with each expert's token count rounded to the "
                                "nearest multiple of the SM-pair tile (L2 flushed between steps); value counts "
                                "6*T*k*d*n like the line's, executed_tflops the rounded rows"}
        del rws, ry

    # ------------------------------------------------ e2e: through moe_forward, host buffers
    # Each step copies its x from pinned host memory, runs moe_forward and
    # copies its y back.  Steps rotate over E2E_STREAMS streams (each with its
    # own buffers and workspace), as a serving loop would run them: the next
    # step's input copy and the previous step's output copy (separate copy
    # engines) overlap this step's compute.  With two streams, step i + 2
    # could not copy its input in before step i's output copy had finished.
    x_cpu = x.cpu()
    streams = [torch.cuda.Stream(dev) for _ in range(E2E_STREAMS)]
    wss = [ws] + [B.Workspace(shape, dev, fp8=args.fp8) for _ in range(E2E_STREAMS - 1)]
    x_host = [torch.empty(T, d, dtype=torch.bfloat16, pin_memory=True) for _ in range(E2E_STREAMS)]
    y_host = [torch.empty(T, d, dtype=torch.float32, pin_memory=True) for _ in range(E2E_STREAMS)]
    for xh in x_host:
        xh.copy_(x_cpu)
    x_dev = [torch.empty_like(x) for _ in range(E2E_STREAMS)]
    y_dev = [torch.empty_like(y) for _ in range(E2E_STREAMS)]

    def e2e_step(i):
        b = i % E2E_STREAMS
        st_b = streams[b]
        with torch.cuda.stream(st_b):
            x_dev[b].copy_(x_host[b], non_blocking=True)
            if args.fp8:
                check(L.moe_forward_fp8(sp, P(x_dev[b]), P(Wr), P(bias), P(W13q), P(sW13), P(W2q), P(sW2),
                                        P(y_dev[b]), wss[b].ptr, wss[b].nbytes, ctypes.c_void_p(st_b.cuda_stream)),
                      "forward_fp8")
            else:
                check(L.moe_forward(sp, P(x_dev[b]), P(Wr), P(bias), P(W13p), P(W2p), P(y_dev[b]), wss[b].ptr,
                                    wss[b].nbytes, ctypes.c_void_p(st_b.cuda_stream)), "forward")
            y_host[b].copy_(y_dev[b], non_blocking=True)

    for i in range(max(E2E_STREAMS, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev_end = [torch.cuda.Event(enable_timing=True) for _ in range(E2E_STREAMS)]
    ev0.record(stream)
    for st_b in streams:
        st_b.wait_event(ev0)
    for i in range(args.steps):
        e2e_step(i)
    for b in range(E2E_STREAMS):
        ev_end[b].record(streams[b])
    torch.cuda.synchronize()
    barrier(world)
    for w_ in wss:
        B.moe_check_device_status(w_)
    e2e_ms = max_over_ranks(max(ev0.elapsed_time(e) for e in ev_end), world, dev)
    e2e_value = world * active * args.steps / (e2e_ms * 1e-3) / 1e12

    if rank != 0:
        return
    # ------------------------------------------------ roofline of the dominant kernel (up-projection)
    up_ms = statistics.mean(stage_ms["up"])
    up_flops = 4.0 * R * d * n
    up_tflops = up_flops / (up_ms * 1e-3) / 1e12
    # peak: the measured burst bf16 figure (the conservative denominator); the
    # fraction of the measured sustained (power-capped) figure rides along
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    peak_t = burst
    peak_kind = "bf16_tflops (burst)"
    up_peak, up_peak_kind = peak_t, peak_kind
    if args.fp8:
        # e4m3 contraction: the measured bf16 burst peak times the nominal
        # dense e4m3 : bf16 ratio (4.5 : 2.25 PFLOP/s)
        up_peak, up_peak_kind = 2.0 * burst, "bf16_tflops (burst) x 2 (nominal e4m3:bf16)"
    roofline = {"bound": "tensor", "kernel": "moe_gemm_kernel<up%s, SwiGLU>" % (" e4m3" if args.fp8 else ""),
                "achieved": up_tflops, "peak": up_peak, "unit": "TFLOP/s", "frac": up_tflops / up_peak,
                "traffic": UP_TRAFFIC.get((cfg.name, args.gather, GEMM_REV))
                if (T, E) == (I.get_config(cfg.name).T, I.get_config(cfg.name).E) and not args.fp8
                and args.round == "off" else None,
                "traffic_unit": "bytes per launch of the main up GEMM kernel (ncu dram read+write)",
                # W13, the A rows (staged rows, or x itself once where the
                # gather is in the operand load), h
                "algorithmic_bytes_per_launch": 2.0 * E * 2 * n * d + (R if args.gather == 0 else T) * d * 2.0
                + R * n * 2.0,
                "peak_source": f"{peak_src} {up_peak_kind}",
                "frac_of_sustained": up_tflops / (sustained * up_peak / peak_t),
                "algorithmic_flops_per_launch": up_flops}
    # HBM-bound stages: algorithmic bytes / time
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    comb_bytes = R * d * 2 + T * d * 4 + A * 4
    comb_gbs = comb_bytes / (statistics.mean(stage_ms["combine"]) * 1e-3) / 1e9
    down_flops = 2.0 * R * n * d
    stage_summary = {s: round(statistics.mean(v), 4) for s, v in stage_ms.items()}
    # routing stage, algorithmic bytes: x and Wr read once; logits, top-k ids
    # and weights written once; with the permutation also counts, offsets and
    # src, dst, row_token, row_w written once
    route_stage = "route_permute" if mode == "off" else "route"
    route_bytes = T * d * 2 + d * E * 4 + T * E * 4 + A * 8
    if mode == "off":
        route_bytes += (2 * E + 1) * 4 + A * 16
    route_gbs = route_bytes / (statistics.mean(stage_ms[route_stage]) * 1e-3) / 1e9
    extra = {
        "stage_ms": stage_summary,
        "down_tflops": down_flops / (statistics.mean(stage_ms["down"]) * 1e-3) / 1e12,
        "combine_gbs": comb_gbs, "combine_frac_hbm": comb_gbs / hbm_peak,
        route_stage + "_gbs": route_gbs, route_stage + "_frac_hbm": route_gbs / hbm_peak,
        route_stage + "_bytes": route_bytes,
        "rows": R,
    }
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 expert GEMMs" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.description, "T": T, "d": d, "n": n, "E": E, "k": k, "round": mode,
                   "up_gather": ["gather_kernel+tma", "tma_gather4",
                                 "cp_async (gather in the operand load)"][args.gather],
                   "expert_gemm_operands": "e4m3 (x per token, W1/W3 per channel, h per row, W2 per channel)"
                   if args.fp8 else "bf16",
                   "tile": cfg.tile if mode != "off" else None,
                   "l2": "256 MiB buffer written between timed steps; expert weights also exceed L2",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": tokens_per_s,
        # rows the expert GEMMs ran on (R = T*k without rounding): executed FLOPs
        "executed_tflops": world * 6.0 * R * d * n * args.steps / (total_ms * 1e-3) / 1e12,
        "frac_of_bf16_peak": value / world / peak_t,
        "frac_of_bf16_sustained_peak": value / world / sustained,
        "roofline": roofline,
        "stages": extra,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "tokens_per_s": world * T * args.steps / (e2e_ms * 1e-3),
                "h2d_bytes_per_step": T * d * 2, "d2h_bytes_per_step": T * d * 4,
                "how": "moe_forward per step with its x H2D from pinned memory and y D2H, steps rotating "
                       f"over {E2E_STREAMS} streams; weights resident (inputs exceed L2, no flush)"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if graph_line is not None:
        line["graph"] = graph_line
    if rounding_line is not None:
        rounding_line["frac_of_bf16_peak"] = rounding_line["value"] / world / burst
        line["token_rounding"] = rounding_line
    if inp_host is not None:
        line["cpu_baseline"] = oracle_baseline(cfg, inp_host, mode, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def launch_ranks(args) -> int:
    """`--gpus N` without a launcher: start N ranks of this script, one per
    GPU, with torch.distributed.run on this node (rendezvous on 127.0.0.1),
    exactly as a torchrun launch of the same command would, and return the
    launcher's exit status.  Rank 0 prints the JSON line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def run_dry(args, world, rank):
    """The replica set-up without the GPU: each rank draws its replica's
    inputs (tiny shapes allowed) on the CPU, the ranks meet at the barrier,
    check that their weights are identical and their tokens are not, and
    reduce a per-rank time with the max, as a measured run does."""
    cfg = I.get_config(args.config)
    inp = I.make_replica_inputs(cfg, rank, device="cpu")
    dev = torch.device("cpu")
    wsum = float(sum(inp[k_].double().abs().sum() for k_ in ("Wr", "W1", "W3", "W2")))
    xsum = float(inp["x"].double().sum())
    barrier(world)
    same_w = max_over_ranks(wsum, world, dev) == -max_over_ranks(-wsum, world, dev)
    distinct_x = world == 1 or max_over_ranks(xsum, world, dev) != -max_over_ranks(-xsum, world, dev)
    t = max_over_ranks(1.0 + rank, world, dev)
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "max_rank_time": t, "weights_identical": same_w,
                          "tokens_distinct": distinct_x, "config": {"workload": cfg.description}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="dsv3", choices=sorted(I.CONFIGS))
    ap.add_argument("--round", default="off", choices=["off", "nearest", "up", "stochastic"])
    ap.add_argument("--seed", type=int, default=0, help="seed of the stochastic rounding draws")
    ap.add_argument("--no-rounding-variant", action="store_true",
                    help="skip the token-rounding variant timed beside the plain layer")
    ap.add_argument("--tile", type=int, default=0, choices=[0, 64, 128, 256],
                    help="token-rounding tile (default: the config's, 128)")
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling of small cases only)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling of small cases only)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8", action="store_true",
                    help="e4m3 expert GEMMs (moe_forward_fp8); the default measures the bf16 layer")
    ap.add_argument("--gather", type=int, default=-1, choices=[-1, 0, 1, 2],
                    help="up-projection A operand: -1 = the path moe_forward takes for the shape (default), "
                         "0 = gather kernel then tiled TMA, 1 = TMA gather4 of token rows, 2 = per-lane "
                         "cp.async of token rows")
    ap.add_argument("--graph", action="store_true",
                    help="also time moe_forward replayed from one captured CUDA graph")
    ap.add_argument("--backward", action="store_true",
                    help="measure the backward pass (moe_backward) instead of the forward")
    ap.add_argument("--dry-run", action="store_true",
                    help="replica set-up, barrier and max-over-ranks only, on the CPU (no kernels)")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args))
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        # the oracle runs on rank 0 only; the other ranks exit without work
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), 0)
        return
    world, rank, local = dist_init(args)
    try:
        if args.dry_run:
            run_dry(args, world, rank)
        else:
            (run_backward if args.backward else run_ours)(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
