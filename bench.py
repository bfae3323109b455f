"""Benchmark: decode-time MoE FFN stage on GB300.

Workload (the one the metric is quoted on): a 40-layer FFN-only decode stack
of Qwen3.6-35B-A3B-shaped layers (hidden 2048, 256 experts, top-8, expert
width 512, Q4_K routed gate/up/down, Q4_K shared expert of width 512 with a
sigmoid gate, bf16 router, residual folded into RMSNorm), 128 sequential
tokens, captured as one CUDA graph. One step = one replay of that graph =
128 x 40 layer-tokens. Weights are seeded synthetic data of those shapes
(18.2 GB resident; every token reads 679 MB of weights, far above the
129 MB L2, so no L2 flush is needed between steps).

Metric: microseconds per layer per token (lower is better), with the
weight-read bandwidth it implies against the measured HBM peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (the plain fp64 restatement of the
method) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import os

# The CPU baseline times the oracle single-threaded: pin numpy's BLAS before
# anything imports numpy.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import hashlib
import json  # noqa: E402
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE FFN decode µs/layer/token; expert weight-read HBM GB/s vs GB300 peak"
UNIT = "us/layer/token"
N_LAYERS, N_TOKENS, SEED = 40, 128, 4040
WORKLOAD = ("40-layer FFN-only decode stack, Qwen3.6-35B-A3B-shaped layers (H=2048, E=256, "
            "top-8, I=512, Q4_K routed + Q4_K shared I=512, bf16 router), 128 sequential "
            "tokens, one CUDA graph")

# Algorithmic bytes per layer-token (weights only; activations are < 20 KB):
# router 256x2048 bf16, 8 routed experts x 3 Q4_K matrices of 512x2048,
# shared expert 3 Q4_K matrices, sigmoid-gate vector.
Q4K_MATRIX = 512 * 2048 // 256 * 144                    # 589,824
BYTES_ROUTER = 256 * 2048 * 2                           # 1,048,576
BYTES_ROUTED = 8 * 3 * Q4K_MATRIX                       # 14,155,776
BYTES_SHARED = 3 * Q4K_MATRIX                           # 1,769,472
BYTES_SIGMOID = 2048 * 2
BYTES_LAYER_TOKEN = BYTES_ROUTER + BYTES_ROUTED + BYTES_SHARED + BYTES_SIGMOID   # 16,977,920
STACK_KERNEL_SOURCES = ["moe_decode_ffn_gb300/csrc/stack.cu", "moe_decode_ffn_gb300/csrc/common.cuh",
                        "moe_decode_ffn_gb300/csrc/topk.cuh"]

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"si_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_max(value: float, pg) -> float:
    """The largest per-rank value over all ranks (the slowest replica bounds
    the job); `pg` is torch.distributed when there are several ranks, else
    None."""
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_us_per_layer_token(ms_step: float, world: int) -> float:
    """Whole-job µs per layer-token: in one step each of `world` replicas runs
    all N_LAYERS x N_TOKENS layer-tokens."""
    return ms_step * 1e3 / (N_LAYERS * N_TOKENS) / world


def _traffic_record(kernel_sources):
    """DRAM bytes per layer-token of the persistent stack kernel from the
    committed ncu record, valid only while the kernel sources match the
    captured ones."""
    path = os.path.join(ROOT, "profiles", "stack_q4k_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    h = hashlib.sha256()
    for src in kernel_sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if rec.get("source_sha256") != h.hexdigest():
        return None
    return rec.get("bytes_per_layer_token")


def oracle_jobs(n_layer_tokens: int, device="cpu"):
    """Inputs of a bounded sample of the workload for the CPU oracle: layer-tokens
    (layer l, token t) of the same stack, with the router weights and the
    selected experts' weights materialised (generated on `device`, then kept
    on the host)."""
    import torch

    import gen
    from oracle import moe as M
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    x = gen.make_tokens(SEED, (n_layer_tokens + N_LAYERS - 1) // N_LAYERS)
    jobs = []
    for i in range(n_layer_tokens):   # distinct (layer, token) pairs
        layer = i % N_LAYERS
        xt = x[i // N_LAYERS]
        w_router = gen.to_bf16(gen.normal([gen.stream_key(SEED, layer, gen.ROLE_ROUTER, 0)],
                                          spec.n_experts * spec.hidden, 0.0, gen.WEIGHT_STD,
                                          device)).reshape(spec.n_experts, spec.hidden).cpu()
        ids = M.topk_sort(M.router_logits(M.as_f64(xt), w_router))
        L = gen.make_layer(spec, SEED, layer, device=device, experts=ids)
        L = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in L.items()}
        jobs.append((L, xt))
    return jobs


def time_oracle(jobs):
    """Seconds per layer-token of the oracle's whole layer (router, top-8,
    softmax, 9 experts in integer mode, residual norm) over `jobs`."""
    from oracle import moe as M
    t0 = time.perf_counter()
    for L, xt in jobs:
        M.layer_forward(L, xt)
    return (time.perf_counter() - t0) / len(jobs)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                v = line.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    return v
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_worker(path, barrier, queue):
    """One host core: load the sample, wait for every worker, time the
    oracle's whole layer over the sample."""
    import torch

    from oracle import moe as M
    jobs = torch.load(path, weights_only=False)
    barrier.wait()
    t0 = time.perf_counter()
    for L, xt in jobs:
        M.layer_forward(L, xt)
    queue.put((t0, time.perf_counter(), len(jobs)))


def time_oracle_all_cores(jobs, n_workers: int):
    """Whole-host throughput of the oracle: n_workers processes (spawned, one
    numpy thread each) each run every job of `jobs`; returns seconds per
    layer-token over all of them (wall time from the first start to the last
    finish, divided by the layer-tokens done)."""
    import multiprocessing as mp

    import torch
    path = os.path.join("/tmp", f"si_oracle_jobs_{os.getpid()}.pt")
    torch.save(jobs, path)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n_workers)
    queue = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(path, barrier, queue)) for _ in range(n_workers)]
    for pr in procs:
        pr.start()
    res = []
    try:
        while len(res) < n_workers:
            try:
                res.append(queue.get(timeout=5))
            except Exception:
                if any(pr.exitcode not in (None, 0) for pr in procs):
                    raise RuntimeError("an oracle worker failed")
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.is_alive():
                pr.kill()
        os.remove(path)
    t0 = min(r[0] for r in res)
    t1 = max(r[1] for r in res)
    return (t1 - t0) / sum(r[2] for r in res)


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    per_lt = []
    n_each = 6
    jobs = oracle_jobs(n_each)
    for _ in range(max(1, args.warmup)):
        time_oracle(jobs[:1])
    t_all = time.perf_counter()
    for _ in range(args.steps):
        per_lt.append(time_oracle(jobs) * 1e6)
    ms_step = (time.perf_counter() - t_all) / args.steps * 1e3
    v = statistics.median(per_lt)
    sample = (f"{n_each} layer-tokens per step (layer l, token t of the 40-layer stack), oracle "
              f"layer_forward in fp64, weights of the selected experts materialised beforehand")
    line = {"metric": METRIC, "value": round(v, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 2),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "layers": N_LAYERS, "tokens": N_TOKENS},
            "cpu_baseline": {"value": round(v, 2), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    m.build()
    lib = m.library()
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    layers = [m.device_layer(spec, SEED, l, device=dev) for l in range(N_LAYERS)]
    x_in = gen.make_tokens(SEED + rank, N_TOKENS, device=dev)
    graph = m.StackGraph(layers, x_in)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()

    def barrier():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    # --- device-resident throughput ----------------------------------------
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.launch(stream)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.launch(stream)
            e1.record(stream)
        barrier()
    ms = e0.elapsed_time(e1)
    status = m.si_workspace_status(graph.ws, stream)
    ids_ok = bool((graph.ids >= 0).all().item() and (graph.ids < 256).all().item())
    ms = job_max(ms, pg)
    ms_step = ms / args.steps
    value_job = job_us_per_layer_token(ms_step, world)
    peak, peak_kind = _peaks()
    gbs_stage = BYTES_LAYER_TOKEN / (ms_step * 1e3 / (N_LAYERS * N_TOKENS)) / 1e3

    # --- end to end through the C ABI with host buffers ------------------------
    h_in = x_in.cpu().pin_memory()
    h_out = torch.empty_like(graph.y, device="cpu").pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            graph.x_in.copy_(h_in, non_blocking=True)
            graph.launch(stream)
            h_out.copy_(graph.y, non_blocking=True)
    barrier()
    t_e2e = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.x_in.copy_(h_in, non_blocking=True)
            graph.launch(stream)
            h_out.copy_(graph.y, non_blocking=True)
    barrier()
    e2e_ms = (time.perf_counter() - t_e2e) * 1e3 / args.steps
    e2e_ms = job_max(e2e_ms, pg)
    e2e_value = job_us_per_layer_token(e2e_ms, world)

    # --- the same stack through four kernels per layer (context) --------------
    per_layer_us = None
    if graph.persistent and not args.no_per_layer_path:
        gl = m.StackGraph(layers, x_in, mode=m.SI_STACK_PER_LAYER)
        with torch.cuda.stream(stream):
            for _ in range(2):
                gl.launch(stream)
            e0.record(stream)
            for _ in range(3):
                gl.launch(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        per_layer_us = e0.elapsed_time(e1) * 1e3 / (3 * N_LAYERS * N_TOKENS)
        gl.close()
    traffic_lt = _traffic_record(STACK_KERNEL_SOURCES) if graph.persistent else None

    if rank != 0:
        return 0
    cpu_us, cpu_n, cpu_all_us, n_cores = None, 0, None, 0
    if world == 1 and not args.no_cpu_baseline:
        jobs = oracle_jobs(args.cpu_layer_tokens, device=dev)
        cpu_us, cpu_n = time_oracle(jobs) * 1e6, len(jobs)
        n_cores = os.cpu_count() or 1
        cpu_all_us = time_oracle_all_cores(jobs[:8], n_cores) * 1e6
    launches = args.steps * (1 if graph.persistent else N_LAYERS * N_TOKENS * 4)
    # The timed path is one persistent kernel launch per step (the dominant and
    # only kernel): algorithmic bytes per launch = weight bytes of all
    # 40 x 128 layer-tokens.
    lt_per_launch = N_LAYERS * N_TOKENS if graph.persistent else 1
    launch_us = ms_step * 1e3 / (1 if graph.persistent else N_LAYERS * N_TOKENS * 4)
    bytes_launch = BYTES_LAYER_TOKEN * lt_per_launch
    achieved = bytes_launch / (launch_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": round(value_job, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "layers": N_LAYERS, "tokens": N_TOKENS,
                   "hidden": 2048, "experts": 256, "top_k": 8, "inter": 512, "shared_inter": 512,
                   "expert_type": "q4_k", "shared_type": "q4_k", "router_type": "bf16",
                   "parallelism": f"replicas{world}",
                   "l2": "no flush: weights 18.2 GB resident, 679 MB read per token > 129 MB L2"},
        "weight_read": {"bytes_per_layer_token": BYTES_LAYER_TOKEN,
                        "gbs": round(gbs_stage, 1), "frac_of_peak": round(gbs_stage / peak, 4),
                        "peak_gbs": peak, "peak_kind": peak_kind},
        "roofline": {"kernel": ("stack_kernel (persistent: router + top-k, routed and shared "
                                "experts, residual + RMSNorm of all 40 layers x 128 tokens)"
                                if graph.persistent else "four kernels per layer"),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": (round(traffic_lt * lt_per_launch) if traffic_lt else None),
                     "bytes_per_launch": bytes_launch, "avg_launch_us": round(launch_us, 1),
                     "peak_kind": peak_kind},
        "e2e": {"value": round(e2e_value, 3), "unit": UNIT,
                "h2d_bytes_per_step": h_in.numel() * h_in.element_size(),
                "d2h_bytes_per_step": h_out.numel() * h_out.element_size()},
        "gpu_launches": launches,
        "per_layer_path": ({"value": round(per_layer_us, 3), "unit": UNIT,
                            "what": "same stack, four kernels per layer and token"}
                           if per_layer_us is not None else None),
        "clocks": clk.summary(),
        "device_status": m.status_string(status), "ids_valid": ids_ok,
    }
    if cpu_us is not None:
        line["cpu_baseline"] = {
            "value": round(cpu_all_us, 1), "unit": UNIT, "cores": n_cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": (f"whole host: {n_cores} processes (one numpy thread each) each run the same 8 "
                       "layer-tokens of the stack through the fp64 oracle layer; wall time over all "
                       "8 x processes layer-tokens"),
            "single_thread": {"value": round(cpu_us, 1), "unit": UNIT, "cores": 1,
                              "sample": f"{cpu_n} layer-tokens of the same stack, one thread"}}
    print(json.dumps(line), flush=True)
    graph.close()
    return 0


# ----------------------------------------------------------------------------
# --configs: one line per workload configuration (not the headline line)
# ----------------------------------------------------------------------------
BYTES_CFG1 = 256 * 2048 * 2 + 8 * 3 * 512 * 2048 * 2 + 3 * 512 * 2048 * 2 + 2048 * 2  # 57,675,776
Q80_MATRIX = 512 * 2048 // 32 * 34                                                   # 1,114,112
BYTES_CFG3_Q80 = BYTES_ROUTER + BYTES_ROUTED + 3 * Q80_MATRIX + BYTES_SIGMOID         # 18,550,784
Q5K_MATRIX = 512 * 2048 // 256 * 176                                                  # 720,896
BYTES_NATIVE = (BYTES_ROUTER + 8 * (2 * Q4K_MATRIX + Q5K_MATRIX) + 3 * Q80_MATRIX
                + BYTES_SIGMOID)                                                      # 19,599,360
Q4K_EXPERT_128E = 3 * (768 * 2048 // 256 * 144)                                       # 2,654,208


def _time_replays(fn, stream, warm=3, reps=10):
    """Device time per call of fn() (which enqueues on `stream`), by CUDA events.
    The device is synchronised first: inputs made on another stream (e.g. by the
    generator on the default stream) must be complete before the timed work."""
    import torch
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def run_configs(args):
    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    m.build()
    lib = m.library()
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(device=dev)
    out = []

    def emit(cfg, what, us, unit, nbytes=None, **extra):
        line = {"config": cfg, "what": what, "value": round(us, 3), "unit": unit}
        if nbytes is not None:
            gbs = nbytes / (us * 1e-6) / 1e9
            line.update({"bytes": nbytes, "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                         "peak_gbs": peak, "peak_kind": peak_kind})
        line.update(extra)
        out.append(line)
        print(json.dumps(line), flush=True)

    # configs 1 and 3: 8 distinct layers x 16 tokens per replay, so every
    # layer-token reads its weights from HBM (8 layers exceed the L2)
    NL, NT = 8, 16
    x = gen.make_tokens(SEED + 7, NT, device=dev)
    for cfg, spec, nbytes in (("1: bf16 layer", gen.BF16_LAYER, BYTES_CFG1),
                              ("3: Q4_K layer, Q8_0 shared", gen.Q4K_LAYER_SHARED_Q8_0, BYTES_CFG3_Q80),
                              ("3: Q4_K layer, Q4_K shared", gen.Q4K_LAYER_SHARED_Q4_K, BYTES_LAYER_TOKEN),
                              ("3n: shipped formats (Q5_K routed down, Q8_0 shared)",
                               gen.NATIVE_LAYER_Q5K_DOWN, BYTES_NATIVE)):
        layers = [m.device_layer(spec, SEED + 100, l, device=dev) for l in range(NL)]
        modes = [m.SI_STACK_AUTO]
        if spec in (gen.Q4K_LAYER_SHARED_Q4_K, gen.Q4K_LAYER_SHARED_Q8_0, gen.BF16_LAYER,
                    gen.NATIVE_LAYER_Q5K_DOWN):
            modes = [m.SI_STACK_PERSISTENT, m.SI_STACK_PER_LAYER]
        for mode in modes:
            g = m.StackGraph(layers, x, mode=mode)
            us = _time_replays(lambda: g.launch(stream), stream) / (NL * NT)
            st = m.si_workspace_status(g.ws, stream)
            emit(cfg, "one layer, one token (8 distinct layers x 16 tokens per graph)", us,
                 "us/layer/token", nbytes,
                 path="persistent kernel" if g.persistent else "four kernels per layer",
                 device_status=m.status_string(st))
            g.close()
        del layers
        torch.cuda.empty_cache()

    # load-time requant of one shipped layer to Q4_K: routed down Q5_K
    # (256 x 2048 rows of 512) and the Q8_0 shared expert
    spec = gen.NATIVE_LAYER_Q5K_DOWN
    Ln = gen.make_layer(spec, SEED + 400, 0, device=dev)
    E, H, I, Is = spec.n_experts, spec.hidden, spec.inter, spec.shared_inter
    jobs = [(Ln["down"].reshape(E * H, -1), "q5_k", E * H, I), (Ln["sh_gate"], "q8_0", Is, H),
            (Ln["sh_up"], "q8_0", Is, H), (Ln["sh_down"], "q8_0", H, Is)]
    outs = [torch.empty(r, c // 256 * 144, dtype=torch.uint8, device=dev) for _, _, r, c in jobs]

    def requant_all():
        for (src, fmt, r, c), o in zip(jobs, outs):
            m.si_requant_q4_k(src, fmt, r, c, out=o, stream=stream)

    us = _time_replays(requant_all, stream, warm=2, reps=5)
    moved = sum(src.numel() for src, _, _, _ in jobs) + sum(o.numel() for o in outs)
    emit("requant", "one shipped layer to Q4_K (Q5_K routed down + Q8_0 shared), load time",
         us, "us/layer", moved, note="bytes = source read + Q4_K written")
    del Ln, jobs, outs
    torch.cuda.empty_cache()

    # config 2: router + top-k on fp32 tie-stress inputs (E = 256 and 128), one
    # token per call, 64 calls per graph over 8 router matrices
    for E in (256, 128):
        mats = [gen.tie_stress_group(SEED, g, E, 8, device=dev) for g in range(8)]
        ws = m.workspace(m.router_workspace_bytes(E, 2048, 1), dev)
        ids = torch.empty(1, 8, dtype=torch.int32, device=dev)
        wts = torch.empty(1, 8, dtype=torch.float32, device=dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for W, X, _ in mats:
                for c in range(8):
                    st = lib.si_moe_router_topk(X[c].data_ptr(), m.SI_F32, W.data_ptr(), m.SI_F32, 2048,
                                                E, 8, 1, ids.data_ptr(), wts.data_ptr(), None,
                                                ws.data_ptr(), ws.numel(), stream.cuda_stream)
                    assert st == 0
        us = _time_replays(graph.replay, stream) / 64
        emit(f"2: router tie stress, E={E}", "fused router GEMV + top-8 + softmax, fp32, 1 token",
             us, "us/call", E * 2048 * 4,
             note="8 distinct router matrices (16 MB at E=256) rotate, L2-resident")
        del graph

    # config 5: 128 experts, I=768, no shared, Q4_K; batched FFN (gate/up + down
    # + combine) for T tokens with per-token routing; 8 distinct layers per graph
    spec = gen.Q4K_LAYER_128E
    layers = [m.device_layer(spec, SEED + 200, l, device=dev) for l in range(8)]
    for T in (1, 4, 16, 64):
        xs = gen.make_tokens(SEED + 300 + T, T, device=dev)
        routs = []
        for l in range(8):
            keys = gen.raw64([gen.stream_key(SEED + l, t, 901) for t in range(T)], 128)
            ids = torch.argsort(keys, dim=1)[:, :8].to(torch.int32).to(dev)
            w = torch.full((T, 8), 0.125, dtype=torch.float32, device=dev)
            routs.append((ids, w))
        U = sum(int(torch.unique(r[0]).numel()) for r in routs) / 8
        for mode, name in ((m.SI_FFN_INT8, "int8 dp4a GEMV"), (m.SI_FFN_TENSOR, "tcgen05 fp16 MMA")):
            if mode == m.SI_FFN_TENSOR and T < 16:
                continue
            wss = [m.workspace(m.ffn_batched_workspace_bytes(L, T), dev) for L in layers]
            outs = [torch.empty(T, 2048, dtype=torch.bfloat16, device=dev) for _ in layers]
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for L, (ids, w), ws, o in zip(layers, routs, wss, outs):
                    st = lib.si_moe_ffn_batched(L.ref, T, mode, xs.data_ptr(), ids.data_ptr(),
                                                w.data_ptr(), o.data_ptr(), ws.data_ptr(), ws.numel(),
                                                stream.cuda_stream)
                    assert st == 0
            us = _time_replays(graph.replay, stream) / 8
            st = max(m.si_workspace_status(ws, stream) for ws in wss)
            emit(f"5: 128 experts, I=768, T={T}", f"batched routed FFN, {name}", us, "us/layer",
                 round(U * Q4K_EXPERT_128E), distinct_experts=U, us_per_layer_token=round(us / T, 3),
                 device_status=m.status_string(st))
            del graph
    del layers
    torch.cuda.empty_cache()

    # config 5 as stated: the 48-layer stack of that layer, T tokens through
    # every layer together (router, grouped experts, norm), one graph
    NL5 = 48
    layers = [m.device_layer(spec, SEED + 600, l, device=dev) for l in range(NL5)]
    for T in (1, 4, 16, 64):
        xs = gen.make_tokens(SEED + 700 + T, T, device=dev)
        g = m.BatchedStackGraph(layers, xs)
        us = _time_replays(lambda: g.launch(stream), stream, warm=3, reps=10) / NL5
        st = m.si_workspace_status(g.ws, stream)
        U = sum(int(torch.unique(g.ids[l]).numel()) for l in range(NL5)) / NL5
        nbytes = round(U * Q4K_EXPERT_128E + 128 * 2048 * 2)
        emit(f"5: 48-layer stack, 128 experts, I=768, T={T}",
             "batched layer stack (router + grouped experts + norm per layer), one graph", us,
             "us/layer", nbytes, distinct_experts=U, us_per_layer_token=round(us / T, 3),
             note="bytes = distinct experts' Q4_K weights + bf16 router, per layer",
             path="persistent kernel" if g.persistent else "batched kernels (router, prep, gate/up, "
                                                           "down, combine, norm)",
             device_status=m.status_string(st))
        g.close()
    # decode of the same 48-layer stack one token at a time on the persistent
    # kernel (16 sequential tokens in one launch)
    xs = gen.make_tokens(SEED + 800, 16, device=dev)
    g = m.StackGraph(layers, xs, mode=m.SI_STACK_PERSISTENT)
    us = _time_replays(lambda: g.launch(stream), stream, warm=3, reps=10) / (NL5 * 16)
    st = m.si_workspace_status(g.ws, stream)
    emit("5: 48-layer stack, 128 experts, I=768, T=1 (sequential tokens)",
         "persistent kernel, one token at a time (16 tokens per launch)", us, "us/layer/token",
         round(8 * Q4K_EXPERT_128E + 128 * 2048 * 2), path="persistent kernel",
         device_status=m.status_string(st))
    g.close()
    return 0


def run_kernels(args):
    """Each kernel of the four-kernel layer on its own: 8 distinct Q4_K layers
    (Q4_K shared expert) x 16 tokens per graph, so every call reads its
    weights from HBM; one JSON line per kernel with its algorithmic bytes and
    fraction of the measured HBM peak. The down kernel is timed as gate/up +
    down minus gate/up."""
    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    m.build()
    lib = m.library()
    peak, peak_kind = _peaks()
    stream = torch.cuda.Stream(device=dev)
    NL, NT = 8, 16
    spec = gen.Q4K_LAYER_SHARED_Q4_K
    H, E, k = spec.hidden, spec.n_experts, spec.top_k
    layers = [m.device_layer(spec, SEED + 100, l, device=dev) for l in range(NL)]
    x = gen.make_tokens(SEED + 7, NT, device=dev)
    ids = torch.empty(NL, NT, k, dtype=torch.int32, device=dev)
    wts = torch.empty(NL, NT, k, dtype=torch.float32, device=dev)
    rws = m.workspace(m.router_workspace_bytes(E, H, 1), dev)
    fws = m.workspace(m.ffn_workspace_bytes(layers[0]), dev)
    routed = torch.empty(H, dtype=torch.bfloat16, device=dev)
    shared = torch.empty(H, dtype=torch.bfloat16, device=dev)
    s_out = torch.empty(H, dtype=torch.bfloat16, device=dev)
    y_out = torch.empty(H, dtype=torch.bfloat16, device=dev)
    q_out = torch.empty(H // 32 * 36, dtype=torch.uint8, device=dev)
    cs = stream.cuda_stream

    def router(L, l, t):
        return lib.si_moe_router_topk(x[t].data_ptr(), m.SI_BF16, L.t["w_router"].data_ptr(), m.SI_BF16,
                                      H, E, k, 1, ids[l, t].data_ptr(), wts[l, t].data_ptr(), None,
                                      rws.data_ptr(), rws.numel(), cs)

    def gateup(L, l, t):
        return lib.si_moe_ffn_gateup(L.ref, 1, x[t].data_ptr(), None, ids[l, t].data_ptr(),
                                     fws.data_ptr(), fws.numel(), cs)

    def ffn(L, l, t):
        return lib.si_moe_ffn_decode(L.ref, 1, x[t].data_ptr(), None, ids[l, t].data_ptr(),
                                     wts[l, t].data_ptr(), routed.data_ptr(), shared.data_ptr(),
                                     fws.data_ptr(), fws.numel(), cs)

    def norm(L, l, t):
        return lib.si_add_rmsnorm3(routed.data_ptr(), shared.data_ptr(), x[t].data_ptr(),
                                   L.t["w_norm"].data_ptr(), H, 1, spec.eps, s_out.data_ptr(),
                                   y_out.data_ptr(), None, cs)

    def quant(L, l, t):
        return lib.si_quantize_q8_1(x[t].data_ptr(), m.SI_BF16, H, q_out.data_ptr(), cs)

    def timed(fn):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for t in range(NT):
                for l, L in enumerate(layers):
                    assert fn(L, l, t) == 0
        us = _time_replays(graph.replay, stream) / (NL * NT)
        del graph
        return us

    def emit(kernel, row, us, nbytes, **extra):
        gbs = nbytes / (us * 1e-6) / 1e9
        line = {"kernel": kernel, "row": row, "value": round(us, 3), "unit": "us/call",
                "bytes": nbytes, "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                "peak_gbs": peak, "peak_kind": peak_kind}
        line.update(extra)
        print(json.dumps(line), flush=True)

    q4k = 512 * 2048 // 256 * 144
    b_router = E * H * 2 + H * 2
    b_gateup = (k + 1) * 2 * q4k
    b_down = (k + 1) * q4k + H * 2
    us_router = timed(router)   # also leaves the ids the experts below read
    emit("router_topk_kernel", "A1-A3", us_router, b_router, note="bf16 router, E=256, T=1")
    us_gu = timed(gateup)
    emit("gateup_q_kernel", "A4-A5, A7", us_gu, b_gateup,
         note="8 routed + shared 32-row units, Q4_K, x quantised to Q8_1 inside")
    us_ffn = timed(ffn)
    emit("gateup_q_kernel + down_q_kernel", "A4-A7", us_ffn, b_gateup + b_down)
    emit("down_q_kernel (by difference)", "A6-A7", us_ffn - us_gu, b_down,
         note="gate/up + down minus gate/up; includes the sigmoid-gate dot")
    emit("add_rmsnorm_kernel", "A8", timed(norm), 5 * H * 2, bound="latency")
    emit("quantize_q8_1_kernel", "A4", timed(quant), H * 2 + H // 32 * 36, bound="latency")
    # Q8_1 of a large vector: the same kernel HBM-bound
    n = 1 << 26
    big = gen.to_bf16(gen.normal([gen.stream_key(SEED, 77, n)], n, 0.0, 1.0, dev)[0])   # seeded
    qb = torch.empty(n // 32 * 36, dtype=torch.uint8, device=dev)

    def quant_big():
        assert lib.si_quantize_q8_1(big.data_ptr(), m.SI_BF16, n, qb.data_ptr(), cs) == 0

    us = _time_replays(quant_big, stream)
    emit("quantize_q8_1_kernel", "A4", us, n * 2 + n // 32 * 36, note=f"n = {n} bf16 values")
    st = max(m.si_workspace_status(w, stream) for w in (rws, fws))
    print(json.dumps({"device_status": m.status_string(st)}), flush=True)
    return 0 if st == m.SI_OK else 1


def run_phase_trace(args):
    """Where the time of one persistent-kernel iteration goes, from the
    profiling build (libsi_moe_trace.so, -DSI_TRACE): thread 0 of every block
    stamps %globaltimer at the start of the last iteration of a launch and at
    one selected phase. Every phase gets `launches` launches of the stack of
    `layers` Q4_K layers x `tokens` tokens; the table gives, per phase, the
    median over blocks of the time after the iteration start (mean over the
    launches), less the stall of one stamp (phase 14 sits right after the
    start stamp). Not a measurement of the product build."""
    import ctypes

    import numpy as np
    import torch

    import gen
    import moe_decode_ffn_gb300 as m
    from moe_decode_ffn_gb300 import _build

    m.LIB = _build.build(trace=True)
    lib = m.library()
    lib.si_trace_dump_stack.argtypes = [ctypes.c_void_p]
    lib.si_trace_stack_phase.argtypes = [ctypes.c_int]
    layers = [m.device_layer(gen.Q4K_LAYER_SHARED_Q4_K, args.seed, l) for l in range(args.layers)]
    x = gen.make_tokens(args.seed, args.tokens, device="cuda")
    g = m.StackGraph(layers, x)
    if not g.persistent:
        print("the persistent kernel does not take these layers")
        return 1
    lib.si_trace_stack_phase(-1)
    for _ in range(3):
        g.launch()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        g.launch()
    e1.record()
    torch.cuda.synchronize()
    lt = args.layers * args.tokens
    print(f"profiling build without stamps: {e0.elapsed_time(e1) * 1e3 / 5 / lt:.3f} us per layer-token")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    names = {1: "fold done (X3 in)", 2: "logits written (X1 out)", 3: "Q8_1 of y done",
             4: "logits in, sorted", 5: "ranked", 6: "copies issued, softmax", 7: "gate/up dots done",
             8: "h written (X2 out)", 9: "h gathered (X2 in)", 10: "down rows ready", 11: "down dots",
             12: "rows written (X3 out)", 13: "next fold done"}
    res = {}
    for ph in [14] + list(range(1, 14)):
        lib.si_trace_stack_phase(ph)
        rows = []
        for _ in range(args.launches):
            g.launch()
            torch.cuda.synchronize()
            buf = np.zeros(4 * 1024 * 16, dtype=np.uint64)
            lib.si_trace_dump_stack(buf.ctypes.data)
            t = buf.reshape(4, 1024, 16)[0, :sms, :].astype(np.float64)
            ok = (t[:, ph] > 0) & (t[:, 0] > 0)
            rows.append(np.where(ok, t[:, ph] - np.median(t[:, 0]), np.nan))
        res[ph] = np.stack(rows)
    st = m.si_workspace_status(g.ws)
    g.close()
    stall = np.nanmean(np.nanmedian(res[14], axis=1))
    print(f"stamp stall {stall / 1e3:.3f} us (subtracted)")
    for ph in range(1, 14):
        v = res[ph] - stall
        print(f"{ph:2d} {names[ph]:26s} {np.nanmean(np.nanmedian(v, 1)) / 1e3:7.3f} us")
    print(f"status={m.status_string(st)}")
    return 0 if st == m.SI_OK else 1


def run_profile_case(args):
    """A bounded run for profilers (ncu), not a measurement: seeded layers,
    n_tokens tokens through n_layers layers captured as one CUDA graph and
    replayed `launches` times (or the batched routed FFN of one 128-expert
    layer for `batched` tokens); exits non-zero if the device recorded an
    error, so a profiler only ever runs a command that has just exited 0."""
    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    m.build()
    if args.quant:
        n = args.quant
        x = gen.to_bf16(gen.normal([gen.stream_key(args.seed, 77, n)], n, 0.0, 1.0, "cuda")[0])
        q = torch.empty(n // 32 * 36, dtype=torch.uint8, device="cuda")
        for _ in range(args.launches):
            m.si_quantize_q8_1(x, out=q)
        torch.cuda.synchronize()
        print(f"quantize n={n} launches={args.launches}")
        return 0
    if args.batched and args.batched_stack:
        T = args.batched
        layers = [m.device_layer(gen.Q4K_LAYER_128E, args.seed, l) for l in range(args.layers)]
        x = gen.make_tokens(args.seed + 1, T, device="cuda")
        mode = m.SI_FFN_TENSOR if args.mode == "tensor" else m.SI_FFN_INT8
        g = m.BatchedStackGraph(layers, x, mode=mode)
        for _ in range(args.launches):
            g.launch()
        torch.cuda.synchronize()
        st = m.si_workspace_status(g.ws)
        print(f"batched stack layers={args.layers} T={T} mode={args.mode} launches={args.launches} "
              f"persistent={g.persistent} status={m.status_string(st)}")
        g.close()
        return 0 if st == m.SI_OK else 1
    if args.batched:
        T = args.batched
        L = m.device_layer(gen.Q4K_LAYER_128E, args.seed, 0)
        x = gen.make_tokens(args.seed + 1, T, device="cuda")
        keys = gen.raw64([gen.stream_key(args.seed, t, 901) for t in range(T)], 128)
        ids = torch.argsort(keys, dim=1)[:, :8].to(torch.int32).cuda()
        w = torch.full((T, 8), 0.125, dtype=torch.float32, device="cuda")
        mode = m.SI_FFN_TENSOR if args.mode == "tensor" else m.SI_FFN_INT8
        ws = m.workspace(m.ffn_batched_workspace_bytes(L, T))
        for _ in range(args.launches):
            m.si_moe_ffn_batched(L, x, ids, w, mode, ws=ws)
        torch.cuda.synchronize()
        st = m.si_workspace_status(ws)
        print(f"batched T={T} mode={args.mode} launches={args.launches} status={m.status_string(st)}")
        return 0 if st == m.SI_OK else 1
    spec = {"q4k": gen.Q4K_LAYER_SHARED_Q4_K, "q4k_q8_0": gen.Q4K_LAYER_SHARED_Q8_0,
            "bf16": gen.BF16_LAYER}[args.spec]
    layers = [m.device_layer(spec, args.seed, l) for l in range(args.layers)]
    x = gen.make_tokens(args.seed + 1, args.tokens, device="cuda")
    mode = m.SI_STACK_PER_LAYER if args.per_layer else m.SI_STACK_AUTO
    g = m.StackGraph(layers, x, mode=mode)
    for _ in range(args.launches):
        g.launch()
    torch.cuda.synchronize()
    st = m.si_workspace_status(g.ws)
    print(f"layers={args.layers} tokens={args.tokens} launches={args.launches} "
          f"persistent={g.persistent} status={m.status_string(st)}")
    g.close()
    return 0 if st == m.SI_OK else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-layer-tokens", type=int, default=120,
                    help="layer-tokens the CPU oracle baseline times (about 10 s on one core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-layer-path", action="store_true",
                    help="skip timing the four-kernels-per-layer path")
    ap.add_argument("--configs", action="store_true",
                    help="instead of the headline line, one line per workload configuration")
    ap.add_argument("--kernels", action="store_true",
                    help="instead of the headline line, one line per kernel of the four-kernel layer")
    pc = ap.add_argument_group("--profile-case", "a bounded run for profilers (not a measurement)")
    pc.add_argument("--profile-case", action="store_true")
    pc.add_argument("--phase-trace", action="store_true",
                    help="phase timings of the persistent kernel from the profiling build (uses --layers, "
                         "--tokens, --launches, --seed)")
    pc.add_argument("--layers", type=int, default=4)
    pc.add_argument("--tokens", type=int, default=8)
    pc.add_argument("--launches", type=int, default=3)
    pc.add_argument("--seed", type=int, default=21)
    pc.add_argument("--per-layer", action="store_true",
                    help="four kernels per layer instead of the persistent kernel")
    pc.add_argument("--spec", default="q4k", choices=["q4k", "q4k_q8_0", "bf16"])
    pc.add_argument("--batched", type=int, default=0, help="T: the batched FFN of T tokens instead")
    pc.add_argument("--batched-stack", action="store_true",
                    help="with --batched T: the batched layer stack (router, grouped experts, combine + "
                         "norm) of --layers 128-expert layers")
    pc.add_argument("--mode", default="tensor", choices=["tensor", "int8"])
    pc.add_argument("--quant", type=int, default=0, help="n: the Q8_1 quantiser on n bf16 values instead")
    args = ap.parse_args()
    if args.profile_case:
        return run_profile_case(args)
    if args.phase_trace:
        return run_phase_trace(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.configs:
        return run_configs(args)
    if args.kernels:
        return run_kernels(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
