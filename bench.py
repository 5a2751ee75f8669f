"""Benchmark of the GB300 Q2_K MoE-FFN layer (one JSON line on stdout).

Default workload: the Qwen3.6-35B-A3B-shaped decode layer at batch 1 (hidden
2048, 256 routed experts, top-8, expert ffn 512, bf16 shared expert ffn 512,
bf16 x), four distinct layer copies cycled, 64-token x pool.  A step is one
call of the whole layer (router, top-k, grouping, routed gate/up + SwiGLU,
down + combine, gated shared expert) on the step's tokens.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--tokens T]
                  [--impl ours|reference] [--l2 cycle|flush] [--format q2k|q4k] [--steer S]

--format q4k runs the layer with Q4_K routed experts (qs_moe_ffn_q4k); --steer S adds the
directional steering of every output row (qs_steer_rows) to each step and reports the
steering kernel alone beside the line.

Timing: W untimed warm-up steps, then K steps.  Inputs are resident in HBM.
Default (--l2 cycle): inputs larger than L2 -- enough distinct layer copies are
cycled that every weight byte a step reads was last touched more than three
L2 capacities of traffic earlier, so it comes from HBM; steps run back to back
(a sleep kernel queued first lets the host enqueue ahead of the GPU) and one
pair of CUDA events brackets all K of them (an event recorded between two
launches lengthens the gap between them, so per-step events would time
themselves too).  --l2 flush: 4 copies, and between timed steps the L2 is
flushed (512 MiB write + 256 MiB read) outside the step's own events; this
also evicts the kernel's own code, so it is the pessimistic figure; it is
reported beside the default as `l2_flush`, with the 10th, 50th and 90th percentile
of its per-step times.  `graph`: the same K steps captured in one CUDA graph and
replayed once inside one event pair.  Time is max over ranks.  `e2e`
times the same K calls through the public API with each step's x copied in
from pinned host memory and y copied back, all inside one event pair.

Weights are drawn N(0, 0.02) on the device with torch's seeded generator
(expert weights then quantised by the library's Q2_K encoder, shared weights
rounded to bf16); x, the Zipf router bias and the steering direction come from the
shared seeded generators (qs_inputs).
`--impl reference` times the oracle (plain C, double precision) on the host
cores on the same workload: that is this layer's reference implementation.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import qs_inputs as qi  # noqa: E402

L2_FLUSH_WRITE = 512 << 20
L2_FLUSH_READ = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_35b_a3b", choices=sorted(qi.WORKLOADS))
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--l2", default="cycle", choices=["cycle", "flush"])
    ap.add_argument("--max-copies", type=int, default=48)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--format", default="q2k", choices=["q2k", "q4k"],
                    help="routed expert format: Q2_K (the workloads' format) or Q4_K")
    ap.add_argument("--steer", type=float, default=0.0,
                    help="directional steering of every output row with this scale (0: off)")
    return ap.parse_args()


KERNEL_SOURCES = ("bit_quantized_moe_router_gb300/csrc/qs_fused.cu", "bit_quantized_moe_router_gb300/csrc/qs_q2k.cuh",
                  "bit_quantized_moe_router_gb300/csrc/qs_common.cuh", "bit_quantized_moe_router_gb300/csrc/qs_fmt.cuh",
                  "bit_quantized_moe_router_gb300/csrc/qs_warp.cuh")


def recorded_traffic(workload):
    """DRAM bytes per launch of the persistent kernel from the committed ncu summary, or None
    when there is none for this workload or the kernel sources changed since it was taken."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", f"fused_decode_kernel_{workload}.md")
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for s in KERNEL_SOURCES:
            h.update(open(os.path.join(ROOT, s), "rb").read())
        m_t = re.search(r"traffic_bytes_per_launch: (\d+)", text)
        m_h = re.search(r"kernel_sources_sha256_16: ([0-9a-f]+)", text)
        if m_t and m_h and m_h.group(1) == h.hexdigest()[:16]:
            return int(m_t.group(1))
    except OSError:
        pass
    return None


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# ------------------------------------------------------------------ distributed plumbing

class Dist:
    """One process per GPU under torchrun (NCCL); `backend="gloo"` runs the same host logic on CPU."""

    def __init__(self, n_gpus, backend="nccl"):
        import torch
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.device = "cuda" if backend == "nccl" else "cpu"
        if self.world > 1:
            import torch.distributed as dist
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist
        elif n_gpus > 1:
            raise SystemExit("--gpus > 1 needs torchrun (one process per GPU)")

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v):
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=self.device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())


def aggregate_throughput(tokens_per_rank_step, steps, world, slowest_seconds):
    """Whole-job tokens/s of independent replicas: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank_step * steps * world / slowest_seconds


def graph_result(dist, local_seconds, local_error, tokens_per_rank_step, steps):
    """The graph-replay figure: every rank takes part in the max over ranks, whatever happened on
    it (a rank whose capture failed passes +inf), and the figure stands only if every rank's
    capture worked."""
    import math
    slowest = dist.max(local_seconds if local_error is None else float("inf"))
    if local_error is not None or not math.isfinite(slowest):
        return {"error": local_error or "graph capture failed on another rank"}
    return {"us_per_layer": slowest / steps * 1e6,
            "value": aggregate_throughput(tokens_per_rank_step, steps, dist.world, slowest),
            "note": "the K timed steps captured in one CUDA graph, one replay timed (launches from the "
                    "graph instead of the host; same layer copies and x rows)"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ the oracle on host cores

def expert_bytes(sh, fmt="q2k"):
    """Bytes of one routed expert (gate, up, down) in Q2_K (84 B) or Q4_K (144 B) blocks of 256 weights."""
    return (144 if fmt == "q4k" else 84) * 3 * sh.expert_ffn * sh.hidden // 256


def oracle_sample_layer(w, T, n_tokens, copy=0, fmt="q2k"):
    """Host layer for the oracle: x pool tokens 0..n_tokens-1, experts those tokens route to."""
    import oracle
    import concurrent.futures as cf
    sh = w.shape
    xb, _ = qi.gen_x(sh, w.seed, n_tokens)
    Wr = qi.gen_router(sh, w.seed, copy)
    bias = qi.gen_bias(sh, w.seed, copy, w.zipf_bias)
    shared = qi.gen_shared(sh, w.seed, copy)
    ids, _, _, _ = oracle.route(xb, oracle.X_BF16 if sh.x_dtype == qi.BF16 else oracle.X_F32, Wr, bias, sh.top_k)
    eb = expert_bytes(sh, fmt)
    blob = np.zeros(sh.n_experts * eb, np.uint8)

    def one(e):
        blob[e * eb:(e + 1) * eb] = oracle.quantize_expert(*qi.gen_expert_f32(sh, w.seed, copy, int(e)), fmt=fmt)

    with cf.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        list(ex.map(one, np.unique(ids)))
    return xb, Wr, bias, shared, blob


def oracle_threads():
    """Host threads for the oracle on many-token calls: every core, at most 64."""
    return max(1, min(64, os.cpu_count() or 1))


def time_oracle(w, T, budget_s, max_calls=None, fmt="q2k", threads=1):
    """Run the oracle for ~budget_s seconds: layer calls of T tokens (at most 16) on one
    thread, or with threads > 1 calls of 2 tokens per thread, the tokens split over them."""
    import oracle
    T = min(T, ORACLE_TOKENS_MAX) if threads == 1 else 2 * threads
    n_pool = 16 if T == 1 else max(T, 16)
    xb, Wr, bias, shared, blob = oracle_sample_layer(w, T, n_pool, fmt=fmt)
    calls, tokens = 0, 0
    t0 = time.perf_counter()
    while True:
        t_start = (calls * T) % max(1, n_pool - T + 1)
        oracle.moe_ffn(w.shape, xb[t_start:t_start + T], Wr, bias, blob, expert_bytes(w.shape, fmt), shared, fmt=fmt,
                       threads=threads)
        calls += 1
        tokens += T
        el = time.perf_counter() - t0
        if el >= budget_s or (max_calls and calls >= max_calls):
            break
    return tokens / el, calls, el


def cpu_model():
    """The host CPU's model (or architecture) and its core count, for the baseline's sample text."""
    import platform
    model = platform.machine()
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return f"{model}, {os.cpu_count() or 1} host cores"


def run_reference(args, w, T):
    """The reference arm: the oracle on host cores, same metric, unit and config."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    T_full = T
    # decode batches: one thread, the call's own tokens; many tokens: calls of 2 tokens per
    # host thread, the tokens split over every core
    nth = oracle_threads() if T_full > ORACLE_TOKENS_MAX else 1
    T = 2 * nth if nth > 1 else min(T, ORACLE_TOKENS_MAX)
    n_pool = max(T, 16)
    xb, Wr, bias, shared, blob = oracle_sample_layer(w, T, n_pool, fmt=args.format)

    def step(i):
        t0 = (i * T) % max(1, n_pool - T + 1)
        oracle.moe_ffn(w.shape, xb[t0:t0 + T], Wr, bias, blob, expert_bytes(w.shape, args.format), shared,
                       fmt=args.format, threads=nth)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    val = T * args.steps / el
    line = {
        "impl": "reference", "metric": metric_name(T_full) + (" [Q4_K experts]" if args.format == "q4k" else ""),
        "value": val,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "us_per_layer": ms * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": config_of(w, T_full, args),
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": f"{args.steps} layer calls of {T} token(s) over a {n_pool}-token x pool, "
                                   f"experts those tokens route to"
                                   + (f", tokens split over {nth} threads" if nth > 1 else "")
                                   + (f" (the oracle's cost per token does not depend on the batch of {T_full})"
                                      if T_full > T else "") + f"; {cpu_model()}"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


ORACLE_TOKENS_MAX = 16  # the oracle works token by token; large batches are timed on 16-token calls


def metric_name(T):
    return ("MoE-FFN layer tokens/s (batch %d decode)" % T) if T <= 16 else \
        ("MoE-FFN layer tokens/s (prefill, %d tokens per call)" % T)


def layer_flops(sh, T):
    """Multiply-adds x2 the layer does per call: router, routed experts (3 matrices per slot), shared."""
    router = 2 * T * sh.n_experts * sh.hidden
    routed = 2 * T * sh.top_k * 3 * sh.expert_ffn * sh.hidden
    shared = 2 * T * (3 * sh.shared_ffn * sh.hidden + sh.hidden)
    return router + routed + shared


def config_of(w, T, args):
    s = w.shape
    return {"workload": w.name, "hidden": s.hidden, "n_experts": s.n_experts, "top_k": s.top_k,
            "expert_ffn": s.expert_ffn, "shared_ffn": s.shared_ffn, "n_tokens": T, "layer_copies": w.copies,
            "x_pool": qi.X_POOL, "zipf_bias": w.zipf_bias,
            "expert_format": "Q4_K (144 B / 256 weights)" if getattr(args, "format", "q2k") == "q4k"
            else "Q2_K (84 B / 256 weights)",
            "layer_copies_cycled": getattr(args, "copies_used", w.copies),
            "l2": ("inputs larger than L2: %d layer copies cycled, no flush" % getattr(args, "copies_used", w.copies))
                  if args.l2 == "cycle" else
                  "flushed between timed steps (512 MiB write + 256 MiB read, outside the events)",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU",
            **({"steer_scale": args.steer} if args.steer else {})}


# ------------------------------------------------------------------ our arm

def device_layers(w, qm, torch, device, copies, fmt="q2k"):
    """Layer copies resident in HBM, drawn on the device (experts quantised by the library's encoder)."""
    sh = w.shape
    H, E, k, F, S = sh.hidden, sh.n_experts, sh.top_k, sh.expert_ffn, sh.shared_ffn
    stride = expert_bytes(sh, fmt)
    gbytes = F * H // 256 * (144 if fmt == "q4k" else 84)
    quantize = qm.qs_q4k_quantize if fmt == "q4k" else qm.qs_q2k_quantize
    layers = []
    for c in range(copies):
        gen = torch.Generator(device=device)
        gen.manual_seed(qi.stream_of(w.seed, c))
        blob = torch.empty(E * stride, dtype=torch.uint8, device=device)
        chunk = max(1, min(E, (256 << 20) // (4 * F * H)))
        for e0 in range(0, E, chunk):
            n = min(chunk, E - e0)
            for rows, cols, off in ((F, H, 0), (F, H, gbytes), (H, F, 2 * gbytes)):
                wts = torch.randn((n, rows, cols), generator=gen, device=device, dtype=torch.float32) * 0.02
                for i in range(n):
                    base = blob.data_ptr() + (e0 + i) * stride + off
                    quantize(wts[i], base)
        Wr = torch.randn((E, H), generator=gen, device=device, dtype=torch.float32) * 0.02
        b = qi.gen_bias(sh, w.seed, c, w.zipf_bias)
        bias = None if b is None else torch.from_numpy(b).to(device)
        shd = {n_: (torch.randn(shp, generator=gen, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
               for n_, shp in (("gate", (S, H)), ("up", (S, H)), ("down", (H, S)), ("sig", (H,)))}
        make = qm.make_q4k_experts if fmt == "q4k" else qm.make_experts
        layers.append({"blob": blob, "experts": make(blob, stride), "Wr": Wr, "bias": bias, "sh": shd,
                       "shared": qm.make_shared(shd["gate"], shd["up"], shd["down"], shd["sig"])})
    torch.cuda.synchronize()
    return layers


def algorithmic_bytes(sh, T, distinct, fmt="q2k"):
    """Bytes the layer must move for one call: router, x, the distinct experts' Q2_K, shared, out."""
    router = sh.n_experts * sh.hidden * 4
    x = T * sh.hidden * (2 if sh.x_dtype == qi.BF16 else 4)
    experts = distinct * expert_bytes(sh, fmt)
    shared = (3 * sh.shared_ffn * sh.hidden + sh.hidden) * 2
    out = T * sh.hidden * 4
    return router + x + experts + shared + out, experts


def run_ours(args, w, T):
    import math
    import torch
    dist = Dist(args.gpus)
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    from bit_quantized_moe_router_gb300 import qs_moe as qm
    qm.load(build_if_missing=False)
    sh = w.shape
    H = sh.hidden
    shape = qm.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.expert_ffn, sh.shared_ffn, sh.x_dtype)
    launches_per_step = qm.qs_moe_ffn_launches(shape, T, True) if args.format == "q2k" else \
        qm.qs_moe_ffn_q4k_launches(shape, T, True)
    if launches_per_step < 1:
        raise SystemExit(f"qs_moe_ffn_launches failed ({launches_per_step})")
    layer_launches = launches_per_step
    if args.steer:
        launches_per_step += 1  # qs_steer_rows after the layer

    # copies: the workload's own count, or enough that nothing a step reads is still in L2
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    per_step_upper = algorithmic_bytes(sh, T, min(sh.n_experts, T * sh.top_k), args.format)[0]
    copies = w.copies
    if args.l2 == "cycle":
        copy_bytes = sh.n_experts * expert_bytes(sh, args.format) + (3 * sh.shared_ffn * H + H) * 2 + sh.n_experts * H * 4
        want = math.ceil(3 * l2 / max(per_step_upper, 1))
        budget = int(0.5 * torch.cuda.get_device_properties(device).total_memory / copy_bytes)
        copies = max(w.copies, min(want, args.max_copies, budget))
    args.copies_used = copies
    layers = device_layers(w, qm, torch, device, copies, args.format)

    # x pool: rows wrap so that rows [j, j+T) are contiguous for every j < X_POOL
    xb, _ = qi.gen_x(sh, w.seed, qi.X_POOL + (T if T > qi.X_POOL else 0))
    xwrap = xb if T > qi.X_POOL else np.concatenate([xb, xb[:T]], axis=0)
    xdev = torch.from_numpy(xwrap.view(np.int16) if xwrap.dtype == np.uint16 else xwrap).to(device)
    ws = qm.alloc_workspace(shape, T)
    out = torch.empty((T, H), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    def xs(i):
        j = (i * T) % qi.X_POOL
        return xdev[j:j + T]

    direction = torch.from_numpy(qi.gen_direction(H, w.seed)).to(device)

    def step(i, x=None, n_layers=None, stream_=None):
        Ld = layers[i % (n_layers or len(layers))]
        ffn = qm.qs_moe_ffn_q4k if args.format == "q4k" else qm.qs_moe_ffn
        st_ = stream if stream_ is None else stream_
        ffn(shape, xs(i) if x is None else x, Ld["Wr"], Ld["bias"], Ld["experts"], Ld["shared"], out, T, ws, st_)
        if args.steer:
            qm.qs_steer_rows(out, direction, args.steer, T, st_)

    # distinct experts per step (routing is a function of the copy and the x rows)
    ids = torch.empty((T, sh.top_k), dtype=torch.int32, device=device)
    pw = torch.empty((T, sh.top_k), dtype=torch.float32, device=device)
    period = math.lcm(len(layers), qi.X_POOL // math.gcd(T, qi.X_POOL))
    distinct = {}
    K = args.steps
    for i in sorted({(args.warmup + j) % period for j in range(K)}):
        Ld = layers[i % len(layers)]
        qm.qs_route_topk(shape, xs(i), Ld["Wr"], Ld["bias"], T, ids, pw, ws, stream)
        distinct[i] = len(torch.unique(ids).tolist())
    qm.qs_workspace_init(ws, stream)

    flush_w = torch.empty(L2_FLUSH_WRITE, dtype=torch.uint8, device=device)
    flush_r = torch.ones(L2_FLUSH_READ // 4, dtype=torch.float32, device=device)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def timed(mode, n_layers, record_clocks):
        """K steps; returns (ms of all K steps, wall seconds, clocks).  With inputs larger than L2
        ("cycle") one event pair brackets the K back-to-back steps: an event recorded between two
        launches lengthens the gap between them, so per-step pairs would time the events too.
        With L2 flushes each step has its own pair, so that the flush kernels stay outside."""
        for i in range(args.warmup):
            if mode == "flush":
                flush()
            step(i, n_layers=n_layers)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        dist.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler(dist.local if dist.world > 1 else torch.cuda.current_device()) if record_clocks else None
        if clocks:
            time.sleep(0.3)
        t_wall = time.perf_counter()
        torch.cuda.nvtx.range_push("timed")
        if mode == "cycle":
            torch.cuda._sleep(int(2e6 + 120000 * K))  # let the host enqueue ahead of the GPU
        if mode == "flush":
            for i in range(K):
                flush()
                evs[i][0].record(stream)
                step(args.warmup + i, n_layers=n_layers)
                evs[i][1].record(stream)
        else:
            evs[0][0].record(stream)
            for i in range(K):
                step(args.warmup + i, n_layers=n_layers)
            evs[0][1].record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        dist.barrier()
        clk = clocks.stop() if clocks else None
        if mode == "flush":
            per_step = [a.elapsed_time(b) for a, b in evs]
            return float(sum(per_step)), wall, clk, per_step
        return float(evs[0][0].elapsed_time(evs[0][1])), wall, clk, None

    total_ms, wall, clk, _ = timed(args.l2, None, True)
    total_s = dist.max(total_ms / 1e3)
    st = qm.qs_read_device_status(ws, stream)
    if st != qm.QS_OK:
        raise SystemExit(f"device status after the timed steps: {qm.status_string(st)}")
    flush_ms = flush_pct = None
    if args.l2 == "cycle":
        fl, _, _, per_step = timed("flush", w.copies, False)
        flush_ms = fl / K
        flush_pct = [float(np.percentile(per_step, q)) * 1e3 for q in (10, 50, 90)]

    # the same K steps captured in one CUDA graph and replayed (eager launches above); the
    # layer's launches keep their programmatic-dependency edges inside the graph
    g_local, g_err = float("inf"), None
    try:
        cap = torch.cuda.Stream(device=device)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for i in range(args.warmup):
                step(i, stream_=cap)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(K):
                step(args.warmup + i, stream_=cap)
        g.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        g.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        g_local = ga.elapsed_time(gb) / 1e3
        del g
    except RuntimeError as exc:   # capture refused (QsError is one too): report it, keep the eager figures
        torch.cuda.synchronize()
        g_err = str(exc).splitlines()[0][:200]
    graph = graph_result(dist, g_local, g_err, T, K)
    st = qm.qs_read_device_status(ws, stream)
    if st != qm.QS_OK:
        raise SystemExit(f"device status after the graph replay: {qm.status_string(st)}")

    # e2e through the public API: pinned host x in, y back out, inside the events.  The Q2_K
    # layer takes host buffers itself (qs_moe_ffn_host queues both copies around the layer);
    # the Q4_K layer and the steered layer copy with torch around their device-buffer calls.
    x_host = torch.from_numpy(xwrap.view(np.int16) if xwrap.dtype == np.uint16 else xwrap).pin_memory()
    y_host = torch.empty((T, H), dtype=torch.float32).pin_memory()
    x_stage = torch.empty_like(xdev[:T])
    host_api = args.format == "q2k" and not args.steer
    ws_host = qm.alloc_host_workspace(shape, T) if host_api else None

    def e2e_step(i):
        j = (i * T) % qi.X_POOL
        if host_api:
            Ld = layers[i % len(layers)]
            qm.qs_moe_ffn_host(shape, x_host[j:j + T], Ld["Wr"], Ld["bias"], Ld["experts"], Ld["shared"], y_host, T,
                               ws_host, stream)
        else:
            x_stage.copy_(x_host[j:j + T], non_blocking=True)
            step(i, x=x_stage)
            y_host.copy_(out, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e6 + 160000 * K))
    e2e_a, e2e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_a.record(stream)
    for i in range(K):
        e2e_step(args.warmup + i)
    e2e_b.record(stream)
    torch.cuda.synchronize()
    e2e_s = dist.max(e2e_a.elapsed_time(e2e_b) / 1e3)
    if ws_host is not None and qm.qs_read_device_status(ws_host, stream) != qm.QS_OK:
        raise SystemExit("device status after the e2e steps: " + qm.status_string(qm.qs_read_device_status(ws_host)))

    steer = None
    if args.steer:
        torch.cuda.synchronize()
        sa, sb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            qm.qs_steer_rows(out, direction, args.steer, T, stream)
        sa.record(stream)
        for _ in range(K):
            qm.qs_steer_rows(out, direction, args.steer, T, stream)
        sb.record(stream)
        torch.cuda.synchronize()
        s_us = sa.elapsed_time(sb) / K * 1e3
        s_bytes = 2 * T * H * 4 + H * 4
        steer = {"kernel": "steer_rows_kernel", "us_per_call": s_us, "bytes_per_call": s_bytes,
                 "achieved_gbs": s_bytes / (s_us * 1e-6) / 1e9,
                 "note": "qs_steer_rows alone, K back-to-back calls on the layer's output rows (L2-resident)"}

    # roofline of the layer kernel: algorithmic bytes over the measured step time
    algo = [algorithmic_bytes(sh, T, distinct[(args.warmup + j) % period], args.format) for j in range(K)]
    algo_bytes = float(np.mean([a for a, _ in algo])) + (H * 4 if args.steer else 0)
    q2k_bytes = float(np.mean([q for _, q in algo]))
    mean_step_s = total_s / K
    pk = peaks()
    hbm_peak = pk["hbm_gbs"] if pk else 6800.0
    achieved = algo_bytes / mean_step_s / 1e9
    tokens_total = T * K * dist.world
    value = aggregate_throughput(T, K, dist.world, total_s)
    if dist.rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and dist.world == 1:
        if T > ORACLE_TOKENS_MAX:   # many tokens per call: the tokens split over every host core
            nth = oracle_threads()
            rate, calls, el = time_oracle(w, T, args.cpu_seconds, fmt=args.format, threads=nth)
            r1, c1, e1 = time_oracle(w, T, args.cpu_seconds / 2, fmt=args.format)
            cpu = {"value": rate, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                   "sample": f"{calls} layer calls of {2 * nth} tokens split over {nth} threads ({el:.1f} s); "
                             f"one thread: {r1:.2f} tokens/s ({c1} calls of {ORACLE_TOKENS_MAX} tokens, {e1:.1f} s); "
                             f"the oracle's cost per token does not depend on the batch; {cpu_model()}"}
        else:
            rate, calls, el = time_oracle(w, T, args.cpu_seconds, fmt=args.format)
            cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                   "sample": f"{calls} layer calls of {T} token(s) ({el:.1f} s, one thread), x pool of 16 tokens "
                             f"and the experts they route to; {cpu_model()}"}
    if args.format == "q2k" and layer_launches > 1 and T > 16:  # tensor-core path: bound by the 16-bit tensor pipe
        flops = layer_flops(sh, T)
        tf_peak = pk["bf16_tflops"] if pk else 1900.0
        tf = flops / mean_step_s / 1e12
        roof = {"bound": "tensor", "kernel": "qs_moe_ffn (whole layer, %d kernels)" % layer_launches,
                "achieved": tf, "peak": tf_peak, "unit": "TFLOP/s", "frac": tf / tf_peak,
                "peak_source": ("MEASURED_PEAKS.json bf16_tflops, dense 16-bit burst (fp16 runs at the bf16 rate; "
                                "of measured)") if pk else "fallback 1.9 PFLOP/s",
                "algorithmic_flops_per_launch": flops, "traffic": None}
    else:
        roof = {"bound": "hbm",
                "kernel": ("fused_decode_kernel" + (" (Q4_K experts)" if args.format == "q4k" else "")
                           if layer_launches == 1 else
                           "qs_moe_ffn (whole layer)" if args.format == "q2k" else
                           "qs_moe_ffn_q4k (whole layer, %d kernels)" % layer_launches),
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else "fallback 6800 GB/s",
                "algorithmic_bytes_per_launch": algo_bytes,
                "traffic": recorded_traffic(w.name) if layer_launches == 1 and T == w.tokens[0] and not args.steer
                and args.format == "q2k" else None}
    line = {
        "metric": metric_name(T) + (" [Q4_K experts]" if args.format == "q4k" else ""),
        "value": value, "unit": "tokens/s", "n_gpus": dist.world, "steps": K, "warmup": args.warmup,
        "ms_per_step": mean_step_s * 1e3, "us_per_layer": mean_step_s * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (("q4k-int16dot-f32" if layer_launches == 1 else "q4k-f32") if args.format == "q4k" else
                  "q2k-int16dot-f32" if roof["bound"] == "hbm" else "q2k-dequant-f16-mma-f32"), "data": "synthetic",
        "config": config_of(w, T, args),
        "achieved_gbs_all_bytes": achieved, "achieved_gbs_q2k_bytes": q2k_bytes / mean_step_s / 1e9,
        "roofline": roof,
        "l2_flush": None if flush_ms is None else {
            "us_per_layer": flush_ms * 1e3, "frac": algo_bytes / (flush_ms / 1e3) / 1e9 / hbm_peak,
            "p10_us": flush_pct[0], "p50_us": flush_pct[1], "p90_us": flush_pct[2],
            "note": "%d layer copies, L2 flushed between steps outside the events (kernel code evicted too); "
                    "per-step events" % w.copies},
        "graph": graph,
        "e2e": {"value": tokens_total / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": int(x_stage.numel() * x_stage.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "api": "qs_moe_ffn_host (pinned host x and y)" if host_api else
                       "device-buffer call with torch copies of pinned host x and y around it"},
        "gpu_launches": launches_per_step * K,
        "kernels_per_step": launches_per_step,
        "clocks": clk,
        "bracket_wall_s": wall,
        "cpu_baseline": cpu,
        **({"steer": steer} if steer else {}),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    w = qi.WORKLOADS[args.workload]
    T = args.tokens or w.tokens[0]
    if args.impl == "reference":
        run_reference(args, w, T)
    else:
        run_ours(args, w, T)


if __name__ == "__main__":
    main()
