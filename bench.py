"""Benchmark of the routed int4 MoE layer (tokens/s per layer and roofline).

python bench.py [--gpus N] [--steps K] [--warmup W] [--config prefill]
                [--workloads decode,latent,exact] [--impl reference]

One step = one full layer forward (router, dispatch, experts, combine, and the
latent projections on the latent workload) over one batch of seeded synthetic
tokens, through ``moe_layer_forward``.  The headline workload is prefill: 8192
tokens through the K2.5-shaped layer (H=7168, 384 experts, top-8, I=2048, int4
g32) with a Zipf(1.1) expert load.  The same JSON line carries, under
``workloads``, the decode (T=32), latent (T=2048, L=3584) and exact (act_bits 8,
T=1024) results, each timed the same way.  Every step reads gigabytes of
distinct expert weights, far more than L2, so no L2 flush is needed.

For N > 1 (torchrun) every rank runs an independent replica of the layer on its
own GPU (no data-path collective); value = total tokens / max-over-ranks time.

--impl reference times the fp64 CPU oracle on the host cores on bounded
samples of the same workload (the oracle is the reference of this build).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "MoE-layer tokens/s (int4 experts, top-8) & % of HBM / tensor-core roofline"
EXPERT_BYTES_PER_ROW_COL = 0.5 + 2.0 / 32  # int4 weight + bf16 scale per 32 columns
L2_BYTES = 129e6  # GB300 L2


def _env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def expert_bytes(w: wl.Workload) -> int:
    """Packed int4 + bf16 scale bytes of one expert (gate, up, down)."""
    D, I = w.D, w.I
    return int(3 * D * I * EXPERT_BYTES_PER_ROW_COL)


def _source_hash() -> str:
    h = hashlib.sha1()
    for name in ("ffn_stream.cu", "ffn_tc.cu", "ffn_tc2.cu", "ffn_tc_q8.cu", "ffn_tc.cuh",
                 "int4_f16.cuh"):
        with open(os.path.join(ROOT, "int4_routed_expert_fp32_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def _profiled_traffic(config: str):
    """DRAM bytes per expert-FFN call from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = _source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == config and parts[1] == src:
                return float(parts[2])
    return None


def visible_gpu_id(visible, local_rank: int, current: int) -> str:
    """The id nvidia-smi knows this rank's GPU by: its entry in
    CUDA_VISIBLE_DEVICES (an index or a UUID), else the current device."""
    if visible:
        ids = [v.strip() for v in visible.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(current)


def roofline(w: wl.Workload, ffn_ms: float, active: int, peaks: dict) -> dict:
    """The expert-FFN call against its binding roofline.

    Algorithmic bytes: the int4 weights and bf16 scales of every active expert
    once, plus the sorted activation rows read (fp16, or int8 with act_bits 8),
    h written and read (fp16), and y written (bf16).  Algorithmic flops:
    2 * rows * 3 * D * I.  The bound is the one their ratio selects against the
    ridge of the measured HBM and sustained bf16 peaks."""
    R = w.T * w.k
    act_bytes = R * w.D * (1 if w.act_bits == 8 else 2) + 2 * R * w.I * 2 + R * w.D * 2
    alg_bytes = active * expert_bytes(w) + act_bytes
    flops = 2.0 * R * 3 * w.D * w.I
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if flops / alg_bytes < ridge:
        achieved = alg_bytes / (ffn_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    else:
        achieved = flops / (ffn_ms / 1000.0) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    roof.update({"traffic": None,
                 "kernel": "expert FFN call (moe_expert_ffn_pairs_bounded, T rows per expert "
                           "at most: schedules; for prefill-shaped batches ffn_tc_pair_kernel "
                           "(CTA pairs, experts of >= 129 rows) and ffn_tc_kernel (the others; "
                           "64-row tiles for experts of <= 64 rows), or ffn_tc_q8_kernel "
                           "(act_bits 8), gate/up and down; for decode-shaped ones "
                           "ffn_stream_fused_kernel)",
                 "kernel_ms": ffn_ms,
                 "algorithmic_bytes": alg_bytes, "algorithmic_flops": flops,
                 "active_experts": active, "peak_source": peaks["source"]})
    return roof


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = str(gpu_id)  # an index or a GPU UUID, as nvidia-smi --id takes
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.6)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [s.strip() for s in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _setup(w: wl.Workload, device):
    import int4_routed_expert_fp32_gb300 as moe
    x = wl.gen_x(w)
    W, b = wl.gen_router(w)
    lat = wl.gen_latent(w)
    weights = {"router_w": W.to(device), "router_bias": b.to(device), **wl.gen_experts(w, device)}
    if lat is not None:
        weights.update({k: v.to(device) for k, v in lat.items()})
    layer = moe.MoeLayer(w.T, w.H, w.E, w.k, w.I, weights, L=w.L, act_bits=w.act_bits,
                         renorm=w.renorm, eps=w.eps)
    return moe, x, layer, weights


def _ffn_pass(moe, w, layer, weights, x_dev, steps):
    """Average duration of the expert-FFN call (moe_expert_ffn_pairs_bounded with
    the layer's bound of T rows per expert: schedules, stream and tensor-core
    kernels) inside a layer step, timed with CUDA events
    on its stream; the step is the work of moe_layer_forward, issued stage by
    stage through the C ABI (on the latent path the layer keeps y in fp32; this
    replay writes bf16 y)."""
    lib = moe.lib
    dev = x_dev.device
    T, k, E, D, I = w.T, w.k, w.E, w.D, w.I
    R = T * k
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    rt, rs, inv = (torch.empty(R, dtype=torch.int32, device=dev) for _ in range(3))
    xs = torch.empty(R, D, dtype=torch.float16 if w.act_bits == 16 else torch.int8, device=dev)
    xsc = torch.empty(R, dtype=torch.float32, device=dev) if w.act_bits == 8 else None
    y = torch.empty(R, D, dtype=torch.bfloat16, device=dev)
    out = torch.empty(T, D, dtype=torch.bfloat16, device=dev)
    u = x_dev
    if w.L:
        u = moe.linear_bf16(x_dev, weights["lat_down"])
    ws_n = max(lib.moe_route_workspace_size(T, w.H, E), lib.moe_dispatch_workspace_size(T, E, k),
               lib.moe_expert_ffn_pairs_workspace_size(E, D, I, R, w.act_bits))
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]

    def step(i=None):
        assert lib.moe_route(p(x_dev), p(weights["router_w"]), p(weights["router_bias"]), T, w.H, E,
                             k, int(w.renorm), p(idx), p(tw), p(ws), ws.numel(), s) == 0
        assert lib.moe_dispatch_pairs(p(idx), p(u), T, D, E, k, w.act_bits, p(counts), p(offsets),
                                      p(rt), p(rs), p(inv), p(xs), p(xsc), p(ws), ws.numel(),
                                      s) == 0
        if i is not None:
            ev[i][0].record()
        # at most T rows per expert, as the layer call knows
        assert lib.moe_expert_ffn_pairs_bounded(p(xs), p(xsc), p(offsets), E, D, I, R, T,
                                                p(weights["gate_packed"]), p(weights["gate_scale"]),
                                                p(weights["up_packed"]), p(weights["up_scale"]),
                                                p(weights["down_packed"]), p(weights["down_scale"]),
                                                w.act_bits, p(y), p(ws), ws.numel(), s) == 0
        if i is not None:
            ev[i][1].record()
        assert lib.moe_combine(p(y), p(inv), p(tw), T, D, k, p(out), s) == 0

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    return statistics.mean(ms), counts.cpu().numpy()


class OracleSampler:
    """The fp64 oracle on the host cores over a fixed token order of the
    workload, one (token, expert slot) pair at a time: the token's routing and
    expert input when its first slot comes up, one expert's gated MLP per slot,
    the latent output after the last slot.

    The expert weights of the pairs about to be timed are generated before the
    clock starts (``prepare``), so the timed region holds oracle arithmetic
    only."""

    def __init__(self, w: wl.Workload):
        import oracle
        from oracle import inputs as oi
        self.O, self.oi, self.w = oracle, oi, w
        x = wl.gen_x(w)
        W, b = wl.gen_router(w)
        lat = wl.gen_latent(w)
        self.params = oi.layer_params(w, router=(W, b), latent=lat)
        self.xf = oi.x_f64(x)
        self.order = np.random.default_rng(0).permutation(w.T)
        self.pair = 0
        self.cur = None
        self.experts = {}

    def _token(self, pair):
        return int(self.order[(pair // self.w.k) % self.w.T])

    def prepare(self, n: int):
        """Generate (untimed) the expert arrays the next n pairs use; keeps
        only those."""
        O, w, p = self.O, self.w, self.params
        need = set()
        for t in sorted({self._token(i) for i in range(self.pair, self.pair + n)}):
            need.update(int(e) for e in O.route(self.xf[t:t + 1], p.w_router, p.bias, w.k,
                                                p.renorm).idx[0])
        self.experts = {e: self.experts[e] if e in self.experts else self.oi.expert_arrays(w, e)
                        for e in need}

    def _one_pair(self):
        O, w, p = self.O, self.w, self.params
        j = self.pair % w.k
        t = self._token(self.pair)
        if j == 0 or self.cur is None:
            xt = self.xf[t:t + 1]
            rt = O.route(xt, p.w_router, p.bias, w.k, p.renorm)
            self.cur = (rt, O.expert_input(xt, p), None)
        rt, u, acc = self.cur
        y = rt.weight[0, j] * O.expert_ffn(u, self.experts[int(rt.idx[0, j])], p.act_bits)
        acc = y if acc is None else acc + y
        if j == w.k - 1:
            O.latent_out(acc, p)
        self.cur = (rt, u, acc)
        self.pair += 1

    def run(self, n: int) -> float:
        """Time exactly n prepared pairs; returns seconds."""
        t0 = time.perf_counter()
        for _ in range(n):
            self._one_pair()
        return time.perf_counter() - t0

    def pairs_for(self, budget_s: float) -> int:
        """Pairs that take about budget_s (from one untimed calibration pair)."""
        self.prepare(1)
        dt = self.run(1)
        return max(1, int(budget_s / max(dt, 1e-9)))

    def describe(self, n: int, dt: float) -> str:
        return (f"{n} (token, expert) pairs = {n / self.w.k:.2f} of {self.w.T} tokens of the "
                f"{self.w.name} workload, fp64 oracle per pair (routing, gated MLP, weighted sum; "
                f"expert weights generated before timing), {dt:.1f} s")


def _cores() -> int:
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def _cpu_baseline(w: wl.Workload, budget_s: float = 20.0):
    """A bounded sample of the workload on the oracle (see OracleSampler)."""
    sampler = OracleSampler(w)
    n = sampler.pairs_for(budget_s)
    sampler.prepare(n)
    dt = sampler.run(n)
    return {"value": n / w.k / dt, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": sampler.describe(n, dt)}


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of the ranks' values (a replicated job takes as long as its
    slowest rank); the value itself with one rank (dist None)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job throughput: every rank processes its own tokens_per_rank
    tokens per step, in ms (the max over ranks)."""
    return world * tokens_per_rank / (ms / 1000.0)


def run_reference(args):
    """The oracle as the reference arm.  One step = one bounded sample of n
    (token, expert) pairs of the workload, n chosen so that all warm-up and
    timed steps take about a minute; ms_per_step is the measured duration of
    those n pairs, and value = n / k tokens per second over the timed steps."""
    rank, world, _ = _env_rank()
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.config]
    sampler = OracleSampler(w)
    n = sampler.pairs_for(60.0 / max(1, args.warmup + args.steps))
    times = []
    for i in range(args.warmup + args.steps):
        sampler.prepare(n)
        dt = sampler.run(n)
        if i >= args.warmup:
            times.append(dt)
    step_s = statistics.mean(times)
    value = n / w.k / step_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * step_s, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "sampled": True,
        "step": f"{n} (token, expert) pairs of the {w.name} workload ({n / w.k:.3f} tokens)",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "I": w.I,
                   "L": w.L, "act_bits": w.act_bits},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
                         "sample": sampler.describe(n * args.steps, sum(times))},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def _measure(args, w, device, dist, world, local):
    """Time one workload on this rank: the layer steps (value, ms_per_step,
    clocks, launches), the expert-FFN call (roofline) and the host-buffer
    path (e2e).  Returns the fields of its JSON entry."""
    import gc
    moe, x, layer, weights = _setup(w, device)
    x_dev = x.to(device)
    out = torch.empty_like(x_dev)

    # the layer call, launched as one captured CUDA graph (moe_layer_graph_*)
    # or kernel by kernel on the stream (--launch stream)
    graph = layer.graph(x_dev, out) if args.launch == "graph" else None
    run = graph.launch if graph else (lambda: layer.forward(x_dev, out))
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    rc = moe.check_error()
    if rc != 0:
        raise RuntimeError(f"{w.name}: device status after warm-up: {moe.status_string(rc)}")

    sampler = ClockSampler(visible_gpu_id(os.environ.get("CUDA_VISIBLE_DEVICES"), local,
                                          torch.cuda.current_device()))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = moe.launch_count()
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    launches = moe.launch_count() - n0
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, device)
    rc = moe.check_error()
    if rc != 0:
        raise RuntimeError(f"{w.name}: device status after timing: {moe.status_string(rc)}")

    # dominant kernel: the expert FFN call
    ffn_ms, counts = _ffn_pass(moe, w, layer, weights, x_dev, min(args.steps, 100))
    roof = roofline(w, ffn_ms, int((counts > 0).sum()), _peaks())
    roof["traffic"] = _profiled_traffic(w.name)

    # end to end through the C ABI with host buffers (pinned), copies inside
    e2e = None
    if not args.no_e2e:
        e2e = _e2e_pass(layer, x, w, world, dist, device, min(args.steps, 100), args.launch)
    cfg = _config(w, world, roof)
    cfg["launch"] = ("one CUDA graph of moe_layer_forward per step (moe_layer_graph_launch)"
                     if graph else "moe_layer_forward, kernels launched on the stream")
    res = {"value": job_tokens_per_s(world, w.T, ms), "ms_per_step": ms, "roofline": roof,
           "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "config": cfg}
    if graph:
        graph.close()
    del layer, weights, x_dev, out, graph, run
    gc.collect()
    torch.cuda.empty_cache()
    return res


def _config(w: wl.Workload, world: int, roof: dict) -> dict:
    wbytes = roof["active_experts"] * expert_bytes(w)
    l2 = (f"no flush: {wbytes / 1e9:.2f} GB of expert weights read per step exceed the "
          f"{L2_BYTES / 1e6:.0f} MB L2" if wbytes > L2_BYTES else
          f"WARNING: {wbytes / 1e6:.0f} MB of expert weights fit in L2 (not flushed)")
    return {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "k": w.k, "I": w.I, "L": w.L,
            "act_bits": w.act_bits, "weights": "int4 g32 bf16 scales", "l2": l2,
            "parallelism": f"replicas x{world}"}


def _parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="prefill", choices=list(wl.WORKLOADS),
                    help="headline workload of the JSON line")
    ap.add_argument("--workloads", default="decode,latent,exact",
                    help="further workloads reported under 'workloads' (comma list, or 'none')")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--launch", default="graph", choices=["graph", "stream"],
                    help="layer calls as one captured CUDA graph each, or kernel by kernel")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling case: replace the workload's expert count (routing uncalibrated)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling case: replace the workload's token count")
    return ap


def main(argv=None):
    ap = _parser()
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    extra = [] if args.workloads in ("", "none") else args.workloads.split(",")
    for name in extra:
        if name not in wl.WORKLOADS:
            ap.error(f"unknown workload {name}")
    extra = [n for n in extra if n != args.config]

    rank, world, local = _env_rank()
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    w = wl.WORKLOADS[args.config]
    if args.experts or args.tokens:
        w = wl.workload(args.config, name=f"{args.config}_small", E=args.experts or w.E,
                        T=args.tokens or w.T)
        extra = []
    from int4_routed_expert_fp32_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if dist:
        dist.barrier()

    head = _measure(args, w, device, dist, world, local)
    others = {name: _measure(args, wl.WORKLOADS[name], device, dist, world, local)
              for name in extra}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = _cpu_baseline(w)
    if rank == 0:
        _report(args, world, head, others, cpu)
    if dist:
        dist.destroy_process_group()
    return 0


def _e2e_pass(layer, x, w, world, dist, device, e_steps, launch="stream"):
    """Every step copies its pinned host input in, runs the layer and copies
    its output out.  --launch graph: through a layer pipe (moe_layer_pipe_*,
    the layer captured as a graph per device slot; a step's copies overlap
    the neighbouring steps' compute); --launch stream: moe_layer_forward_host,
    copies and layer in order on one stream."""
    xh = x.pin_memory()
    oh = torch.empty_like(x).pin_memory()
    pipe = layer.pipe() if launch == "graph" else None
    run = (lambda: pipe.submit(xh, oh)) if pipe else (lambda: layer.forward_host(xh, oh))
    for _ in range(3):
        run()
    if pipe:
        pipe.join()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(e_steps):
        run()
    if pipe:
        pipe.join()  # the last step's output copy is inside the timed region
    e1.record()
    torch.cuda.synchronize()
    wall = (time.perf_counter() - t0) / e_steps
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dist, device)
    if pipe:
        pipe.close()
    return {"value": job_tokens_per_s(world, w.T, e2e_ms), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x.numel() * 2), "d2h_bytes_per_step": int(x.numel() * 2),
            "host_wall_ms_per_step": wall * 1000.0,
            "api": ("moe_layer_pipe_submit per step (its copies overlap the neighbouring steps' "
                    "compute), moe_layer_pipe_join after the last" if launch == "graph"
                    else "moe_layer_forward_host per step")}


def _report(args, world, head, others, cpu):
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16", "data": "synthetic",
        "config": head["config"],
        "roofline": head["roofline"],
        "cpu_baseline": cpu,
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "workloads": {name: {**r, "unit": "tokens/s", "steps": args.steps, "warmup": args.warmup}
                      for name, r in others.items()},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    sys.exit(main())
