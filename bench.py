#!/usr/bin/env python
"""Benchmark of the quantized MoE expert layer on GB300.

One step = one full pass of the layer (router + top-k, counting sort + permute, FC1 with
fused dequant and activation, FC2, shared expert, un-permute/combine) over one batch of T
synthetic tokens; for a stacked config (Phi-shaped, 32 layers) one step runs every layer.

Default workload: the largest single-GPU configuration, the Phi-3.5-MoE-shaped layer (d=4096,
ffn=6400, E=16, top-2, SwiGLU, INT4 group-128, bf16 activations) at T = 8192 tokens, 32
stacked layers with distinct weights run back to back on one stream per step.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead, on a
bounded token sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from weight_only_int4_route_gb300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300; % of HBM (decode) / tensor (prefill) roofline"
L2_BYTES = 129 * 1024 * 1024
GRAPH_MAX_T = 32   # steps of at most this many tokens replay each layer's chain as a CUDA graph
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# A timed region at least this long runs under the sustained (power-capped) clocks; a shorter
# one is compared with the burst tensor peak.
SUSTAINED_REGION_S = 1.0


def tensor_peak(peaks: dict, region_s: float, src: str):
    """Dense 16-bit tensor peak that applies to a kernel timed inside a region of region_s seconds."""
    if region_s >= SUSTAINED_REGION_S and "bf16_tflops_sustained" in peaks:
        return peaks["bf16_tflops_sustained"], (f"{src} bf16 sustained (timed region {region_s:.2f} s >= "
                                                f"{SUSTAINED_REGION_S:.0f} s)")
    return peaks["bf16_tflops"], f"{src} bf16 burst (timed region {region_s:.2f} s < {SUSTAINED_REGION_S:.0f} s)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="phi", choices=sorted(synth.CONFIGS))
    ap.add_argument("--T", type=int, default=0, help="tokens per step (default: the config's largest)")
    ap.add_argument("--layers", type=int, default=0, help="stacked layers per step (default: the config's)")
    ap.add_argument("--cpu-sample", type=int, default=256, help="tokens in the oracle's timed sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="decode-sized steps: launch kernels one by one")
    ap.add_argument("--decode-chain", action="store_true",
                    help="decode-sized steps: always the chain of kernels")
    ap.add_argument("--decode-launch", action="store_true",
                    help="decode-sized steps: always the one-launch layer kernel (where the layer allows it)")
    ap.add_argument("--elb", action="store_true",
                    help="time ELB counting + top-M for one chunk boundary instead of the layer (separate metric)")
    ap.add_argument("--codec", action="store_true",
                    help="time the BF16 bit-field recombine kernel instead of the layer (separate metric)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """Largest value of x over all ranks (the step time that bounds the whole job)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, T: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own T tokens per step."""
    return world * T / (ms_per_step * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------- algorithmic work


def packed_bytes(K, N, bits, group):
    G = 1 if group == 0 else K // group
    return K * N * bits // 8 + G * N * 2


def work_model(cfg, T, counts):
    """Algorithmic bytes and FLOPs of one layer and of its two grouped GEMM launches.

    Weights are counted once per active expert (experts with no routed rows load none);
    FC1 reads Xp (R x d) and writes H (R x F) in 16-bit; FC2 reads H and writes fp32 Yp."""
    R = T * cfg.k
    act_e = sum(1 for c in counts if c > 0)
    w1 = packed_bytes(cfg.d, cfg.F1, cfg.bits, cfg.group)
    w2 = packed_bytes(cfg.F, cfg.d, cfg.bits, cfg.group)
    fc1 = dict(bytes=act_e * w1 + R * cfg.d * 2 + R * cfg.F * 2, flops=2 * R * cfg.d * cfg.F1)
    fc2 = dict(bytes=act_e * w2 + R * cfg.F * 2 + R * cfg.d * 4, flops=2 * R * cfg.F * cfg.d)
    sh_w = 3 * cfg.d * cfg.Fs * 2
    router_w = cfg.d * cfg.E * (4 if cfg.router_dtype == "f32" else 2)
    layer = dict(bytes=act_e * (w1 + w2) + sh_w + router_w + 2 * T * cfg.d * 2,
                 flops=2 * R * (cfg.d * cfg.F1 + cfg.F * cfg.d) + 2 * T * 3 * cfg.d * cfg.Fs + 2 * T * cfg.d * cfg.E)
    return dict(fc1=fc1, fc2=fc2, layer=layer, active_experts=act_e)


# ---------------------------------------------------------------- clocks


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        self.error = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.ferr = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=self.ferr)
        except Exception as e:   # no nvidia-smi: the line says so instead of carrying clocks
            self.proc = None
            self.error = f"nvidia-smi not started: {e}"

    def stop(self):
        if self.proc is None:
            return {"error": self.error} if self.error else None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        self.ferr.seek(0)
        err = self.ferr.read().strip()
        self.ferr.close()
        if not rows:
            return {"error": "nvidia-smi gave no samples" + (f": {err[:200]}" if err else "")}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- our arm


def run_ours(args, cfg, T, n_layers, world, rank, local):
    from weight_only_int4_route_gb300 import build as B
    from weight_only_int4_route_gb300 import moe as M

    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.decode_chain:
        M.set_decode_mode("chain")
    elif args.decode_launch:
        M.set_decode_mode("launch")
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ---- weights: distinct layers for a stack; else rotate copies so the step's weight
    # stream never fits in L2 (inputs larger than L2 between timed iterations)
    est_touch = None
    w0 = synth.layer_weights(cfg, 0, device=dev)
    packed = [M.PackedLayer.from_weights(cfg, w0, dev)]
    per_layer = sum(t.numel() for t in (packed[0].w1, packed[0].w2)) + sum(
        t.numel() * t.element_size() for t in (packed[0].ws_gu, packed[0].ws_d) if t is not None)
    del w0
    if n_layers > 1:
        copies = n_layers
    else:
        # bytes one step touches: active experts' weights + shared + activations
        R = T * cfg.k
        act_e = min(cfg.E, R)
        act_e = cfg.E * (1 - (1 - min(1.0, cfg.k / cfg.E)) ** T) if act_e < cfg.E else cfg.E
        est_touch = act_e * (packed_bytes(cfg.d, cfg.F1, cfg.bits, cfg.group) + packed_bytes(cfg.F, cfg.d, cfg.bits, cfg.group)) \
            + 3 * cfg.d * cfg.Fs * 2 + T * cfg.d * 2 * 4
        copies = max(2, math.ceil(3 * L2_BYTES / max(est_touch, 1)))
        copies = min(copies, 16)
    for i in range(1, copies):
        wi = synth.layer_weights(cfg, i, device=dev)
        packed.append(M.PackedLayer.from_weights(cfg, wi, dev))
        del wi
    nx = copies if n_layers == 1 else 1
    xs = [synth.normal(cfg, "x", (T, cfg.d), 1.0, cfg.torch_dtype, layer=i, extra=T, device=dev) for i in range(nx)]
    outs = [torch.empty((T, cfg.d), dtype=cfg.torch_dtype, device=dev) for _ in range(max(1, n_layers if n_layers > 1 else 1))]
    ws_bytes = M.Layer(packed[0], T).ws_bytes
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    layers = [M.Layer(p, T, workspace=ws) for p in packed]
    # decode-sized steps run each layer's chain as one CUDA graph (fixed buffers, input resident)
    use_graph = T <= GRAPH_MAX_T and not args.no_graph
    graphs = []
    if use_graph:
        for li, layer in enumerate(layers):
            g = M.LayerGraph(layer, T)
            g.x.copy_(xs[0] if n_layers > 1 else xs[li % nx])
            graphs.append(g)
    torch.cuda.synchronize()

    def step(i):
        if use_graph:
            if n_layers > 1:
                for g in graphs:
                    g.launch()
            else:
                graphs[i % copies].launch()
        elif n_layers > 1:
            for li, layer in enumerate(layers):
                layer.forward(xs[0], outs[li])
        else:
            j = i % copies
            layers[j].forward(xs[j % nx], outs[0])

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        step(args.warmup + i)
    t1.record()
    barrier()
    elapsed_ms = t0.elapsed_time(t1)

    # ---- per-stage durations inside the same workload (roofline of the dominant kernel)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in M.STAGES] for _ in range(len(layers))]
    for ring in evs:
        for e in ring:
            e.record()
    torch.cuda.synchronize()
    stage_ms = {s: 0.0 for s in M.STAGES[1:]}
    n_prof = 0
    for i in range(args.steps):
        if n_layers > 1:
            for li, layer in enumerate(layers):
                layer.forward_profiled(xs[0], outs[li], evs[li])
            torch.cuda.synchronize()
            for li in range(len(layers)):
                for a, b, s in zip(evs[li][:-1], evs[li][1:], M.STAGES[1:]):
                    stage_ms[s] += a.elapsed_time(b)
                n_prof += 1
        else:
            j = i % copies
            layers[j].forward_profiled(xs[j % nx], outs[0], evs[0])
            torch.cuda.synchronize()
            for a, b, s in zip(evs[0][:-1], evs[0][1:], M.STAGES[1:]):
                stage_ms[s] += a.elapsed_time(b)
            n_prof += 1
    stage_ms = {s: v / max(n_prof, 1) for s, v in stage_ms.items()}
    clk = clocks.stop()

    # ---- end to end through the public call with host buffers: every step copies its input
    # from pinned host memory and its output back, inside the timed region.  The copies run on
    # their own streams, double-buffered, so step i's download and step i+1's upload overlap the
    # neighbouring steps' compute, as a serving loop would run them.
    e2e = None
    if not args.no_e2e:
        nbuf = 2
        xh = [xs[0].cpu().pin_memory() for _ in range(nbuf)]
        oh = [torch.empty((T, cfg.d), dtype=cfg.torch_dtype).pin_memory() for _ in range(nbuf)]
        comp = torch.cuda.current_stream(dev)
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ksteps = max(3, min(args.steps, 50))
        if use_graph:   # graph j owns its input / output buffers; the step uses graph i % copies
            nslot = copies if n_layers == 1 else 1
            x_dev = [graphs[j].x for j in range(nslot)] if n_layers == 1 else [graphs[0].x]
            o_dev = [graphs[j].out for j in range(nslot)] if n_layers == 1 else [graphs[-1].out]
        else:
            nslot = nbuf
            x_dev = [torch.empty_like(xs[0]) for _ in range(nbuf)]
            o_dev = [torch.empty((T, cfg.d), dtype=cfg.torch_dtype, device=dev) for _ in range(nbuf)]
        read_done = [None] * nslot    # compute finished reading slot j's input
        dl_done = [None] * nslot      # download finished reading slot j's output

        def e2e_step(i):
            j = i % nslot
            with torch.cuda.stream(up):
                if read_done[j] is not None:
                    up.wait_event(read_done[j])
                x_dev[j].copy_(xh[i % nbuf], non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
            comp.wait_event(uploaded)
            if dl_done[j] is not None:
                comp.wait_event(dl_done[j])
            if use_graph:
                if n_layers > 1:
                    for g in graphs:
                        g.launch()
                else:
                    graphs[j].launch()
            elif n_layers > 1:
                for li, layer in enumerate(layers):
                    layer.forward(x_dev[j], outs[li] if li < n_layers - 1 else o_dev[j])
            else:
                layers[i % copies].forward(x_dev[j], o_dev[j])
            done = torch.cuda.Event()
            done.record(comp)
            read_done[j] = done
            with torch.cuda.stream(down):
                down.wait_event(done)
                oh[i % nbuf].copy_(o_dev[j], non_blocking=True)
                fin = torch.cuda.Event()
                fin.record(down)
                dl_done[j] = fin
            return fin

        for i in range(3):
            e2e_step(i)
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        up.wait_event(a)
        last = None
        for i in range(ksteps):
            last = e2e_step(i)
        comp.wait_event(last)
        b.record(comp)
        barrier()
        e2e_ms = a.elapsed_time(b) / ksteps
        e2e = dict(ms=e2e_ms, h2d=T * cfg.d * 2, d2h=T * cfg.d * 2)

    # routing counts of layer 0 for the algorithmic work
    layers[0].forward(xs[0], outs[0])
    torch.cuda.synchronize()
    offs = layers[0].routing(T)["offsets"].cpu().tolist()
    counts = [offs[i + 1] - offs[i] for i in range(cfg.E)]
    launches_per_layer = layers[0].launch_count(T)
    one_launch = launches_per_layer == 1
    # a kernel that gave up on a bounded wait leaves a code in the device error word: the run's
    # outputs and times are then not valid, so no number is reported
    derr = M.device_error(dev)
    if derr:
        raise SystemExit(f"bench: device error word {derr} set during the run (a bounded wait expired); "
                         "no result reported")
    kinds = {"tcgen05": "gemm_tc_kernel", "gemv": "gemv_kernel", "mma": "gemm_mma_kernel"}
    F1 = 2 * cfg.F if cfg.act == "swiglu" else cfg.F
    R = T * cfg.k
    kernels = {"fc1": kinds[M.gemm_path(R, cfg.E, cfg.d, F1, cfg.bits, cfg.group, cfg.act)],
               "fc2": kinds[M.gemm_path(R, cfg.E, cfg.F, cfg.d, cfg.bits, cfg.group, "none")]}

    ms = max_over_ranks(elapsed_ms / args.steps, dist, dev)
    if e2e is not None:
        e2e["ms"] = max_over_ranks(e2e["ms"], dist, dev)
    for g in graphs:
        g.close()
    return dict(ms=ms, stage_ms=stage_ms, counts=counts, clocks=clk, e2e=e2e, copies=copies,
                launch=("one kernel launch per layer" + (" (replayed from a CUDA graph)" if use_graph else "")
                        if one_launch else
                        "one CUDA graph per layer chain" if use_graph else "kernels launched one by one"),
                one_launch=one_launch,
                launches=launches_per_layer * n_layers * args.steps, per_layer_bytes=per_layer, kernels=kernels,
                est_touch=est_touch, dist=dist)


# DRAM bytes (read + write) per launch of a grouped GEMM, from one ncu capture of this bench's
# own command on the named workload (summaries are kept with the profiles); null elsewhere.
# An entry is valid only for the kernel version it was taken on: it is removed whenever that
# kernel changes.
MEASURED_TRAFFIC = {
    ("phi", 8192, "fc1"): 567_240_704 + 197_445_632,
    ("encdec_int4", 3840, "fc1"): 75_360_256 + 5_082_624,
    ("encdec_int4", 3840, "fc2"): 98_776_064 + 3_428_864,
    # decode weight stream (gemv_kernel): several tokens on a graph replay, one token on the
    # graph-creation call (one token's routing always touches k experts)
    ("phi", 16, "fc1"): 351_766_784 + 8_243_712,
    ("phi", 1, "fc1"): 54_117_888 + 119_296,
    ("qwen", 8, "fc1"): 71_535_616 + 1_062_912,
    ("dsv2", 32, "fc1"): 84_102_912 + 2_102_784,
}


def cpu_baseline(cfg, T, sample, n_layers, min_seconds=10.0, max_rounds=200):
    """Time the CPU oracle, as it stands, on a bounded token sample of the workload: one round
    routes all T tokens and runs the expert FFNs and combine for `sample` seeded tokens; rounds
    (each on a fresh seeded sample) repeat until at least `min_seconds` of CPU work."""
    from oracle import moe_oracle as O
    w = synth.layer_weights(cfg, 0)
    x = synth.activations(cfg, T)
    O.moe_layer(x[:8], w, cfg)     # warm the allocator
    gen = torch.Generator().manual_seed(T)
    tokens, dt, rounds = 0, 0.0, 0
    while dt < min_seconds and rounds < max_rounds:
        sub = torch.randperm(T, generator=gen)[:min(sample, T)].sort().values
        t = time.perf_counter()
        O.moe_layer(x, w, cfg, token_subset=sub)
        dt += time.perf_counter() - t
        tokens += len(sub)
        rounds += 1
    # one layer of a stack per sample: tokens/s of the whole stack = per-layer rate / layers
    value = tokens / dt / n_layers
    return {"value": value, "unit": "tokens/s", "cores": torch.get_num_threads(), "kind": "oracle",
            "sample": f"{rounds} rounds of the float64 oracle, each routing all {T} tokens and running the expert "
                      f"FFNs and combine for {min(sample, T)} seeded tokens of layer 0"
                      + (f", rate divided by {n_layers} layers" if n_layers > 1 else ""),
            "seconds": dt}


def run_elb(args, world, rank, local):
    """Specter's expert lookahead buffer at one chunk boundary: accumulate the routed ids of a
    32-step draft window for every MoE layer of a Qwen-shaped stack (24 layers, E=60, top-4),
    then take each layer's top-8 experts.  Latency-bound (a few KB), so the metric is time."""
    from weight_only_int4_route_gb300 import build as B
    from weight_only_int4_route_gb300 import moe as M
    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L, S, k, E, Mtop = 24, 32, 4, 60, 8
    g = torch.Generator(device=dev).manual_seed(9)
    ids = torch.argsort(torch.rand((L, S, E), generator=g, device=dev), dim=-1)[..., :k].to(torch.int32).contiguous()
    counts = torch.zeros((L, E), dtype=torch.int32, device=dev)
    experts = torch.empty((L, Mtop), dtype=torch.int32, device=dev)
    vals = torch.empty((L, Mtop), dtype=torch.int32, device=dev)
    lib, st = M.lib(), M._stream(dev)
    args_c = (M._ptr(ids), L, S, k, E, M._ptr(counts), Mtop, M._ptr(experts), M._ptr(vals), st)

    def step():   # one launch through the C ABI: accumulate + top-M
        M._check(lib.moe_elb_step(*args_c), "moe_elb_step")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    if M.device_error(dev):
        raise SystemExit("bench: device error word set during the run; no result reported")
    peaks, src = load_peaks()
    nbytes = ids.numel() * 4 + 3 * counts.numel() * 4 + 2 * L * Mtop * 4
    line = {"metric": "ELB boundary latency (accumulate a 32-step draft window for 24 layers + top-8 per layer)",
            "value": ms * 1e3, "unit": "us", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
            "data": "synthetic", "config": {"workload": f"L={L} layers, S={S} draft steps, top-{k} of E={E}, M={Mtop}"},
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "traffic": None,
                         "peak_source": f"{src} HBM copy bandwidth", "kernel": "elb_step_kernel",
                         "algorithmic_bytes": nbytes,
                         "note": "a few KB per boundary: the launch's latency, not bandwidth, is the cost"},
            "gpu_launches": args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_codec(args, world, rank, local):
    """BF16 bit-field recombine (exponent bytes + sign|mantissa bytes -> BF16): an HBM stream of
    4 bytes per element; 256 M elements per launch (1 GB moved, far above L2)."""
    from weight_only_int4_route_gb300 import build as B
    from weight_only_int4_route_gb300 import moe as M
    B.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n = 256 << 20
    g = torch.Generator(device=dev).manual_seed(5)
    w = (torch.randn(n, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    exp, sm = M.bf16_split(w)
    out = torch.empty_like(w)
    del w
    lib = M.lib()
    st = M._stream(dev)

    def step():
        M._check(lib.moe_bf16_recombine(M._ptr(exp), M._ptr(sm), n, M._ptr(out), st), "moe_bf16_recombine")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        step()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    if M.device_error(dev):
        raise SystemExit("bench: device error word set during the run; no result reported")
    peaks, src = load_peaks()
    gbs = 4.0 * n / (ms * 1e-3) / 1e9
    line = {"metric": "BF16 bit-field recombine bandwidth (exponent + sign|mantissa bytes -> BF16)", "value": gbs,
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": f"{n} BF16 elements (N(0, 0.02) weights), 1 GB moved per launch"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_source": f"{src} HBM copy bandwidth",
                         "kernel": "recombine_kernel", "algorithmic_bytes": 4 * n},
            "gpu_launches": args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_env()
    cfg = synth.CONFIGS[args.config]
    T = args.T or max(cfg.T)
    n_layers = args.layers or cfg.layers
    workload = (f"{cfg.name}: d={cfg.d} ffn={cfg.F} E={cfg.E} top-{cfg.k} {cfg.act} INT{cfg.bits} "
                f"{'per-channel' if cfg.group == 0 else 'group-128'} {cfg.dtype} activations"
                + (f" + shared expert Fs={cfg.Fs}" if cfg.Fs else "") + (f", Zipf({cfg.zipf}) logit bias" if cfg.zipf else "")
                + f", T={T} tokens" + (f", {n_layers} stacked layers" if n_layers > 1 else ""))
    base_cfg = {"workload": workload, "config": cfg.name, "T": T, "layers": n_layers}

    if args.impl == "reference":
        if rank != 0:
            return
        from oracle import moe_oracle as O
        w = synth.layer_weights(cfg, 0)
        x = synth.activations(cfg, T)
        sample = min(64, T)
        gen = torch.Generator().manual_seed(7)
        times = []
        for i in range(args.warmup + args.steps):
            sub = torch.randperm(T, generator=gen)[:sample].sort().values
            t = time.perf_counter()
            O.moe_layer(x, w, cfg, token_subset=sub)
            if i >= args.warmup:
                times.append(time.perf_counter() - t)
        per_step = sum(times) / len(times)
        value = sample / per_step / n_layers
        cores = torch.get_num_threads()
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": dict(base_cfg, l2="CPU run"),
                "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"each step: float64 oracle routing all {T} tokens, expert FFNs + combine "
                                           f"for {sample} seeded tokens of layer 0"},
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if args.codec:
        return run_codec(args, world, rank, local)
    if args.elb:
        return run_elb(args, world, rank, local)
    r = run_ours(args, cfg, T, n_layers, world, rank, local)
    peaks, peak_src = load_peaks()
    wm = work_model(cfg, T, r["counts"])
    value = job_tokens_per_s(world, T, r["ms"])
    # dominant kernel: the longer of the two grouped GEMM stages; a decode step that runs as one
    # launch is its own dominant kernel (the whole layer's bytes over the layer's time)
    st = r["stage_ms"]
    dom = "fc1" if st["fc1"] >= st["fc2"] else "fc2"
    dom_ms = st[dom]
    work = wm[dom]
    if r["one_launch"]:
        dom, dom_ms, work = "layer", r["ms"] / n_layers, wm["layer"]
    intensity = work["flops"] / work["bytes"]
    # the stage times come from a run of args.steps profiled steps, as long as the timed region
    tpeak, tpeak_src = tensor_peak(peaks, r["ms"] * args.steps * 1e-3, peak_src)
    ridge = tpeak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if intensity >= ridge:
        peak = tpeak
        achieved = work["flops"] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": tpeak_src}
    else:
        peak = peaks["hbm_gbs"]
        achieved = work["bytes"] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_src} HBM copy bandwidth"}
    roof.update({"traffic": MEASURED_TRAFFIC.get((cfg.name, T, dom)),
                 "kernel": ("decode_layer_kernel (the whole layer in one launch)" if dom == "layer" else
                            f"grouped GEMM {dom.upper()} ({r['kernels'][dom]})"),
                 "algorithmic_bytes": work["bytes"], "algorithmic_flops": work["flops"], "ms_per_launch": dom_ms})
    layer_ms = r["ms"] / n_layers
    lw = wm["layer"]
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
            "config": dict(base_cfg, launch=r["launch"], l2=(f"inputs larger than L2: {r['copies']} rotating weight/activation copies"
                                         if n_layers == 1 else f"{n_layers} distinct layers per step"),
                           active_experts=wm["active_experts"],
                           layer_roofline={"hbm_frac": lw["bytes"] / (layer_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                           "tensor_frac": lw["flops"] / (layer_ms * 1e-3) / 1e12 / tpeak,
                                           "bytes": lw["bytes"], "flops": lw["flops"]},
                           **({"stage_ms_kernel_chain": st} if r["one_launch"] else {"stage_ms": st}),
                           parallelism=f"replicas x{world} (token data parallel)"),
            "roofline": roof, "gpu_launches": r["launches"]}
    if r["clocks"]:
        line["clocks"] = r["clocks"]
    if r["e2e"]:
        e = r["e2e"]
        line["e2e"] = {"value": job_tokens_per_s(world, T, e["ms"]), "unit": "tokens/s", "h2d_bytes_per_step": e["h2d"],
                       "d2h_bytes_per_step": e["d2h"],
                       "copies": "pinned host <-> device every step, on upload / download streams, double-buffered"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, T, args.cpu_sample, n_layers)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if r["dist"] is not None:
        r["dist"].destroy_process_group()


if __name__ == "__main__":
    main()
