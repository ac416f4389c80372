"""Benchmark of the GB300 W4A16 MoE layer: MoE-layer tokens/s, INT4 weight-stream
GB/s and roofline fraction, one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode1]
                    [--impl ours|reference]

A step is one forward of the whole layer (router, histogram/scan/permute,
gate/up+SwiGLU, down, combine with the shared expert) over one batch. The
default workload is decode at 1 token on the DeepSeek-V4-Flash-shaped layer
(hidden 4096, 256 routed experts top-6 + 1 shared, intermediate 2048, INT4
g128). Inputs are synthetic (seeded), resident in HBM before timing; the L2
is flushed (a 512 MB read) before every timed step, outside the timed span.
The forward is captured once in a CUDA graph and replayed.
"""
from __future__ import annotations

import argparse
import dataclasses
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

import moe_synth as ms  # noqa: E402

PROFILE_DIR = os.path.join(ROOT, "profiles")
METRIC = "MoE-layer tokens/s; INT4 weight-stream GB/s & % roofline (bs 1..8192)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ------------------------------------------------------------ algorithmic work
def expert_bytes(shape, inter):
    H = shape.hidden
    w13 = 2 * inter * H // 2 + 2 * inter * (H // 128) * 2
    w2 = H * inter // 2 + H * (inter // 128) * 2
    return w13, w2


def layer_work(shape, counts):
    """Algorithmic bytes and flops of one forward given per-expert row counts."""
    T, H, E, k, I, Is = (shape.tokens, shape.hidden, shape.experts, shape.top_k, shape.inter,
                         shape.shared_inter)
    hit = int((np.asarray(counts) > 0).sum())
    r13, r2 = expert_bytes(shape, I)
    s13, s2 = expert_bytes(shape, Is) if Is else (0, 0)
    w13_bytes = hit * r13 + s13
    w2_bytes = hit * r2 + s2
    act = T * H * 2 * 2                      # x in, out
    router = E * H * 4 + E * 4
    flops = 2 * T * E * H + 2 * 3 * H * (T * k * I + (T * Is if Is else 0))
    return {"hit": hit, "w13_bytes": w13_bytes, "w2_bytes": w2_bytes,
            "weight_bytes": w13_bytes + w2_bytes, "act_bytes": act, "router_bytes": router,
            "bytes": w13_bytes + w2_bytes + act + router, "flops": flops}


def kernel_work(name, shape, work, y_bytes=None):
    """Algorithmic DRAM bytes and useful FLOPs of one launch of a kernel.

    Bytes: the INT4 weights and scales of the experts hit, plus each
    activation operand read once and each result written once. FLOPs: 2 per
    multiply-add of the layer's own arithmetic (no padding, no re-reads).
    y, the per-expert down output, is bf16 (2 bytes) after the tensor-core
    down GEMM and fp32 (4) after the GEMV one; y_bytes says which one the
    combine read (default: bf16).
    """
    T, H, E, k, I, Is = (shape.tokens, shape.hidden, shape.experts, shape.top_k, shape.inter,
                         shape.shared_inter)
    rows = T * k + (T if Is else 0)
    hrows = T * k * I + T * Is               # h elements
    f13 = 2 * H * 2 * hrows                  # gate + up
    f2 = 2 * H * hrows                       # down
    if name == "decode_fused":
        return work["bytes"], work["flops"]
    if name.startswith("gemv_gate_up"):
        return work["w13_bytes"] + T * H * 2 + hrows * 2, f13
    if name.startswith("tc_gate_up"):
        # activations counted once (T rows); the expert-ordered copy of x the
        # GEMM reads instead is an implementation choice (implementation_bytes)
        return work["w13_bytes"] + T * H * 2 + hrows * 2, f13
    if name.startswith("gemv_down"):
        return work["w2_bytes"] + hrows * 2 + rows * H * 4, f2
    if name.startswith("tc_down"):
        return work["w2_bytes"] + hrows * 2 + rows * H * 2, f2
    # W4A8-FP8 experts: e4m3 activations (1 byte) in, fp32 h and y out
    if name == "w4a8_quantize_x":
        return T * H * 2 + T * H + T * (H // 128) * 4, 0
    if name == "w4a8_gate_up_swiglu":
        return work["w13_bytes"] + T * H + T * (H // 128) * 4 + hrows * 4, f13
    if name == "w4a8_quantize_h":
        return hrows * 4 + hrows + hrows // 128 * 4, 0
    if name == "w4a8_down":
        return work["w2_bytes"] + hrows + hrows // 128 * 4 + rows * H * 4, f2
    if name.startswith("route") or name.startswith("router"):
        return work["router_bytes"] + T * H * 2 * 2, 2 * T * E * H
    if name == "combine":
        return rows * H * (2 if y_bytes is None else y_bytes) + T * H * 2, 2 * T * k * H
    return 0, 0


def implementation_bytes(name, shape):
    """DRAM bytes a kernel moves beyond its algorithmic ones by design (not
    counted in the roofline): the tensor-core gate/up GEMM reads x gathered
    into expert order (T*k + T rows) instead of the T token rows."""
    if name.startswith("tc_gate_up"):
        rows = shape.tokens * shape.top_k + (shape.tokens if shape.shared_inter else 0)
        return (rows - shape.tokens) * shape.hidden * 2
    return 0


def roofline(name, shape, work, seconds, pk, y_bytes=None):
    """Roofline entry of one kernel: whichever of the HBM and bf16 tensor
    bounds is slower for its algorithmic work decides the bound."""
    nbytes, flops = kernel_work(name, shape, work, y_bytes)
    extra = implementation_bytes(name, shape)
    # fp8 kernels: the measured bf16 peak times the nominal fp8 / bf16 ratio (2)
    fp8 = name.startswith("w4a8")
    tpk = pk["bf16_tflops"] * (2.0 if fp8 else 1.0)
    t_mem = nbytes / (pk["hbm_gbs"] * 1e9)
    t_mma = flops / (tpk * 1e12)
    if t_mma > t_mem:
        ach = flops / seconds / 1e12
        return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tpk,
                "unit": "TFLOP/s", "frac": ach / tpk, "algorithmic_flops": flops,
                "algorithmic_bytes": nbytes, "implementation_bytes": extra,
                "peak_source": pk["source"] + (" bf16 x 2 (fp8, nominal ratio)" if fp8 else "")
                               + " (burst)"}
    ach = nbytes / seconds / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
            "algorithmic_flops": flops, "implementation_bytes": extra,
            "peak_source": pk["source"]}


# ------------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        self.path = f"/tmp/moe_bench_clocks_{os.getpid()}.csv"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}", "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                smax = float(f[2].split()[0])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------- ncu traffic
def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture (else None)."""
    path = os.path.join(PROFILE_DIR, f"{kernel}_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        prof = json.load(f)
    src = os.path.join(ROOT, "w4a16_routed_expert_router_gb300", "csrc", prof.get("source", ""))
    if not os.path.exists(src):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if digest != prof.get("source_sha256_16"):
        return None
    return prof.get("dram_bytes_per_launch")


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def maybe_init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(value, dist, device=None):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle arm
def oracle_sample(shape, budget_s=15.0, w4a8=False):
    """Time the fp64 oracle on the host on a bounded sample of the workload.

    Routing is computed for the whole batch; outputs token by token until the
    time budget is spent. Drawing the synthetic weights is not timed. w4a8:
    the W4A8-FP8 oracle's layer instead of the W4A16 one.
    """
    from oracle import moe_oracle as mo
    from oracle import w4a8_oracle as w8
    layer_fn = w8.moe_forward_w4a8 if w4a8 else mo.moe_forward
    x = ms.tokens(shape)
    rw, rb = ms.router_weights(shape), ms.router_bias(shape)
    shared = ms.expert_weights(shape, shape.experts) if shape.shared_inter else None
    wall = cpu = 0.0
    t0, c0 = time.perf_counter(), time.process_time()
    route = mo.route(x, rw, rb, shape.experts, shape.top_k)
    wall += time.perf_counter() - t0
    cpu += time.process_time() - c0
    done = 0
    while wall < budget_s and (done < shape.tokens or shape.tokens < 8):
        if done and done % shape.tokens == 0:   # tiny batches: time further draws
            x = ms.tokens(dataclasses.replace(shape, token_seed=shape.token_seed + 7919 * done))
            t0, c0 = time.perf_counter(), time.process_time()
            route = mo.route(x, rw, rb, shape.experts, shape.top_k)
            wall += time.perf_counter() - t0
            cpu += time.process_time() - c0
        t = done % shape.tokens
        experts = [None] * shape.experts
        for e in route["ids"][t]:
            experts[int(e)] = ms.expert_weights(shape, int(e))
        t0, c0 = time.perf_counter(), time.process_time()
        layer_fn(x[t:t + 1], rw, rb, experts, shared, shape.top_k)
        wall += time.perf_counter() - t0
        cpu += time.process_time() - c0
        done += 1
    return {"tokens": done, "wall_s": wall, "cpu_s": cpu,
            "cores": max(1, round(cpu / wall)) if wall > 0 else 1}


def config_of(shape, args):
    """The workload description both arms print (the same dict, so that the
    two lines can be compared key by key)."""
    return {"workload": shape.name, "tokens": shape.tokens, "hidden": shape.hidden,
            "experts": shape.experts, "top_k": shape.top_k, "inter": shape.inter,
            "shared_inter": shape.shared_inter, "weights": "int4 g128 symmetric",
            "l2": "flushed before every step (512 MB read, untimed)",
            "graph": "one forward per CUDA-graph replay", "parallelism": "replicas",
            "expert_path": args.expert_path}


def run_reference(args, shape):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    r = oracle_sample(shape, budget_s=max(5.0, min(60.0, 10.0 + 2.0 * args.steps)))
    value = r["tokens"] / r["wall_s"]
    sample = (f"{r['tokens']} tokens of {shape.name} batches (routing of every batch, "
              f"outputs token by token), {r['wall_s']:.1f} s wall")
    line = {"impl": "reference", "metric": METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * r["wall_s"] / max(r["tokens"], 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": config_of(shape, args),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": r["cores"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU arm
class Bench:
    """One device, one uploaded copy of each distinct layer's weights; measures
    workloads on it."""

    def __init__(self, args, dev, dist):
        import torch
        self.torch = torch
        self.args = args
        self.dev = dev
        self.dist = dist
        self.layers = {}
        # L2 flush: reading a 512 MB buffer (4x the 129 MB L2) leaves only
        # clean lines of that buffer in L2, so the timed step starts cold and
        # pays no write-back of someone else's dirty lines.
        self.flush = torch.ones(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.flush_out = torch.empty((), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)

    def flush_l2(self):
        self.torch.sum(self.flush, dim=0, out=self.flush_out)

    def tensors(self, shape):
        from moe_synth.device import upload_layer
        key = (shape.layer_seed, shape.hidden, shape.experts, shape.inter, shape.shared_inter)
        if key not in self.layers:
            base = ms.make_layer(shape.with_tokens(0), x=np.zeros((0, shape.hidden), np.uint16))
            self.layers[key] = upload_layer(base, self.dev)[0]
        t = dict(self.layers[key])
        t["router_bias"] = self.torch.from_numpy(ms.router_bias(shape)).to(self.dev)
        return t

    def measure(self, shape, steps, warmup, clocks):
        """Time one workload: CUDA-graph replays (L2 flushed before each), the
        per-kernel durations, and the host-buffer entry point end to end."""
        import w4a16_routed_expert_router_gb300 as moe
        from moe_synth.device import upload_tokens
        torch, dev, dist, stream = self.torch, self.dev, self.dist, self.stream
        tensors = self.tensors(shape)
        T, H = shape.tokens, shape.hidden
        # distinct token batches (same distribution), resident in HBM before timing
        nx = min(steps, 8)
        xs = [upload_tokens(ms.tokens(dataclasses.replace(shape, token_seed=shape.token_seed + 7919 * i)),
                            dev) for i in range(nx)]
        out = torch.empty((T, H), dtype=torch.int16, device=dev)
        path_flags = {"auto": 0, "tc": moe.MOE_W4A16_FLAG_FORCE_TC,
                      "gemv": moe.MOE_W4A16_FLAG_FORCE_GEMV,
                      "w4a8": moe.MOE_W4A16_FLAG_W4A8}[self.args.expert_path]
        obj = moe.MoeLayer(shape.hidden, shape.experts, shape.top_k, shape.inter,
                           shape.shared_inter, T, tensors, flags=path_flags)
        prof = moe.MoeLayer(shape.hidden, shape.experts, shape.top_k, shape.inter,
                            shape.shared_inter, T, tensors,
                            flags=path_flags | moe.MOE_W4A16_FLAG_PROFILE)
        xin = torch.empty_like(xs[0])

        # --- capture one forward in a CUDA graph (input copied into xin first)
        with torch.cuda.stream(stream):
            xin.copy_(xs[0])
            obj.forward(xin, out, stream=stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            obj.forward(xin, out, stream=torch.cuda.current_stream())
        launches_per_fwd = len(moe.moe_w4a16_last_launches(obj.handle))

        def step(i, timed, ev=None):
            with torch.cuda.stream(stream):
                self.flush_l2()
                xin.copy_(xs[i % nx])
                if timed:
                    ev[0].record(stream)
                graph.replay()
                if timed:
                    ev[1].record(stream)

        for i in range(warmup):
            step(i, False)
        stream.synchronize()
        assert moe.moe_w4a16_check_device_errors(obj.handle) == 0

        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with clocks:
            for i in range(steps):
                step(i, True, evs[i])
            torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        total_ms = sum(a.elapsed_time(b) for a, b in evs)
        total_ms = max_over_ranks(total_ms, dist, dev)
        world = dist.get_world_size() if dist is not None else 1
        ms_per_step = total_ms / steps
        value = world * T * steps / (total_ms / 1000.0)

        # --- routing stats of the timed inputs (for the algorithmic bytes)
        rt_counts = []
        for i in range(nx):
            with torch.cuda.stream(stream):
                obj.forward(xs[i], out, stream=stream)
            stream.synchronize()
            rt_counts.append(np.diff(obj.routing(T, stream=stream)["offsets"]))
        works = [layer_work(shape, c) for c in rt_counts]
        work = {k_: float(np.mean([w[k_] for w in works])) for k_ in works[0]}

        # --- per-kernel durations with CUDA events (no graph), same flush
        kernel_ms = {}
        nprof = min(steps, 50)
        for i in range(warmup + nprof):
            with torch.cuda.stream(stream):
                self.flush_l2()
                prof.forward(xs[i % nx], out, stream=stream)
            stream.synchronize()
            if i >= warmup:
                for name, t_ms in moe.moe_w4a16_last_launches(prof.handle):
                    kernel_ms.setdefault(name, []).append(t_ms)
        kernel_avg = {n: float(np.mean(v)) for n, v in kernel_ms.items()}
        dominant = max(kernel_avg, key=kernel_avg.get)

        # --- end to end through the host-buffer entry point
        xh = torch.from_numpy(ms.tokens(shape).view(np.int16)).pin_memory()
        oh = torch.empty((T, H), dtype=torch.int16).pin_memory()
        for _ in range(3):
            obj.forward_host(xh, oh, stream=stream)
        e2e_s = 0.0
        n_e2e = min(steps, 100)
        for i in range(n_e2e):
            with torch.cuda.stream(stream):
                self.flush_l2()
            stream.synchronize()
            t0 = time.perf_counter()
            obj.forward_host(xh, oh, stream=stream)
            e2e_s += time.perf_counter() - t0
        e2e_s = max_over_ranks(e2e_s, dist, dev)
        e2e_value = world * T * n_e2e / e2e_s
        assert moe.moe_w4a16_check_device_errors(obj.handle) == 0
        obj.close()
        prof.close()

        pk = peaks()
        y_bytes = 4 if any(n.startswith(("gemv_down", "w4a8_down")) for n in kernel_avg) else 2
        roof = roofline(dominant, shape, work, kernel_avg[dominant] / 1000.0, pk, y_bytes)
        roof["traffic"] = profiled_traffic(dominant, shape.name)
        layer_roof_s = max(work["bytes"] / (pk["hbm_gbs"] * 1e9),
                           work["flops"] / (pk["bf16_tflops"] * 1e12))
        return {
            "value": value, "unit": "tokens/s", "ms_per_step": ms_per_step, "steps": steps,
            "weight_stream_gbs": work["weight_bytes"] / (ms_per_step / 1000.0) / 1e9,
            "layer_roofline_frac": layer_roof_s / (ms_per_step / 1000.0),
            "layer_bound": "tensor" if work["flops"] / (pk["bf16_tflops"] * 1e12) >
                           work["bytes"] / (pk["hbm_gbs"] * 1e9) else "hbm",
            "algorithmic_bytes": work["bytes"], "algorithmic_flops": work["flops"],
            "experts_hit": work["hit"],
            "roofline": roof,
            "kernels_ms": kernel_avg,
            "gpu_launches": launches_per_fwd * steps,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                    "d2h_bytes_per_step": T * H * 2},
        }


def run_ours(args, shape):
    import torch

    import w4a16_routed_expert_router_gb300 as moe
    from w4a16_routed_expert_router_gb300 import _build

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = maybe_init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    moe.lib()

    b = Bench(args, dev, dist)
    clocks = ClockSampler(local)
    head = b.measure(shape, args.steps, args.warmup, clocks)
    clk = clocks.summary()
    others = {}
    for name in args.per_config:
        if name == shape.name:
            continue
        c = ClockSampler(local)
        r = b.measure(ms.CONFIGS[name], min(args.steps, 100), args.warmup, c)
        r["clocks"] = c.summary()
        others[name] = r

    if rank == 0:
        cpu = oracle_sample(shape, budget_s=15.0, w4a8=args.expert_path == "w4a8") if world == 1 else None
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if args.expert_path == "w4a8" else "bf16",
            "data": "synthetic",
            "config": config_of(shape, args),
        }
        for k_ in ("weight_stream_gbs", "layer_roofline_frac", "layer_bound", "experts_hit",
                   "roofline", "kernels_ms", "gpu_launches", "e2e"):
            line[k_] = head[k_]
        line["clocks"] = clk
        if cpu is not None:
            line["cpu_baseline"] = {"value": cpu["tokens"] / cpu["wall_s"], "unit": "tokens/s",
                                    "cores": cpu["cores"], "kind": "oracle",
                                    "sample": f"{cpu['tokens']} tokens of {shape.name} batches "
                                              f"({cpu['wall_s']:.1f} s wall)"}
        if others:
            line["per_config"] = others
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default="decode1", choices=ms.CONFIG_ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--expert-path", default="auto", choices=["auto", "tc", "gemv", "w4a8"],
                    help="expert kernels: the library's choice, tensor-core, split-K GEMV, "
                         "or the W4A8-FP8 experts (e4m3 activations)")
    ap.add_argument("--per-config", default="decode64,prefill8192,zipf2048",
                    help="further workloads measured after the headline one and reported "
                         "under per_config (comma-separated; 'none' for none)")
    args = ap.parse_args()
    args.per_config = [] if args.per_config in ("", "none") else args.per_config.split(",")
    for name in args.per_config:
        if name not in ms.CONFIGS:
            ap.error(f"unknown workload {name}")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    shape = ms.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, shape)
    else:
        run_ours(args, shape)


if __name__ == "__main__":
    main()
