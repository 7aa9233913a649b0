#!/usr/bin/env python3
"""Benchmark of the fused a8w4 MoE layer forward on GB300.

One step = one layer forward (routing, EPLB remap/record, MXFP8 quant,
dispatch, GEMM1+SwiGLU+requant, GEMM2, combine) over one batch of seeded
synthetic tokens.  Default workload: the largest one-GPU layer, T=16384
tokens, H=7168, I=2048, 256 logical experts on 320 physical (64 redundant
replicas), top-6, Zipf-skewed routing with load recording (the large-input
path); --config 1 is the decode (small-input) layer, T=64.  The expert
weights (6-7.5 GB of MXFP4) and the dispatched rows are larger than L2, so
consecutive steps stream them from HBM; no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

Under torchrun each rank runs its own batch (independent replicas, no
collective on the data path): weak scaling, value = tokens of all ranks /
max-over-ranks time.  Prints one JSON line on rank 0.
"""
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

import synthetic  # noqa: E402

METRIC = "MoE-layer tokens/s"
EXPERT_BYTES_PER_ELEM = 0.5 + 1.0 / 32      # packed e2m1 + one e8m0 byte per 32


def strip_c_comments(text: str) -> str:
    """C/C++ source without its // and /* */ comments and with every run of
    whitespace outside string and character literals made one space (the
    literals are kept as they are)."""
    out, i, n = [], 0, len(text)

    def space():
        if out and out[-1] != " ":
            out.append(" ")

    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            space()
            i = n if j < 0 else j + 2
        elif c.isspace():
            space()
            i += 1
        else:
            out.append(c)
            i += 1
    return "".join(out).strip()


def sources_digest() -> str:
    """sha256 over the kernel sources (csrc/*.cu, *.cuh, *.h and the C header)
    with comments removed and whitespace collapsed: editing a comment or the
    layout does not change a kernel."""
    import hashlib
    csrc = os.path.join(ROOT, "moe_layer_serving_gb300", "csrc")
    files = sorted(os.path.join("moe_layer_serving_gb300", "csrc", f) for f in os.listdir(csrc)
                   if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join("include", "megamoe.h"))
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(strip_c_comments(fh.read()).encode())
    return h.hexdigest()


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary (profiles/traffic.json), or None when there is none or the kernel
    sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path)).get(kernel, {}).get(workload)
    if not entry or entry.get("sources_sha256") != sources_digest():
        return None
    return entry["bytes_per_launch"]


def expert_bytes(cfg) -> int:
    return int((2 * cfg.I * cfg.H + cfg.H * cfg.I) * EXPERT_BYTES_PER_ELEM)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-sample", type=int, default=64,
                    help="tokens per step in the reference arm's sample (the oracle dequantises each touched "
                         "expert once per call, so a whole decode batch is the representative sample)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work the oracle baseline leg runs (its token sample doubles up to the batch)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baseline leg")
    ap.add_argument("--route", choices=["auto", "small", "large"], default="auto",
                    help="path: auto (fused kernel up to 512 tokens), or force the fused or the multi-launch path")
    ap.add_argument("--shared", type=int, default=0,
                    help="fused shared experts: slots per token beyond top-k, weight 1 (mm_set_shared_experts)")
    ap.add_argument("--act", choices=["mxfp8", "bf16"], default="mxfp8",
                    help="activation format: mxfp8 (a8w4, the fused operator) or bf16 (the a16w4 variant)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E = P (a smaller case of the same kernels, for profiler captures)")
    ap.add_argument("--scale-down", type=int, default=1,
                    help="divide T, E and P by this factor, keeping the routing shape, the rows per expert and "
                         "the redundant-replica share (a smaller case for profiler captures)")
    return ap.parse_args()


def scaled_down(cfg, f: int):
    """The same workload with T, E and P divided by f: equal rows per expert
    (T k / E), the same routing recipe and the same share of redundant
    replicas, so its kernels do 1/f of the work of the full one."""
    import dataclasses
    if cfg.T % f or cfg.E % f or cfg.P % f or cfg.E // f < cfg.k:
        raise SystemExit(f"--scale-down {f} does not divide config {cfg.cid}")
    return dataclasses.replace(cfg, T=cfg.T // f, E=cfg.E // f, P=cfg.P // f)


def routing_label(cfg) -> str:
    if cfg.zipf_s:
        return f"zipf s={cfg.zipf_s:g} logit offset + N(0,1)"
    return "N(0,1) logits" + (f" + N(0,{cfg.bias_std:g}) selection bias" if cfg.bias_std else "")


def workload_config(cfg, act="mxfp8", route="auto", shared=0):
    name = "a8w4" if act == "mxfp8" else "a16w4"
    suffix = ("" if route == "auto" else f"-{route}-path") + (f"-shared{shared}" if shared else "")
    full = synthetic.CONFIGS.get(cfg.cid)
    if full is not None and (cfg.E, cfg.P) != (full.E, full.P):
        suffix += f"-E{cfg.E}-P{cfg.P}"          # a reduced case of the workload (profiler captures)
    return {"workload": f"moe-layer-{name}-T{cfg.T}{suffix}", "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E,
            "P": cfg.P, "topk": cfg.k, "shared_experts": shared, "routing": routing_label(cfg),
            "eplb_redundant": cfg.P - cfg.E, "recording": bool(cfg.recording),
            "l2": "weights and dispatched rows > L2, no flush", "parallelism": "replicas"}


class ClockSampler:
    """nvidia-smi samples (200 ms apart) of the SM clock and throttle reasons;
    stop(since, until) keeps the samples taken between the two (time.monotonic())."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.monotonic(), parts))

    def stop(self, since=None, until=None):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = [r for t, r in self.rows if (since is None or t >= since) and (until is None or t <= until)]
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


SOAK_S = 1.0


def oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, n_tokens, act="mxfp8", shared=0):
    """Tokens/s of the CPU oracle on the first n_tokens of the batch."""
    import oracle
    sel = np.arange(min(n_tokens, hidden.shape[0]))
    m, rc = pmap if pmap else (None, None)
    t0 = time.perf_counter()
    oracle.forward(hidden[sel], logits[sel], bias, cfg.k, W, m, rc, token_ids=sel, act=act, shared=shared)
    dt = time.perf_counter() - t0
    return sel.size / dt, dt, sel.size


def with_shared_weights(cfg, W, shared):
    """W (the P routed physical experts) followed by `shared` further experts,
    drawn as logical experts E .. E+shared-1 of the same seeded generator."""
    if not shared:
        return W
    extra = [synthetic.make_expert_weights(cfg, cfg.E + s) for s in range(shared)]
    return tuple(np.concatenate([a, np.stack([x[i] for x in extra])]) for i, a in enumerate(W))


def oracle_bounded_rate(cfg, hidden, logits, bias, W, pmap, seconds, act="mxfp8", shared=0):
    """Tokens/s of the CPU oracle over about `seconds` of work: the token sample
    doubles from 8 until one run takes a quarter of that or covers the batch,
    then that sample runs until the time is spent (at most 8 runs)."""
    n = min(8, cfg.T)
    rate, dt, n = oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, n, act, shared)
    while dt < seconds / 4 and n < cfg.T:
        rate, dt, n = oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, min(2 * n, cfg.T), act, shared)
    toks, total, reps = n, dt, 1
    while total < seconds and reps < 8:
        _, d, _ = oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, n, act, shared)
        toks, total, reps = toks + n, total + d, reps + 1
    return toks / total, total, n, reps


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s: every rank processed its own batch in at most max_ms."""
    return tokens_per_rank * world / (max_ms / 1e3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The oracle (plain C, fp64) timed on this machine's CPU cores."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    cfg = synthetic.CONFIGS[args.config]
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = with_shared_weights(cfg, synthetic.make_all_weights(cfg), args.shared)
    pmap = synthetic.make_eplb_map(cfg)[:2] if cfg.P != cfg.E else None
    n = min(args.cpu_sample, cfg.T)
    for _ in range(max(0, args.warmup and 1)):
        oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, 1, args.act, args.shared)
    times = []
    for _ in range(args.steps):
        _, dt, _ = oracle_sample_rate(cfg, hidden, logits, bias, W, pmap, n, args.act, args.shared)
        times.append(dt)
    per_tok = statistics.median(times) / n
    value = 1.0 / per_tok
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_tok * cfg.T * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(cfg, args.act, shared=args.shared),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"first {n} of {cfg.T} tokens per step, all stages"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch

    import moe_layer_serving_gb300 as mm
    from moe_layer_serving_gb300 import build as mbuild

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    mbuild.build()
    dev = torch.device("cuda", local)
    cfg = synthetic.CONFIGS[args.config]
    if args.experts:
        import dataclasses
        cfg = dataclasses.replace(cfg, E=args.experts, P=args.experts, zipf_s=0.0)
    if args.scale_down > 1:
        cfg = scaled_down(cfg, args.scale_down)
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = with_shared_weights(cfg, synthetic.make_all_weights(cfg), args.shared)
    pmap = synthetic.make_eplb_map(cfg)[:2] if cfg.P != cfg.E else None

    op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
    if args.shared:
        op.set_shared_experts(args.shared)
    wt = [torch.from_numpy(a).to(dev) for a in W]
    op.set_weights(*wt)
    del wt
    torch.cuda.empty_cache()
    if pmap:
        op.set_eplb_map(*pmap)
    a16 = args.act == "bf16"
    if a16:
        op.set_activation_format(mm.ACT_BF16)
    op.set_route({"auto": mm.ROUTE_AUTO, "small": mm.ROUTE_SMALL, "large": mm.ROUTE_LARGE}[args.route])
    op.reserve(cfg.T)
    op.set_recording(cfg.recording)
    x = torch.from_numpy(hidden.view(np.int16)).to(dev).view(torch.bfloat16)
    lg = torch.from_numpy(logits).to(dev)
    b = torch.from_numpy(bias).to(dev)
    out = torch.empty_like(x)
    stream = torch.cuda.Stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident inputs: the kernel-level number ------------------
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            op.forward(x, lg, b, out, stream=stream)
    stream.synchronize()
    assert op.get_status() == 0
    route, launches, _ = op.last_info()
    gemm_kind = op.last_gemm()
    phys = op.debug_dump(2)
    touched = int(np.unique(phys).size)

    op.profile_begin(args.steps)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_load = time.monotonic()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            op.forward(x, lg, b, out, stream=stream)
        ev1.record(stream)
    stream.synchronize()
    kern = op.profile_end()
    # a short timed region falls between two clock samples: the same steps run on,
    # untimed, for SOAK_S more seconds so that the clocks are sampled under this load
    t_soak = time.monotonic()
    with torch.cuda.stream(stream):
        while time.monotonic() - t_soak < SOAK_S:
            for i in range(args.steps):
                op.forward(x, lg, b, out, stream=stream)
            stream.synchronize()
    clk = clocks.stop(since=t_load, until=time.monotonic())
    clk["window"] = f"the timed steps and {SOAK_S:.0f} s more of them"
    torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    kern_ms = float(np.mean(kern))
    assert op.get_status() == 0
    value = weak_scaling_value(cfg.T, world, ms)

    # ---- end to end through the public call, host buffers ------------------
    xh = torch.from_numpy(hidden.view(np.int16)).pin_memory()
    lh = torch.from_numpy(logits).pin_memory()
    oh = torch.empty((cfg.T, cfg.H), dtype=torch.int16).pin_memory()
    xd = torch.empty_like(x)
    ld = torch.empty_like(lg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            if i == args.warmup:
                e0.record(stream)
            xd.view(torch.int16).copy_(xh, non_blocking=True)
            ld.copy_(lh, non_blocking=True)
            op.forward(xd, ld, b, out, stream=stream)
            oh.copy_(out.view(torch.int16), non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e = weak_scaling_value(cfg.T, world, e2e_ms)
    h2d = hidden.nbytes + logits.nbytes
    d2h = cfg.T * cfg.H * 2

    # ---- roofline of the dominant kernel ------------------------------------
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))
    kname = {0: "small_kernel", 1: "gemm_kernel", 2: "gemm2_kernel", 3: "gemm16_kernel"}[gemm_kind]
    wname = workload_config(cfg, args.act, args.route, args.shared)["workload"]
    if cfg.T <= 512:
        alg = touched * expert_bytes(cfg)           # weight streaming: the touched experts' bytes
        achieved = alg / (kern_ms / 1e3) / 1e9
        peak = peaks.get("hbm_gbs", 6800.0)
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": measured_traffic(kname, wname), "kernel": kname, "algorithmic_bytes": alg,
                "peak_source": "measured" if "hbm_gbs" in peaks else "fallback"}
    else:
        flops = 6.0 * cfg.T * (cfg.k + args.shared) * cfg.H * cfg.I
        achieved = flops / (kern_ms / 1e3) / 1e12
        # bf16 MMAs (a16w4) against the measured bf16 rate; fp8-class MMAs at 2x it
        mult = 1.0 if a16 else 2.0
        peak = peaks.get("bf16_tflops", 1900.0) * mult
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": measured_traffic(kname, wname), "kernel": kname, "algorithmic_flops": flops,
                "step_frac": flops / (ms / 1e3) / 1e12 / peak,
                "peak_source": ("measured bf16" if a16 else "measured bf16 x 2") if "bf16_tflops" in peaks
                else ("fallback" if a16 else "fallback x 2")}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16xe2m1->f32" if a16 else "e4m3xe2m1->f32",
        "data": "synthetic (seeded, random-init weights)", "config": workload_config(cfg, args.act, args.route, args.shared), "clocks": clk, "gpu_launches": launches * args.steps,
        "route": "small" if route == 1 else "large", "kernel_ms": kern_ms, "touched_experts": touched,
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "roofline": roof,
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        rate, total, n, reps = oracle_bounded_rate(cfg, hidden, logits, bias, W, pmap, args.cpu_seconds, args.act,
                                                   args.shared)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": oracle.threads(), "kind": "oracle",
                                "sample": f"{reps} x first {n} of {cfg.T} tokens, all stages, {total:.1f} s timed"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    op.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
