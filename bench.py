#!/usr/bin/env python3
"""Benchmark of the fused FP4-weight MoE layer on GB300.

Workload: the decode layer E=512, H=2560, I=320, top_k=10, M=1 token, NVFP4
weights (an E4M3 scale per 16 K-elements plus FP32 per-tensor multipliers),
BF16 activations, softmax top-k routing with distinct experts per token.  A
step is one whole layer (routing inside the kernels, FC1, SiLU*up, FC2,
router-weighted sum) on one routing draw.  Metric: routed-weight HBM GB/s
(the routed experts' weight + scale bytes, plus activations, ids and output,
divided by the layer time), with microseconds per layer alongside.

Cold L2: the K timed layers cycle through K routing draws in which no expert
repeats within 20 consecutive layers (20 x 13.8 MB = 276 MB > 2 x L2), so
every layer streams its experts from HBM.  The K layers are captured in one
CUDA graph and replayed once between two device syncs.

--impl reference runs the FP64 CPU oracle (the only other implementation of
this layer here) on the host cores on the same workload.
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

METRIC = "fused FP4 MoE µs/layer & routed-weight HBM GB/s at M=1..8; prefill TFLOP/s"
WORKLOAD = "decode_e512"
WINDOW = 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default=WORKLOAD, help="workload name (default: the decode_e512 headline)")
    ap.add_argument("--M", type=int, default=None, help="override the token count")
    ap.add_argument("--E", type=int, default=None, help="override the expert count (profiling on smaller memory)")
    ap.add_argument("--fmt", choices=["mxfp4", "nvfp4"], default=None)
    return ap.parse_args()


def workload_config(args):
    from workload import gen
    c = dict(gen.CONFIGS[args.workload])
    if args.M is not None:
        c["M"] = args.M
    if args.E is not None:
        c["E"] = args.E
    if args.fmt is not None:
        c["fmt"] = gen.MXFP4 if args.fmt == "mxfp4" else gen.NVFP4
    return c


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_time_and_units(ms, units, ws, device):
    """Whole-job timing of the replicas: the slowest rank's time (every rank
    times its own K layers with CUDA events) and the units all ranks
    processed (each rank draws its own routing, so their bytes differ)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, units], dtype=torch.float64, device=device)
    if ws > 1:
        tmax = t[:1].clone()
        tsum = t[1:].clone()
        dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
        dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
        return float(tmax.item()), float(tsum.item())
    return float(t[0].item()), float(t[1].item())


def layer_flops(ids, E, H, I):
    """2 * (gate + up + down) multiply-adds per valid routed row."""
    n = int(((ids >= 0) & (ids < E)).sum())
    return 2 * 3 * H * I * n


def load_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def layer_bytes(ids, E, H, I, M, top_k, fmt):
    from workload import gen
    uniq = len(gen.routed_unique_experts(ids, E))
    return uniq * gen.expert_bytes(H, I, fmt) + M * H * 2 * 2 + M * top_k * 8, uniq


# ------------------------------------------------------------------ CPU oracle
def oracle_layers(c, seed, ids_pool, w_pool, x_host, seconds, max_layers):
    """Time the FP64 oracle on successive routing draws (bounded sample)."""
    import oracle
    from workload import gen
    E, H, I, k, M, fmt = c["E"], c["H"], c["I"], c["top_k"], c["M"], c["fmt"]
    done, total_s, total_bytes = 0, 0.0, 0
    for i in range(min(max_layers, len(ids_pool))):
        ids = ids_pool[i]
        used = gen.routed_unique_experts(ids, E)
        sub = gen.make_expert_weights(E, H, I, fmt, seed, device="cpu", experts=used)
        remap = {e: j for j, e in enumerate(used)}
        ids_c = [[remap.get(e, -1) for e in row] for row in ids.tolist()]
        t0 = time.perf_counter()
        oracle.forward(x_host, sub, ids_c, w_pool[i], len(used), H, I, k, fmt)
        total_s += time.perf_counter() - t0
        total_bytes += layer_bytes(ids, E, H, I, M, k, fmt)[0]
        done += 1
        if total_s >= seconds:
            break
    threads = min(oracle.num_threads(), M)  # the oracle parallelises over tokens
    return done, total_s, total_bytes, threads


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from workload import gen
    c = workload_config(args)
    seed = gen.CONFIG_SEED[args.workload]
    n = args.warmup + args.steps
    window = max(1, min(WINDOW, c["E"] // (c["top_k"] * c["M"])))
    ids_pool, w_pool = gen.draw_routing_pool(max(n, window), c["M"], c["E"], c["top_k"], seed + 29, window)
    x = gen.draw_activations(c["M"], c["H"], seed + 17)
    # warm-up layers, then the timed layers (each step = one oracle layer)
    oracle_layers(c, seed, ids_pool[:args.warmup], w_pool[:args.warmup], x, 1e9, args.warmup)
    done, secs, nbytes, threads = oracle_layers(c, seed, ids_pool[args.warmup:n], w_pool[args.warmup:n], x, 1e9,
                                                args.steps)
    gbs = nbytes / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": done, "warmup": args.warmup, "ms_per_step": secs / done * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "E": c["E"], "H": c["H"], "I": c["I"], "top_k": c["top_k"],
                   "M": c["M"], "fmt": gen.FMT_NAMES[c["fmt"]]},
        "us_per_layer": secs / done * 1e6,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{done} layers of {args.workload}, one routing draw each"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
def decode_src_sha256():
    """Hash of the decode kernels' code: a stored ncu traffic figure is used
    only while the kernels it was measured on are unchanged.  Line comments
    and blank lines are left out (they do not change the kernels)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("common.cuh", "tcgen05.cuh", "decode_tc.cu", "decode.cu"):
        text = open(os.path.join(ROOT, "fp4_weight_moe_gb300", "csrc", f)).read()
        code = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()


def decode_kernel_label(m, M, E, H, I, k):
    """What one decode layer of this shape launches (for the JSON line)."""
    c = m._capi
    if M <= m.MOE_FP4_DECODE_MAX_M and c.moe_fp4_debug_decode_family_of(M, E, H, I, k) == 1:
        return "decode layer: streaming-GEMV FC1 + FC2 (PDL-chained)"
    head = "decode layer" if M <= m.MOE_FP4_DECODE_MAX_M else \
        f"decode layer in {-(-M // m.MOE_FP4_DECODE_MAX_M)} chunks"
    return f"{head}: x pre-pass + FC1 + " + ("" if M < 2 else "h pre-pass + ") + "FC2 (tcgen05, PDL-chained)"


def run_ours(args):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import build as b
    from workload import gen
    b.build()

    c = workload_config(args)
    E, H, I, k, M, fmt = c["E"], c["H"], c["I"], c["top_k"], c["M"], c["fmt"]
    seed = gen.CONFIG_SEED[args.workload]
    K, W = args.steps, args.warmup
    window = max(1, min(WINDOW, E // (k * M)))
    weights = gen.make_expert_weights(E, H, I, fmt, seed, device=dev)
    pw = m.prepare_weights(weights, E, H, I, fmt)
    del weights
    x = gen.draw_activations(M, H, seed + 17, device=dev)
    ids_pool, w_pool = gen.draw_routing_pool(max(K, window), M, E, k, seed + 29 + 1000 * rank, window)
    ids_d = [t.to(dev) for t in ids_pool]
    w_d = [t.to(dev) for t in w_pool]
    m.reserve_workspace(M, E, H, I, k, fmt)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()

    # eager warm-up, then capture the K timed layers in one graph
    for i in range(W):
        m.forward(x, pw, ids_d[i % K], w_d[i % K], out=out)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(K):
            m.forward(x, pw, ids_d[i], w_d[i], out=out)
    torch.cuda.synchronize()
    g.replay()  # untimed: graph upload and one more warm pass
    torch.cuda.synchronize()

    per_layer_bytes = [layer_bytes(ids_pool[i], E, H, I, M, k, fmt)[0] for i in range(K)]
    step_bytes = sum(per_layer_bytes)
    # batches past the decode band that run as decode-band chunks report like the decode band
    prefill = M > m.MOE_FP4_DECODE_MAX_M and m._capi.moe_fp4_debug_decode_launches(M, E, H, I, k) == 0
    step_flops = sum(layer_flops(ids_pool[i], E, H, I) for i in range(K))

    sampler = ClockSampler(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()
    ev0.record(cur)
    g.replay()
    ev1.record(cur)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if ws > 1:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    ms_max, job_units = job_time_and_units(ms, step_flops if prefill else step_bytes, ws, dev)
    ms_per_step = ms_max / K
    value = job_units / (ms_max * 1e-3) / (1e12 if prefill else 1e9)

    e2e_value = None
    # end to end through the C ABI's host-buffer entry point, one eager call
    # per layer: H2D of x, ids and router weights, the layer, D2H of the
    # output, all enqueued by moe_fp4_forward_host on the current stream.
    xh = x.cpu().pin_memory()
    idh = [t.contiguous().pin_memory() for t in ids_pool[:K]]
    wh = [t.contiguous().pin_memory() for t in w_pool[:K]]
    outh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
    hws = m.alloc_host_workspace(M, E, H, I, k, fmt, device=dev)
    torch.cuda.synchronize()

    def e2e_step(i):
        m.forward_host(xh, pw, idh[i], wh[i], outh, hws)

    e2e_ms = float("nan")
    if not args.no_e2e:
        for i in range(W):
            e2e_step(i % K)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for i in range(K):
            e2e_step(i)
        e1.record(cur)
        torch.cuda.synchronize()
        e2e_ms, job_units = job_time_and_units(e0.elapsed_time(e1), step_flops if prefill else step_bytes, ws, dev)
        e2e_value = job_units / (e2e_ms * 1e-3) / (1e12 if prefill else 1e9)

    peak, peak_kind = load_peaks()
    achieved = (step_bytes / K) / (ms_per_step * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_e512_traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                pd = json.load(f)
            key = f"{args.workload}/M={M}/{gen.FMT_NAMES[fmt]}"
            if (args.E is None and pd.get("decode_src_sha256") == decode_src_sha256()
                    and key in pd.get("configs", {})):
                traffic = pd["configs"][key]["dram_bytes_per_layer"]
        except Exception:
            traffic = None

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp32-accum e2m1 x bf16", "data": "synthetic",
        "config": {"workload": args.workload, "E": E, "H": H, "I": I, "top_k": k, "M": M,
                   "fmt": gen.FMT_NAMES[fmt],
                   "l2": f"routing draws rotate; no expert repeats within {window} layers "
                         f"({window} x {per_layer_bytes[0] / 1e6:.1f} MB)",
                   "timing": "K layers in one CUDA graph, one replay, CUDA events"},
        "us_per_layer": ms_per_step * 1e3,
        "routed_bytes_per_layer": step_bytes / K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"hbm_gbs of {peak_kind}", "traffic": traffic,
                     "kernel": decode_kernel_label(m, M, E, H, I, k)},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": M * H * 2 + M * k * 8,
                "d2h_bytes_per_step": M * H * 2, "us_per_layer": e2e_ms * 1e3 / K},
        "gpu_launches": m._capi.moe_fp4_debug_decode_launches(M, E, H, I, k) * K,
        "clocks": clocks,
    }

    if prefill:
        # Roofline = min(FP4 tensor peak, arithmetic intensity x HBM): the
        # layer's algorithmic bytes are the routed experts' weights and
        # scales plus x read and out written once (the intermediates could
        # stay on chip).  At prefill_e128 the intensity (~870 flop/B) is below
        # the ridge (FP4 peak / HBM), so HBM bounds it; the FP4-peak view is
        # reported beside it.  FP4 peak: measured BF16 dense peak x the
        # nominal FP4/BF16 ratio (13.5 / 2.25 = 6).
        bf16, bf16_kind = load_bf16_peak()
        fp4_peak = 6.0 * bf16
        ach_tf = (step_flops / K) / (ms_per_step * 1e-3) / 1e12
        n_exp = [len(gen.routed_unique_experts(ids_pool[i], E)) for i in range(K)]
        alg_bytes = sum(n * gen.expert_bytes(H, I, fmt) + 2 * M * H * 2 for n in n_exp) / K
        ach_gbs = alg_bytes / (ms_per_step * 1e-3) / 1e9
        ai = (step_flops / K) / alg_bytes
        line["unit"] = "TFLOP/s"
        line["dtype"] = "e2m1 x e2m1 (nvfp4 activations), fp32 accumulate"
        line["config"]["l2"] = f"inputs larger than L2 (expert weights {E * gen.expert_bytes(H, I, fmt) / 1e9:.2f} GB)"
        line["flops_per_layer"] = step_flops / K
        line["algorithmic_bytes_per_layer"] = alg_bytes
        bound = "hbm" if ai * peak * 1e9 < fp4_peak * 1e12 else "tensor"
        line["roofline"] = {"bound": bound, "achieved": ach_gbs if bound == "hbm" else ach_tf,
                            "peak": peak if bound == "hbm" else fp4_peak,
                            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                            "frac": ach_gbs / peak if bound == "hbm" else ach_tf / fp4_peak,
                            "peak_source": f"hbm_gbs of {peak_kind}" if bound == "hbm"
                            else f"bf16_tflops of {bf16_kind} x 6 (nominal fp4/bf16)",
                            "traffic": None, "kernel": "prefill layer (8 launches), per layer",
                            "arithmetic_intensity_flop_per_byte": ai,
                            "ceiling_tflops": min(fp4_peak, ai * peak * 1e9 / 1e12),
                            "tensor_view": {"achieved": ach_tf, "peak": fp4_peak, "unit": "TFLOP/s",
                                            "frac": ach_tf / fp4_peak,
                                            "peak_source": f"bf16_tflops of {bf16_kind} x 6 (nominal fp4/bf16)"}}
        line["e2e"]["unit"] = "TFLOP/s"
        line["gpu_launches"] = 8 * K
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and prefill:
        # the oracle on a bounded sample: the first 4 tokens of the first draw
        import oracle
        tok = [0, 1, 2, 3]
        ids_s = ids_pool[0][tok]
        used = gen.routed_unique_experts(ids_s, E)
        sub = gen.make_expert_weights(E, H, I, fmt, seed, device="cpu", experts=used)
        remap = {e: j for j, e in enumerate(used)}
        ids_c = [[remap.get(e, -1) for e in row] for row in ids_s.tolist()]
        t1 = time.perf_counter()
        oracle.forward_prefill(x.cpu()[tok], sub, ids_c, w_pool[0][tok], len(used), H, I, k)
        secs = time.perf_counter() - t1
        fl = layer_flops(ids_s, E, H, I)
        line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": min(oracle.num_threads(), 4),
                                "kind": "oracle", "sample": f"4 tokens of {args.workload} (mirrored activation "
                                                            f"quantisation), {secs:.1f} s"}
    elif rank == 0 and ws == 1 and not args.no_cpu_baseline:
        done, secs, nbytes, threads = oracle_layers(c, seed, ids_pool, w_pool, x.cpu(), args.cpu_seconds, K)
        line["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{done} layers of {args.workload} (one routing draw each), "
                                          f"{secs:.1f} s; us/layer {secs / done * 1e6:.0f}"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
