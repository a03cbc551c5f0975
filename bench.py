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
# decode-band kernel plans of moe_fp4_debug_set_decode_family
DECODE_PLANS = {"auto": 0, "gemv": 1, "chain": 2, "single": 3}
MID_BANDS = {"auto": 0, "prefill": 1, "chunks": 2, "mid": 3}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-sweep", action="store_true", help="time the headline workload only")
    ap.add_argument("--min-timed-s", type=float, default=0.6,
                    help="device time of the headline's timed replays (at least 15 replays); sweep entries a quarter")
    ap.add_argument("--workload", default=WORKLOAD, help="workload name (default: the decode_e512 headline)")
    ap.add_argument("--M", type=int, default=None, help="override the token count")
    ap.add_argument("--E", type=int, default=None, help="override the expert count (profiling on smaller memory)")
    ap.add_argument("--fmt", choices=["mxfp4", "nvfp4"], default=None)
    ap.add_argument("--prefill-mode", choices=["nvfp4", "bf16", "w4a8"], default="nvfp4",
                    help="prefill-band activation precision of the headline (bf16: the exact band; w4a8: MXFP8 "
                         "activations, MXFP4 weights)")
    ap.add_argument("--decode-plan", choices=list(DECODE_PLANS), default="auto",
                    help="decode-band kernel plan (auto: by shape)")
    ap.add_argument("--mid-band", choices=list(MID_BANDS), default="auto",
                    help="kernels of batches past 8 tokens (auto: by shape; prefill: the prefill band's GEMMs; "
                         "chunks: decode kernels on chunks of 8; mid: the mid band's swapped GEMMs)")
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
    """nvidia-smi clock / throttle sampling during the timed regions: start()
    before a timed region, pause() after it; stop() summarises every sample
    taken."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.available = True

    def start(self):
        if self.proc is not None or not self.available:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, args=(self.proc,), daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
            self.available = False

    def _read(self, proc):
        for line in proc.stdout:
            self.lines.append(line.strip())

    def pause(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        self.proc = None

    def stop(self):
        self.pause()
        if not self.available:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
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
def oracle_layers(c, seed, ids_pool, w_pool, x_host, seconds, max_layers, threads=0):
    """Time the FP64 oracle on successive routing draws (bounded sample), on
    `threads` OpenMP threads (0: the affinity cores)."""
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
        oracle.forward(x_host, sub, ids_c, w_pool[i], len(used), H, I, k, fmt, nthreads=threads)
        total_s += time.perf_counter() - t0
        total_bytes += layer_bytes(ids, E, H, I, M, k, fmt)[0]
        done += 1
        if total_s >= seconds:
            break
    # the oracle spreads each layer over (token, slot, row) and (token, output row)
    return done, total_s, total_bytes, threads if threads > 0 else affinity_cores()


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
def _src_sha256(files):
    import hashlib
    import re
    h = hashlib.sha256()
    for f in files:
        text = open(os.path.join(ROOT, "fp4_weight_moe_gb300", "csrc", f)).read()
        code = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in text.splitlines()]
        h.update("\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()


def decode_src_sha256():
    """Hash of the decode kernels' code: a stored ncu traffic figure is used
    only while the kernels it was measured on are unchanged.  Line comments
    and blank lines are left out (they do not change the kernels)."""
    return _src_sha256(("common.cuh", "tcgen05.cuh", "decode_tc.cu", "decode.cu"))


def decode_kernel_label(m, M, E, H, I, k):
    """What one decode layer of this shape launches (for the JSON line)."""
    c = m._capi
    fam = c.moe_fp4_debug_decode_family_of(M, E, H, I, k) if M <= m.MOE_FP4_DECODE_MAX_M else 0
    if fam == 1:
        return "decode layer: streaming-GEMV FC1 + FC2 (PDL-chained)"
    if fam == 3:
        return "decode layer: one tcgen05 launch (FC1, h handed over by flags, FC2)"
    head = "decode layer" if M <= m.MOE_FP4_DECODE_MAX_M else \
        f"decode layer in {-(-M // m.MOE_FP4_DECODE_MAX_M)} chunks"
    return f"{head}: x pre-pass + FC1 + " + ("" if M < 2 else "h pre-pass + ") + "FC2 (tcgen05, PDL-chained)"


COS_MIN, MAXABS_REL_RMS = 0.99995, 2e-2  # the parity bound of the layer output against the FP64 oracle

# The sweep: every workload configuration beside the headline, each checked
# against the oracle before it is timed.  (label, workload, overrides)
SWEEP = [("C0", "tiny_decode", {}),
         ("C1/M=8", "decode_e512", dict(M=8)),
         # the C1 expert shape past the decode band: the mid band's GEMMs
         ("C1/M=64", "decode_e512", dict(M=64)),
         ("C2", "decode_e288_m4", {})] + \
    [(f"C3/M={M}/{f}", "decode_e256", dict(M=M, fmt=fmt)) for fmt, f in ((0, "mxfp4"), (1, "nvfp4"))
     for M in (1, 2, 4, 8)] + \
    [("C4", "prefill_e128", {}), ("C4/bf16-exact", "prefill_e128", dict(prefill_mode=1)),
     ("C4/w4a8-mx", "prefill_e128", dict(prefill_mode=2, fmt=0))]


def affinity_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:  # pragma: no cover
        return os.cpu_count() or 1


def parity_metrics(got, want):
    """(cosine, max |got - want| / RMS(want), the same beyond the output's own
    BF16 rounding (half a BF16 ulp of want), zero rows exact) over the
    flattened output; ok when cosine >= 0.99995 and the error beyond the
    BF16 rounding is <= 2e-2 RMS."""
    import numpy as np
    g = np.asarray(got, np.float64).reshape(-1)
    w = np.asarray(want, np.float64).reshape(-1)
    rms = float(np.sqrt(np.mean(w * w)))
    ng, nw = float(np.linalg.norm(g)), float(np.linalg.norm(w))
    cos = float(np.dot(g, w) / (ng * nw)) if ng > 0 and nw > 0 else (1.0 if ng == nw == 0 else 0.0)
    aw = np.abs(w)
    half_ulp = np.where(aw > 0, np.ldexp(1.0, (np.floor(np.log2(np.where(aw > 0, aw, 1.0))) - 8).astype(np.int64)),
                        0.0)
    err = float(np.max(np.abs(g - w))) / rms if rms > 0 else float(np.max(np.abs(g)))
    excess = float(np.max(np.abs(g - w) - half_ulp)) / rms if rms > 0 else err
    rows_w = np.asarray(want).reshape(np.asarray(got).shape)
    zero_rows = ~np.any(rows_w != 0, axis=-1)
    zero_ok = not np.any(np.asarray(got)[zero_rows])
    ok = bool(np.all(np.isfinite(g))) and zero_ok and (rms == 0 or (cos >= COS_MIN and excess <= MAXABS_REL_RMS))
    return {"cos": cos, "maxabs_over_rms": err, "maxabs_beyond_bf16_rounding_over_rms": excess,
            "zero_rows_exact": zero_ok, "ok": ok}


def oracle_check(m, gen, weights, c, x, ids, tw, got, prefill, threads, mode=0):
    """The layer of one routing draw on the FP64 oracle (routed experts only;
    the prefill band on a spread of 16 tokens: against the definition of its
    activation precision, the NVFP4 mirror (mode 0), the plain layer (mode 1,
    exact BF16) or the W4A8-MX mirror (mode 2)) against the GPU output of the
    same draw."""
    exact = mode != 0
    import numpy as np
    import oracle
    import torch
    E, H, I, k, M, fmt = c["E"], c["H"], c["I"], c["top_k"], c["M"], c["fmt"]
    tokens = None
    if prefill:
        tokens = sorted(set(int(t) for t in np.linspace(0, M - 1, 16)))
        ids_used = ids[tokens]
    else:
        ids_used = ids
    used = gen.routed_unique_experts(ids_used, E)
    remap = {e: j for j, e in enumerate(used)}
    ids_c = np.array([[remap.get(e, -1) for e in row] for row in ids.tolist()], dtype=np.int32)
    idx = torch.tensor(used if used else [0], dtype=torch.long, device=weights["w13"].device)
    sub = {kk: v.index_select(0, idx).cpu() for kk, v in weights.items() if v is not None}
    t0 = time.perf_counter()
    if prefill and not exact:
        want = oracle.forward_prefill(x.cpu(), sub, ids_c, tw.cpu(), max(1, len(used)), H, I, k, tokens=tokens,
                                      nthreads=threads, fmt=fmt)[0]
        got_rows = got.float().cpu().double().numpy()[tokens]
    elif prefill and mode == 2:
        want = oracle.forward_w4a8(x.cpu()[tokens], sub, ids_c[tokens], tw.cpu()[tokens], max(1, len(used)), H, I, k,
                                   nthreads=threads)
        got_rows = got.float().cpu().double().numpy()[tokens]
    elif prefill:
        want = oracle.forward(x.cpu()[tokens], sub, ids_c[tokens], tw.cpu()[tokens], max(1, len(used)), H, I, k, fmt,
                              nthreads=threads)
        got_rows = got.float().cpu().double().numpy()[tokens]
    else:
        want = oracle.forward(x.cpu(), sub, ids_c, tw.cpu(), max(1, len(used)), H, I, k, fmt, nthreads=threads)
        got_rows = got.float().cpu().double().numpy()
    secs = time.perf_counter() - t0
    r = parity_metrics(got_rows, want)
    r["oracle_s"] = secs
    r["checked"] = (f"{len(tokens)} sampled tokens ({'W4A8-MX mirror' if mode == 2 else 'plain definition'})"
                    if exact else
                    f"{len(tokens)} sampled tokens (mirrored activation quantisation)") if prefill else \
        f"all {M} tokens"
    return r


def measure(m, name, ov, K, W, dev, rank, ws_world, min_timed_s, threads, do_e2e, sampler):
    """One workload: draw it, check it against the oracle, then time K layers
    in a CUDA graph replayed R >= 15 times (and at least min_timed_s of device
    time), each replay between CUDA events; and, end to end, K calls of the
    host-buffer entry point.  Returns a dict (or the parity failure)."""
    import statistics as st
    import torch
    from workload import gen
    c = dict(gen.CONFIGS[name])
    c.update({kk: v for kk, v in ov.items() if v is not None})
    E, H, I, k, M, fmt = c["E"], c["H"], c["I"], c["top_k"], c["M"], c["fmt"]
    mode = int(c.get("prefill_mode", 0))  # 1: the exact BF16 prefill band
    seed = gen.CONFIG_SEED[name]
    window = max(1, min(WINDOW, E // (k * M)))
    weights = gen.make_expert_weights(E, H, I, fmt, seed, device=dev)
    pw = m.prepare_weights(weights, E, H, I, fmt)
    x = gen.draw_activations(M, H, seed + 17, device=dev)
    ids_pool, w_pool = gen.draw_routing_pool(max(K, window), M, E, k, seed + 29 + 1000 * rank, window)
    ids_d = [t.to(dev) for t in ids_pool]
    w_d = [t.to(dev) for t in w_pool]
    ws = m.alloc_workspace_mode(M, E, H, I, k, fmt, mode, device=dev)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device=dev)
    decode = M <= m.MOE_FP4_DECODE_MAX_M or (mode == 0 and m._capi.moe_fp4_debug_decode_launches(M, E, H, I, k) > 0)
    prefill = not decode
    exact = prefill and mode in (1, 2)  # the 16-bit bands (exact BF16, W4A8-MX)

    def layer(i):
        if mode:
            m.forward_mode(x, pw, ids_d[i], w_d[i], ws, mode, out=out)
        else:
            m.forward(x, pw, ids_d[i], w_d[i], out=out, workspace=ws)

    res = {"workload": name, "E": E, "H": H, "I": I, "top_k": k, "M": M, "fmt": gen.FMT_NAMES[fmt]}
    if exact:
        res["prefill_mode"] = "bf16-exact" if mode == 1 else "w4a8-mx"
        # W4A8-MX runs on the FP8 tensor cores where I % 128 == 0
        res["engine"] = "fp8" if mode == 2 and I % 128 == 0 else "16-bit"
    # correctness first: one layer against the oracle, and a clean status word
    layer(0)
    torch.cuda.synchronize()
    res["parity"] = oracle_check(m, gen, weights, c, x, ids_pool[0], w_pool[0], out, prefill, threads,
                                 mode if exact else 0)
    res["parity"]["status_word"] = m.workspace_status(ws)
    del weights
    if not res["parity"]["ok"] or res["parity"]["status_word"] != 0:
        res["timed"] = False
        res["_state"] = (c, seed, ids_pool, w_pool, x)
        return res
    # batches of at most 8192 routing entries route in one kernel, larger in three
    route_launches = 1 if M * k <= 8192 else 3
    mid = prefill and not exact and m._capi.moe_fp4_debug_mid_band_of(M, E, H, I, k) == 3
    per_layer_bytes = [layer_bytes(ids_pool[i], E, H, I, M, k, fmt)[0] for i in range(K)]
    step_flops = sum(layer_flops(ids_pool[i], E, H, I) for i in range(K))
    for i in range(W):
        layer(i % K)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(K):
            layer(i)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    g.replay()
    e1.record(cur)
    torch.cuda.synchronize()
    R = max(15, int(min_timed_s * 1e3 / max(e0.elapsed_time(e1), 1e-3)) + 1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    if ws_world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    for a, b in evs:
        a.record(cur)
        g.replay()
        b.record(cur)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.pause()
    if ws_world > 1:
        import torch.distributed as dist
        dist.barrier()
    times = [a.elapsed_time(b) for a, b in evs]
    med = st.median(times)
    ms_max, job_units = job_time_and_units(med, step_flops if prefill else sum(per_layer_bytes), ws_world, dev)
    res.update({"timed": True, "replays": R, "layers_per_replay": K,
                "us_per_layer": ms_max * 1e3 / K, "us_per_layer_min": min(times) * 1e3 / K,
                "us_per_layer_max": max(times) * 1e3 / K, "routed_bytes_per_layer": sum(per_layer_bytes) / K,
                "flops_per_layer": step_flops / K, "job_units": job_units, "ms_per_replay": ms_max,
                "launches_per_layer": m._capi.moe_fp4_debug_decode_launches(M, E, H, I, k) if decode else
                route_launches + (4 if res.get("engine") == "fp8" else 5),
                "plan": decode_kernel_label(m, M, E, H, I, k) if decode else
                ("W4A8-MX prefill layer: route, x to MXFP8 per routed row, FC1 and FC2 on tcgen05 kind::mxf8f6f4 "
                 "(E4M3 x E2M1 as stored, h to MXFP8 in FC1's epilogue), cast"
                 if res.get("engine") == "fp8" else
                 "16-bit prefill layer: route, x staged in row-scaled FP16 per routed row, FC1 GEMM, h rescaled to "
                 "FP16, FC2 GEMM (FP16 tensor cores, FP4 weights decoded to FP16 in shared memory), cast"
                 if exact else
                 "mid-band layer: route (32-row routing tiles), x quantiser, FC1 and FC2 GEMMs with the weights on "
                 "the MMA's 128-row side and the routed rows on N, h quantiser, cast"
                 if mid else
                 "prefill layer: route, x quantiser, FC1 GEMM, h quantiser, FC2 GEMM, cast")
                + f" ({route_launches} routing launch{'es' if route_launches > 1 else ''})",
                "window": window, "prefill": prefill})
    if do_e2e and not exact:
        # end to end through the host-buffer entry point, one eager call per
        # layer: H2D of x, ids and router weights, the layer, D2H of the output
        xh = x.cpu().pin_memory()
        idh = [t.contiguous().pin_memory() for t in ids_pool[:K]]
        wh = [t.contiguous().pin_memory() for t in w_pool[:K]]
        outh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
        hws = m.alloc_host_workspace(M, E, H, I, k, fmt, device=dev)
        torch.cuda.synchronize()
        for i in range(W):
            m.forward_host(xh, pw, idh[i % K], wh[i % K], outh, hws)
        torch.cuda.synchronize()
        if ws_world > 1:
            import torch.distributed as dist
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for i in range(K):
            m.forward_host(xh, pw, idh[i], wh[i], outh, hws)
        b.record(cur)
        torch.cuda.synchronize()
        e2e_ms, units = job_time_and_units(a.elapsed_time(b), step_flops if prefill else sum(per_layer_bytes),
                                           ws_world, dev)
        res["e2e"] = {"value": units / (e2e_ms * 1e-3) / (1e12 if prefill else 1e9),
                      "unit": "TFLOP/s" if prefill else "GB/s", "h2d_bytes_per_step": M * H * 2 + M * k * 8,
                      "d2h_bytes_per_step": M * H * 2, "us_per_layer": e2e_ms * 1e3 / K}
        res["e2e_status_word"] = m.workspace_status(hws)
        del hws
    res["_state"] = (c, seed, ids_pool, w_pool, x)
    del pw, ws, g
    torch.cuda.empty_cache()
    return res


def roofline_of(res, peak, peak_kind, traffic):
    """The roofline object of one measured workload (decode: HBM on routed
    bytes; prefill: min(FP4 peak, intensity x HBM) with the tensor view)."""
    us = res["us_per_layer"]
    if not res["prefill"]:
        ach = res["routed_bytes_per_layer"] / (us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "peak_source": f"hbm_gbs of {peak_kind}", "traffic": traffic, "kernel": res["plan"]}
    from workload import gen
    bf16, bf16_kind = load_bf16_peak()
    exact = res.get("prefill_mode") in ("bf16-exact", "w4a8-mx")  # 16-bit or FP8 tensor cores
    fp8 = res.get("engine") == "fp8"
    fp4_peak = (2.0 * bf16 if fp8 else bf16) if exact else 6.0 * bf16
    c = res["_state"][0]
    E, H, I, M, fmt = c["E"], c["H"], c["I"], c["M"], c["fmt"]
    ids_pool = res["_state"][2]
    K = res["layers_per_replay"]
    n_exp = [len(gen.routed_unique_experts(ids_pool[i], E)) for i in range(K)]
    alg_bytes = sum(n * gen.expert_bytes(H, I, fmt) + 2 * M * H * 2 for n in n_exp) / K
    ach_tf = res["flops_per_layer"] / (us * 1e-6) / 1e12
    ach_gbs = alg_bytes / (us * 1e-6) / 1e9
    ai = res["flops_per_layer"] / alg_bytes
    bound = "hbm" if ai * peak * 1e9 < fp4_peak * 1e12 else "tensor"
    return {"bound": bound, "achieved": ach_gbs if bound == "hbm" else ach_tf,
            "peak": peak if bound == "hbm" else fp4_peak, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": ach_gbs / peak if bound == "hbm" else ach_tf / fp4_peak,
            "peak_source": f"hbm_gbs of {peak_kind}" if bound == "hbm"
            else (f"bf16_tflops of {bf16_kind} x 2 (nominal fp8/bf16)" if fp8 else f"bf16_tflops of {bf16_kind}"
                  if exact else f"bf16_tflops of {bf16_kind} x 6 (nominal fp4/bf16)"),
            "traffic": traffic, "kernel": res["plan"], "algorithmic_bytes_per_layer": alg_bytes,
            "arithmetic_intensity_flop_per_byte": ai, "ceiling_tflops": min(fp4_peak, ai * peak * 1e9 / 1e12),
            "tflops": ach_tf,
            "tensor_view": {"achieved": ach_tf, "peak": fp4_peak, "unit": "TFLOP/s", "frac": ach_tf / fp4_peak,
                            "peak_source": f"bf16_tflops of {bf16_kind} x 2 (nominal fp8/bf16)" if fp8 else
                            f"bf16_tflops of {bf16_kind}" if exact else
                            f"bf16_tflops of {bf16_kind} x 6 (nominal fp4/bf16)"}}


def prefill_src_sha256():
    """Hash of the prefill kernels' code (line comments and blank lines left
    out), the key of the stored prefill traffic figures."""
    return _src_sha256(("common.cuh", "tcgen05.cuh", "gemm_fp4.cuh", "gemm_f16w4.cuh", "gemm_mxf8.cuh", "prefill.cu"))


def stored_traffic(args_workload, M, fmt_name, E_override, prefill_mode=None):
    """Per-layer DRAM bytes from a stored ncu capture of this workload, or None
    when there is none or the kernels changed since (decode and prefill keep
    separate files keyed on their sources' code)."""
    name, key_src = (("prefill_e128_traffic.json", prefill_src_sha256) if prefill_mode is not None else
                     ("decode_e512_traffic.json", decode_src_sha256))
    prof = os.path.join(ROOT, "profiles", name)
    if E_override is not None or not os.path.exists(prof):
        return None
    try:
        with open(prof) as f:
            pd = json.load(f)
        key = f"{args_workload}/M={M}/{fmt_name}" + (f"/{prefill_mode}" if prefill_mode is not None else "")
        if pd.get("src_sha256", pd.get("decode_src_sha256")) == key_src() and key in pd.get("configs", {}):
            return pd["configs"][key]["dram_bytes_per_layer"]
    except Exception:
        return None
    return None


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
    m._capi.moe_fp4_debug_set_decode_family(DECODE_PLANS[args.decode_plan])
    m._capi.moe_fp4_debug_set_mid_band(MID_BANDS[args.mid_band])
    threads = affinity_cores()
    K, W = args.steps, args.warmup
    sampler = ClockSampler(local)
    ov = {"M": args.M, "E": args.E, "fmt": None if args.fmt is None else (0 if args.fmt == "mxfp4" else 1),
          "prefill_mode": {"bf16": 1, "w4a8": 2}.get(args.prefill_mode)}
    head = measure(m, args.workload, ov, K, W, dev, rank, ws, args.min_timed_s, threads, not args.no_e2e, sampler)
    c, seed, ids_pool, w_pool, x = head.pop("_state")
    E, H, I, k, M, fmt = c["E"], c["H"], c["I"], c["top_k"], c["M"], c["fmt"]
    peak, peak_kind = load_peaks()
    line = {"metric": METRIC, "n_gpus": ws, "steps": K, "warmup": W, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32-accum e2m1 x bf16", "data": "synthetic",
            "config": {"workload": args.workload, "E": E, "H": H, "I": I, "top_k": k, "M": M,
                       "fmt": gen.FMT_NAMES[fmt],
                       "l2": f"routing draws rotate; no expert repeats within {head.get('window')} layers "
                             f"({head.get('window')} x {head.get('routed_bytes_per_layer', 0) / 1e6:.1f} MB)",
                       "timing": "K layers in one CUDA graph, replayed R times between CUDA events; "
                                 "median replay (min/max beside it)"},
            "parity": head["parity"]}
    if not head["timed"]:
        line.update({"value": None, "unit": "GB/s", "ms_per_step": None,
                     "error": "the oracle check failed: not timed"})
    else:
        prefill = head["prefill"]
        head["_state"] = (c, seed, ids_pool, w_pool, x)
        traffic = stored_traffic(args.workload, M, gen.FMT_NAMES[fmt], args.E,
                                 head.get("prefill_mode", "nvfp4") if prefill else None)
        rl = roofline_of(head, peak, peak_kind, traffic)
        head.pop("_state")
        line.update({"value": head["job_units"] / (head["ms_per_replay"] * 1e-3) / (1e12 if prefill else 1e9),
                     "unit": "TFLOP/s" if prefill else "GB/s", "ms_per_step": head["ms_per_replay"] / K,
                     "us_per_layer": head["us_per_layer"], "us_per_layer_min": head["us_per_layer_min"],
                     "us_per_layer_max": head["us_per_layer_max"], "replays": head["replays"],
                     "routed_bytes_per_layer": head["routed_bytes_per_layer"], "roofline": rl,
                     "e2e": head.get("e2e"),
                     "gpu_launches": head["launches_per_layer"] * K * head["replays"]})
        if prefill:
            line["dtype"] = {"bf16-exact": "bf16 activations as row-scaled fp16 x (e2m1 decoded to fp16), fp32 "
                                           "accumulate",
                             "w4a8-mx": "e4m3 x e2m1 with ue8m0 scales (mxfp8 activations), fp32 accumulate"
                             if head.get("engine") == "fp8" else
                             "mxfp8 activations as row-scaled fp16 x (e2m1 decoded to fp16), fp32 "
                             "accumulate"}.get(head.get("prefill_mode"),
                                               "e2m1 x e2m1 (nvfp4 activations), fp32 accumulate")
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and head["timed"] and not head["prefill"]:
        done, secs, nbytes, used_threads = oracle_layers(c, seed, ids_pool, w_pool, x.cpu(), args.cpu_seconds, K,
                                                         threads)
        d1, s1, b1, _ = oracle_layers(c, seed, ids_pool, w_pool, x.cpu(), 0.0, 1, 1)
        line["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": used_threads,
                                "kind": "oracle",
                                "sample": f"{done} layers of {args.workload} (one routing draw each), {secs:.2f} s "
                                          f"on {used_threads} threads; us/layer {secs / done * 1e6:.0f}",
                                "single_thread": {"value": b1 / s1 / 1e9, "unit": "GB/s", "cores": 1,
                                                  "us_per_layer": s1 / d1 * 1e6}}
    if not args.no_sweep:
        sweep = []
        for label, name, sov in SWEEP:
            if name == args.workload and all(sov.get(kk, c[kk]) == c[kk] for kk in ("M", "fmt")) \
                    and not sov.get("prefill_mode") and args.E is None:
                continue  # the headline itself
            try:
                r = measure(m, name, sov, K, W, dev, rank, ws, args.min_timed_s / 4, threads, not args.no_e2e,
                            sampler)
            except Exception as exc:  # report, keep going
                sweep.append({"config": label, "workload": name, "error": repr(exc)[:300]})
                torch.cuda.empty_cache()
                continue
            ent = {"config": label}
            if r["timed"]:
                tr = stored_traffic(name, r["M"], r["fmt"], None, r.get("prefill_mode", "nvfp4") if r["prefill"] else None)
                r["roofline"] = roofline_of(r, peak, peak_kind, tr)
            r.pop("_state", None)
            r.pop("job_units", None)
            ent.update(r)
            sweep.append(ent)
        line["sweep"] = sweep
    line["clocks"] = sampler.stop()
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
