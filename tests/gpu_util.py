"""Shared helpers of the GPU parity tests: build the library, make seeded
workloads on the device, and compare the CUDA path with the FP64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workload import gen

# Acceptance bound of the layer output against the FP64 oracle: cosine
# similarity over the flattened [M, H] output >= 0.99995 and the largest
# absolute error <= 2e-2 * RMS(oracle output), the error counted beyond the
# output's own BF16 rounding: |got - want| <= 2e-2 * RMS + ulp_bf16(want) / 2
# (a correctly rounded BF16 output already misses an FP64 value by up to
# half a BF16 unit in the last place, which exceeds 2e-2 * RMS wherever |want|
# is above about ten times the RMS).
COS_MIN = 0.99995
MAXABS_REL_RMS = 2e-2


def bf16_half_ulp(w: np.ndarray) -> np.ndarray:
    """Half a BF16 unit in the last place at each |w| (8 significant bits)."""
    a = np.abs(np.asarray(w, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)

_built = False


def ensure_built():
    global _built
    if not _built:
        from fp4_weight_moe_gb300 import build as b
        b.build()
        _built = True


def layer_metrics(got: torch.Tensor, want: np.ndarray):
    g = got.detach().float().cpu().double().numpy().reshape(-1)
    w = np.asarray(want, dtype=np.float64).reshape(-1)
    rms = float(np.sqrt(np.mean(w * w)))
    ng, nw = float(np.linalg.norm(g)), float(np.linalg.norm(w))
    cos = float(np.dot(g, w) / (ng * nw)) if ng > 0 and nw > 0 else (1.0 if ng == nw == 0 else 0.0)
    maxabs = float(np.max(np.abs(g - w))) if g.size else 0.0
    return cos, maxabs, rms


def assert_layer_close(got: torch.Tensor, want: np.ndarray, what: str = ""):
    g = got.detach().float().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    w = np.asarray(want)
    if not np.any(w):
        assert not np.any(g), f"{what}: oracle output is zero but the GPU output is not"
        return
    cos, maxabs, rms = layer_metrics(got, want)
    assert cos >= COS_MIN, f"{what}: cosine {cos:.7f} < {COS_MIN}"
    excess = float(np.max(np.abs(g.astype(np.float64) - w.reshape(g.shape)) - bf16_half_ulp(w.reshape(g.shape))))
    assert excess <= MAXABS_REL_RMS * rms, \
        f"{what}: max abs err beyond the BF16 rounding {excess:.3e} > {MAXABS_REL_RMS} * rms {rms:.3e} (raw {maxabs:.3e})"
    # zero rows of the oracle (tokens without a valid route) must be exact zeros
    zero_rows = ~np.any(w.reshape(g.shape) != 0, axis=-1)
    assert not np.any(g[zero_rows]), f"{what}: tokens without valid routes are not exactly zero"


def compact_for_oracle(weights: dict, ids: torch.Tensor, E: int, fmt: int):
    """Copy only the routed experts' bytes to the host and remap ids, so the
    oracle sees a small expert table (invalid ids stay invalid)."""
    flat = ids.reshape(-1).tolist()
    used = sorted({e for e in flat if 0 <= e < E})
    remap = {e: i for i, e in enumerate(used)}
    ids_c = np.array([[remap.get(e, -1) for e in row] for row in ids.tolist()], dtype=np.int32)
    idx = torch.tensor(used, dtype=torch.long, device=weights["w13"].device)
    sub = {}
    for k, v in weights.items():
        if v is None:
            continue
        sub[k] = v.index_select(0, idx).cpu().numpy() if len(used) else v[:0].cpu().numpy()
    if not used:  # oracle needs E >= 1; give it one unused expert
        sub = {k: v[:1].cpu().numpy() for k, v in weights.items() if v is not None}
    return sub, ids_c, max(1, len(used))


def oracle_layer(wl: gen.Workload, tokens=None):
    sub, ids_c, Ec = compact_for_oracle(wl.weights, wl.topk_ids, wl.E, wl.fmt)
    return oracle.forward(wl.x, sub, ids_c, wl.topk_weights.cpu(), Ec, wl.H, wl.I, wl.top_k, wl.fmt, tokens=tokens)
