"""Seeded synthetic workloads shaped like the pages' MoE geometries.

Everything here is input synthesis:

* float expert weights drawn from N(0, 0.02) and written out as a synthetic
  FP4 checkpoint (packed E2M1 nibbles plus block scales), the way a quantised
  model file would arrive at the layer;
* BF16 activations drawn from N(0, 1);
* top-k routing from N(0, 1) router logits (optionally with a Zipf expert
  popularity bias and with invalid expert ids injected).

The layer itself never quantises weights: the pages keep the checkpoint's
"exact FP4 nibbles and caller-owned scale buffers" and slice "native E2M1
experts ... without requantization" (b12x PR #459, "Reduce NVFP4-CSF scale
reconstruction overhead", commit notes).  So the encoder below only produces
inputs; both the CUDA path and the oracle consume the same bytes and decode
them with their own, independent code.

Checkpoint layout written here (the layer's logical input format):

* ``w13``  uint8 ``[E][2I][H/2]``: rows ``[0, I)`` are the gate projection,
  rows ``[I, 2I)`` the up projection; the low nibble of byte ``j`` holds the
  element at K index ``2j``, the high nibble the one at ``2j + 1``.
* ``s13``  uint8 ``[E][2I][H/B]``: one scale byte per (row, K-block of B).
* ``w2``   uint8 ``[E][H][I/2]`` and ``s2`` uint8 ``[E][H][I/B]`` likewise.
* NVFP4 only: ``g13`` float32 ``[E][2]`` (gate, up) and ``g2`` float32 ``[E]``:
  the per-tensor FP32 multipliers.

MXFP4: B = 32, UE8M0 scale bytes.  NVFP4: B = 16, E4M3 scale bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

MXFP4 = 0
NVFP4 = 1
FMT_NAMES = {MXFP4: "mxfp4", NVFP4: "nvfp4"}
BLOCK = {MXFP4: 32, NVFP4: 16}

# Magnitudes on the E2M1 grid, used only to write the synthetic checkpoint
# (a nearest-grid-point search).  Codes 0..7 in order.
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)

# The five workloads: geometry, format and routing recipe.
CONFIGS = {
    "tiny_decode": dict(E=8, H=256, I=128, top_k=2, M=1, fmt=MXFP4, routing="softmax"),
    "decode_e512": dict(E=512, H=2560, I=320, top_k=10, M=1, fmt=NVFP4, routing="softmax"),
    "decode_e288_m4": dict(E=288, H=4096, I=512, top_k=10, M=4, fmt=MXFP4, routing="softmax_invalid"),
    "decode_e256": dict(E=256, H=7168, I=2048, top_k=8, M=1, fmt=MXFP4, routing="zipf"),
    "prefill_e128": dict(E=128, H=4096, I=1536, top_k=8, M=4096, fmt=NVFP4, routing="softmax"),
}
CONFIG_SEED = {name: 1234 + i for i, name in enumerate(CONFIGS)}


# --------------------------------------------------------------------------
# synthetic checkpoint writer
# --------------------------------------------------------------------------
def _nearest_e2m1_code(a: torch.Tensor) -> torch.Tensor:
    """Code (0..7) of the grid point nearest to |a| (a >= 0), ties to the
    even code; values beyond 6 saturate to code 7."""
    grid = torch.tensor(_E2M1_GRID, dtype=a.dtype, device=a.device)
    mids = (grid[1:] + grid[:-1]) / 2  # 7 decision points
    above = (a.unsqueeze(-1) > mids).sum(-1)
    # at an exact midpoint between codes i and i+1 the even one wins
    odd_i = torch.arange(7, device=a.device) % 2 == 1  # i odd -> i+1 even
    tie_up = ((a.unsqueeze(-1) == mids) & odd_i).sum(-1)
    return (above + tie_up).to(torch.uint8)


def _pack_codes(sign: torch.Tensor, code: torch.Tensor) -> torch.Tensor:
    nib = code | (sign.to(torch.uint8) << 3)
    lo = nib[..., 0::2]
    hi = nib[..., 1::2]
    return lo | (hi << 4)


def encode_mxfp4(w: torch.Tensor):
    """float32 ``[..., K]`` -> (nibbles ``[..., K/2]``, UE8M0 scales ``[..., K/32]``).

    Scale per 32 K-elements is ``2^ceil(log2(amax/6))`` (an all-zero block
    gets exponent 0, i.e. byte 127), so every scaled element lies within the
    grid's range."""
    K = w.shape[-1]
    assert K % 32 == 0
    blk = w.reshape(*w.shape[:-1], K // 32, 32)
    amax = blk.abs().amax(-1).to(torch.float64)
    mant, ex = torch.frexp(amax / 6.0)
    # amax/6 = mant * 2^ex with mant in [0.5, 1): ceil(log2) = ex, or ex-1 at mant == 0.5
    e = torch.where(mant == 0.5, ex - 1, ex)
    e = torch.where(amax == 0, torch.zeros_like(e), e)
    e = e.clamp(-127, 127)
    sbyte = (e + 127).to(torch.uint8)
    scaled = blk / torch.ldexp(torch.ones_like(amax), e).to(torch.float32).unsqueeze(-1)
    code = _nearest_e2m1_code(scaled.abs())
    sign = scaled < 0
    sign = sign & (code != 0)
    return _pack_codes(sign, code).reshape(*w.shape[:-1], K // 2), sbyte.reshape(*w.shape[:-1], K // 32)


def encode_nvfp4(w: torch.Tensor):
    """float32 ``[..., K]`` (one tensor, e.g. one expert's gate projection) ->
    (nibbles ``[..., K/2]``, E4M3 scales ``[..., K/16]``, FP32 global multiplier).

    ``g = amax/(6*448)``, block scale ``s = e4m3(amax_blk/(6 g))``, element
    ``q = e2m1(x/(s g))`` saturating to 6; an all-zero block has s = 0, q = 0."""
    K = w.shape[-1]
    assert K % 16 == 0
    amax_t = w.abs().amax()
    g = (amax_t / (6.0 * 448.0)).to(torch.float32)
    if float(g) == 0.0:
        g = torch.tensor(1.0, dtype=torch.float32, device=w.device)
    blk = w.reshape(*w.shape[:-1], K // 16, 16)
    amax_b = blk.abs().amax(-1)
    s_f = (amax_b / (6.0 * g)).clamp(max=448.0)
    s8 = s_f.to(torch.float8_e4m3fn)
    s_back = s8.to(torch.float32)
    denom = (s_back * g).unsqueeze(-1)
    scaled = torch.where(denom > 0, blk / torch.where(denom > 0, denom, torch.ones_like(denom)),
                         torch.zeros_like(blk))
    code = _nearest_e2m1_code(scaled.abs())
    sign = (scaled < 0) & (code != 0)
    nib = _pack_codes(sign, code).reshape(*w.shape[:-1], K // 2)
    return nib, s8.view(torch.uint8).reshape(*w.shape[:-1], K // 16), g


def _expert_generator(seed: int, expert: int, proj: int, device) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed((seed * 1_000_003 + expert * 7919 + proj * 104_729) % (2**62))
    return gen


def make_expert_weights(E: int, H: int, I: int, fmt: int, seed: int, device="cpu", std: float = 0.02,
                        experts=None):
    """Draw and encode all experts' weights. Returns a dict of logical tensors on
    ``device``: w13, s13, w2, s2 and (NVFP4) g13, g2.

    Each expert's floats come from its own counter-seeded generator, so a
    subset of experts can be generated alone: with ``experts`` (a list of ids)
    only those are drawn, in that order, and the leading dimension is
    ``len(experts)``."""
    B = BLOCK[fmt]
    expert_ids = list(range(E)) if experts is None else list(experts)
    E = len(expert_ids)
    w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=device)
    s13 = torch.empty((E, 2 * I, H // B), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, H, I // B), dtype=torch.uint8, device=device)
    g13 = torch.ones((E, 2), dtype=torch.float32, device=device) if fmt == NVFP4 else None
    g2 = torch.ones((E,), dtype=torch.float32, device=device) if fmt == NVFP4 else None
    for e, eid in enumerate(expert_ids):
        for proj, rows, K in ((0, I, H), (1, I, H), (2, H, I)):
            gen = _expert_generator(seed, eid, proj, device)
            wf = torch.randn((rows, K), generator=gen, device=device, dtype=torch.float32) * std
            if fmt == MXFP4:
                nib, sc = encode_mxfp4(wf)
            else:
                nib, sc, g = encode_nvfp4(wf)
            if proj == 0:
                w13[e, :I], s13[e, :I] = nib, sc
                if g13 is not None:
                    g13[e, 0] = g
            elif proj == 1:
                w13[e, I:], s13[e, I:] = nib, sc
                if g13 is not None:
                    g13[e, 1] = g
            else:
                w2[e], s2[e] = nib, sc
                if g2 is not None:
                    g2[e] = g
    out = dict(w13=w13, s13=s13, w2=w2, s2=s2)
    if fmt == NVFP4:
        out.update(g13=g13, g2=g2)
    return out


def make_relu2_weights(E: int, H: int, I: int, fmt: int, seed: int, device="cpu", std: float = 0.02,
                       experts=None):
    """Non-gated (squared-ReLU) experts: w1 [E][I][H/2], s1 [E][I][H/B] from
    N(0, std) floats of their own counter-seeded stream per expert, and w2, s2
    drawn like the gated experts' down projection; NVFP4 adds g1 [E], g2 [E]."""
    B = BLOCK[fmt]
    expert_ids = list(range(E)) if experts is None else list(experts)
    E = len(expert_ids)
    w1 = torch.empty((E, I, H // 2), dtype=torch.uint8, device=device)
    s1 = torch.empty((E, I, H // B), dtype=torch.uint8, device=device)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=device)
    s2 = torch.empty((E, H, I // B), dtype=torch.uint8, device=device)
    g1 = torch.ones((E,), dtype=torch.float32, device=device) if fmt == NVFP4 else None
    g2 = torch.ones((E,), dtype=torch.float32, device=device) if fmt == NVFP4 else None
    for e, eid in enumerate(expert_ids):
        for proj, rows, K in ((3, I, H), (2, H, I)):
            gen = _expert_generator(seed, eid, proj, device)
            wf = torch.randn((rows, K), generator=gen, device=device, dtype=torch.float32) * std
            if fmt == MXFP4:
                nib, sc = encode_mxfp4(wf)
                g = None
            else:
                nib, sc, g = encode_nvfp4(wf)
            if proj == 3:
                w1[e], s1[e] = nib, sc
                if g1 is not None:
                    g1[e] = g
            else:
                w2[e], s2[e] = nib, sc
                if g2 is not None:
                    g2[e] = g
    out = dict(w1=w1, s1=s1, w2=w2, s2=s2)
    if fmt == NVFP4:
        out.update(g1=g1, g2=g2)
    return out


# --------------------------------------------------------------------------
# activations and routing
# --------------------------------------------------------------------------
def draw_activations(M: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """BF16 activations N(0, 1), shape [M, H]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, H), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).to(device)


def _softmax_topk(logits: np.ndarray, top_k: int):
    z = logits - logits.max(-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(-1, keepdims=True)
    # highest probabilities first; ties go to the lower expert index (stable sort)
    order = np.argsort(-p, axis=-1, kind="stable")[:, :top_k]
    pk = np.take_along_axis(p, order, -1)
    wk = pk / pk.sum(-1, keepdims=True)
    return order.astype(np.int32), wk.astype(np.float32)


def draw_routing(M: int, E: int, top_k: int, seed: int, mode: str = "softmax", n_invalid: Optional[int] = None):
    """Router output: (topk_ids int32 [M, top_k], topk_weights float32 [M, top_k]).

    modes:
      ``softmax``          N(0,1) logits -> softmax -> top-k (distinct experts), renormalised
      ``zipf``             as softmax, plus a Zipf(1.1) popularity bias -1.1*ln(rank_e),
                           rank a seeded permutation of 1..E
      ``softmax_invalid``  as softmax, then round(5%) of the M*top_k slots are made invalid:
                           the first gets id -1, the next id E, alternating; weights kept
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    logits = rng.standard_normal((M, E))
    if mode == "zipf":
        rank = rng.permutation(E) + 1
        logits = logits + (-1.1 * np.log(rank))[None, :]
    ids, w = _softmax_topk(logits, top_k)
    if mode == "softmax_invalid" or n_invalid:
        n = n_invalid if n_invalid is not None else int(round(0.05 * M * top_k))
        slots = rng.choice(M * top_k, size=n, replace=False)
        flat = ids.reshape(-1)
        for i, s in enumerate(sorted(slots)):
            flat[s] = -1 if i % 2 == 0 else E
    return torch.from_numpy(ids), torch.from_numpy(w)


def draw_routing_pool(n_draws: int, M: int, E: int, top_k: int, seed: int, window: int):
    """``n_draws`` routings for a timing loop, drawn like ``draw_routing`` in
    softmax mode except that no expert appears in two draws closer than
    ``window`` positions apart, cyclically (draw i and draw (i + d) mod n for
    0 < d < window share no expert; the excluded experts get logit -inf
    before the top-k).  Replaying the sequence in a loop, the bytes touched by
    any ``window`` consecutive layers then exceed the L2 cache, so every timed
    layer streams its experts from HBM."""
    assert window <= 1 or window * top_k * M <= E, "window too large for E"
    assert n_draws >= 1
    rng = np.random.Generator(np.random.PCG64(seed))
    sets = [None] * n_draws
    ids_all, w_all = [None] * n_draws, [None] * n_draws
    for i in range(n_draws):
        logits = rng.standard_normal((M, E))
        banned = set()
        for d in range(1, min(window, n_draws)):
            for j in ((i - d) % n_draws, (i + d) % n_draws):
                if sets[j] is not None and j != i:
                    banned.update(sets[j])
        if banned:
            logits[:, sorted(banned)] = -np.inf
        ids, w = _softmax_topk(logits, top_k)
        sets[i] = set(ids.reshape(-1).tolist())
        ids_all[i] = torch.from_numpy(ids)
        w_all[i] = torch.from_numpy(w)
    return ids_all, w_all


# --------------------------------------------------------------------------
# a whole workload
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    name: str
    E: int
    H: int
    I: int
    top_k: int
    M: int
    fmt: int
    seed: int
    weights: dict
    x: torch.Tensor
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor

    @property
    def block(self) -> int:
        return BLOCK[self.fmt]


def make_workload(name: str, device="cpu", M: Optional[int] = None, fmt: Optional[int] = None,
                  E: Optional[int] = None, H: Optional[int] = None, I: Optional[int] = None,
                  top_k: Optional[int] = None, routing: Optional[str] = None,
                  seed: Optional[int] = None) -> Workload:
    """Build a named workload (see ``CONFIGS``); any field may be overridden,
    e.g. ``M`` for the decode sweep or a smaller ``E`` for a quick test."""
    c = dict(CONFIGS[name])
    for k, v in dict(M=M, fmt=fmt, E=E, H=H, I=I, top_k=top_k, routing=routing).items():
        if v is not None:
            c[k] = v
    s = CONFIG_SEED[name] if seed is None else seed
    weights = make_expert_weights(c["E"], c["H"], c["I"], c["fmt"], s, device=device)
    x = draw_activations(c["M"], c["H"], s + 17, device=device)
    ids, w = draw_routing(c["M"], c["E"], c["top_k"], s + 29, mode=c["routing"])
    return Workload(name=name, E=c["E"], H=c["H"], I=c["I"], top_k=c["top_k"], M=c["M"], fmt=c["fmt"],
                    seed=s, weights=weights, x=x, topk_ids=ids.to(device), topk_weights=w.to(device))


def routed_unique_experts(topk_ids: torch.Tensor, E: int) -> list:
    ids = topk_ids.reshape(-1).tolist()
    return sorted({e for e in ids if 0 <= e < E})


def expert_bytes(H: int, I: int, fmt: int) -> int:
    """Weight + scale bytes of one expert (and its FP32 multipliers for NVFP4)."""
    B = BLOCK[fmt]
    nib = (2 * I * H + H * I) // 2
    sc = 3 * I * H // B
    return nib + sc + (12 if fmt == NVFP4 else 0)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [
    "MXFP4", "NVFP4", "FMT_NAMES", "BLOCK", "CONFIGS", "CONFIG_SEED", "Workload", "make_workload",
    "make_expert_weights", "make_relu2_weights", "encode_mxfp4", "encode_nvfp4", "draw_activations", "draw_routing",
    "draw_routing_pool", "routed_unique_experts", "expert_bytes", "ceil_div", "math",
]
