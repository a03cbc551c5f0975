"""FP64 CPU oracle for the fused FP4-weight MoE layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product (the CUDA
library and its binding) never imports this package, and this package never
imports the product.

The arithmetic lives in ``moe_oracle.c`` (plain C, FP64); this module builds it
with gcc and wraps it with ctypes, converting torch/numpy arrays to pointers.
Pins that tie it to the pages and to mathematics live in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

MXFP4 = 0
NVFP4 = 1


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP, no fast-math, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math", "-ffp-contract=off",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        _lib = _bind(ctypes.CDLL(build()))
        return _lib


class using_library:
    """Context manager: route every call of this module through another build
    of the oracle source (used by the mutation tests, which compile
    deliberately broken copies and check that the pins reject them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _bind(lib):
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.moe_oracle_e2m1.restype = ctypes.c_double
    lib.moe_oracle_e2m1.argtypes = [ctypes.c_uint]
    lib.moe_oracle_ue8m0.restype = ctypes.c_double
    lib.moe_oracle_ue8m0.argtypes = [ctypes.c_uint]
    lib.moe_oracle_e4m3.restype = ctypes.c_double
    lib.moe_oracle_e4m3.argtypes = [ctypes.c_uint]
    lib.moe_oracle_e4m3_round.restype = ctypes.c_uint8
    lib.moe_oracle_e4m3_round.argtypes = [ctypes.c_float]
    lib.moe_oracle_e2m1_round.restype = ctypes.c_uint8
    lib.moe_oracle_e2m1_round.argtypes = [ctypes.c_float]
    lib.moe_oracle_dequant.restype = None
    lib.moe_oracle_dequant.argtypes = [P, P, i, i, i, ctypes.c_double, P]
    lib.moe_oracle_forward.restype = i
    lib.moe_oracle_forward.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, i]
    lib.moe_oracle_forward_prefill.restype = i
    lib.moe_oracle_forward_prefill.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, P, P, P, i]
    d = ctypes.c_double
    lib.moe_oracle_forward_act.restype = i
    lib.moe_oracle_forward_act.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, i, i, d, d, d]
    lib.moe_oracle_forward_prefill_act.restype = i
    lib.moe_oracle_forward_prefill_act.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, P, P, P, i,
                                                   i, d, d, d]
    lib.moe_oracle_fc1.restype = i
    lib.moe_oracle_fc1.argtypes = [P, P, P, P, i, i, i, i, P, P]
    lib.moe_oracle_quant_nvfp4_row.restype = None
    lib.moe_oracle_quant_nvfp4_row.argtypes = [P, i, P, P, P]
    lib.moe_oracle_quant_mxfp8_row.restype = None
    lib.moe_oracle_quant_mxfp8_row.argtypes = [P, i, P, P]
    lib.moe_oracle_forward_w4a8_act.restype = i
    lib.moe_oracle_forward_w4a8_act.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, P, i, P, i, i, d, d, d]
    lib.moe_oracle_forward_relu2.restype = i
    lib.moe_oracle_forward_relu2.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, i]
    lib.moe_oracle_forward_prefill_relu2.restype = i
    lib.moe_oracle_forward_prefill_relu2.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, P, i, P, i]
    lib.moe_oracle_route.restype = i
    lib.moe_oracle_route.argtypes = [P, i, i, i, P, P]
    lib.moe_oracle_num_threads.restype = i
    lib.moe_oracle_num_threads.argtypes = []
    return lib


# ---------------------------------------------------------------- helpers
def _np(a, dtype):
    """torch tensor / numpy array -> C-contiguous numpy array of dtype."""
    if a is None:
        return None
    if hasattr(a, "detach"):
        t = a.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            import torch
            a = t.view(torch.int16).numpy().view(np.uint16)
        else:
            a = t.numpy()
    return np.ascontiguousarray(np.asarray(a).astype(dtype, copy=False))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def e2m1(code: int) -> float:
    return _load().moe_oracle_e2m1(code)


def ue8m0(b: int) -> float:
    return _load().moe_oracle_ue8m0(b)


def e4m3(b: int) -> float:
    return _load().moe_oracle_e4m3(b)


def e4m3_round(v: float) -> int:
    return int(_load().moe_oracle_e4m3_round(v))


def e2m1_round(v: float) -> int:
    return int(_load().moe_oracle_e2m1_round(v))


def dequant(nib, sc, K: int, fmt: int, g: float = 1.0) -> np.ndarray:
    """One projection ``[rows][K/2]`` nibbles + ``[rows][K/B]`` scales -> FP64 ``[rows][K]``."""
    nib = _np(nib, np.uint8)
    sc = _np(sc, np.uint8)
    rows = nib.shape[0] if nib.ndim > 1 else 1
    out = np.empty((rows, K), dtype=np.float64)
    _load().moe_oracle_dequant(_ptr(nib), _ptr(sc), rows, K, fmt, float(g), _ptr(out))
    return out


def _weights_np(weights: dict, fmt: int):
    w13 = _np(weights["w13"], np.uint8)
    s13 = _np(weights["s13"], np.uint8)
    w2 = _np(weights["w2"], np.uint8)
    s2 = _np(weights["s2"], np.uint8)
    g13 = _np(weights.get("g13"), np.float32) if fmt == NVFP4 else None
    g2 = _np(weights.get("g2"), np.float32) if fmt == NVFP4 else None
    return w13, s13, g13, w2, s2, g2


# Gated activations: SiLU (the layer's own), GELU (tanh form), SwiGLU-OAI
# (parameters alpha, beta, limit).  ``act`` arguments take None (SiLU) or a
# tuple (kind, alpha, beta, limit).
ACT_SILU, ACT_GELU_TANH, ACT_SWIGLUOAI = 0, 1, 2


def _act_args(act):
    if act is None:
        return None
    kind, alpha, beta, limit = act
    return int(kind), float(alpha), float(beta), float(limit)


def forward(x_bf16, weights: dict, topk_ids, topk_weights, E: int, H: int, I: int, top_k: int, fmt: int,
            tokens: Optional[Sequence[int]] = None, nthreads: int = 0, act=None) -> np.ndarray:
    """Decode-band definition of the layer in FP64: returns ``[n_tok][H]`` (all tokens if ``tokens`` is None)."""
    x = _np(x_bf16, np.uint16)
    M = x.shape[0]
    w13, s13, g13, w2, s2, g2 = _weights_np(weights, fmt)
    ids = _np(topk_ids, np.int32)
    tw = _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n_tok = M if tok is None else len(tok)
    out = np.full((n_tok, H), np.nan, dtype=np.float64)  # poisoned: the oracle must overwrite
    args = (_ptr(x), _ptr(w13), _ptr(s13), _ptr(g13), _ptr(w2), _ptr(s2), _ptr(g2), _ptr(ids), _ptr(tw), M, E, H, I,
            top_k, fmt, _ptr(tok), n_tok, _ptr(out), nthreads)
    a = _act_args(act)
    rc = _load().moe_oracle_forward(*args) if a is None else _load().moe_oracle_forward_act(*args, *a)
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return out


def forward_prefill(x_bf16, weights: dict, topk_ids, topk_weights, E: int, H: int, I: int, top_k: int,
                    tokens: Optional[Sequence[int]] = None, nthreads: int = 0, fmt: int = NVFP4, act=None):
    """Prefill-band definition (NVFP4 activations, mirrored; weights in either
    format): returns (out ``[n_tok][H]`` FP64, x_q ``[n_tok][H/2]``,
    x_s ``[n_tok][H/16]``, x_G ``[n_tok]``)."""
    x = _np(x_bf16, np.uint16)
    M = x.shape[0]
    w13, s13, g13, w2, s2, g2 = _weights_np(weights, fmt)
    ids = _np(topk_ids, np.int32)
    tw = _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n_tok = M if tok is None else len(tok)
    out = np.full((n_tok, H), np.nan, dtype=np.float64)  # poisoned: the oracle must overwrite
    xq = np.zeros((n_tok, H // 2), dtype=np.uint8)
    xs = np.zeros((n_tok, H // 16), dtype=np.uint8)
    xg = np.zeros((n_tok,), dtype=np.float32)
    args = (_ptr(x), _ptr(w13), _ptr(s13), _ptr(g13), _ptr(w2), _ptr(s2), _ptr(g2), _ptr(ids), _ptr(tw), M, E, H, I,
            top_k, fmt, _ptr(tok), n_tok, _ptr(out), _ptr(xq), _ptr(xs), _ptr(xg), nthreads)
    a = _act_args(act)
    rc = (_load().moe_oracle_forward_prefill(*args) if a is None
          else _load().moe_oracle_forward_prefill_act(*args, *a))
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return out, xq, xs, xg


def fc1(x_row_bf16, weights: dict, e: int, H: int, I: int, fmt: int):
    """FC1 stage for one token row and expert e: (gate[I], up[I]) in FP64."""
    x = _np(x_row_bf16, np.uint16).reshape(-1)
    w13, s13, g13, _, _, _ = _weights_np(weights, fmt)
    gate = np.zeros(I, dtype=np.float64)
    up = np.zeros(I, dtype=np.float64)
    _load().moe_oracle_fc1(_ptr(x), _ptr(w13), _ptr(s13), _ptr(g13), e, H, I, fmt, _ptr(gate), _ptr(up))
    return gate, up


def quant_nvfp4_row(a) -> tuple:
    """FP32 row -> (packed nibbles, E4M3 scale bytes, FP32 multiplier)."""
    a = _np(a, np.float32).reshape(-1)
    K = a.shape[0]
    q = np.zeros(K // 2, dtype=np.uint8)
    s = np.zeros(K // 16, dtype=np.uint8)
    g = np.zeros(1, dtype=np.float32)
    _load().moe_oracle_quant_nvfp4_row(_ptr(a), K, _ptr(q), _ptr(s), _ptr(g))
    return q, s, float(g[0])


def quant_mxfp8_row(a) -> tuple:
    """FP32 row -> (E4M3 bytes [K], UE8M0 scale bytes [K/32])."""
    a = _np(a, np.float32).reshape(-1)
    K = a.shape[0]
    q = np.zeros(K, dtype=np.uint8)
    s = np.zeros(K // 32, dtype=np.uint8)
    _load().moe_oracle_quant_mxfp8_row(_ptr(a), K, _ptr(q), _ptr(s))
    return q, s


def forward_w4a8(x_bf16, weights: dict, topk_ids, topk_weights, E: int, H: int, I: int, top_k: int,
                 tokens: Optional[Sequence[int]] = None, nthreads: int = 0, act=None):
    """W4A8-MX definition (MXFP4 weights, MXFP8 activations, mirrored):
    returns out ``[n_tok][H]`` FP64."""
    x = _np(x_bf16, np.uint16)
    M = x.shape[0]
    w13, s13, _, w2, s2, _ = _weights_np(weights, MXFP4)
    ids = _np(topk_ids, np.int32)
    tw = _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n_tok = M if tok is None else len(tok)
    out = np.full((n_tok, H), np.nan, dtype=np.float64)  # poisoned: the oracle must overwrite
    a = _act_args(act) or (ACT_SILU, 0.0, 0.0, 0.0)
    rc = _load().moe_oracle_forward_w4a8_act(_ptr(x), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(ids), _ptr(tw),
                                             M, E, H, I, top_k, _ptr(tok), n_tok, _ptr(out), nthreads, *a)
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return out


def forward_relu2(x_bf16, weights: dict, topk_ids, topk_weights, E: int, H: int, I: int, top_k: int, fmt: int,
                  tokens: Optional[Sequence[int]] = None, nthreads: int = 0) -> np.ndarray:
    """Non-gated experts with the squared ReLU in FP64: ``weights`` holds w1
    ``[E][I][H/2]``, s1 ``[E][I][H/B]``, (NVFP4) g1 ``[E]``, and w2, s2, g2 as
    for the gated layer.  Returns ``[n_tok][H]``."""
    x = _np(x_bf16, np.uint16)
    M = x.shape[0]
    w1, s1 = _np(weights["w1"], np.uint8), _np(weights["s1"], np.uint8)
    g1 = _np(weights.get("g1"), np.float32) if fmt == NVFP4 else None
    w2, s2 = _np(weights["w2"], np.uint8), _np(weights["s2"], np.uint8)
    g2 = _np(weights.get("g2"), np.float32) if fmt == NVFP4 else None
    ids = _np(topk_ids, np.int32)
    tw = _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n_tok = M if tok is None else len(tok)
    out = np.full((n_tok, H), np.nan, dtype=np.float64)  # poisoned: the oracle must overwrite
    rc = _load().moe_oracle_forward_relu2(_ptr(x), _ptr(w1), _ptr(s1), _ptr(g1), _ptr(w2), _ptr(s2), _ptr(g2),
                                          _ptr(ids), _ptr(tw), M, E, H, I, top_k, fmt, _ptr(tok), n_tok, _ptr(out),
                                          nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return out


def forward_prefill_relu2(x_bf16, weights: dict, topk_ids, topk_weights, E: int, H: int, I: int, top_k: int,
                          fmt: int, tokens: Optional[Sequence[int]] = None, nthreads: int = 0) -> np.ndarray:
    """Prefill-band definition for non-gated experts (NVFP4 activations,
    mirrored; h = max(u, 0)^2 staged in BF16): ``weights`` as for
    ``forward_relu2``.  Returns ``[n_tok][H]`` FP64."""
    x = _np(x_bf16, np.uint16)
    M = x.shape[0]
    w1, s1 = _np(weights["w1"], np.uint8), _np(weights["s1"], np.uint8)
    g1 = _np(weights.get("g1"), np.float32) if fmt == NVFP4 else None
    w2, s2 = _np(weights["w2"], np.uint8), _np(weights["s2"], np.uint8)
    g2 = _np(weights.get("g2"), np.float32) if fmt == NVFP4 else None
    ids = _np(topk_ids, np.int32)
    tw = _np(topk_weights, np.float32)
    tok = None if tokens is None else np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    n_tok = M if tok is None else len(tok)
    out = np.full((n_tok, H), np.nan, dtype=np.float64)  # poisoned: the oracle must overwrite
    rc = _load().moe_oracle_forward_prefill_relu2(_ptr(x), _ptr(w1), _ptr(s1), _ptr(g1), _ptr(w2), _ptr(s2),
                                                  _ptr(g2), _ptr(ids), _ptr(tw), M, E, H, I, top_k, fmt, _ptr(tok),
                                                  n_tok, _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the shapes")
    return out


def route(topk_ids, E: int):
    """Stable grouping of routed rows by expert -> (perm[n_valid], expert_offset[E+1])."""
    ids = _np(topk_ids, np.int32)
    M, top_k = ids.shape
    perm = np.zeros(M * top_k, dtype=np.int32)
    off = np.zeros(E + 1, dtype=np.int32)
    n = _load().moe_oracle_route(_ptr(ids), M, E, top_k, _ptr(perm), _ptr(off))
    return perm[:n], off


def num_threads() -> int:
    return int(_load().moe_oracle_num_threads())
