"""ctypes binding of libmoe_fp4.so: one Python function per C entry point,
same names, arguments marshalled as integers (device pointers, sizes,
stream handles).  No arithmetic of the layer happens here.

The library is loaded from this package directory (built in-tree by
``fp4_weight_moe_gb300.build``).  If it is missing, every call raises: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_fp4.so")

MOE_FP4_OK = 0
MOE_FP4_EINVAL = 1
MOE_FP4_EUNSUPPORTED = 2
MOE_FP4_ECUDA = 3
MOE_FP4_EWORKSPACE = 4
MOE_FP4_MXFP4 = 0
MOE_FP4_NVFP4 = 1
MOE_FP4_DECODE_MAX_M = 8
MOE_FP4_NOALLOC_SCRATCH_BYTES = 16 << 20
MOE_FP4_ACT_SILU = 0
MOE_FP4_ACT_GELU_TANH = 1
MOE_FP4_ACT_SWIGLUOAI = 2
MOE_FP4_ACT_RELU2 = 3
MOE_FP4_PREFILL_NVFP4 = 0
MOE_FP4_PREFILL_BF16 = 1
MOE_FP4_PREFILL_W4A8_MX = 2
MOE_FP4_STATUS_OK = 0
MOE_FP4_STATUS_TEST_WAIT = 8192


class MoeFp4Activation(ctypes.Structure):
    """struct moe_fp4_activation."""
    _fields_ = [("kind", ctypes.c_int), ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("limit", ctypes.c_float)]


# (name, restype, argtypes) for every symbol declared in include/moe_fp4.h
_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_PZ = ctypes.POINTER(ctypes.c_size_t)
SIGNATURES = {
    "moe_fp4_status_string": (ctypes.c_char_p, [_I]),
    "moe_fp4_last_cuda_error": (_I, []),
    "moe_fp4_version": (_I, []),
    "moe_fp4_prepared_sizes": (_I, [_I, _I, _I, _I, _PZ, _PZ, _PZ, _PZ]),
    "moe_fp4_prepare_weights": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_fp4_prepared_sizes_relu2": (_I, [_I, _I, _I, _I, _PZ, _PZ, _PZ, _PZ]),
    "moe_fp4_prepare_weights_relu2": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_fp4_unprepare_weights_relu2": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_fp4_unprepare_weights": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_fp4_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I]),
    "moe_fp4_workspace_zero_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "moe_fp4_workspace_bytes_mode": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_fp4_debug_set_w4a8_engine": (_I, [_I]),
    "moe_fp4_forward_mode": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                                  ctypes.POINTER(MoeFp4Activation), _I, _P, _Z, _P]),
    "moe_fp4_reserve_workspace": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "moe_fp4_release_workspace": (_I, []),
    "moe_fp4_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moe_fp4_forward_ws": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "moe_fp4_forward_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                ctypes.POINTER(MoeFp4Activation), _P, _Z, _P]),
    "moe_fp4_forward_ex_i64": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                    ctypes.POINTER(MoeFp4Activation), _P, _Z, _P]),
    "moe_fp4_forward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "moe_fp4_host_workspace_bytes": (_Z, [_I, _I, _I, _I, _I, _I]),
    "moe_fp4_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "moe_fp4_debug_set_decode_family": (_I, [_I, ctypes.POINTER(ctypes.c_int)]),
    "moe_fp4_debug_set_mid_band": (_I, [_I, ctypes.POINTER(ctypes.c_int)]),
    "moe_fp4_debug_decode_gemv_fits": (_I, [_I, _I, _I, _I, _I]),
    "moe_fp4_debug_decode_launches": (_I, [_I, _I, _I, _I, _I]),
    "moe_fp4_debug_mid_band_of": (_I, [_I, _I, _I, _I, _I]),
    "moe_fp4_debug_decode_family_of": (_I, [_I, _I, _I, _I, _I]),
    "moe_fp4_debug_dequant": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moe_fp4_debug_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_fp4_debug_route": (_I, [_P, _I, _I, _I, _P, _P, _P, _Z, _P]),
"moe_fp4_debug_route_small": (_I, [_P, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "moe_fp4_debug_route_workspace_bytes": (_Z, [_I, _I, _I]),
    "moe_fp4_debug_quant_mxfp8_rows": (_I, [_P, _I, _I, _P, _P, _P]),
    "moe_fp4_debug_quant_rows": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "moe_fp4_workspace_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint32), _I, _P]),
    "moe_fp4_noalloc_status": (_I, [ctypes.POINTER(ctypes.c_uint32), _I, _P]),
    "moe_fp4_debug_wait_timeout": (_I, [_P, ctypes.c_uint, _P]),
    "moe_fp4_debug_decode_plan": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
}

_lock = threading.Lock()
_lib = None


class MoeFp4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = _load()
        msg = lib.moe_fp4_status_string(status).decode()
        if status == MOE_FP4_ECUDA:
            msg += f" (cudaError {lib.moe_fp4_last_cuda_error()})"
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libmoe_fp4.so is not built ({LIB_PATH}); run fp4_weight_moe_gb300.build.build()")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
        return _lib


def lib():
    return _load()


def _check(fn: str, status: int) -> int:
    if status != MOE_FP4_OK:
        raise MoeFp4Error(fn, status)
    return status


# ------------------------------------------------------------- entry points
def moe_fp4_status_string(status: int) -> str:
    return _load().moe_fp4_status_string(status).decode()


def moe_fp4_version() -> int:
    return _load().moe_fp4_version()


def moe_fp4_prepared_sizes(E, H, I, fmt):
    sizes = [ctypes.c_size_t() for _ in range(4)]
    _check("moe_fp4_prepared_sizes",
           _load().moe_fp4_prepared_sizes(E, H, I, fmt, *[ctypes.byref(s) for s in sizes]))
    return tuple(int(s.value) for s in sizes)


def moe_fp4_prepare_weights(w13_l, s13_l, g13, w2_l, s2_l, g2, E, H, I, fmt, w13, s13, w2, s2, stream):
    return _check("moe_fp4_prepare_weights",
                  _load().moe_fp4_prepare_weights(w13_l, s13_l, g13, w2_l, s2_l, g2, E, H, I, fmt, w13, s13, w2, s2,
                                                  stream))


def moe_fp4_unprepare_weights(w13, s13, w2, s2, E, H, I, fmt, w13_l, s13_l, g13, w2_l, s2_l, g2, stream):
    return _check("moe_fp4_unprepare_weights",
                  _load().moe_fp4_unprepare_weights(w13, s13, w2, s2, E, H, I, fmt, w13_l, s13_l, g13, w2_l, s2_l,
                                                    g2, stream))


def moe_fp4_prepared_sizes_relu2(E, H, I, fmt):
    out = [ctypes.c_size_t(0) for _ in range(4)]
    _check("moe_fp4_prepared_sizes_relu2",
           lib().moe_fp4_prepared_sizes_relu2(E, H, I, fmt, *[ctypes.byref(o) for o in out]))
    return tuple(o.value for o in out)


def moe_fp4_prepare_weights_relu2(w1_l, s1_l, g1, w2_l, s2_l, g2, E, H, I, fmt, w1, s1, w2, s2, stream):
    _check("moe_fp4_prepare_weights_relu2",
           lib().moe_fp4_prepare_weights_relu2(w1_l, s1_l, g1, w2_l, s2_l, g2, E, H, I, fmt, w1, s1, w2, s2, stream))


def moe_fp4_unprepare_weights_relu2(w1, s1, w2, s2, E, H, I, fmt, w1_l, s1_l, g1, w2_l, s2_l, g2, stream):
    _check("moe_fp4_unprepare_weights_relu2",
           lib().moe_fp4_unprepare_weights_relu2(w1, s1, w2, s2, E, H, I, fmt, w1_l, s1_l, g1, w2_l, s2_l, g2, stream))


def moe_fp4_workspace_bytes(M_max, E, H, I, top_k, fmt) -> int:
    return int(_load().moe_fp4_workspace_bytes(M_max, E, H, I, top_k, fmt))


def moe_fp4_debug_set_w4a8_engine(fp8: int) -> int:
    return int(lib().moe_fp4_debug_set_w4a8_engine(fp8))


def moe_fp4_workspace_bytes_mode(M_max, E, H, I, top_k, fmt, prefill_mode) -> int:
    return int(lib().moe_fp4_workspace_bytes_mode(M_max, E, H, I, top_k, fmt, prefill_mode))


def moe_fp4_forward_mode(x, w13, s13, w2, s2, ids, ids64, tw, out, M, E, H, I, top_k, fmt, act, prefill_mode, ws,
                         ws_bytes, stream):
    _check("moe_fp4_forward_mode", lib().moe_fp4_forward_mode(x, w13, s13, w2, s2, ids, ids64, tw, out, M, E, H, I,
                                                               top_k, fmt, act, prefill_mode, ws, ws_bytes, stream))


def moe_fp4_workspace_zero_bytes(E, H, I, top_k, fmt) -> int:
    return int(lib().moe_fp4_workspace_zero_bytes(E, H, I, top_k, fmt))


def moe_fp4_reserve_workspace(M_max, E, H, I, top_k, fmt, stream):
    return _check("moe_fp4_reserve_workspace", _load().moe_fp4_reserve_workspace(M_max, E, H, I, top_k, fmt, stream))


def moe_fp4_release_workspace():
    return _check("moe_fp4_release_workspace", _load().moe_fp4_release_workspace())


def moe_fp4_forward(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, stream):
    return _check("moe_fp4_forward",
                  _load().moe_fp4_forward(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, stream))


def moe_fp4_forward_ws(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, ws, ws_bytes, stream):
    return _check("moe_fp4_forward_ws",
                  _load().moe_fp4_forward_ws(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, ws, ws_bytes,
                                             stream))


def moe_fp4_forward_ex(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, act, ws, ws_bytes, stream):
    """``act``: None (SiLU) or a MoeFp4Activation."""
    return _check("moe_fp4_forward_ex",
                  _load().moe_fp4_forward_ex(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt,
                                             None if act is None else ctypes.byref(act), ws, ws_bytes, stream))


def moe_fp4_forward_ex_i64(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, act, ws, ws_bytes, stream):
    """moe_fp4_forward_ex with int64 ``ids``."""
    return _check("moe_fp4_forward_ex_i64",
                  _load().moe_fp4_forward_ex_i64(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt,
                                                 None if act is None else ctypes.byref(act), ws, ws_bytes, stream))


def moe_fp4_forward_noalloc(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, stream):
    return _check("moe_fp4_forward_noalloc",
                  _load().moe_fp4_forward_noalloc(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, stream))


def moe_fp4_host_workspace_bytes(M_max, E, H, I, top_k, fmt) -> int:
    return int(_load().moe_fp4_host_workspace_bytes(M_max, E, H, I, top_k, fmt))


def moe_fp4_forward_host(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, ws, ws_bytes, stream):
    return _check("moe_fp4_forward_host",
                  _load().moe_fp4_forward_host(x, w13, s13, w2, s2, ids, tw, out, M, E, H, I, top_k, fmt, ws,
                                               ws_bytes, stream))


def moe_fp4_debug_set_decode_family(family: int) -> int:
    prev = ctypes.c_int()
    _check("moe_fp4_debug_set_decode_family", _load().moe_fp4_debug_set_decode_family(family, ctypes.byref(prev)))
    return prev.value


def moe_fp4_debug_set_mid_band(mode: int) -> int:
    prev = ctypes.c_int()
    _check("moe_fp4_debug_set_mid_band", _load().moe_fp4_debug_set_mid_band(mode, ctypes.byref(prev)))
    return prev.value


def moe_fp4_debug_decode_gemv_fits(M, E, H, I, top_k) -> bool:
    return bool(_load().moe_fp4_debug_decode_gemv_fits(M, E, H, I, top_k))


def moe_fp4_debug_decode_family_of(M, E, H, I, top_k) -> int:
    return int(_load().moe_fp4_debug_decode_family_of(M, E, H, I, top_k))


def moe_fp4_debug_decode_launches(M, E, H, I, top_k) -> int:
    return int(_load().moe_fp4_debug_decode_launches(M, E, H, I, top_k))


def moe_fp4_debug_mid_band_of(M, E, H, I, top_k) -> int:
    """1 the prefill band's GEMMs, 2 decode-band chunks, 3 the mid band's
    GEMMs, 0 for the decode band or invalid shapes."""
    return int(_load().moe_fp4_debug_mid_band_of(M, E, H, I, top_k))


def moe_fp4_debug_dequant(w, s, which, expert, E, H, I, fmt, out, stream):
    return _check("moe_fp4_debug_dequant",
                  _load().moe_fp4_debug_dequant(w, s, which, expert, E, H, I, fmt, out, stream))


def moe_fp4_debug_gemm(a_q, a_sf, b_q, b_sf, d, M_rows, N_rows, K, fmt, status, stream):
    return _check("moe_fp4_debug_gemm",
                  _load().moe_fp4_debug_gemm(a_q, a_sf, b_q, b_sf, d, M_rows, N_rows, K, fmt, status, stream))


def moe_fp4_debug_route(ids, M, E, top_k, perm, offset, ws, ws_bytes, stream):
    return _check("moe_fp4_debug_route", _load().moe_fp4_debug_route(ids, M, E, top_k, perm, offset, ws, ws_bytes,
                                                                       stream))


def moe_fp4_debug_route_small(ids, M, E, top_k, perm, offset, ws, ws_bytes, stream):
    return _check("moe_fp4_debug_route_small",
                  _load().moe_fp4_debug_route_small(ids, M, E, top_k, perm, offset, ws, ws_bytes, stream))


def moe_fp4_debug_route_workspace_bytes(M, E, top_k) -> int:
    return int(_load().moe_fp4_debug_route_workspace_bytes(M, E, top_k))


def moe_fp4_debug_quant_mxfp8_rows(inp, rows, K, q, s, stream):
    return _check("moe_fp4_debug_quant_mxfp8_rows", _load().moe_fp4_debug_quant_mxfp8_rows(inp, rows, K, q, s, stream))


def moe_fp4_debug_quant_rows(inp, rows, K, q, s, G, stream):
    return _check("moe_fp4_debug_quant_rows", _load().moe_fp4_debug_quant_rows(inp, rows, K, q, s, G, stream))


def moe_fp4_workspace_status(ws, clear: bool, stream) -> int:
    v = ctypes.c_uint32(0)
    _check("moe_fp4_workspace_status", lib().moe_fp4_workspace_status(ws, ctypes.byref(v), int(bool(clear)), stream))
    return v.value


def moe_fp4_noalloc_status(clear: bool, stream) -> int:
    v = ctypes.c_uint32(0)
    _check("moe_fp4_noalloc_status", lib().moe_fp4_noalloc_status(ctypes.byref(v), int(bool(clear)), stream))
    return v.value


def moe_fp4_debug_wait_timeout(status_word, polls: int, stream):
    _check("moe_fp4_debug_wait_timeout", lib().moe_fp4_debug_wait_timeout(status_word, polls, stream))


def moe_fp4_debug_decode_plan(M, E, H, I, top_k):
    """(C, s1, Q, cap) of the single-launch plan on the current device, zeros if none."""
    v = (ctypes.c_int * 4)()
    _check("moe_fp4_debug_decode_plan", lib().moe_fp4_debug_decode_plan(M, E, H, I, top_k, v))
    return tuple(v)


def raw_status(name: str, *args) -> int:
    """Call an entry point and return its status without raising (tests of the error contract)."""
    return getattr(_load(), name)(*args)
