"""GB300-native fused FP4-weight mixture-of-experts layer.

The compute path is ``libmoe_fp4.so`` (hand-written CUDA for sm_103a behind a
C ABI, see ``include/moe_fp4.h``).  This package is its thin Python binding:
``_capi`` mirrors the C entry points one to one, and the helpers below only
allocate torch device tensors and pass their pointers.  PyTorch provides device
memory and streams; no step of the layer runs in PyTorch.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import _capi
from ._capi import (  # noqa: F401
    MOE_FP4_DECODE_MAX_M,
    MOE_FP4_MXFP4,
    MOE_FP4_NVFP4,
    MoeFp4Error,
)

MXFP4 = MOE_FP4_MXFP4
NVFP4 = MOE_FP4_NVFP4


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: Optional[torch.device] = None) -> Optional[int]:
    """Raw cudaStream_t of ``stream`` (None: the current stream of ``device``,
    else of the current device)."""
    if stream is None:
        if _raw_stream is not None:
            idx = device.index if device is not None and device.index is not None else torch.cuda.current_device()
            return _raw_stream(idx)
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libmoe_fp4 takes CUDA tensors only (there is no CPU path)")


@dataclasses.dataclass
class PreparedWeights:
    """Resident (repacked) expert weights on one device."""
    w13: torch.Tensor
    s13: torch.Tensor
    w2: torch.Tensor
    s2: torch.Tensor
    E: int
    H: int
    I: int
    fmt: int

    def __post_init__(self):
        self._ptrs = (_ptr(self.w13), _ptr(self.s13), _ptr(self.w2), _ptr(self.s2))

    def ptrs(self):
        return self._ptrs


def prepared_sizes(E: int, H: int, I: int, fmt: int):
    return _capi.moe_fp4_prepared_sizes(E, H, I, fmt)


def prepare_weights(weights: dict, E: int, H: int, I: int, fmt: int, stream=None) -> PreparedWeights:
    """Repack logical checkpoint tensors (dict with w13, s13, w2, s2 and, for
    NVFP4, g13, g2; CUDA tensors) into the resident layout."""
    w13_l, s13_l, w2_l, s2_l = (weights[k].contiguous() for k in ("w13", "s13", "w2", "s2"))
    g13 = weights.get("g13") if fmt == NVFP4 else None
    g2 = weights.get("g2") if fmt == NVFP4 else None
    if g13 is not None:
        g13 = g13.contiguous().float()
        g2 = g2.contiguous().float()
    _require_cuda(w13_l, s13_l, w2_l, s2_l, g13, g2)
    dev = w13_l.device
    n13, ns13, n2, ns2 = prepared_sizes(E, H, I, fmt)
    out = [torch.empty(n, dtype=torch.uint8, device=dev) for n in (n13, ns13, n2, ns2)]
    _capi.moe_fp4_prepare_weights(_ptr(w13_l), _ptr(s13_l), _ptr(g13), _ptr(w2_l), _ptr(s2_l), _ptr(g2), E, H, I,
                                  fmt, *[_ptr(t) for t in out], _stream(stream))
    return PreparedWeights(*out, E=E, H=H, I=I, fmt=fmt)


def unprepare_weights(pw: PreparedWeights, stream=None) -> dict:
    """Resident -> logical tensors (test support)."""
    E, H, I, fmt = pw.E, pw.H, pw.I, pw.fmt
    B = 32 if fmt == MXFP4 else 16
    dev = pw.w13.device
    w13 = torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev)
    s13 = torch.empty((E, 2 * I, H // B), dtype=torch.uint8, device=dev)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev)
    s2 = torch.empty((E, H, I // B), dtype=torch.uint8, device=dev)
    g13 = torch.empty((E, 2), dtype=torch.float32, device=dev) if fmt == NVFP4 else None
    g2 = torch.empty((E,), dtype=torch.float32, device=dev) if fmt == NVFP4 else None
    _capi.moe_fp4_unprepare_weights(*pw.ptrs(), E, H, I, fmt, _ptr(w13), _ptr(s13), _ptr(g13), _ptr(w2), _ptr(s2),
                                    _ptr(g2), _stream(stream))
    out = dict(w13=w13, s13=s13, w2=w2, s2=s2)
    if fmt == NVFP4:
        out.update(g13=g13, g2=g2)
    return out


def prepare_weights_relu2(weights: dict, E: int, H: int, I: int, fmt: int, stream=None) -> PreparedWeights:
    """Repack a non-gated (squared-ReLU) expert checkpoint: dict with w1
    [E][I][H/2], s1, w2, s2 and, for NVFP4, g1, g2 (CUDA tensors).  The
    result's w13/s13 fields hold the resident w1/s1; run it with
    ``forward_act(..., kind=ACT_RELU2)``."""
    w1_l, s1_l, w2_l, s2_l = (weights[k].contiguous() for k in ("w1", "s1", "w2", "s2"))
    g1 = weights.get("g1") if fmt == NVFP4 else None
    g2 = weights.get("g2") if fmt == NVFP4 else None
    if g1 is not None:
        g1 = g1.contiguous().float()
        g2 = g2.contiguous().float()
    _require_cuda(w1_l, s1_l, w2_l, s2_l, g1, g2)
    dev = w1_l.device
    sizes = _capi.moe_fp4_prepared_sizes_relu2(E, H, I, fmt)
    out = [torch.empty(n, dtype=torch.uint8, device=dev) for n in sizes]
    _capi.moe_fp4_prepare_weights_relu2(_ptr(w1_l), _ptr(s1_l), _ptr(g1), _ptr(w2_l), _ptr(s2_l), _ptr(g2), E, H,
                                        I, fmt, *[_ptr(t) for t in out], _stream(stream))
    return PreparedWeights(*out, E=E, H=H, I=I, fmt=fmt)


def unprepare_weights_relu2(pw: PreparedWeights, stream=None) -> dict:
    """Resident -> logical tensors of a non-gated checkpoint (test support)."""
    E, H, I, fmt = pw.E, pw.H, pw.I, pw.fmt
    B = 32 if fmt == MXFP4 else 16
    dev = pw.w13.device
    w1 = torch.empty((E, I, H // 2), dtype=torch.uint8, device=dev)
    s1 = torch.empty((E, I, H // B), dtype=torch.uint8, device=dev)
    w2 = torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev)
    s2 = torch.empty((E, H, I // B), dtype=torch.uint8, device=dev)
    g1 = torch.empty((E,), dtype=torch.float32, device=dev) if fmt == NVFP4 else None
    g2 = torch.empty((E,), dtype=torch.float32, device=dev) if fmt == NVFP4 else None
    _capi.moe_fp4_unprepare_weights_relu2(*pw.ptrs(), E, H, I, fmt, _ptr(w1), _ptr(s1), _ptr(g1), _ptr(w2), _ptr(s2),
                                          _ptr(g2), _stream(stream))
    out = dict(w1=w1, s1=s1, w2=w2, s2=s2)
    if fmt == NVFP4:
        out.update(g1=g1, g2=g2)
    return out


def workspace_bytes(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int) -> int:
    return _capi.moe_fp4_workspace_bytes(M_max, E, H, I, top_k, fmt)


def alloc_workspace(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int, device=None) -> torch.Tensor:
    """A zero-filled caller-owned workspace for ``forward(..., workspace=...)``."""
    n = workspace_bytes(M_max, E, H, I, top_k, fmt)
    if n == 0:
        raise MoeFp4Error("moe_fp4_workspace_bytes", _capi.MOE_FP4_EUNSUPPORTED)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def reserve_workspace(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int, stream=None):
    _capi.moe_fp4_reserve_workspace(M_max, E, H, I, top_k, fmt, _stream(stream))


def _check_dtypes(x, topk_ids, topk_weights):
    if x.dtype != torch.bfloat16 or topk_ids.dtype not in (torch.int32, torch.int64) or \
            topk_weights.dtype != torch.float32:
        raise TypeError("x must be bfloat16, topk_ids int32 or int64, topk_weights float32")


def forward(x: torch.Tensor, pw: PreparedWeights, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
            out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The fused MoE layer: bf16 ``x [M, H]`` -> bf16 ``out [M, H]``.  int64
    ``topk_ids`` need a caller ``workspace`` (moe_fp4_forward_ex_i64)."""
    _check_dtypes(x, topk_ids, topk_weights)
    _require_cuda(x, topk_ids, topk_weights, out, workspace)
    M, H = x.shape
    top_k = topk_ids.shape[1]
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    if topk_ids.dtype == torch.int64:
        if workspace is None:
            raise TypeError("int64 topk_ids need a caller workspace (alloc_workspace)")
        _capi.moe_fp4_forward_ex_i64(_ptr(x), *pw.ptrs(), _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, pw.E,
                                     pw.H, pw.I, top_k, pw.fmt, None, _ptr(workspace), workspace.nbytes,
                                     _stream(stream, x.device))
        return out
    args = (_ptr(x), *pw.ptrs(), _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, pw.E, pw.H, pw.I, top_k, pw.fmt)
    if workspace is None:
        _capi.moe_fp4_forward(*args, _stream(stream, x.device))
    else:
        _capi.moe_fp4_forward_ws(*args, _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream, x.device))
    return out


ACT_SILU, ACT_GELU_TANH, ACT_SWIGLUOAI, ACT_RELU2 = (_capi.MOE_FP4_ACT_SILU, _capi.MOE_FP4_ACT_GELU_TANH,
                                                   _capi.MOE_FP4_ACT_SWIGLUOAI, _capi.MOE_FP4_ACT_RELU2)


def forward_act(x: torch.Tensor, pw: PreparedWeights, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                workspace: torch.Tensor, kind: int = ACT_SILU, alpha: float = 0.0, beta: float = 1.0,
                limit: float = 0.0, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The layer with a chosen activation (ACT_SILU, ACT_GELU_TANH, or
    ACT_SWIGLUOAI with alpha, beta, limit; ACT_RELU2 with weights from
    prepare_weights_relu2), on a caller-owned workspace."""
    _check_dtypes(x, topk_ids, topk_weights)
    _require_cuda(x, topk_ids, topk_weights, out, workspace)
    M, H = x.shape
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    act = _capi.MoeFp4Activation(kind, alpha, beta, limit)
    call = _capi.moe_fp4_forward_ex_i64 if topk_ids.dtype == torch.int64 else _capi.moe_fp4_forward_ex
    call(_ptr(x), *pw.ptrs(), _ptr(topk_ids), _ptr(topk_weights), _ptr(out), M, pw.E, pw.H, pw.I, topk_ids.shape[1],
         pw.fmt, act, _ptr(workspace), workspace.nbytes, _stream(stream, x.device))
    return out


PREFILL_NVFP4, PREFILL_BF16, PREFILL_W4A8_MX = (_capi.MOE_FP4_PREFILL_NVFP4, _capi.MOE_FP4_PREFILL_BF16,
                                                _capi.MOE_FP4_PREFILL_W4A8_MX)


def alloc_workspace_mode(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int, prefill_mode: int,
                         device=None) -> torch.Tensor:
    """A zero-filled workspace for ``forward_mode`` with this prefill precision."""
    n = _capi.moe_fp4_workspace_bytes_mode(M_max, E, H, I, top_k, fmt, prefill_mode)
    if n == 0:
        raise MoeFp4Error("moe_fp4_workspace_bytes_mode", _capi.MOE_FP4_EUNSUPPORTED)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def forward_mode(x: torch.Tensor, pw: PreparedWeights, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                 workspace: torch.Tensor, prefill_mode: int = PREFILL_BF16, kind: int = ACT_SILU, alpha: float = 0.0,
                 beta: float = 1.0, limit: float = 0.0, out: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """The layer with a chosen prefill precision (PREFILL_NVFP4, the exact
    PREFILL_BF16, or PREFILL_W4A8_MX with MXFP8 activations and MXFP4
    weights) and activation, on a workspace from alloc_workspace_mode."""
    _check_dtypes(x, topk_ids, topk_weights)
    _require_cuda(x, topk_ids, topk_weights, out, workspace)
    M, H = x.shape
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    act = _capi.MoeFp4Activation(kind, alpha, beta, limit)
    _capi.moe_fp4_forward_mode(_ptr(x), *pw.ptrs(), _ptr(topk_ids), 1 if topk_ids.dtype == torch.int64 else 0,
                               _ptr(topk_weights), _ptr(out), M, pw.E, pw.H, pw.I, topk_ids.shape[1], pw.fmt, act,
                               prefill_mode, _ptr(workspace), workspace.nbytes, _stream(stream, x.device))
    return out


def host_workspace_bytes(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int) -> int:
    return _capi.moe_fp4_host_workspace_bytes(M_max, E, H, I, top_k, fmt)


def alloc_host_workspace(M_max: int, E: int, H: int, I: int, top_k: int, fmt: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace for ``forward_host``."""
    n = host_workspace_bytes(M_max, E, H, I, top_k, fmt)
    if n == 0:
        raise MoeFp4Error("moe_fp4_host_workspace_bytes", _capi.MOE_FP4_EUNSUPPORTED)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def forward_host(x: torch.Tensor, pw: PreparedWeights, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                 out: torch.Tensor, workspace: torch.Tensor, stream=None) -> torch.Tensor:
    """The layer on HOST tensors (pinned for asynchronous copies): enqueues the
    input copies, the layer and the output copy on ``stream``; ``out`` holds
    the result once the stream has been synchronised."""
    if x.dtype != torch.bfloat16 or topk_ids.dtype != torch.int32 or topk_weights.dtype != torch.float32:
        raise TypeError("x must be bfloat16, topk_ids int32, topk_weights float32")
    if out.dtype != torch.bfloat16 or out.shape != x.shape:
        raise TypeError("out must be bfloat16 of x's shape")
    if not (x.is_contiguous() and topk_ids.is_contiguous() and topk_weights.is_contiguous() and out.is_contiguous()):
        raise ValueError("host tensors must be contiguous")
    if not workspace.is_cuda:
        raise ValueError("the workspace must be a CUDA tensor")
    M, H = x.shape
    _capi.moe_fp4_forward_host(x.data_ptr(), *pw.ptrs(), topk_ids.data_ptr(), topk_weights.data_ptr(), out.data_ptr(),
                               M, pw.E, pw.H, pw.I, topk_ids.shape[1], pw.fmt, workspace.data_ptr(),
                               workspace.nbytes, _stream(stream, workspace.device))
    return out


def debug_dequant(pw: PreparedWeights, which: int, expert: int, stream=None) -> torch.Tensor:
    """which: 0 w13, 1 w2, 2 the w1 of non-gated (squared-ReLU) weights."""
    rows, K = {0: (2 * pw.I, pw.H), 1: (pw.H, pw.I), 2: (pw.I, pw.H)}[which]
    out = torch.empty((rows, K), dtype=torch.float32, device=pw.w13.device)
    w, s = (pw.w2, pw.s2) if which == 1 else (pw.w13, pw.s13)
    _capi.moe_fp4_debug_dequant(_ptr(w), _ptr(s), which, expert, pw.E, pw.H, pw.I, pw.fmt, _ptr(out),
                                _stream(stream))
    return out


def workspace_status(workspace: Optional[torch.Tensor] = None, clear: bool = False, stream=None) -> int:
    """Status word of a workspace (None: the reserved library workspace): 0,
    or bits of kernel waits that gave up (the outputs since the last clear
    are not valid).  Synchronises ``stream``; ``clear`` resets the word."""
    dev = workspace.device if workspace is not None else None
    return _capi.moe_fp4_workspace_status(_ptr(workspace), clear, _stream(stream, dev))


def noalloc_status(clear: bool = False, stream=None) -> int:
    """Status word of moe_fp4_forward_noalloc's scratch array on the current device."""
    return _capi.moe_fp4_noalloc_status(clear, _stream(stream))
