"""moe_fp4_forward_noalloc: the decode-band layer without device allocation.

Callers that cannot allocate device memory where they run the layer (inside a
stream capture, under a runtime that owns all device memory, on a path that
cannot take an allocation's synchronisation) use this entry point; its
scratch is a fixed array in the library's device image.  These tests call it
through the C ABI and compare it with moe_fp4_forward_ws on the same inputs,
twice in a row (the array keeps the previous call's contents), and check that
shapes needing more scratch than the array holds are rejected.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_util import COS_MIN, MAXABS_REL_RMS, ensure_built, layer_metrics
from workload import gen

pytestmark = pytest.mark.gpu


def _args(wl, pw, out):
    return (wl.x.data_ptr(), pw.w13.data_ptr(), pw.s13.data_ptr(), pw.w2.data_ptr(), pw.s2.data_ptr(),
            wl.topk_ids.data_ptr(), wl.topk_weights.data_ptr(), out.data_ptr(), wl.M, wl.E, wl.H, wl.I, wl.top_k,
            wl.fmt)


@pytest.mark.parametrize("name,ov", [("decode_e512", dict(E=32, M=1)), ("decode_e288_m4", dict(E=24)),
                                     ("tiny_decode", dict(M=8, top_k=2, fmt=gen.NVFP4))])
def test_noalloc_matches_forward_twice(name, ov):
    ensure_built()
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    lib = _capi.lib()
    wl = gen.make_workload(name, device="cuda", **ov)
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    ref = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws).clone()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        st = lib.moe_fp4_forward_noalloc(*_args(wl, pw, out), stream)
        assert st == 0, _capi.moe_fp4_status_string(st)
        torch.cuda.synchronize()
        want = ref.float().cpu().double().numpy()
        assert np.all(np.isfinite(out.float().cpu().numpy()))
        cos, maxabs, rms = layer_metrics(out, want)
        assert cos >= COS_MIN and maxabs <= MAXABS_REL_RMS * rms, (call, cos, maxabs, rms)
        # same kernels on the same inputs: the two entry points agree bitwise
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), call


def test_noalloc_rejects_oversized_scratch():
    ensure_built()
    from fp4_weight_moe_gb300 import _capi
    lib = _capi.lib()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # M=8, top_k=16, I=8192 (MXFP4): needs 8*16*8*8192*4 bytes = 32 MiB > 16 MiB
    need = lib.moe_fp4_workspace_bytes(8, 4, 256, 8192, 16, 0)
    assert need > _capi.MOE_FP4_NOALLOC_SCRATCH_BYTES
    st = lib.moe_fp4_forward_noalloc(p, p, p, p, p, p, p, p, 8, 4, 256, 8192, 16, 0, ctypes.c_void_p(0))
    assert st == _capi.MOE_FP4_EWORKSPACE
    # the prefill band is not served by this entry point
    st = lib.moe_fp4_forward_noalloc(p, p, p, p, p, p, p, p, 9, 4, 256, 128, 2, 0, ctypes.c_void_p(0))
    assert st == _capi.MOE_FP4_EUNSUPPORTED
