"""moe_fp4_forward_host: the layer on host buffers.

In the decode band the kernels read page-locked host inputs and write a
page-locked host output in place; other buffers (and all of them in the
prefill band) are copied through the workspace.  Either way the layer runs
the same kernels as moe_fp4_forward_ws, on one stream.  These tests check
that its result equals moe_fp4_forward_ws on device copies of the same inputs (bitwise in the
decode band, whose kernels are deterministic; within the parity bound in the
prefill band, whose FP32 token accumulator takes atomic adds), with pinned,
pageable and mixed host tensors, across batch sizes sharing one workspace, and
that a short workspace is refused before anything runs.
"""
import ctypes

import pytest
import torch

from tests.gpu_util import assert_layer_close, ensure_built
from workload import gen

pytestmark = pytest.mark.gpu


def _host(t, pinned):
    h = t.cpu().contiguous()
    return h.pin_memory() if pinned else h


# pinned: (x, ids, router weights, out) page-locked (read or written in place
# by the kernels) or pageable (staged through the workspace)
@pytest.mark.parametrize("name,ov,pinned", [("decode_e512", dict(E=32, M=1), (True,) * 4),
                                            ("decode_e288_m4", dict(E=24), (False,) * 4),
                                            ("decode_e288_m4", dict(E=24, M=3), (True, False, True, False)),
                                            ("tiny_decode", dict(M=8, fmt=gen.NVFP4), (False, True, False, True))])
def test_host_entry_matches_device_entry(name, ov, pinned):
    ensure_built()
    import fp4_weight_moe_gb300 as m
    wl = gen.make_workload(name, device="cuda", **ov)
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    ref = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws).clone()
    hws = m.alloc_host_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    xh, idh, twh = (_host(t, p) for t, p in zip((wl.x, wl.topk_ids, wl.topk_weights), pinned))
    for call in range(2):
        outh = _host(torch.full_like(ref, float("nan")), pinned[3])
        m.forward_host(xh, pw, idh, twh, outh, hws)
        torch.cuda.current_stream().synchronize()
        assert torch.equal(outh.view(torch.int16), ref.cpu().view(torch.int16)), call


def test_host_entry_shared_workspace_across_batches():
    """One workspace sized for the largest batch serves smaller and larger
    calls in any order, including the prefill band."""
    ensure_built()
    import fp4_weight_moe_gb300 as m
    E, H, I, k, fmt = 16, 512, 256, 4, gen.NVFP4
    hws = m.alloc_host_workspace(40, E, H, I, k, fmt)
    weights = gen.make_expert_weights(E, H, I, fmt, 7, device="cuda")
    pw = m.prepare_weights(weights, E, H, I, fmt)
    for M in (8, 1, 40, 12, 3, 8):
        x = gen.draw_activations(M, H, 100 + M, device="cuda")
        ids, tw = gen.draw_routing(M, E, k, 200 + M, mode="softmax")
        ids, tw = ids.cuda(), tw.cuda()
        ws = m.alloc_workspace(M, E, H, I, k, fmt)
        ref = m.forward(x, pw, ids, tw, workspace=ws).clone()
        outh = torch.empty((M, H), dtype=torch.bfloat16).pin_memory()
        m.forward_host(_host(x, True), pw, _host(ids, True), _host(tw, True), outh, hws)
        torch.cuda.current_stream().synchronize()
        if m._capi.moe_fp4_debug_decode_launches(M, E, H, I, k) > 0:  # decode kernels
            assert torch.equal(outh.view(torch.int16), ref.cpu().view(torch.int16)), M
        else:
            assert_layer_close(outh, ref.float().cpu().double().numpy(), f"prefill M={M} host vs device")


def test_host_entry_rejects_short_workspace():
    ensure_built()
    from fp4_weight_moe_gb300 import _capi
    lib = _capi.lib()
    E, H, I, k, fmt = 8, 256, 128, 2, gen.MXFP4
    need = lib.moe_fp4_host_workspace_bytes(4, E, H, I, k, fmt)
    assert need > lib.moe_fp4_workspace_bytes(4, E, H, I, k, fmt)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    xh = torch.zeros((4, H), dtype=torch.bfloat16)
    p = ctypes.c_void_p(ws.data_ptr())
    # the size check comes before any copy or launch: host pointers of the
    # right kind are passed, weights stand in with the workspace pointer
    st = lib.moe_fp4_forward_host(xh.data_ptr(), p, p, p, p, xh.data_ptr(), xh.data_ptr(), xh.data_ptr(), 4, E, H,
                                  I, k, fmt, p, need - 256, None)
    assert st == _capi.MOE_FP4_EWORKSPACE
    st = lib.moe_fp4_forward_host(xh.data_ptr(), p, p, p, p, xh.data_ptr(), xh.data_ptr(), xh.data_ptr(), 0, E, H,
                                  I, k, fmt, p, need, None)
    assert st == _capi.MOE_FP4_OK
