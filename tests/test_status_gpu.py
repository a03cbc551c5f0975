"""The device status word: a bounded wait that gives up is visible to the
caller through moe_fp4_workspace_status (and moe_fp4_noalloc_status for the
no-allocation entry point), and clean layers leave it at zero.

The wait that runs out is one the test entry moe_fp4_debug_wait_timeout
starts on a barrier nothing completes, with a short poll limit: nothing is
faulted or hung, the kernel records its bit and returns.
"""
import pytest
import torch

from tests.gpu_util import ensure_built
from workload import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def test_timed_out_wait_is_reported_and_cleared():
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    wl = gen.make_workload("tiny_decode", device="cuda")
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    assert m.workspace_status(ws) == 0
    stream = torch.cuda.current_stream().cuda_stream
    _capi.moe_fp4_debug_wait_timeout(ws.data_ptr(), 64, stream)
    st = m.workspace_status(ws)
    assert st & _capi.MOE_FP4_STATUS_TEST_WAIT
    assert m.workspace_status(ws, clear=True) == st  # returns the word, then clears it
    assert m.workspace_status(ws) == 0


@pytest.mark.parametrize("family", [1, 2, 3], ids=["gemv", "chain", "single"])
def test_clean_layers_leave_status_zero(family):
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    prev = _capi.moe_fp4_debug_set_decode_family(family)
    try:
        for name, ov in (("tiny_decode", {}), ("decode_e512", dict(E=24)), ("decode_e512", dict(E=24, M=4))):
            wl = gen.make_workload(name, device="cuda", **ov)
            pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
            ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
            for _ in range(3):
                m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws)
            assert m.workspace_status(ws) == 0, (name, ov)
    finally:
        _capi.moe_fp4_debug_set_decode_family(prev)


def test_library_workspace_and_noalloc_status():
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    wl = gen.make_workload("decode_e512", device="cuda", E=24)
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    m.reserve_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights)
    assert m.workspace_status() == 0
    out = torch.empty((wl.M, wl.H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    _capi.moe_fp4_forward_noalloc(wl.x.data_ptr(), *pw.ptrs(), wl.topk_ids.data_ptr(), wl.topk_weights.data_ptr(),
                                  out.data_ptr(), wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, stream)
    assert m.noalloc_status() == 0
