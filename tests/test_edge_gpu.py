"""Edge cases of the layer against the FP64 oracle, through the C ABI.

The largest decode batch with the largest top_k, one expert taking every
route (all of a layer's tokens in one expert: the GEMV family's 8-token path),
the smallest H and I the boundary accepts, the band boundary (M = 8, and
the first batches past it on the mid band), and routings whose slots all
repeat one expert.  Each decode case runs on both kernel families.
"""
import pytest
import torch

from tests.gpu_util import assert_layer_close, ensure_built, oracle_layer
from workload import gen

pytestmark = pytest.mark.gpu

GEMV, TC, SINGLE = 1, 2, 3  # decode plans: streaming GEMV, tcgen05 chain, tcgen05 single launch


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def _run(wl, family=0):
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    prev = _capi.moe_fp4_debug_set_decode_family(family)
    try:
        m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, out=out, workspace=ws)
        torch.cuda.synchronize()
    finally:
        _capi.moe_fp4_debug_set_decode_family(prev)
    return out


def _with_ids(wl, ids, seed=0):
    wl.topk_ids = torch.tensor(ids, dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(seed)
    wl.topk_weights = torch.rand(wl.topk_ids.shape, generator=g).cuda()
    return wl


@pytest.mark.parametrize("family", [0, GEMV, TC, SINGLE], ids=["auto", "gemv", "chain", "single"])
@pytest.mark.parametrize("case", ["max_batch_topk16", "one_expert_all_routes", "min_shape", "same_expert_slots"])
def test_decode_edges(case, family):
    if case == "max_batch_topk16":
        wl = gen.make_workload("tiny_decode", device="cuda", M=8, E=40, top_k=16, fmt=gen.NVFP4)
    elif case == "one_expert_all_routes":
        wl = gen.make_workload("decode_e512", device="cuda", E=1, M=8, top_k=1)
        wl = _with_ids(wl, [[0]] * 8, seed=1)
    elif case == "min_shape":
        wl = gen.make_workload("tiny_decode", device="cuda", M=5, E=4, H=256, I=64, top_k=2)
    else:  # every slot of every token names expert 3 (or an invalid id)
        wl = gen.make_workload("tiny_decode", device="cuda", M=4, E=6, top_k=4, fmt=gen.NVFP4)
        wl = _with_ids(wl, [[3, 3, 3, 3], [3, -1, 3, 6], [3, 3, 3, 3], [-1, -1, -1, -1]], seed=2)
    got = _run(wl, family)
    assert_layer_close(got, oracle_layer(wl), f"{case} family {family}")


@pytest.mark.parametrize("M", [8, 9, 12, 13, 17])
def test_band_boundary(M):
    """The last decode batch and the first batches past it, on the mid band's
    GEMMs (9 on)."""
    from fp4_weight_moe_gb300 import _capi
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=M)
    assert _capi.moe_fp4_debug_mid_band_of(wl.M, wl.E, wl.H, wl.I, wl.top_k) == (0 if M <= 8 else 3)
    got = _run(wl)
    if M <= 8:
        want = oracle_layer(wl)
    else:  # the mid band quantises the activations; the oracle mirrors it
        import oracle
        want, _, _, _ = oracle.forward_prefill(wl.x, wl.weights, wl.topk_ids, wl.topk_weights, wl.E, wl.H, wl.I,
                                               wl.top_k, fmt=wl.fmt)
    assert_layer_close(got, want, f"decode_e512 M={M}")
