"""Parity of the other gated activations with the FP64 oracle.

moe_fp4_forward_ex takes FC1's activation: SiLU (the layer's own), GELU in
its tanh form, and SwiGLU-OAI (alpha, beta, limit), the activations the SM12x
sync PR's kernels accept.  Each runs through the streaming-GEMV and the
tcgen05 decode kernels and the prefill band, against the oracle with the same
activation (the prefill band against the oracle's mirrored activation
quantisation).  The limit is chosen so that both clamps bind on part of the
outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, compact_for_oracle, ensure_built
from workload import gen

pytestmark = pytest.mark.gpu

GEMV, TC, SINGLE = 1, 2, 3  # decode plans: streaming GEMV, tcgen05 chain, tcgen05 single launch
ACTS = [("gelu_tanh", (oracle.ACT_GELU_TANH, 0.0, 0.0, 0.0)),
        ("swigluoai", (oracle.ACT_SWIGLUOAI, 1.702, 1.0, 0.25))]


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def _family(f):
    from fp4_weight_moe_gb300 import _capi
    return _capi.moe_fp4_debug_set_decode_family(f)


def _run(wl, act, family=0):
    import fp4_weight_moe_gb300 as m
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    prev = _family(family)
    try:
        m.forward_act(wl.x, pw, wl.topk_ids, wl.topk_weights, ws, *act, out=out)
        torch.cuda.synchronize()
    finally:
        _family(prev)
    return out


def _oracle_decode(wl, act):
    w, ids_c, E_c = compact_for_oracle(wl.weights, wl.topk_ids, wl.E, wl.fmt)
    return oracle.forward(wl.x, w, ids_c, wl.topk_weights, E_c, wl.H, wl.I, wl.top_k, wl.fmt, act=act)


@pytest.mark.parametrize("family", [GEMV, TC, SINGLE], ids=["gemv", "chain", "single"])
@pytest.mark.parametrize("name,ov", [("tiny_decode", dict(M=3, E=12, top_k=3)),
                                     ("decode_e512", dict(E=24)),
                                     ("decode_e288_m4", dict(E=24))])
@pytest.mark.parametrize("aname,act", ACTS, ids=[a for a, _ in ACTS])
def test_decode_activation_parity(name, ov, aname, act, family):
    wl = gen.make_workload(name, device="cuda", **ov)
    got = _run(wl, act, family)
    assert_layer_close(got, _oracle_decode(wl, act), f"{name} {ov} {aname} family {family}")


def test_silu_through_forward_ex_matches_forward_ws():
    import fp4_weight_moe_gb300 as m
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=2)
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    a = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws).clone()
    b = m.forward_act(wl.x, pw, wl.topk_ids, wl.topk_weights, ws, m.ACT_SILU)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("aname,act", ACTS, ids=[a for a, _ in ACTS])
@pytest.mark.parametrize("M,E,H,I,k", [(64, 8, 512, 256, 4), (24, 12, 512, 320, 4)])
def test_prefill_activation_parity(aname, act, M, E, H, I, k):
    import fp4_weight_moe_gb300 as m
    fmt = gen.NVFP4
    weights = gen.make_expert_weights(E, H, I, fmt, 41 + M, device="cuda")
    x = gen.draw_activations(M, H, 42 + M, device="cuda")
    ids, tw = gen.draw_routing(M, E, k, 43 + M, mode="softmax")
    ids, tw = ids.cuda(), tw.cuda()
    pw = m.prepare_weights(weights, E, H, I, fmt)
    ws = m.alloc_workspace(M, E, H, I, k, fmt)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward_act(x, pw, ids, tw, ws, *act, out=out)
    torch.cuda.synchronize()
    want, _, _, _ = oracle.forward_prefill(x, weights, ids, tw, E, H, I, k, fmt=fmt, act=act)
    assert_layer_close(got, want, f"prefill {aname} M={M} I={I}")
    assert np.isfinite(got.float().cpu().numpy()).all()
