"""Batches past the decode band (M > MOE_FP4_DECODE_MAX_M).

They run on the prefill band's GEMMs or on the mid band's swapped GEMMs
(weights on the MMA's 128-row side, an expert's routed rows on N), and on
request (a test switch) on the decode-band kernels over balanced chunks of
at most MOE_FP4_DECODE_MAX_M tokens.  The chunked path keeps the decode band's
numerics (BF16 activations, no activation quantisation), so it is held to
the unquantised FP64 oracle, and it must be bitwise the concatenation of the
chunks run as separate decode calls.  The prefill and mid bands quantise the
activations to NVFP4 and are held to the oracle that mirrors it.
"""
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, ensure_built, oracle_layer
from workload import gen

pytestmark = pytest.mark.gpu

PREFILL, CHUNKS, MID = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def _run(wl, mode, ids=None, tw=None, x=None):
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    xx = wl.x if x is None else x
    M = xx.shape[0]
    ws = m.alloc_workspace(max(M, 1), wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    out = torch.full((M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    prev = _capi.moe_fp4_debug_set_mid_band(mode)
    try:
        m.forward(xx, pw, wl.topk_ids if ids is None else ids, wl.topk_weights if tw is None else tw, out=out,
                  workspace=ws)
        torch.cuda.synchronize()
    finally:
        _capi.moe_fp4_debug_set_mid_band(prev)
    return out


@pytest.mark.parametrize("name,ov", [("decode_e512", dict(E=48, M=9)), ("decode_e512", dict(E=64, M=16)),
                                     ("decode_e288_m4", dict(E=40, M=13)), ("tiny_decode", dict(M=24, E=10,
                                                                                               top_k=3))])
def test_chunked_mid_band_parity(name, ov):
    wl = gen.make_workload(name, device="cuda", **ov)
    got = _run(wl, CHUNKS)
    assert_layer_close(got, oracle_layer(wl), f"{name} {ov} chunked")


def test_chunks_equal_separate_decode_calls():
    wl = gen.make_workload("decode_e512", device="cuda", E=40, M=11)
    whole = _run(wl, CHUNKS)
    # balanced chunks of 11 tokens: 5 + 6
    parts = [_run(wl, CHUNKS, ids=wl.topk_ids[a:b].contiguous(), tw=wl.topk_weights[a:b].contiguous(),
                  x=wl.x[a:b].contiguous()) for a, b in ((0, 5), (5, 11))]
    assert torch.equal(whole.view(torch.int16), torch.cat(parts).view(torch.int16))


@pytest.mark.parametrize("M", [9, 16])
def test_mid_band_prefill_mode(M):
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=M)
    got = _run(wl, PREFILL)
    want, _, _, _ = oracle.forward_prefill(wl.x, wl.weights, wl.topk_ids, wl.topk_weights, wl.E, wl.H, wl.I,
                                           wl.top_k, fmt=wl.fmt)
    assert_layer_close(got, want, f"decode_e512 M={M} prefill band")


def test_int64_ids_through_chunks():
    wl = gen.make_workload("decode_e512", device="cuda", E=48, M=12)
    a = _run(wl, CHUNKS)
    b = _run(wl, CHUNKS, ids=wl.topk_ids.long())
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# The mid band on the decode workloads' expert shapes: routed rows per expert
# from about one (N = 16) to past a 128-row routing tile, invalid slots,
# MXFP4 and NVFP4 weights.
@pytest.mark.parametrize("name,ov", [("decode_e512", dict(M=64)), ("decode_e512", dict(E=64, M=200)),
                                     ("decode_e288_m4", dict(E=96, M=40)),
                                     ("decode_e256", dict(E=16, H=2048, I=1024, M=24)),
                                     ("tiny_decode", dict(M=700, E=8, top_k=2)),
                                     # the smallest K of both GEMMs (H = 256: one stage without its second
                                     # box; I = 64: one scale group)
                                     ("tiny_decode", dict(M=40, E=3, H=256, I=64, top_k=2)),
                                     # FC2's K of 256 + 128 and 256 + 64 (one stage, its second box ragged),
                                     # and 512 + 64 (a second stage of one scale group)
                                     ("tiny_decode", dict(M=90, E=6, H=512, I=384, top_k=3)),
                                     ("decode_e288_m4", dict(E=20, H=768, I=320, M=50, fmt=gen.MXFP4)),
                                     ("tiny_decode", dict(M=70, E=5, H=256, I=576, top_k=2)),
                                     # every expert on every token, past the one-kernel routing's 8192
                                     # entries (the three-kernel routing with 32-row tiles)
                                     ("tiny_decode", dict(M=600, E=16, H=512, I=192, top_k=16))])
def test_mid_band_swapped_gemms_parity(name, ov):
    wl = gen.make_workload(name, device="cuda", **ov)
    got = _run(wl, MID)
    want, _, _, _ = oracle.forward_prefill(wl.x, wl.weights, wl.topk_ids, wl.topk_weights, wl.E, wl.H, wl.I,
                                           wl.top_k, fmt=wl.fmt)
    assert_layer_close(got, want, f"{name} {ov} mid band")
    got64 = _run(wl, MID, ids=wl.topk_ids.long())
    assert_layer_close(got64, want, f"{name} {ov} mid band, int64 ids")


@pytest.mark.parametrize("M", [9, 32])
def test_mid_band_by_shape_matches_its_plan(M):
    """decode_e512 past 8 tokens runs the mid band's GEMMs by shape."""
    from fp4_weight_moe_gb300 import _capi
    wl = gen.make_workload("decode_e512", device="cuda", M=M)
    assert _capi.moe_fp4_debug_mid_band_of(wl.M, wl.E, wl.H, wl.I, wl.top_k) == MID
    got = _run(wl, 0)
    want, _, _, _ = oracle.forward_prefill(wl.x, wl.weights, wl.topk_ids, wl.topk_weights, wl.E, wl.H, wl.I,
                                           wl.top_k, fmt=wl.fmt)
    assert_layer_close(got, want, f"decode_e512 M={M} by shape")
