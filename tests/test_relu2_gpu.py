"""Non-gated experts with the squared ReLU (h = max(x . W1[e][n], 0)^2) on the
GPU against the FP64 oracle, through the C ABI: the resident layout's round
trip (bitwise) and dequantised w1 (bit-exact), the decode band (tcgen05
launch chain; int32 and int64 ids, invalid slots, several batches, a w1 whose
last 128-row tile is half padding), and the prefill band against its
mirrored oracle (NVFP4 activations, h staged in BF16 and quantised with the
exact row quantiser).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, ensure_built
from workload import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def fm():
    import fp4_weight_moe_gb300 as m
    return m


def _case(E, H, I, k, M, fmt, seed, invalid=0):
    w = gen.make_relu2_weights(E, H, I, fmt, seed, device="cuda")
    x = gen.draw_activations(M, H, seed + 1, device="cuda")
    ids, tw = gen.draw_routing(M, E, k, seed + 2, n_invalid=invalid or None)
    return w, x, ids.cuda(), tw.cuda()


def _oracle(w, x, ids, tw, E, H, I, k, fmt, prefill=False):
    used = sorted({int(e) for e in ids.reshape(-1).tolist() if 0 <= e < E}) or [0]
    remap = {e: j for j, e in enumerate(used)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids.tolist()], dtype=np.int32)
    idx = torch.tensor(used, dtype=torch.long, device=w["w1"].device)
    sub = {kk: v.index_select(0, idx).cpu().numpy() for kk, v in w.items()}
    f = oracle.forward_prefill_relu2 if prefill else oracle.forward_relu2
    return f(x, sub, ids_c, tw.cpu(), len(used), H, I, k, fmt)


@pytest.mark.parametrize("fmt", [gen.MXFP4, gen.NVFP4])
@pytest.mark.parametrize("H,I", [(256, 128), (512, 320)])
def test_relu2_prepare_round_trip_and_dequant(fmt, H, I):
    m = fm()
    E = 3
    w = gen.make_relu2_weights(E, H, I, fmt, 5, device="cuda")
    pw = m.prepare_weights_relu2(w, E, H, I, fmt)
    back = m.unprepare_weights_relu2(pw)
    torch.cuda.synchronize()
    for kk in ("w1", "s1", "w2", "s2") + (("g1", "g2") if fmt == gen.NVFP4 else ()):
        assert torch.equal(back[kk], w[kk]), kk
    wn = {kk: v.cpu().numpy() for kk, v in w.items()}
    for e in range(E):
        got = m.debug_dequant(pw, 2, e).cpu().numpy()
        g = float(wn["g1"][e]) if fmt == gen.NVFP4 else 1.0
        want = oracle.dequant(wn["w1"][e], wn["s1"][e], H, fmt, g)
        assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32)), e


DECODE = [  # E, H, I, top_k, M, fmt, invalid slots
    (8, 256, 128, 2, 1, gen.MXFP4, 0),
    (16, 512, 320, 4, 3, gen.NVFP4, 1),
    (24, 2560, 320, 10, 1, gen.NVFP4, 0),
    (24, 2560, 320, 10, 4, gen.MXFP4, 2),
    (16, 4096, 512, 10, 2, gen.MXFP4, 1),
    (12, 1792, 512, 8, 8, gen.NVFP4, 0),
]


@pytest.mark.parametrize("E,H,I,k,M,fmt,invalid", DECODE)
def test_relu2_decode_parity(E, H, I, k, M, fmt, invalid):
    m = fm()
    w, x, ids, tw = _case(E, H, I, k, M, fmt, seed=E * 7 + M, invalid=invalid)
    pw = m.prepare_weights_relu2(w, E, H, I, fmt)
    ws = m.alloc_workspace(M, E, H, I, k, fmt)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward_act(x, pw, ids, tw, ws, kind=m.ACT_RELU2, out=out)
    torch.cuda.synchronize()
    assert m.workspace_status(ws) == 0
    assert_layer_close(got, _oracle(w, x, ids, tw, E, H, I, k, fmt), f"relu2 decode E={E} H={H} I={I} M={M}")
    # int64 ids: the same result bitwise (the decode kernels are deterministic)
    got64 = m.forward_act(x, pw, ids.to(torch.int64), tw, ws, kind=m.ACT_RELU2)
    torch.cuda.synchronize()
    assert torch.equal(got64.view(torch.int16), got.view(torch.int16))


@pytest.mark.parametrize("band", [1, 3], ids=["prefill", "mid"])
@pytest.mark.parametrize("M,E,H,I,k,fmt", [(40, 12, 512, 320, 4, gen.NVFP4), (64, 8, 1024, 256, 2, gen.MXFP4),
                                           (24, 6, 256, 128, 3, gen.NVFP4), (300, 4, 512, 192, 2, gen.NVFP4)])
def test_relu2_prefill_parity(M, E, H, I, k, fmt, band):
    m = fm()
    w, x, ids, tw = _case(E, H, I, k, M, fmt, seed=M + E)
    pw = m.prepare_weights_relu2(w, E, H, I, fmt)
    ws = m.alloc_workspace(M, E, H, I, k, fmt)
    # batches past 8 tokens: the prefill band's GEMMs, or the mid band's
    prev = m._capi.moe_fp4_debug_set_mid_band(band)
    try:
        got = m.forward_act(x, pw, ids, tw, ws, kind=m.ACT_RELU2)
        torch.cuda.synchronize()
    finally:
        m._capi.moe_fp4_debug_set_mid_band(prev)
    assert m.workspace_status(ws) == 0
    want = _oracle(w, x, ids, tw, E, H, I, k, fmt, prefill=True)
    assert_layer_close(got, want, f"relu2 prefill M={M} E={E} H={H} I={I}")
