"""The W4A8-MX prefill band (MOE_FP4_PREFILL_W4A8_MX: MXFP4 weights, MXFP8
activations) on the GPU against the oracle's W4A8-MX definition, through the
C ABI, on both of its engines.

The band quantises x per token and h (staged in BF16) per routed row to MXFP8
(E4M3 elements, one UE8M0 scale per 32).  Where I % 128 == 0 both GEMMs run
on the FP8 tensor cores (tcgen05.mma kind::mxf8f6f4, the MXFP4 weights as
stored); otherwise, or with the engine switch at 0, on the 16-bit engine with
the MXFP8 values carried exactly; ``oracle.forward_w4a8`` is the same
definition in FP64.  Cases: several tiles per expert, I % 128 != 0, empty
experts, invalid and int64 ids, the three gated activations, outlier-heavy
activations (wide block exponents), a full-size E=128 / H=4096 / I=1536 /
M=4096 layer on sampled tokens; the mode's format and activation limits;
and the accuracy against the plain definition next to the other modes.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, compact_for_oracle, ensure_built, layer_metrics, oracle_layer
from workload import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


@pytest.fixture(params=[1, 0], ids=["fp8", "16bit"])
def engine(request):
    """The W4A8-MX engine: 1 the FP8 tensor cores where I % 128 == 0, 0 the
    16-bit engine."""
    c = fm()._capi
    prev = c.moe_fp4_debug_set_w4a8_engine(request.param)
    yield request.param
    c.moe_fp4_debug_set_w4a8_engine(prev)


def fm():
    import fp4_weight_moe_gb300 as m
    return m


def _run(wl, mode, ids=None, kind=0, alpha=0.0, beta=1.0, limit=0.0, pw=None):
    m = fm()
    if pw is None:
        pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace_mode(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, mode)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward_mode(wl.x, pw, wl.topk_ids if ids is None else ids, wl.topk_weights, ws, mode, kind=kind,
                         alpha=alpha, beta=beta, limit=limit, out=out)
    torch.cuda.synchronize()
    assert m.workspace_status(ws) == 0
    return got, pw


def _want(wl, tokens=None, act=None):
    ids = wl.topk_ids if tokens is None else wl.topk_ids[tokens]
    x = wl.x if tokens is None else wl.x[tokens]
    tw = wl.topk_weights if tokens is None else wl.topk_weights[tokens]
    sub, ids_c, Ec = compact_for_oracle(wl.weights, ids, wl.E, wl.fmt)
    return oracle.forward_w4a8(x, sub, ids_c, tw.cpu(), Ec, wl.H, wl.I, wl.top_k, act=act)


CASES = [  # M, E, H, I, top_k, invalid slots
    (9, 8, 256, 128, 2, 0),
    (40, 12, 512, 320, 4, 3),
    (300, 16, 1024, 256, 4, 20),
    (700, 48, 2560, 320, 8, 0),
    (200, 6, 2048, 768, 2, 0),
]


@pytest.mark.parametrize("M,E,H,I,k,invalid", CASES)
def test_w4a8_prefill_parity(M, E, H, I, k, invalid, engine):
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=M, E=E, H=H, I=I, top_k=k, fmt=gen.MXFP4)
    if invalid:
        ids, tw = gen.draw_routing(M, E, k, seed=M + E, n_invalid=invalid)
        wl.topk_ids, wl.topk_weights = ids.cuda(), tw.cuda()
    if E > 8:  # an expert without rows
        wl.topk_ids[wl.topk_ids == 5] = 6
    got, _ = _run(wl, m.PREFILL_W4A8_MX)
    want = _want(wl)
    assert_layer_close(got, want, f"W4A8-MX prefill M={M} E={E} H={H} I={I}")
    got64, _ = _run(wl, m.PREFILL_W4A8_MX, ids=wl.topk_ids.to(torch.int64))
    assert_layer_close(got64, want, f"W4A8-MX prefill, int64 ids, M={M}")


@pytest.mark.parametrize("kind,alpha,beta,limit", [(1, 0.0, 1.0, 0.0), (2, 1.702, 1.0, 7.0)])
def test_w4a8_prefill_activations(kind, alpha, beta, limit, engine):
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=96, E=10, H=1024, I=384, top_k=4, fmt=gen.MXFP4)
    got, _ = _run(wl, m.PREFILL_W4A8_MX, kind=kind, alpha=alpha, beta=beta, limit=limit)
    assert_layer_close(got, _want(wl, act=(kind, alpha, beta, limit)), f"W4A8-MX prefill, activation {kind}")


def test_w4a8_prefill_outlier_activations(engine):
    """Per 256-wide K stage two channels at 2^8 .. 2^12 and one block near
    2^-20 of the RMS: block exponents spread over the row."""
    from tests.test_hardening_gpu import outlier_activations
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=48, E=12, H=2560, I=384, top_k=4, fmt=gen.MXFP4)
    wl.x = outlier_activations(wl.M, wl.H, seed=9).cuda()
    got, _ = _run(wl, m.PREFILL_W4A8_MX)
    assert_layer_close(got, _want(wl), "W4A8-MX prefill, outlier activations")


def test_w4a8_prefill_full_size_sampled(engine):
    m = fm()
    wl = gen.make_workload("prefill_e128", device="cuda", fmt=gen.MXFP4)
    got, _ = _run(wl, m.PREFILL_W4A8_MX)
    ids = wl.topk_ids.cpu().numpy()
    tokens = set(range(0, wl.M, wl.M // 24))
    for e in range(wl.E):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if rows.size:
            tokens.update((int(rows[0]), int(rows[-1])))
    tokens = sorted(tokens)
    assert_layer_close(got[tokens], _want(wl, tokens=tokens), "prefill_e128 MXFP4 W4A8-MX band, sampled")


def test_w4a8_mode_limits():
    """NVFP4 weights and non-gated experts are not part of the mode."""
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=32, E=8, H=512, I=128, top_k=2, fmt=gen.NVFP4)
    assert m._capi.moe_fp4_workspace_bytes_mode(32, 8, 512, 128, 2, gen.NVFP4, m.PREFILL_W4A8_MX) == 0
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace_mode(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, m.PREFILL_BF16)
    with pytest.raises(m.MoeFp4Error):
        m.forward_mode(wl.x, pw, wl.topk_ids, wl.topk_weights, ws, m.PREFILL_W4A8_MX)
    w = gen.make_relu2_weights(8, 512, 128, gen.MXFP4, 3, device="cuda")
    pr = m.prepare_weights_relu2(w, 8, 512, 128, gen.MXFP4)
    with pytest.raises(m.MoeFp4Error):
        m.forward_mode(wl.x, pr, wl.topk_ids, wl.topk_weights, ws, m.PREFILL_W4A8_MX, kind=m.ACT_RELU2)


def test_w4a8_accuracy_between_exact_and_nvfp4():
    """Against the plain FP64 layer the W4A8-MX band sits between the exact
    BF16 band and the NVFP4-activation band (MXFP8 keeps three mantissa bits
    per element where NVFP4 keeps one)."""
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=256, E=16, H=2048, I=512, top_k=4, fmt=gen.MXFP4)
    got_mx, pw = _run(wl, m.PREFILL_W4A8_MX)
    got_x, _ = _run(wl, m.PREFILL_BF16, pw=pw)
    prev = m._capi.moe_fp4_debug_set_mid_band(1)
    try:
        got_q, _ = _run(wl, m.PREFILL_NVFP4, pw=pw)
    finally:
        m._capi.moe_fp4_debug_set_mid_band(prev)
    want = oracle_layer(wl)
    cx, _, _ = layer_metrics(got_x, want)
    cm, _, _ = layer_metrics(got_mx, want)
    cq, _, _ = layer_metrics(got_q, want)
    print(f"cosine vs the plain FP64 layer: exact {cx:.8f}, W4A8-MX {cm:.8f}, NVFP4 activations {cq:.8f}")
    assert cx > cm > cq
