"""The exact-numerics prefill band (MOE_FP4_PREFILL_BF16) on the GPU against
the plain FP64 definition of the layer, through the C ABI.

This band quantises no activation: x keeps its BF16 values (carried in FP16
rows scaled by a power of two), the FP4 weights are decoded to FP16 exactly,
both GEMMs sum in FP32 on the FP16 tensor cores and only h (staged in BF16
for FC2) and the output are rounded.  So it is compared with
``oracle.forward`` / ``oracle.forward_relu2`` (the decode band's reference:
no activation quantisation anywhere), not with the mirrored-quantisation
prefill definition.  Cases: several tiles per expert, I % 128 != 0 (a
half-used last tile of the non-gated w1), empty experts, invalid ids, both
weight formats, all activations, int64 ids, the full E=128 / H=4096 /
I=1536 / M=4096 layer on sampled tokens, and the accuracy against the NVFP4
band on the same inputs.
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


def fm():
    import fp4_weight_moe_gb300 as m
    return m


def _run_exact(wl, ids=None, kind=None, alpha=0.0, beta=1.0, limit=0.0, pw=None, relu2=False):
    m = fm()
    if pw is None:
        prep = m.prepare_weights_relu2 if relu2 else m.prepare_weights
        pw = prep(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace_mode(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, m.PREFILL_BF16)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward_mode(wl.x, pw, wl.topk_ids if ids is None else ids, wl.topk_weights, ws, m.PREFILL_BF16,
                         kind=m.ACT_RELU2 if relu2 else (m.ACT_SILU if kind is None else kind), alpha=alpha, beta=beta,
                         limit=limit, out=out)
    torch.cuda.synchronize()
    assert m.workspace_status(ws) == 0
    return got, pw


CASES = [  # M, E, H, I, top_k, fmt, invalid slots
    (9, 8, 256, 128, 2, gen.NVFP4, 0),
    (40, 12, 512, 320, 4, gen.NVFP4, 3),
    (300, 16, 1024, 256, 4, gen.MXFP4, 20),
    (1000, 64, 2560, 320, 8, gen.NVFP4, 0),
    (200, 6, 2048, 768, 2, gen.MXFP4, 0),
]


@pytest.mark.parametrize("M,E,H,I,k,fmt,invalid", CASES)
def test_exact_prefill_parity(M, E, H, I, k, fmt, invalid):
    wl = gen.make_workload("decode_e512", device="cuda", M=M, E=E, H=H, I=I, top_k=k, fmt=fmt)
    if invalid:
        ids, tw = gen.draw_routing(M, E, k, seed=M + E, n_invalid=invalid)
        wl.topk_ids, wl.topk_weights = ids.cuda(), tw.cuda()
    if E > 8:  # an expert without rows
        wl.topk_ids[wl.topk_ids == 5] = 6
    got, _ = _run_exact(wl)
    assert_layer_close(got, oracle_layer(wl), f"exact prefill M={M} E={E} H={H} I={I}")
    # int64 ids: the same layer (FC2's FP32 reductions land in any order, so
    # the tolerance rather than bit equality)
    got64, _ = _run_exact(wl, ids=wl.topk_ids.to(torch.int64))
    assert_layer_close(got64, oracle_layer(wl), f"exact prefill, int64 ids, M={M}")


@pytest.mark.parametrize("kind,alpha,beta,limit", [(1, 0.0, 1.0, 0.0), (2, 1.702, 1.0, 7.0)])
def test_exact_prefill_activations(kind, alpha, beta, limit):
    M, E, H, I, k = 96, 10, 1024, 384, 4
    wl = gen.make_workload("decode_e512", device="cuda", M=M, E=E, H=H, I=I, top_k=k)
    got, _ = _run_exact(wl, kind=kind, alpha=alpha, beta=beta, limit=limit)
    sub, ids_c, Ec = compact_for_oracle(wl.weights, wl.topk_ids, wl.E, wl.fmt)
    want = oracle.forward(wl.x, sub, ids_c, wl.topk_weights.cpu(), Ec, H, I, k, wl.fmt, act=(kind, alpha, beta, limit))
    assert_layer_close(got, want, f"exact prefill, activation {kind}")


@pytest.mark.parametrize("M,E,H,I,k,fmt", [(40, 12, 512, 320, 4, gen.NVFP4), (64, 8, 1024, 256, 2, gen.MXFP4),
                                           (130, 5, 768 + 256, 192, 3, gen.NVFP4)])
def test_exact_prefill_relu2(M, E, H, I, k, fmt):
    w = gen.make_relu2_weights(E, H, I, fmt, M + 1, device="cuda")
    x = gen.draw_activations(M, H, M + 2, device="cuda")
    ids, tw = gen.draw_routing(M, E, k, M + 3, n_invalid=2)
    wl = gen.Workload(name="relu2", E=E, H=H, I=I, top_k=k, M=M, fmt=fmt, seed=M + 1, weights=w, x=x,
                      topk_ids=ids.cuda(), topk_weights=tw.cuda())
    got, _ = _run_exact(wl, relu2=True)
    used = sorted({int(e) for e in ids.reshape(-1).tolist() if 0 <= e < E}) or [0]
    remap = {e: j for j, e in enumerate(used)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids.tolist()], dtype=np.int32)
    sub = {kk: v.index_select(0, torch.tensor(used, device="cuda")).cpu().numpy() for kk, v in w.items()}
    want = oracle.forward_relu2(x, sub, ids_c, tw, len(used), H, I, k, fmt)
    assert_layer_close(got, want, f"exact prefill relu2 M={M} E={E} H={H} I={I}")


def test_exact_prefill_more_accurate_than_nvfp4_band():
    """On the same layer the exact band sits much closer to the plain
    definition than the NVFP4-activation band (which quantises x and h)."""
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=256, E=16, H=2048, I=512, top_k=4)
    got_exact, pw = _run_exact(wl)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    prev = m._capi.moe_fp4_debug_set_mid_band(1)
    try:
        got_q = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws)
        torch.cuda.synchronize()
    finally:
        m._capi.moe_fp4_debug_set_mid_band(prev)
    want = oracle_layer(wl)
    ce, me, rms = layer_metrics(got_exact, want)
    cq, mq, _ = layer_metrics(got_q, want)
    print(f"vs the plain FP64 layer: exact band cosine {ce:.8f} max/rms {me / rms:.3e}; "
          f"NVFP4 band cosine {cq:.8f} max/rms {mq / rms:.3e}")
    assert 1.0 - ce < 0.2 * (1.0 - cq)
    assert me < mq


def test_exact_prefill_decode_sizes_take_the_decode_band():
    """Batches of at most eight tokens run the decode band in either mode."""
    for M in (1, 8):
        wl = gen.make_workload("decode_e512", device="cuda", M=M, E=24)
        got, _ = _run_exact(wl)
        assert_layer_close(got, oracle_layer(wl), f"forward_mode M={M}")


def test_exact_prefill_full_size_sampled():
    wl = gen.make_workload("prefill_e128", device="cuda")
    got, _ = _run_exact(wl)
    ids = wl.topk_ids.cpu().numpy()
    tokens = set(range(0, wl.M, wl.M // 24))
    for e in range(wl.E):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if rows.size:
            tokens.update((int(rows[0]), int(rows[-1])))
    tokens = sorted(tokens)
    sub, ids_c, Ec = compact_for_oracle(wl.weights, wl.topk_ids[tokens], wl.E, wl.fmt)
    want = oracle.forward(wl.x[tokens], sub, ids_c, wl.topk_weights[tokens].cpu(), Ec, wl.H, wl.I, wl.top_k, wl.fmt)
    assert_layer_close(got[tokens], want, "prefill_e128 exact band, sampled")


def test_exact_prefill_rejects_small_workspace():
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", M=64, E=8, H=512, I=128, top_k=2)
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    n_q = m._capi.moe_fp4_workspace_bytes_mode(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, m.PREFILL_NVFP4)
    n_x = m._capi.moe_fp4_workspace_bytes_mode(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt, m.PREFILL_BF16)
    assert n_x > n_q
    ws = torch.zeros(n_q, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeFp4Error):
        m.forward_mode(wl.x, pw, wl.topk_ids, wl.topk_weights, ws, m.PREFILL_BF16)
