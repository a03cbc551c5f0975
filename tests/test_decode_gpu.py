"""Parity of the decode band (M <= 8) with the FP64 oracle, through the C ABI.

Covers: the resident-layout round trip (bitwise), dequantised weights
(bit-exact), every decode workload shape at oracle-friendly sizes spanning
several tiles and ragged K-block groups, the full-size workloads, invalid and
duplicate routes, all-invalid tokens, NaN-poisoned outputs, determinism,
untouched inputs, CUDA-graph replay and the workspace contract.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, compact_for_oracle, ensure_built, oracle_layer
from workload import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def fm():
    import fp4_weight_moe_gb300 as m
    return m


def _prepare(wl):
    return fm().prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)


def _run(wl, pw=None, out=None, ws=None):
    m = fm()
    pw = pw or _prepare(wl)
    ws = ws if ws is not None else m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    return m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, out=out, workspace=ws)


# ------------------------------------------------------------------ resident layout
@pytest.mark.parametrize("fmt", [gen.MXFP4, gen.NVFP4])
@pytest.mark.parametrize("H,I", [(256, 128), (512, 320)])
def test_prepare_round_trip(fmt, H, I):
    wl = gen.make_workload("tiny_decode", device="cuda", fmt=fmt, E=3, H=H, I=I)
    pw = _prepare(wl)
    back = fm().unprepare_weights(pw)
    torch.cuda.synchronize()
    for k in ("w13", "s13", "w2", "s2") + (("g13", "g2") if fmt == gen.NVFP4 else ()):
        assert torch.equal(back[k], wl.weights[k]), k


@pytest.mark.parametrize("fmt", [gen.MXFP4, gen.NVFP4])
def test_dequant_bit_exact(fmt):
    wl = gen.make_workload("tiny_decode", device="cuda", fmt=fmt, E=3, H=512, I=320)
    pw = _prepare(wl)
    B = gen.BLOCK[fmt]
    w = {k: v.cpu().numpy() for k, v in wl.weights.items()}
    for e in range(wl.E):
        for which in (0, 1):
            got = fm().debug_dequant(pw, which, e).cpu().numpy()
            if which == 0:
                rows = []
                for proj, sl in ((0, slice(0, wl.I)), (1, slice(wl.I, 2 * wl.I))):
                    g = float(w["g13"][e, proj]) if fmt == gen.NVFP4 else 1.0
                    rows.append(oracle.dequant(w["w13"][e, sl], w["s13"][e, sl], wl.H, fmt, g))
                want = np.concatenate(rows)
            else:
                g = float(w["g2"][e]) if fmt == gen.NVFP4 else 1.0
                want = oracle.dequant(w["w2"][e], w["s2"][e], wl.I, fmt, g)
            # FP64 product rounded once to FP32 must equal the kernel's bits
            assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32)), (e, which, B)


def test_mx_scale_range_in_resident_layout():
    """MXFP4 block scales are carried as E4M3 powers of two relative to a
    per-projection power-of-two multiplier: exactly within 2^17 of the
    projection's largest block scale, as zero below (the resident layout's
    documented limit)."""
    E, H, I = 1, 256, 128
    w = gen.make_expert_weights(E, H, I, gen.MXFP4, 11, device="cuda")
    for key, rows, kb in (("s13", 2 * I, H // 32), ("s2", H, I // 32)):
        exps = 140 - (torch.arange(rows * kb, device="cuda") % 30)  # 140 .. 111 in every projection
        w[key] = exps.reshape(1, rows, kb).to(torch.uint8)
    pw = fm().prepare_weights(w, E, H, I, gen.MXFP4)
    wn = {k: v.cpu().numpy() for k, v in w.items() if v is not None}
    for which, (wk, sk, K) in enumerate((("w13", "s13", H), ("w2", "s2", I))):
        got = fm().debug_dequant(pw, which, 0).cpu().numpy()
        want = oracle.dequant(wn[wk][0], wn[sk][0], K, gen.MXFP4, 1.0)
        blk_exp = np.repeat(wn[sk][0].astype(np.int64), 32, axis=1)
        keep = blk_exp >= 140 - 17
        assert np.array_equal(got[keep], want[keep].astype(np.float32)), which
        assert not np.any(got[~keep]), which
    back = fm().unprepare_weights(pw)
    s_back = back["s13"].cpu().numpy()[0]
    kept = wn["s13"][0] >= 123
    assert np.array_equal(s_back[kept], wn["s13"][0][kept])


# ------------------------------------------------------------------ layer parity
DECODE_CASES = [
    # name, overrides
    ("tiny_decode", {}),
    ("tiny_decode", dict(fmt=gen.NVFP4)),
    ("tiny_decode", dict(M=3, E=16, top_k=4)),
    ("decode_e512", dict(E=24)),                      # NVFP4, H=2560 (split K), I=320
    ("decode_e512", dict(E=24, fmt=gen.MXFP4)),       # MX with a ragged K-block group in FC2
    ("decode_e512", dict(E=40, M=8)),
    ("decode_e288_m4", dict(E=24)),                   # 2 invalid slots (-1 and E)
    ("decode_e288_m4", dict(E=24, M=8, fmt=gen.NVFP4)),
    ("decode_e256", dict(E=12, H=1792, I=512, M=2)),  # Zipf routing
    ("decode_e256", dict(E=12, H=1792, I=512, M=5, fmt=gen.NVFP4)),
]


GEMV, TC, FUSED = 1, 2, 3  # decode plans (streaming GEMV, tcgen05 launch chain, tcgen05 single launch)
FAMILY_IDS = {GEMV: "gemv", TC: "chain", FUSED: "single"}


class decode_family:
    """Route the decode band through one kernel family inside a with-block."""

    def __init__(self, family):
        self.family = family

    def __enter__(self):
        from fp4_weight_moe_gb300 import _capi
        self.prev = _capi.moe_fp4_debug_set_decode_family(self.family)

    def __exit__(self, *exc):
        from fp4_weight_moe_gb300 import _capi
        _capi.moe_fp4_debug_set_decode_family(self.prev)


def _fits_gemv(wl):
    from fp4_weight_moe_gb300 import _capi
    return _capi.moe_fp4_debug_decode_gemv_fits(wl.M, wl.E, wl.H, wl.I, wl.top_k)


def _fits_single(wl):
    from fp4_weight_moe_gb300 import _capi
    with decode_family(FUSED):
        return _capi.moe_fp4_debug_decode_family_of(wl.M, wl.E, wl.H, wl.I, wl.top_k) == FUSED


def _skip_unless_fits(wl, family):
    if family == GEMV and not _fits_gemv(wl):
        pytest.skip("shape outside the streaming GEMV kernels' shared memory (served by tcgen05)")
    if family == FUSED and not _fits_single(wl):
        pytest.skip("grid of the single-launch plan not resident at once on this GPU (served by the chain)")


@pytest.mark.parametrize("family", [GEMV, TC, FUSED], ids=lambda f: FAMILY_IDS[f])
@pytest.mark.parametrize("name,ov", DECODE_CASES, ids=[f"{n}-{i}" for i, (n, _) in enumerate(DECODE_CASES)])
def test_decode_parity(name, ov, family):
    wl = gen.make_workload(name, device="cuda", **ov)
    _skip_unless_fits(wl, family)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    with decode_family(family):
        got = _run(wl, out=out)
        torch.cuda.synchronize()
    assert_layer_close(got, oracle_layer(wl), f"{name} {ov} family {family}")


@pytest.mark.parametrize("name,ov", [("decode_e512", dict(E=64, M=8)), ("decode_e288_m4", dict(E=24)),
                                     ("tiny_decode", dict(M=8, E=4, top_k=4, fmt=gen.NVFP4))])
def test_families_agree(name, ov):
    """The two families compute the same layer: their outputs agree within
    the parity bound (they sum in different orders)."""
    wl = gen.make_workload(name, device="cuda", **ov)
    with decode_family(GEMV):
        a = _run(wl).clone()
    with decode_family(TC):
        b = _run(wl).clone()
    torch.cuda.synchronize()
    assert_layer_close(a, b.float().cpu().double().numpy(), f"{name} gemv vs tc")


def test_duplicate_and_invalid_routes():
    wl = gen.make_workload("tiny_decode", device="cuda", M=4, E=6, top_k=4)
    ids = torch.tensor([[0, 0, 3, -1], [5, 6, 2, 2], [1, 1, 1, 1], [-5, 100, 6, 4]], dtype=torch.int32)
    wl.topk_ids = ids.cuda()
    wl.topk_weights = torch.rand((4, 4), generator=torch.Generator().manual_seed(0)).cuda()
    got = _run(wl)
    torch.cuda.synchronize()
    assert_layer_close(got, oracle_layer(wl), "duplicates/invalid")


def test_all_invalid_gives_exact_zero():
    wl = gen.make_workload("tiny_decode", device="cuda", M=3, E=8, top_k=2)
    wl.topk_ids = torch.tensor([[-1, 8], [9, -3], [-1, -1]], dtype=torch.int32, device="cuda")
    out = torch.full((3, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = _run(wl, out=out)
    torch.cuda.synchronize()
    assert torch.all(got.float() == 0) and not torch.any(torch.signbit(got.float()))


def test_deterministic_and_inputs_untouched():
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=4)
    pw = _prepare(wl)
    snap = [t.clone() for t in (wl.x, wl.topk_ids, wl.topk_weights, pw.w13, pw.s13, pw.w2, pw.s2)]
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    a = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws).clone()
    b = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for s, t in zip(snap, (wl.x, wl.topk_ids, wl.topk_weights, pw.w13, pw.s13, pw.w2, pw.s2)):
        assert torch.equal(s, t)


def test_library_workspace_and_graph_replay():
    m = fm()
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=2)
    pw = _prepare(wl)
    m.reserve_workspace(8, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    eager = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, out=out)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_workspace_too_small_is_rejected():
    m = fm()
    wl = gen.make_workload("tiny_decode", device="cuda")
    pw = _prepare(wl)
    n = m.workspace_bytes(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    small = torch.zeros(n - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MoeFp4Error) as ei:
        m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=small)
    assert ei.value.status == 4


# ------------------------------------------------------------------ full-size workloads
FULL = [
    ("decode_e512", {}),
    ("decode_e288_m4", {}),
]


@pytest.mark.parametrize("family", [GEMV, TC, FUSED], ids=lambda f: FAMILY_IDS[f])
@pytest.mark.parametrize("name,ov", FULL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(FULL)])
def test_decode_full_size(name, ov, family):
    wl = gen.make_workload(name, device="cuda", **ov)
    _skip_unless_fits(wl, family)
    with decode_family(family):
        got = _run(wl)
        torch.cuda.synchronize()
    assert_layer_close(got, oracle_layer(wl), f"{name} {ov} family {family}")
    del wl
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", [gen.MXFP4, gen.NVFP4], ids=["mxfp4", "nvfp4"])
def test_decode_e256_full_size_every_batch(fmt):
    """The full E=256, H=7168, I=2048, top_k=8 layer (Zipf routing) at every
    batch of the sweep, M = 1, 2, 4, 8, in both weight formats, on the plan
    each batch takes by shape; the weights are drawn once per format."""
    m = fm()
    c = gen.CONFIGS["decode_e256"]
    E, H, I, k = c["E"], c["H"], c["I"], c["top_k"]
    seed = gen.CONFIG_SEED["decode_e256"]
    weights = gen.make_expert_weights(E, H, I, fmt, seed, device="cuda")
    pw = m.prepare_weights(weights, E, H, I, fmt)
    ws = m.alloc_workspace(8, E, H, I, k, fmt)
    for M in (1, 2, 4, 8):
        wl = gen.Workload(name="decode_e256", E=E, H=H, I=I, top_k=k, M=M, fmt=fmt, seed=seed, weights=weights,
                          x=gen.draw_activations(M, H, seed + 17 + M, device="cuda"),
                          topk_ids=None, topk_weights=None)
        ids, tw = gen.draw_routing(M, E, k, seed + 29 + M, mode="zipf")
        wl.topk_ids, wl.topk_weights = ids.cuda(), tw.cuda()
        got = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws)
        torch.cuda.synchronize()
        assert m.workspace_status(ws) == 0
        assert_layer_close(got, oracle_layer(wl), f"decode_e256 M={M} fmt={fmt}")
    del weights, pw, ws
    torch.cuda.empty_cache()

