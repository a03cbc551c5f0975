"""Parity of the prefill band (M > 8) with the oracle, through the C ABI.

* routing compaction: perm and expert offsets bit-exact against the oracle's
  stable counting sort (invalid ids excluded);
* the NVFP4 activation quantiser: codes, scale bytes and FP32 multipliers
  bit-exact against the oracle's FP32 quantiser;
* the layer: against the oracle's mirrored-quantisation prefill definition
  (x quantised per token, h = SiLU(gate)*up staged in BF16 and quantised per
  routed row), within the layer tolerance; shapes with several tiles per
  expert, empty experts, invalid ids and ragged row counts; and the full
  E=128/H=4096/I=1536/M=4096 workload on sampled tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, compact_for_oracle, ensure_built, layer_metrics
from workload import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True, params=[1, 3], ids=["prefill", "mid"])
def _build(request):
    """Build, and send every batch past the decode band to one set of GEMMs:
    the prefill band's (routed rows on the MMA's 128-row side) or the mid
    band's (weights there, an expert's routed rows on N).  Both compute the
    same layer, so every case here runs on both."""
    ensure_built()
    from fp4_weight_moe_gb300 import _capi as c
    prev = c.moe_fp4_debug_set_mid_band(request.param)
    yield
    c.moe_fp4_debug_set_mid_band(prev)


def fm():
    import fp4_weight_moe_gb300 as m
    return m


def _capi():
    from fp4_weight_moe_gb300 import _capi as c
    return c


@pytest.mark.parametrize("M,E,k", [(16, 8, 2), (300, 16, 4), (1000, 64, 8), (600, 512, 10), (4096, 128, 8)])
def test_route_bit_exact(M, E, k):
    rng = np.random.default_rng(M + E)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    ids[rng.random((M, k)) < 0.03] = -1
    ids[rng.random((M, k)) < 0.03] = E + 3
    if E > 8:
        ids[ids == 5] = 6  # expert 5 gets no rows
    c = _capi()
    dev = torch.device("cuda")
    tids = torch.from_numpy(ids).to(dev)
    perm = torch.empty(M * k, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    nws = c.moe_fp4_debug_route_workspace_bytes(M, E, k)
    ws = torch.zeros(nws, dtype=torch.uint8, device=dev)
    c.moe_fp4_debug_route(tids.data_ptr(), M, E, k, perm.data_ptr(), off.data_ptr(), ws.data_ptr(), nws,
                          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want_perm, want_off = oracle.route(ids, E)
    assert np.array_equal(off.cpu().numpy(), want_off)
    n = int(want_off[-1])
    got = perm.cpu().numpy()
    assert np.array_equal(got[:n], want_perm)
    assert np.all(got[n:] == -1)
    if M * k > 8192:
        return
    # the single-CTA routing of small batches: the same offsets, and per
    # expert the same entries (in the order they won the expert's counter)
    perm.fill_(-7)
    off.fill_(-7)
    c.moe_fp4_debug_route_small(tids.data_ptr(), M, E, k, perm.data_ptr(), off.data_ptr(), ws.data_ptr(), nws,
                                torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(off.cpu().numpy(), want_off)
    got = perm.cpu().numpy()
    for e in range(E):
        a, b = int(want_off[e]), int(want_off[e + 1])
        assert np.array_equal(np.sort(got[a:b]), np.sort(want_perm[a:b])), e
    assert np.all(got[n:] == -1)


def test_quant_rows_bit_exact():
    rng = np.random.default_rng(7)
    rows, K = 64, 512
    a = (rng.standard_normal((rows, K)) * np.exp(rng.uniform(-8, 8, (rows, 1)))).astype(np.float32)
    a[3] = 0.0                                            # all-zero row
    a[4, :16] = 0.0                                       # one all-zero block
    a[5] = (np.float32(1e-30) * rng.standard_normal(K)).astype(np.float32)  # tiny row
    a[6, ::7] = np.float32(5.0)                           # exact ties after scaling
    a[7] = np.round(a[7] * 4) / 4
    # G = 1 (row max 2688) and a block with block max 6 (scale 1): the
    # quotients are the values themselves, placed on every E2M1 rounding
    # midpoint and one unit in the last place to either side of it
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    a[8] = 0.0
    a[8, 0] = 2688.0
    a[8, 16:32] = np.concatenate([[6.0], mids, -mids, [-6.0]])
    a[8, 32:48] = np.concatenate([[6.0], np.nextafter(mids, np.float32(np.inf)),
                                  -np.nextafter(mids, np.float32(0)), [0.0]])
    a[8, 48:64] = np.concatenate([[6.0], np.nextafter(mids, np.float32(0)),
                                  -np.nextafter(mids, np.float32(np.inf)), [-0.0]])
    c = _capi()
    dev = torch.device("cuda")
    ta = torch.from_numpy(a).to(dev)
    q = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    g = torch.empty(rows, dtype=torch.float32, device=dev)
    c.moe_fp4_debug_quant_rows(ta.data_ptr(), rows, K, q.data_ptr(), s.data_ptr(), g.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    qg, sg, gg = q.cpu().numpy(), s.cpu().numpy(), g.cpu().numpy()
    for r in range(rows):
        wq, ws_, wg = oracle.quant_nvfp4_row(a[r])
        assert np.float32(gg[r]).view(np.uint32) == np.float32(wg).view(np.uint32), r
        assert np.array_equal(sg[r], ws_), r
        assert np.array_equal(qg[r], wq), r


def _prefill_case(M, E, H, I, k, seed, invalid=0.0, fmt=gen.NVFP4):
    w = gen.make_expert_weights(E, H, I, fmt, seed, device="cuda")
    x = gen.draw_activations(M, H, seed + 1, device="cuda")
    ids, tw = gen.draw_routing(M, E, k, seed + 2)
    if invalid:
        rng = np.random.default_rng(seed)
        idn = ids.numpy()
        idn[rng.random(idn.shape) < invalid] = -1
        ids = torch.from_numpy(idn)
    return w, x, ids.cuda(), tw.cuda()


# The last cases have I % 256 != 0: FC1 runs 128-wide tiles (2I % 256 != 0)
# and FC2's last K stage holds 1 or 2 of 4 groups (I = 320, 128), the
# shapes of the decode workloads above 8 tokens (the mid band).
@pytest.mark.parametrize("M,E,H,I,k,invalid,fmt", [(16, 4, 256, 256, 2, 0.0, gen.NVFP4),
                                                   (200, 8, 512, 256, 4, 0.05, gen.NVFP4),
                                                   (600, 6, 768, 512, 3, 0.0, gen.NVFP4),
                                                   (300, 8, 512, 512, 4, 0.05, gen.MXFP4),
                                                   (16, 12, 512, 320, 4, 0.0, gen.NVFP4),
                                                   (40, 8, 256, 128, 2, 0.05, gen.MXFP4),
                                                   (64, 24, 2560, 320, 10, 0.0, gen.NVFP4),
                                                   (9, 6, 512, 192, 3, 0.0, gen.NVFP4)])
def test_prefill_parity(M, E, H, I, k, invalid, fmt):
    m = fm()
    w, x, ids, tw = _prefill_case(M, E, H, I, k, seed=M + E, invalid=invalid, fmt=fmt)
    pw = m.prepare_weights(w, E, H, I, fmt)
    ws = m.alloc_workspace(M, E, H, I, k, fmt)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward(x, pw, ids, tw, out=out, workspace=ws)
    torch.cuda.synchronize()
    want, _, _, _ = oracle.forward_prefill(x, w, ids, tw, E, H, I, k, fmt=fmt)
    assert_layer_close(got, want, f"prefill M={M} E={E} H={H} I={I} k={k} fmt={fmt}")


def test_prefill_repeat_and_library_workspace():
    m = fm()
    M, E, H, I, k = 64, 4, 256, 256, 2
    w, x, ids, tw = _prefill_case(M, E, H, I, k, seed=5)
    pw = m.prepare_weights(w, E, H, I, gen.NVFP4)
    m.reserve_workspace(M, E, H, I, k, gen.NVFP4)
    a = m.forward(x, pw, ids, tw).float()
    b = m.forward(x, pw, ids, tw).float()
    torch.cuda.synchronize()
    cos, maxabs, rms = layer_metrics(b, a.double().cpu().numpy())
    assert cos > 0.999999 and maxabs <= 1e-3 * rms


def test_prefill_full_size_sampled():
    m = fm()
    wl = gen.make_workload("prefill_e128", device="cuda")
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    got = m.forward(wl.x, pw, wl.topk_ids, wl.topk_weights, workspace=ws)
    torch.cuda.synchronize()
    # every expert's first and last routed row (its lowest and highest
    # token: the first row of its first 128-row tile and the last valid row
    # of its last tile), plus every 170th token
    ids = wl.topk_ids.cpu().numpy()
    tokens = set(range(0, wl.M, wl.M // 24))
    for e in range(wl.E):
        rows = np.nonzero((ids == e).any(axis=1))[0]
        if rows.size:
            tokens.update((int(rows[0]), int(rows[-1])))
    tokens = sorted(tokens)
    sub_ids = wl.topk_ids[tokens]
    sub, ids_c, Ec = compact_for_oracle(wl.weights, sub_ids, wl.E, wl.fmt)
    want, _, _, _ = oracle.forward_prefill(wl.x[tokens], sub, ids_c, wl.topk_weights[tokens].cpu(), Ec, wl.H, wl.I,
                                           wl.top_k)
    assert_layer_close(got[tokens], want, "prefill_e128 sampled")
