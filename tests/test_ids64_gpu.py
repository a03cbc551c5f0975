"""int64 routing ids (moe_fp4_forward_ex_i64) against the FP64 oracle.

The b12x PR #459 page (Reduce NVFP4-CSF scale reconstruction overhead, its
commit list) keeps kernel programs for both integer types of the routing
ids.  Here every path reads either width.  Each case plants ids that only
int64 can hold: values at or past 2^31 whose low 32 bits name a valid expert
(2^32 + e), large negatives, and E itself.  All of them must contribute
exactly zero, as the oracle does with those slots invalid.  Ids that fit in
int32 must give bitwise the int32 result on the decode band, which is
deterministic.
"""
import pytest
import torch

import oracle
from tests.gpu_util import assert_layer_close, ensure_built, oracle_layer
from workload import gen

pytestmark = pytest.mark.gpu

GEMV, TC, SINGLE = 1, 2, 3  # decode plans: streaming GEMV, tcgen05 chain, tcgen05 single launch


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def _wide_ids(ids32: torch.Tensor, E: int, seed: int) -> torch.Tensor:
    """int64 copy of the ids with about a quarter of the slots replaced by
    invalid values that int32 cannot hold or that alias a valid expert in
    their low 32 bits."""
    g = torch.Generator().manual_seed(seed)
    ids = ids32.cpu().long()
    pick = torch.rand(ids.shape, generator=g) < 0.25
    bad = torch.tensor([2 ** 32, -(2 ** 40), 2 ** 31, E], dtype=torch.long)
    choice = bad[torch.randint(0, len(bad), ids.shape, generator=g)]
    # 2^32 + e keeps the low word of a valid expert
    choice = torch.where(choice == 2 ** 32, choice + ids, choice)
    return torch.where(pick, choice, ids)


def _as_oracle_ids(ids64: torch.Tensor, E: int) -> torch.Tensor:
    valid = (ids64 >= 0) & (ids64 < E)
    return torch.where(valid, ids64, torch.full_like(ids64, -1)).int()


def _run(wl, ids, family=0):
    import fp4_weight_moe_gb300 as m
    from fp4_weight_moe_gb300 import _capi
    pw = m.prepare_weights(wl.weights, wl.E, wl.H, wl.I, wl.fmt)
    ws = m.alloc_workspace(wl.M, wl.E, wl.H, wl.I, wl.top_k, wl.fmt)
    out = torch.full((wl.M, wl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    prev = _capi.moe_fp4_debug_set_decode_family(family)
    try:
        m.forward(wl.x, pw, ids.cuda().contiguous(), wl.topk_weights, out=out, workspace=ws)
        torch.cuda.synchronize()
    finally:
        _capi.moe_fp4_debug_set_decode_family(prev)
    return out


@pytest.mark.parametrize("family", [GEMV, TC, SINGLE], ids=["gemv", "chain", "single"])
@pytest.mark.parametrize("name,ov", [("tiny_decode", dict(M=3, E=12, top_k=3)),
                                     ("decode_e512", dict(E=40, M=2)),
                                     ("decode_e288_m4", dict(E=24))])
def test_decode_int64_ids(name, ov, family):
    wl = gen.make_workload(name, device="cuda", **ov)
    ids64 = _wide_ids(wl.topk_ids, wl.E, seed=7 + family)
    got = _run(wl, ids64, family)
    wl.topk_ids = _as_oracle_ids(ids64, wl.E).cuda()
    assert_layer_close(got, oracle_layer(wl), f"{name} {ov} int64 ids family {family}")


@pytest.mark.parametrize("family", [GEMV, TC, SINGLE], ids=["gemv", "chain", "single"])
def test_decode_int64_matches_int32_bitwise(family):
    wl = gen.make_workload("decode_e512", device="cuda", E=32, M=4, top_k=6)
    ids32 = wl.topk_ids.clone()
    ids32[0, 1] = -3  # invalid ids that int32 holds too
    ids32[2, 0] = wl.E + 5
    a = _run(wl, ids32, family)
    b = _run(wl, ids32.long(), family)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("M,E,H,I,k", [(24, 12, 512, 320, 4), (64, 8, 512, 256, 4)])
def test_prefill_int64_ids(M, E, H, I, k):
    import fp4_weight_moe_gb300 as m
    fmt = gen.NVFP4
    weights = gen.make_expert_weights(E, H, I, fmt, 61 + M, device="cuda")
    x = gen.draw_activations(M, H, 62 + M, device="cuda")
    ids, tw = gen.draw_routing(M, E, k, 63 + M, mode="softmax")
    ids64 = _wide_ids(ids, E, seed=M)
    ids_o = _as_oracle_ids(ids64, E)
    pw = m.prepare_weights(weights, E, H, I, fmt)
    ws = m.alloc_workspace(M, E, H, I, k, fmt)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    got = m.forward(x, pw, ids64.cuda(), tw.cuda(), out=out, workspace=ws)
    torch.cuda.synchronize()
    want, _, _, _ = oracle.forward_prefill(x, weights, ids_o, tw, E, H, I, k, fmt=fmt)
    assert_layer_close(got, want, f"prefill int64 ids M={M} I={I}")
