"""The seeded input recipe (workload/gen.py) against its stated rules, on CPU.

The generators hold no layer arithmetic, but every parity case and bench line
depends on them producing what the design record's input recipe says:
synthetic FP4 checkpoints quantised by the stated rules (MXFP4:
scale 2^ceil(log2(amax/6)), round to the nearest E2M1 point with ties to the
even code; NVFP4: g = amax/(6*448), s = e4m3(amax_blk/(6 g)), saturating
codes), N(0, 1) BF16 activations, and top-k routing from N(0, 1) logits by
value with ties to the lower index, renormalised, with the E=288 workload's
exact count of invalid slots, the Zipf(1.1) popularity bias, and the bench's
no-repeat window.  Each rule is checked here from its own definition (the
E2M1 table, Python's math, an argsort of the logits), not through the
generator's helpers.
"""
import math

import numpy as np
import pytest
import torch

from workload import gen

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _decode_nibbles(packed: np.ndarray) -> np.ndarray:
    lo, hi = packed & 0xF, packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], -1)
    mag = np.array(E2M1)[codes & 7]
    return np.where(codes & 8, -mag, mag)


def _nearest_even(v: float) -> float:
    """The E2M1 magnitude nearest to v >= 0 (ties to the even code, beyond 6: 6)."""
    best = min(range(8), key=lambda c: (abs(E2M1[c] - v), c % 2))
    return E2M1[best]


def _e4m3_decode(b: int) -> float:
    e, m = (b >> 3) & 15, b & 7
    v = m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if b & 0x80 else v


def test_mxfp4_scale_rule_and_nearest_codes():
    g = torch.Generator().manual_seed(3)
    w = torch.randn(6, 256, generator=g) * torch.logspace(-3, 1, 6).unsqueeze(1)
    w[2, :32] = 0.0                                            # an all-zero block
    w[3, 32:64] = torch.tensor([6.0 * 2 ** -4] + [0.0] * 31)   # amax/6 an exact power of two
    nib, sc = gen.encode_mxfp4(w)
    vals = _decode_nibbles(nib.numpy())
    for r in range(w.shape[0]):
        for b in range(w.shape[1] // 32):
            blk = w[r, 32 * b:32 * (b + 1)].double().numpy()
            amax = float(np.abs(blk).max())
            want = 127 if amax == 0 else 127 + math.ceil(math.log2(amax / 6))
            assert int(sc[r, b]) == want, (r, b)
            scale = 2.0 ** (want - 127)
            for i in range(32):
                got = vals[r, 32 * b + i]
                q = abs(float(np.float32(blk[i])) / scale)
                assert abs(got) == _nearest_even(q), (r, b, i)
                if got != 0:
                    assert (got < 0) == (blk[i] < 0)
    assert not np.any(vals[2, :32])


def test_nvfp4_scale_rule_and_saturating_codes():
    g = torch.Generator().manual_seed(4)
    w = torch.randn(8, 128, generator=g) * 0.02
    w[1, 16:32] = 0.0
    nib, sc, gm = gen.encode_nvfp4(w)
    amax = float(w.abs().max())
    assert float(gm) == float(np.float32(np.float32(amax) / np.float32(6 * 448)))
    vals = _decode_nibbles(nib.numpy())
    G = float(gm)
    for r in range(8):
        for b in range(8):
            blk = w[r, 16 * b:16 * (b + 1)].numpy()
            s_exact = float(np.abs(blk).max()) / (6 * G)
            s = _e4m3_decode(int(sc[r, b]))
            want_s = float(torch.tensor(min(s_exact, 448.0)).to(torch.float8_e4m3fn).float())
            assert s == want_s, (r, b)
            for i in range(16):
                got = vals[r, 16 * b + i]
                if s == 0:
                    assert got == 0
                    continue
                q = abs(float(blk[i]) / (s * G))
                assert abs(got) == _nearest_even(q), (r, b, i)
    assert not np.any(vals[1, 16:32]) and int(sc[1, 1]) == 0


def test_activations_are_seeded_standard_normal_bf16():
    a = gen.draw_activations(64, 1024, 11)
    b = gen.draw_activations(64, 1024, 11)
    assert a.dtype == torch.bfloat16 and torch.equal(a.view(torch.int16), b.view(torch.int16))
    x = a.float().numpy()
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1.0) < 0.02


@pytest.mark.parametrize("M,E,k", [(4, 64, 8), (1, 512, 10), (32, 16, 4)])
def test_routing_is_topk_of_the_logits_renormalised(M, E, k):
    ids, w = gen.draw_routing(M, E, k, 123)
    rng = np.random.Generator(np.random.PCG64(123))
    logits = rng.standard_normal((M, E))
    for t in range(M):
        want = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        assert ids[t].tolist() == want
        p = np.exp(logits[t] - logits[t].max())
        p /= p.sum()
        np.testing.assert_allclose(w[t].numpy(), p[want] / p[want].sum(), rtol=1e-6)
    assert w.dtype == torch.float32 and ids.dtype == torch.int32


def test_zipf_bias_shifts_the_logits():
    M, E, k = 6, 256, 8
    ids, _ = gen.draw_routing(M, E, k, 77, mode="zipf")
    rng = np.random.Generator(np.random.PCG64(77))
    logits = rng.standard_normal((M, E))
    rank = rng.permutation(E) + 1
    biased = logits - 1.1 * np.log(rank)[None, :]
    for t in range(M):
        assert ids[t].tolist() == sorted(range(E), key=lambda e: (-biased[t, e], e))[:k]


def test_invalid_slots_of_the_e288_workload():
    ids, w = gen.draw_routing(4, 288, 10, 5, mode="softmax_invalid")
    flat = ids.reshape(-1).tolist()
    bad = [(i, e) for i, e in enumerate(flat) if not 0 <= e < 288]
    assert len(bad) == round(0.05 * 40) == 2
    assert sorted(e for _, e in bad) == [-1, 288]
    assert all(float(w.reshape(-1)[i]) > 0 for i, _ in bad)


def test_bench_pool_has_no_repeat_within_the_window():
    n, M, E, k, window = 12, 1, 512, 10, 5
    ids, w = gen.draw_routing_pool(n, M, E, k, 9, window)
    sets = [set(t.reshape(-1).tolist()) for t in ids]
    for i in range(n):
        assert len(sets[i]) == M * k
        for d in range(1, window):
            assert not sets[i] & sets[(i + d) % n], (i, d)


def test_expert_bytes_of_the_pages_geometries():
    # per-expert weight + scale bytes as the scope table states them
    assert gen.expert_bytes(2560, 320, gen.NVFP4) == 1_382_412
    assert gen.expert_bytes(4096, 512, gen.MXFP4) == 3_342_336
    assert gen.expert_bytes(7168, 2048, gen.MXFP4) == 23_396_352
    assert gen.expert_bytes(7168, 2048, gen.NVFP4) == 24_772_620
