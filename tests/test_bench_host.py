"""Host-side pieces of bench.py, on CPU.

The reported metric's units (routed-weight bytes and FLOPs per layer), the
key that ties a stored ncu traffic figure to the decode kernels' code (line
comments do not count, code does), and the stored traffic file's shape.
"""
import json
import os
import shutil
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workload import gen  # noqa: E402


def test_layer_bytes_count_unique_valid_experts_once():
    ids = torch.tensor([[3, 7, -1], [7, 9, 12]], dtype=torch.int32)  # 12 is invalid for E = 12
    E, H, I, M, k = 12, 512, 256, 2, 3
    b, uniq = bench.layer_bytes(ids, E, H, I, M, k, gen.NVFP4)
    assert uniq == 3  # experts 3, 7, 9
    assert b == 3 * gen.expert_bytes(H, I, gen.NVFP4) + M * H * 2 * 2 + M * k * 8


def test_layer_flops_count_valid_routed_rows():
    ids = torch.tensor([[0, 1], [1, -1], [5, 2]], dtype=torch.int32)
    assert bench.layer_flops(ids, 5, 256, 128) == 2 * 3 * 256 * 128 * 4


def test_traffic_key_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "fp4_weight_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("common.cuh", "tcgen05.cuh", "decode_tc.cu", "decode.cu"):
        shutil.copy(os.path.join(ROOT, "fp4_weight_moe_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.decode_src_sha256()
    assert base == bench.decode_src_sha256()
    p = csrc / "decode_tc.cu"
    text = p.read_text()
    p.write_text("// a new comment line\n\n" + text.replace("\n", "  // trailing note\n", 1))
    assert bench.decode_src_sha256() == base
    p.write_text(text.replace("constexpr int kRing = 4;", "constexpr int kRing = 3;"))
    assert bench.decode_src_sha256() != base


def test_stored_traffic_file_shape():
    with open(os.path.join(ROOT, "profiles", "decode_e512_traffic.json")) as f:
        d = json.load(f)
    assert len(d["decode_src_sha256"]) == 64
    for key, c in d["configs"].items():
        workload, m, fmt = key.split("/")
        assert workload in gen.CONFIGS and m.startswith("M=") and fmt in gen.FMT_NAMES.values()
        assert c["dram_bytes_per_layer"] == sum(c["kernels_per_layer"].values())
        assert c["algorithmic_bytes_per_layer"] > 0 and "ncu" in c["command"]
        # each routed byte is read about once on the tcgen05 decode layers
        if workload == "decode_e512":
            assert 1.0 <= c["dram_bytes_per_layer"] / c["algorithmic_bytes_per_layer"] < 1.05
    # ten distinct routed experts plus x, out, ids and router weights of one token
    assert np.isclose(d["configs"]["decode_e512/M=1/nvfp4"]["algorithmic_bytes_per_layer"],
                      10 * gen.expert_bytes(2560, 320, gen.NVFP4) + 2560 * 2 * 2 + 10 * 8)


def test_bf16_half_ulp_bounds_the_bf16_rounding():
    """The parity tests' allowance for the BF16 output's own rounding: half a
    BF16 unit in the last place bounds |bf16(w) - w| (torch's
    round-to-nearest-even conversion), and the bound is reached at midpoints."""
    import numpy as np
    import torch
    from tests.gpu_util import bf16_half_ulp
    rng = np.random.default_rng(3)
    # FP32 values (what the kernels round to BF16); torch converts FP64 via
    # FP32, which would round twice
    w = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32).astype(np.float64)
    r = torch.tensor(w, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.all(np.abs(r - w) <= bf16_half_ulp(w))
    mid = np.array([1.0 + 2.0 ** -8, 0.75 + 2.0 ** -9, -(3.0 + 2.0 ** -7)])  # halfway between BF16 neighbours
    rm = torch.tensor(mid, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.allclose(np.abs(rm - mid), bf16_half_ulp(mid), rtol=0, atol=0)
    assert bf16_half_ulp(np.array([0.0]))[0] == 0.0


def _prefill_res(mode=None, engine=None, us=1000.0):
    c = dict(gen.CONFIGS["prefill_e128"])
    ids = [torch.tensor([[0, 1], [2, 3]], dtype=torch.int32)]
    res = {"us_per_layer": us, "prefill": True, "plan": "p", "layers_per_replay": 1,
           "flops_per_layer": 1e12, "_state": (c, 0, ids, None, None)}
    if mode:
        res["prefill_mode"] = mode
    if engine:
        res["engine"] = engine
    return res


def test_prefill_roofline_peaks_follow_the_tensor_core_kind(monkeypatch):
    """The NVFP4 band is judged against the FP4 peak (measured BF16 x 6), the
    exact mode against the BF16 peak, the W4A8-MX FP8 engine against the FP8
    peak (measured BF16 x 2); each above its ridge reports TFLOP/s."""
    monkeypatch.setattr(bench, "load_bf16_peak", lambda: (1000.0, "measured"))
    hbm = 1e9  # so high that every case sits above the ridge: the tensor bound
    r = bench.roofline_of(_prefill_res(), hbm, "measured", None)
    assert r["bound"] == "tensor" and r["peak"] == 6000.0 and abs(r["achieved"] - 1000.0) < 1e-6
    r = bench.roofline_of(_prefill_res("bf16-exact", "16-bit"), hbm, "measured", None)
    assert r["peak"] == 1000.0 and abs(r["frac"] - 1.0) < 1e-9
    r = bench.roofline_of(_prefill_res("w4a8-mx", "fp8"), hbm, "measured", None)
    assert r["peak"] == 2000.0 and "x 2" in r["peak_source"]
    r = bench.roofline_of(_prefill_res("w4a8-mx", "16-bit"), hbm, "measured", None)
    assert r["peak"] == 1000.0


def test_stored_prefill_traffic_file_shape_and_lookup():
    with open(os.path.join(ROOT, "profiles", "prefill_e128_traffic.json")) as f:
        d = json.load(f)
    assert len(d["src_sha256"]) == 64
    for key, c in d["configs"].items():
        workload, m, fmt, mode = key.split("/")
        assert workload in gen.CONFIGS and m.startswith("M=") and fmt in gen.FMT_NAMES.values()
        assert mode in ("nvfp4", "bf16-exact", "w4a8-mx")
        assert c["dram_bytes_per_layer"] == sum(c["kernels_per_layer"].values())
        assert c["algorithmic_bytes_per_layer"] > 0 and "ncu" in c["command"]
        assert "--clock-control none" in c["command"]
    # the bench finds a figure exactly while the prefill sources hash to the stored key
    got = bench.stored_traffic("prefill_e128", 4096, "nvfp4", None, "nvfp4")
    if d["src_sha256"] == bench.prefill_src_sha256():
        assert got == d["configs"]["prefill_e128/M=4096/nvfp4/nvfp4"]["dram_bytes_per_layer"]
    else:
        assert got is None
    assert bench.stored_traffic("prefill_e128", 4096, "nvfp4", 32, "nvfp4") is None  # another E: no figure
