"""The W4A8-MX activation quantiser (MXFP8) on the GPU against the oracle.

Bit-exact: E4M3 element bytes and UE8M0 scale bytes of every 32-block, on
rows with a wide spread of magnitudes, all-zero and negative-zero blocks,
blocks whose maximum sits exactly on 448 * 2^j and one unit in the last
place above it, values on every E4M3 rounding midpoint after scaling,
values below the normal FP32 range, and blocks in the top FP32 binade
(FLT_MAX, 448 * 2^119 and one unit above it).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    ensure_built()


def _rows():
    rng = np.random.default_rng(17)
    rows, K = 24, 512
    a = (rng.standard_normal((rows, K)) * np.exp(rng.uniform(-25, 25, (rows, 1)))).astype(np.float32)
    a[1] = 0.0
    a[2, :32] = np.float32(-0.0)
    a[2, 40] = np.float32(-1e-30)
    for j, r in zip((-20, 0, 7), (3, 4, 5)):
        a[r, :32] = np.linspace(-1, 1, 32, dtype=np.float32) * np.float32(448.0 * 2.0 ** j)
        a[r, 31] = np.float32(448.0 * 2.0 ** j)
        a[r, 32:64] = a[r, :32]
        a[r, 63] = np.nextafter(np.float32(448.0 * 2.0 ** j), np.float32(np.inf))
    # midpoints between neighbouring E4M3 values (scale 1: block max 448)
    grid = np.array([oracle.e4m3(c) for c in range(0x7F)], np.float64)
    mids = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)
    a[6, :] = 0.0
    for b in range((len(mids) + 30) // 31):
        chunk = mids[31 * b:31 * b + 31] * (1 if b % 2 else -1)
        a[6, 32 * b] = 448.0
        a[6, 32 * b + 1:32 * b + 1 + len(chunk)] = chunk
    a[7] = np.float32(1e-40) * rng.standard_normal(K).astype(np.float32)  # below the normal range
    # the top FP32 binade: a block holding FLT_MAX (largest scale exponent),
    # one whose maximum is 448 * 2^119 exactly and one a unit above it
    fmax = np.finfo(np.float32).max
    a[8, :32] = rng.standard_normal(32).astype(np.float32) * np.float32(1e37)
    a[8, 5] = fmax
    a[8, 6] = -fmax
    top = np.float32(448.0 * 2.0 ** 119)
    a[8, 32:64] = np.linspace(-1, 1, 32, dtype=np.float32) * top
    a[8, 63] = top
    a[8, 64:96] = a[8, 32:64]
    a[8, 95] = np.nextafter(top, np.float32(np.inf))
    return a


def test_mxfp8_quantiser_bit_exact():
    from fp4_weight_moe_gb300 import _capi
    a = _rows()
    rows, K = a.shape
    dev = torch.device("cuda")
    ta = torch.from_numpy(a).to(dev)
    q = torch.empty((rows, K), dtype=torch.uint8, device=dev)
    s = torch.empty((rows, K // 32), dtype=torch.uint8, device=dev)
    _capi.moe_fp4_debug_quant_mxfp8_rows(ta.data_ptr(), rows, K, q.data_ptr(), s.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    qg, sg = q.cpu().numpy(), s.cpu().numpy()
    for r in range(rows):
        wq, ws = oracle.quant_mxfp8_row(a[r])
        assert np.array_equal(sg[r], ws), r
        assert np.array_equal(qg[r], wq), r


def test_mxfp8_quantiser_argument_errors():
    from fp4_weight_moe_gb300 import _capi
    assert _capi.raw_status("moe_fp4_debug_quant_mxfp8_rows", 0x1000, 4, 48, 0x1000, 0x1000, None) == \
        _capi.MOE_FP4_EUNSUPPORTED
    assert _capi.raw_status("moe_fp4_debug_quant_mxfp8_rows", 0x1000, 4, 64, 0x1008, 0x1000, None) == \
        _capi.MOE_FP4_EINVAL
