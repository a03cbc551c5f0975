"""The prefill band's tcgen05 block-scaled FP4 GEMM in isolation, through the
C ABI: D = A * B^T with E2M1 operands and per-16 E4M3 block scales, compared
with the FP64 oracle's dequantisation of the same bytes times a NumPy
float64 matmul.  Several 128x256 tiles and a K longer than the 4-stage ring
are covered."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import ensure_built

pytestmark = pytest.mark.gpu


def chunk_layout(scales: np.ndarray) -> np.ndarray:
    """[rows][K/16] scale bytes -> 512-byte chunks [rows/128][K/64][512],
    byte (r%32)*16 + (r//32)*4 + b for row r of a 128-row tile, K-block b of
    a group of 4 (the resident layout of the scale tensors)."""
    rows, kb = scales.shape
    kg = kb // 4
    out = np.zeros((rows // 128, kg, 512), dtype=np.uint8)
    r = np.arange(rows)
    for b in range(kb):
        pos = (r % 128 % 32) * 16 + (r % 128 // 32) * 4 + (b % 4)
        out[r // 128, b // 4, pos] = scales[:, b]
    return out


def random_case(rows, K, rng):
    nib = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    # E4M3 scales with exponent field 4..9 (values 2^-3 .. 2^2 with mantissa), no NaN
    e = rng.integers(4, 10, (rows, K // 16))
    m = rng.integers(0, 8, (rows, K // 16))
    sc = ((e << 3) | m).astype(np.uint8)
    return nib, sc


@pytest.mark.parametrize("M_rows,N_rows,K", [(128, 256, 256), (256, 512, 1280), (384, 256, 2048)])
def test_block_scaled_gemm(M_rows, N_rows, K):
    ensure_built()
    from fp4_weight_moe_gb300 import _capi
    rng = np.random.default_rng(M_rows + N_rows + K)
    a_q, a_s = random_case(M_rows, K, rng)
    b_q, b_s = random_case(N_rows, K, rng)
    dev = torch.device("cuda")
    ta_q = torch.from_numpy(a_q).to(dev)
    tb_q = torch.from_numpy(b_q).to(dev)
    ta_s = torch.from_numpy(chunk_layout(a_s)).to(dev)
    tb_s = torch.from_numpy(chunk_layout(b_s)).to(dev)
    d = torch.full((M_rows, N_rows), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _capi.moe_fp4_debug_gemm(ta_q.data_ptr(), ta_s.data_ptr(), tb_q.data_ptr(), tb_s.data_ptr(), d.data_ptr(),
                             M_rows, N_rows, K, 1, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"internal wait timed out (status {int(status.item())})"
    A = oracle.dequant(a_q, a_s, K, 1)
    B = oracle.dequant(b_q, b_s, K, 1)
    want = A @ B.T
    got = d.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    err = np.abs(got - want)
    scale = np.sqrt(np.mean(want ** 2))
    # FP32 accumulation of exact products over K terms
    assert err.max() <= 1e-5 * scale * np.sqrt(K / 256) + 1e-6, (err.max(), scale)
