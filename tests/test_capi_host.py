"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every symbol that include/moe_fp4.h declares, and rejects bad
arguments with the documented status codes before touching the GPU."""
import ctypes
import os
import re

import pytest

from fp4_weight_moe_gb300 import _capi
from fp4_weight_moe_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fp4.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _capi.lib()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_FP4_API\s+[\w\s\*]*?\b(moe_fp4_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = _declared()
    for must in ("moe_fp4_prepare_weights", "moe_fp4_forward", "moe_fp4_forward_ws", "moe_fp4_workspace_bytes",
                 "moe_fp4_prepared_sizes", "moe_fp4_debug_dequant", "moe_fp4_debug_route"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _capi.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for s in range(5):
        assert _capi.moe_fp4_status_string(s)
    assert _capi.moe_fp4_status_string(99) == "unknown status"
    assert _capi.moe_fp4_version() >= 100


@pytest.mark.parametrize("fmt,B", [(0, 32), (1, 16)])
def test_prepared_sizes_closed_form(lib, fmt, B):
    E, H, I = 5, 512, 192
    w13, s13, w2, s2 = _capi.moe_fp4_prepared_sizes(E, H, I, fmt)
    assert w13 == E * 2 * I * H // 2
    assert w2 == E * H * I // 2
    # resident scales: one E4M3 byte per 16 elements for both formats
    kg13 = -(-(H // 16) // 4)
    kg2 = -(-(I // 16) // 4)
    pad = lambda v: (v + 15) // 16 * 16  # noqa: E731
    assert s13 == pad(E * (2 * I // 128) * kg13 * 512 + 8 * E)
    assert s2 == pad(E * (H // 128) * kg2 * 512 + 4 * E)


def _fwd_status(M=1, E=8, H=256, I=128, k=2, fmt=0, ptr=0x1000, ws=0x10000, ws_bytes=1 << 20, out=None):
    p = ptr
    return _capi.raw_status("moe_fp4_forward_ws", p, p, p, p, p, p, p, out if out is not None else p, M, E, H, I, k,
                            fmt, ws, ws_bytes, None)


def test_forward_argument_errors(lib):
    assert _fwd_status(M=-1) == _capi.MOE_FP4_EINVAL
    assert _fwd_status(fmt=7) == _capi.MOE_FP4_EINVAL
    assert _fwd_status(E=0) == _capi.MOE_FP4_EINVAL
    assert _fwd_status(H=384) == _capi.MOE_FP4_EUNSUPPORTED  # H % 256
    assert _fwd_status(I=96) == _capi.MOE_FP4_EUNSUPPORTED  # I % 64
    assert _fwd_status(k=17) == _capi.MOE_FP4_EUNSUPPORTED
    assert _fwd_status(ptr=0) == _capi.MOE_FP4_EINVAL  # null pointers
    assert _fwd_status(ptr=0x1008) == _capi.MOE_FP4_EINVAL  # x / weights not 16-byte aligned
    assert _fwd_status(M=0) == _capi.MOE_FP4_OK  # empty batch is a no-op
    assert _fwd_status(ws=0) == _capi.MOE_FP4_EWORKSPACE
    assert _fwd_status(ws=0x10010) == _capi.MOE_FP4_EWORKSPACE  # not 256-byte aligned


def test_prepare_argument_errors(lib):
    st = _capi.raw_status("moe_fp4_prepare_weights", 0x1000, 0x1000, None, 0x1000, 0x1000, None, 4, 256, 128, 1,
                          0x1000, 0x1000, 0x1000, 0x1000, None)
    assert st == _capi.MOE_FP4_EINVAL  # NVFP4 needs the FP32 multipliers
    st = _capi.raw_status("moe_fp4_prepare_weights", 0x1000, 0x1000, None, 0x1000, 0x1000, None, 4, 200, 128, 0,
                          0x1000, 0x1000, 0x1000, 0x1000, None)
    assert st == _capi.MOE_FP4_EUNSUPPORTED
    st = _capi.raw_status("moe_fp4_debug_dequant", 0x1000, 0x1000, 3, 0, 4, 256, 128, 0, 0x1000, None)
    assert st == _capi.MOE_FP4_EINVAL  # which: 0 w13, 1 w2, 2 w1 (non-gated)
    # non-gated (squared-ReLU) weights: the same checks
    st = _capi.raw_status("moe_fp4_prepare_weights_relu2", 0x1000, 0x1000, None, 0x1000, 0x1000, None, 4, 256, 128,
                          1, 0x1000, 0x1000, 0x1000, 0x1000, None)
    assert st == _capi.MOE_FP4_EINVAL  # NVFP4 needs the FP32 multipliers
    st = _capi.raw_status("moe_fp4_prepare_weights_relu2", 0x1000, 0x1000, None, 0x1000, 0x1000, None, 4, 200, 128,
                          0, 0x1000, 0x1000, 0x1000, 0x1000, None)
    assert st == _capi.MOE_FP4_EUNSUPPORTED
    st = _capi.raw_status("moe_fp4_prepare_weights_relu2", 0x1000, 0x1000, None, 0x1000, 0x1000, None, 4, 256, 128,
                          0, 0x1008, 0x1000, 0x1000, 0x1000, None)
    assert st == _capi.MOE_FP4_EINVAL  # resident buffers 16-byte aligned
    st = _capi.raw_status("moe_fp4_debug_dequant", 0x1000, 0x1000, 0, 4, 4, 256, 128, 0, 0x1000, None)
    assert st == _capi.MOE_FP4_EINVAL  # expert out of range


def test_forward_ex_rejects_bad_activation(lib):
    """The activation is validated before anything else touches the device."""
    import ctypes
    p = ctypes.c_void_p(16)
    bad = [_capi.MoeFp4Activation(7, 0.0, 0.0, 0.0),
           _capi.MoeFp4Activation(_capi.MOE_FP4_ACT_SWIGLUOAI, 1.702, 1.0, 0.0),
           _capi.MoeFp4Activation(_capi.MOE_FP4_ACT_SWIGLUOAI, float("nan"), 1.0, 7.0),
           _capi.MoeFp4Activation(_capi.MOE_FP4_ACT_SWIGLUOAI, 1.702, float("inf"), 7.0)]
    for act in bad:
        st = lib.moe_fp4_forward_ex(p, p, p, p, p, p, p, p, 1, 8, 256, 128, 2, 1, ctypes.byref(act), p, 1 << 20, None)
        assert st == _capi.MOE_FP4_EINVAL


def test_forward_ex_i64_argument_errors(lib):
    """int64 routing ids: an ids pointer that is not 8-byte aligned, null
    pointers and bad shapes are rejected on the host; an empty batch is a
    no-op."""
    import ctypes
    p = ctypes.c_void_p(0x1000)

    def st(ids=0x1000, x=0x1000, M=1, H=256):
        return lib.moe_fp4_forward_ex_i64(ctypes.c_void_p(x), p, p, p, p, ctypes.c_void_p(ids), p, p, M, 8, H, 128, 2,
                                          1, None, p, 1 << 20, None)

    assert st(ids=0x1004) == _capi.MOE_FP4_EINVAL  # 4-byte aligned only
    assert st(x=0) == _capi.MOE_FP4_EINVAL
    assert st(ids=0) == _capi.MOE_FP4_EINVAL
    assert st(H=384) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(M=0) == _capi.MOE_FP4_OK


def test_band_policy_by_shape(lib):
    """Which kernels a batch takes (host logic only): the decode band up to 8
    tokens (streaming GEMV for one token with few routed bytes, else tcgen05
    with 3 launches, 4 from two tokens), everything else the mid or prefill
    band (0 decode launches); the test knobs force the decode kernels in
    balanced chunks of at most 8 tokens for up to 24 tokens, or the GEMV."""
    c = _capi
    e512 = (512, 2560, 320, 10)     # 1.38 MB experts
    e256 = (256, 7168, 2048, 8)     # 22 MB experts
    tiny = (8, 256, 128, 2)
    assert c.moe_fp4_debug_decode_family_of(1, *tiny) == 1
    assert c.moe_fp4_debug_decode_launches(1, *tiny) == 2
    # tcgen05 beyond that (the launch chain by default; the single launch
    # only where its grid is resident at once on the current GPU, never
    # without one)
    prev_family = c.moe_fp4_debug_set_decode_family(3)
    try:
        single = c.moe_fp4_debug_decode_family_of(1, *e512) == 3
        assert c.moe_fp4_debug_decode_family_of(1, *e512) in (2, 3)
        assert c.moe_fp4_debug_decode_launches(1, *e512) == (1 if single else 3)
    finally:
        c.moe_fp4_debug_set_decode_family(prev_family)
    assert c.moe_fp4_debug_decode_family_of(1, *e512) == 2
    prev_family = c.moe_fp4_debug_set_decode_family(2)  # the chain: 3 launches, 4 from two tokens
    try:
        assert c.moe_fp4_debug_decode_family_of(1, *e512) == 2
        assert [c.moe_fp4_debug_decode_launches(M, *e512) for M in (1, 2, 8)] == [3, 4, 4]
        assert [c.moe_fp4_debug_decode_launches(M, *e512) for M in (9, 12, 13, 16, 24)] == [0, 0, 0, 0, 0]
        assert [c.moe_fp4_debug_decode_launches(M, *e256) for M in (8, 9, 16)] == [4, 0, 0]
        prev = c.moe_fp4_debug_set_mid_band(2)
        try:
            assert [c.moe_fp4_debug_decode_launches(M, *e512) for M in (9, 12, 13, 24, 25)] == [8, 8, 8, 12, 0]
        finally:
            c.moe_fp4_debug_set_mid_band(prev)
    finally:
        c.moe_fp4_debug_set_decode_family(prev_family)
    assert c.moe_fp4_debug_decode_family_of(9, *e512) == 0
    prev = c.moe_fp4_debug_set_mid_band(2)
    try:
        assert [c.moe_fp4_debug_decode_launches(M, *e256) for M in (9, 17, 24, 25)] == [8, 12, 12, 0]
        c.moe_fp4_debug_set_mid_band(1)
        assert c.moe_fp4_debug_decode_launches(9, *e512) == 0
    finally:
        c.moe_fp4_debug_set_mid_band(prev)
    with pytest.raises(c.MoeFp4Error):
        c.moe_fp4_debug_set_mid_band(4)
    with pytest.raises(c.MoeFp4Error):
        c.moe_fp4_debug_set_decode_family(4)


def test_mid_band_plan_by_shape(lib):
    """Past the decode band: the mid band's GEMMs while the experts average
    at most 28 routed rows (36 with I <= 384), the prefill band's beyond; the switch overrides
    the rule (decode-kernel chunks only when forced)."""
    c = _capi
    e512, e288, e256, e128 = (512, 2560, 320, 10), (288, 4096, 512, 10), (256, 7168, 2048, 8), (128, 4096, 1536, 8)
    assert [c.moe_fp4_debug_mid_band_of(M, *e512) for M in (1, 8, 9, 12, 13, 1843, 1844)] == [0, 0, 3, 3, 3, 3, 1]
    assert [c.moe_fp4_debug_mid_band_of(M, *e288) for M in (806, 807)] == [3, 1]  # I = 512: 28 rows
    assert [c.moe_fp4_debug_mid_band_of(M, *e256) for M in (9, 896, 897)] == [3, 3, 1]
    assert [c.moe_fp4_debug_mid_band_of(M, *e128) for M in (9, 448, 449, 4096)] == [3, 3, 1, 1]
    assert [c.moe_fp4_debug_mid_band_of(M, *e288) for M in (9, 12)] == [3, 3]
    assert c.moe_fp4_debug_mid_band_of(9, 512, 2560, 320, 0) == 0  # invalid top_k
    prev = c.moe_fp4_debug_set_mid_band(1)
    try:
        assert [c.moe_fp4_debug_mid_band_of(M, *e512) for M in (9, 17, 4096)] == [1, 1, 1]
        c.moe_fp4_debug_set_mid_band(3)
        assert [c.moe_fp4_debug_mid_band_of(M, *e512) for M in (9, 17, 4096)] == [3, 3, 3]
        c.moe_fp4_debug_set_mid_band(2)
        assert [c.moe_fp4_debug_mid_band_of(M, *e512) for M in (9, 24, 25)] == [2, 2, 3]
    finally:
        c.moe_fp4_debug_set_mid_band(prev)


def test_status_query_argument_errors(lib):
    """The status queries and the wait-timeout test entry reject bad
    arguments on the host: a null flags pointer, a workspace that is not
    256-byte aligned, no reserved library workspace, a null or misaligned
    status word, a poll limit out of range."""
    import ctypes
    v = ctypes.c_uint32(7)
    assert lib.moe_fp4_workspace_status(ctypes.c_void_p(0x1000), None, 0, None) == _capi.MOE_FP4_EINVAL
    assert lib.moe_fp4_workspace_status(ctypes.c_void_p(0x1010), ctypes.byref(v), 0, None) == \
        _capi.MOE_FP4_EWORKSPACE
    assert lib.moe_fp4_noalloc_status(None, 0, None) == _capi.MOE_FP4_EINVAL
    assert lib.moe_fp4_debug_wait_timeout(None, 16, None) == _capi.MOE_FP4_EINVAL
    assert lib.moe_fp4_debug_wait_timeout(ctypes.c_void_p(0x1002), 16, None) == _capi.MOE_FP4_EINVAL
    assert lib.moe_fp4_debug_wait_timeout(ctypes.c_void_p(0x1000), 0, None) == _capi.MOE_FP4_EINVAL
    assert lib.moe_fp4_debug_wait_timeout(ctypes.c_void_p(0x1000), (1 << 20) + 1, None) == _capi.MOE_FP4_EINVAL
    assert v.value == 7


def test_noalloc_shape_limits(lib):
    """moe_fp4_forward_noalloc applies the same shape limits as the other
    forward calls, including one projection's 2I x H elements within 2^31
    (I = 2^19 at H = 4096 would fit the scratch array at one token)."""
    import ctypes
    p = ctypes.c_void_p(0x1000)

    def st(E=8, H=256, I=128, top_k=2, M=1, fmt=1):
        return lib.moe_fp4_forward_noalloc(p, p, p, p, p, p, p, p, M, E, H, I, top_k, fmt, None)

    assert st(H=4096, I=1 << 19, top_k=1) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(H=384) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(I=96) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(top_k=17) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(E=65537) == _capi.MOE_FP4_EUNSUPPORTED
    assert st(fmt=2) == _capi.MOE_FP4_EINVAL
    assert st(M=-1) == _capi.MOE_FP4_EINVAL
    assert st(M=0) == _capi.MOE_FP4_OK
    assert st(M=9) == _capi.MOE_FP4_EUNSUPPORTED


def test_header_is_plain_c_and_links(lib, tmp_path):
    """include/moe_fp4.h compiles as C99 (-pedantic, no warnings) and a C
    program links against libmoe_fp4.so and calls a host-only entry point."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text("""
#include <stddef.h>
#include <stdint.h>
#include "moe_fp4.h"
int main(void) {
  size_t w13, s13, w2, s2;
  moe_fp4_activation act = {MOE_FP4_ACT_SWIGLUOAI, 1.702f, 1.0f, 7.0f};
  int st = moe_fp4_prepared_sizes(8, 256, 128, MOE_FP4_MXFP4, &w13, &s13, &w2, &s2);
  (void)act;
  if (st != MOE_FP4_OK) return 1;
  if (w13 != (size_t)8 * 256 * 128 || w2 != (size_t)8 * 256 * 64) return 2;
  return moe_fp4_status_string(MOE_FP4_EWORKSPACE)[0] ? 0 : 3;
}
""")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(_capi.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lmoe_fp4", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert subprocess.run([str(exe)]).returncode == 0


def test_relu2_prepared_sizes(lib):
    """Non-gated layout sizes: w1 [E][I][H/2]; its scale chunks cover each
    expert's rows padded to a multiple of 128, then the FP32 multipliers [E];
    w2 and s2 as for the gated layout."""
    E, H, I = 5, 512, 320
    w1, s1, w2, s2 = _capi.moe_fp4_prepared_sizes_relu2(E, H, I, 1)
    assert w1 == E * I * H // 2
    chunks = E * ((I + 127) // 128) * (H // 64) * 512
    assert s1 == (chunks + 4 * E + 15) // 16 * 16
    g13 = _capi.moe_fp4_prepared_sizes(E, H, I, 1)
    assert (w2, s2) == (g13[2], g13[3])



def test_prefill_mode_argument_errors(lib):
    """An unknown prefill precision is rejected before anything touches the
    device, by both the forward call and the workspace query."""
    import ctypes
    p = ctypes.c_void_p(0x1000)
    for mode in (-1, 3, 7):
        st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 0, p, p, 16, 8, 256, 128, 2, 1, None, mode, p, 1 << 20, None)
        assert st == _capi.MOE_FP4_EINVAL
        assert lib.moe_fp4_workspace_bytes_mode(16, 8, 256, 128, 2, 1, mode) == 0
    # the shape checks of every entry point apply
    st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 0, p, p, 16, 8, 384, 128, 2, 1, None, _capi.MOE_FP4_PREFILL_BF16,
                                  p, 1 << 20, None)
    assert st == _capi.MOE_FP4_EUNSUPPORTED
    st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 2, p, p, 16, 8, 256, 128, 2, 1, None, _capi.MOE_FP4_PREFILL_BF16,
                                  p, 1 << 20, None)
    assert st == _capi.MOE_FP4_EINVAL  # ids_int64 is 0 or 1
    st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 0, p, p, 0, 8, 256, 128, 2, 1, None, _capi.MOE_FP4_PREFILL_BF16,
                                  p, 1 << 20, None)
    assert st == _capi.MOE_FP4_OK  # empty batch


def test_w4a8_mode_limits_on_host(lib):
    """The W4A8-MX prefill mode takes MXFP4 weights and gated activations
    only; both limits are checked before anything touches the device."""
    import ctypes
    p = ctypes.c_void_p(0x1000)
    mode = _capi.MOE_FP4_PREFILL_W4A8_MX
    st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 0, p, p, 16, 8, 256, 128, 2, _capi.MOE_FP4_NVFP4, None, mode, p,
                                  1 << 20, None)
    assert st == _capi.MOE_FP4_EUNSUPPORTED
    relu2 = _capi.MoeFp4Activation(_capi.MOE_FP4_ACT_RELU2, 0.0, 0.0, 0.0)
    st = lib.moe_fp4_forward_mode(p, p, p, p, p, p, 0, p, p, 16, 8, 256, 128, 2, _capi.MOE_FP4_MXFP4,
                                  ctypes.byref(relu2), mode, p, 1 << 20, None)
    assert st == _capi.MOE_FP4_EUNSUPPORTED
    assert lib.moe_fp4_workspace_bytes_mode(16, 8, 256, 128, 2, _capi.MOE_FP4_NVFP4, mode) == 0


def test_w4a8_engine_switch(lib):
    """The W4A8-MX engine switch returns the previous setting and is restored."""
    prev = _capi.moe_fp4_debug_set_w4a8_engine(0)
    assert prev in (0, 1)
    assert _capi.moe_fp4_debug_set_w4a8_engine(1) == 0
    assert _capi.moe_fp4_debug_set_w4a8_engine(prev) == 1
