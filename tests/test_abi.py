"""CPU-side checks of the C ABI: the library loads without a GPU and exports
every entry point that include/pgg.h declares; no compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgg.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pgg_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from precision_grouped_gemm_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for name in ["pgg_grouped_gemm_fwd", "pgg_grouped_gemm_dgrad", "pgg_grouped_gemm_wgrad",
                 "pgg_grouped_fc1_swiglu", "pgg_grouped_fc2_dgrad_swiglu_bwd",
                 "pgg_mx_quantize_rowwise", "pgg_mx_quantize_colwise", "pgg_mx_grouped_gemm",
                 "pgg_grouped_gemm_wgrad_accumulate", "pgg_moe_permute", "pgg_moe_combine",
                 "pgg_moe_combine_bwd"]:
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_binding_signatures_cover_header():
    from precision_grouped_gemm_gb300 import _binding
    for s in declared_symbols():
        if s not in ("pgg_status_string", "pgg_moe_permute_workspace_size",
                     "pgg_fp8_workspace_size"):  # non-int returns
            assert s in _binding.SIGNATURES, s


def test_status_strings_and_version(lib):
    lib.pgg_status_string.restype = ctypes.c_char_p
    assert lib.pgg_status_string(0) == b"ok"
    assert b"group_lens" in lib.pgg_status_string(16)
    assert lib.pgg_version() >= 100


def test_host_validation_without_gpu(lib):
    # argument checks run before any CUDA call, so they answer on a machine without a GPU
    P = ctypes.c_void_p
    f = lib.pgg_grouped_gemm_fwd
    f.argtypes = [P, P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P]
    good = 1 << 20
    assert f(None, good, good, good, 8, 64, 64, 1, None, None) == 1       # null X
    assert f(None, None, good, None, 0, 64, 64, 1, None, None) == 0       # M == 0 is a no-op
    assert f(good, good, good, good, 8, 64, 60, 1, None, None) == 3       # K % 8
    assert f(good, good, good, good, 8, 64, 64, 2000, None, None) == 1    # G > 1024
    assert f(good + 8, good, good, good, 8, 64, 64, 1, None, None) == 3   # misaligned
    q = lib.pgg_mx_quantize_rowwise
    q.argtypes = [P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, P, P, P]
    assert q(good, 4, 48, 1, good, good, None) == 3                        # C % 32
    assert q(good, 4, 64, 7, good, good, None) == 1                        # bad format


def test_moe_glue_host_validation_without_gpu(lib):
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    ws = lib.pgg_moe_permute_workspace_size
    ws.argtypes, ws.restype = [I64, I32], ctypes.c_size_t
    assert ws(4096, 256) == 128 * 256 * 4            # ceil(T / 32) chunks x E experts x int32
    assert ws(33, 3) == 2 * 3 * 4
    f = lib.pgg_moe_permute
    f.argtypes = [P, P, I64, I32, I64, I32, P, P, P, P, ctypes.c_size_t, P, P]
    g = 1 << 20
    assert f(g, g, 100, 0, 64, 8, g, g, g, g, 1 << 20, None, None) == 1        # k < 1
    assert f(g, g, 100, 33, 64, 8, g, g, g, g, 1 << 20, None, None) == 1       # k > 32
    assert f(g, g, 100, 4, 64, 2000, g, g, g, g, 1 << 20, None, None) == 1     # E > 1024
    assert f(g, g, 100, 4, 60, 8, g, g, g, g, 1 << 20, None, None) == 3        # H % 8
    assert f(g, g, 100, 4, 64, 8, g, g, g, g, 16, None, None) == 1             # workspace too small
    assert f(g, g, 100, 4, 64, 8, g + 8, g, g, g, 1 << 20, None, None) == 3    # misaligned Xs
    assert f(g, g, 100, 4, 64, 8, g, None, g, g, 1 << 20, None, None) == 1     # null group_lens
    c = lib.pgg_moe_combine
    c.argtypes = [P, P, P, P, I64, I32, I64, P]
    assert c(None, None, None, None, 0, 4, 64, None) == 0                      # T == 0 is a no-op
    assert c(g, g, None, None, 8, 4, 64, None) == 1                            # null out
    assert c(g, g, None, g, 8, 4, 12, None) == 3                               # H % 8
    b = lib.pgg_moe_combine_bwd
    b.argtypes = [P, P, P, P, P, P, I64, I32, I64, P]
    assert b(g, g, g, None, g, g, 8, 4, 64, None) == 1                         # w required
    assert b(g, g, g, g, g + 4, g, 8, 4, 64, None) == 3                        # misaligned dYs


def test_blocked_scale_layout_helpers():
    # the tests' view of the blocked column-wise scale layout (pgg.h): atom (r // 128, j // 4)
    # of 512 bytes, byte 16 (m % 32) + 4 (m // 32) + j % 4 inside it, m = r % 128
    import numpy as np
    import util
    C, M_pad = 200, 384
    s = (np.arange(C * (M_pad // 32)) % 251 + 1).astype(np.uint8).reshape(C, M_pad // 32)
    b = util.block_scales(s, M_pad)
    assert b.shape == (256, M_pad // 32)
    flat = b.reshape(-1)
    assert flat[0] == s[0, 0] and flat[1] == s[0, 1] and flat[4] == s[32, 0] and flat[16] == s[1, 0]
    assert flat[512] == s[0, 4]                                  # next k-block atom of row block 0
    assert flat[3 * 512 + 16 * 5 + 4 * 2 + 3] == s[128 + 69, 3]  # row block 1, m = 69
    np.testing.assert_array_equal(util.unblock_scales(b, C, M_pad), s)


def test_new_entry_points_host_validation_without_gpu(lib):
    P, I64, I32, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.pgg_status_string.restype = ctypes.c_char_p
    assert b"expert" in lib.pgg_status_string(19)
    assert b"scratch" in lib.pgg_status_string(6)
    g = 1 << 20
    fc1 = lib.pgg_grouped_fc1_swiglu_clamped
    fc1.argtypes = [P, P, P, P, P, I64, I64, I64, I32, F32, P, P]
    assert fc1(g, g, g, g, g, 64, 64, 64, 2, -1.0, None, None) == 1           # negative limit
    assert fc1(g, g, g, g, g, 64, 64, 64, 2, float("nan"), None, None) == 1   # NaN limit
    assert fc1(g, g, g, g, g, 0, 64, 64, 2, 1.0, None, None) == 0             # M == 0 is a no-op
    fc2 = lib.pgg_grouped_fc2_dgrad_swiglu_bwd_clamped
    fc2.argtypes = [P, P, P, P, P, I64, I64, I64, I32, F32, P, P]
    assert fc2(g, g, g, g, g, 64, 64, 64, 2, float("inf"), None, None) == 1   # non-finite limit
    mxc = lib.pgg_mx_grouped_gemm_clamped
    mxc.argtypes = [I32, I32, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I32, F32, P, P]
    assert mxc(2, 1, g, g, g, g, None, g, g, None, None, None, 64, 128, 128, 1, 1.0, None, None) == 1  # wgrad
    q = lib.pgg_mx_quantize_rowwise_blocked
    q.argtypes = [P, I64, I64, I32, P, P, P]
    assert q(g, 4, 96, 1, g, g, None) == 3          # C % 128
    assert q(g, 4, 128, 7, g, g, None) == 1         # bad format
    assert q(g, 0, 128, 1, g, g, None) == 0         # R == 0 is a no-op


def test_fp8_entry_points_host_validation_without_gpu(lib):
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    g = 1 << 20
    ws = lib.pgg_fp8_workspace_size
    ws.argtypes, ws.restype = [I64, I64, I32, I64], ctypes.c_size_t
    # the plain FP8 MMAs read no scale factors: no scratch in any mode
    assert ws(4096, 4096, 256, 0) == 0
    assert ws(64, 64, 2, 24576 + 256) == 0
    t = lib.pgg_fp8_tensor_scale
    t.argtypes = [P, I64, P, P]
    assert t(g, 12, g, None) == 3                        # n % 8
    assert t(g, 16, None, None) == 1                     # no output
    assert t(g, 16, g + 4, None) == 3                    # misaligned {s, amax}
    r = lib.pgg_fp8_quantize_rowwise
    r.argtypes = [P, I64, I64, P, P, P]
    assert r(g, 4, 12, g, g, None) == 3                  # C % 8
    assert r(g, 4, 16, None, g, None) == 1               # no scale
    assert r(g, 0, 16, g, g, None) == 0                  # R == 0 is a no-op
    c = lib.pgg_fp8_quantize_colwise
    c.argtypes = [P, I64, I64, P, I32, P, P, I64, P, P]
    assert c(g, 64, 16, g, 2, g, g, 100, None, None) == 3    # M_pad % 128
    assert c(g, 64, 16, g + 2, 2, g, g, 128, None, None) == 3  # misaligned group_lens
    assert c(g, 64, 16, None, 3, g, g, 128, None, None) == 1  # G > 1 without group_lens
    f = lib.pgg_fp8_grouped_gemm
    f.argtypes = [I32, I32, P, P, P, P, P, P, P, P, I64, I64, I64, I32, I64, ctypes.c_float, P, ctypes.c_size_t,
                  P, P]
    ok = dict(mode=0, epi=0, sa=g, ws=g, wsb=1 << 20, K=256, M=64, lim=0.0)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["mode"], a["epi"], g, a["sa"], g, g, None, g, g, None, a["M"], 128, a["K"], 2, 0, a["lim"],
                 a["ws"], a["wsb"], None, None)
    assert call(sa=None) == 1                    # no scale_a
    assert call(sa=g + 2) == 3                   # misaligned scale_a
    assert call(ws=None, wsb=0, M=0) == 0        # the reserved workspace may be absent
    assert call(K=200) == 3                      # fwd K % 128
    assert call(M=0) == 0                        # M == 0 is a no-op
    assert call(mode=3) == 1                     # bad mode
    assert call(lim=1.0) == 1                    # a clamp limit needs the SwiGLU epilogue
    assert call(epi=1, lim=-1.0) == 1            # negative limit
    assert call(mode=2, epi=1) == 1              # no SwiGLU wgrad


def test_scalar_operand_alignment_is_checked(lib):
    # 4-byte operands read by scalar or 4-byte copies: group_lens, the row-major MX scales,
    # the combine's positions and weights
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    g = 1 << 20
    f = lib.pgg_grouped_gemm_fwd
    f.argtypes = [P, P, P, P, I64, I64, I64, I32, P, P]
    assert f(g, g, g + 2, g, 8, 64, 64, 1, None, None) == 3           # group_lens
    mx = lib.pgg_mx_grouped_gemm
    mx.argtypes = [I32, I32, I32, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, I32, I64, P, P]
    assert mx(0, 1, 0, g, g + 2, g, g, None, g, g, None, None, None, 8, 64, 128, 1, 0, None, None) == 3  # SA
    assert mx(0, 1, 0, g, g, g, g, None, g, g, None, None, None, 8, 64, 128, 1, 0, g + 1, None) == 3  # err
    c = lib.pgg_moe_combine
    c.argtypes = [P, P, P, P, I64, I32, I64, P]
    assert c(g, g + 2, None, g, 8, 4, 64, None) == 3                  # pos
    assert c(g, g, g + 1, g, 8, 4, 64, None) == 3                     # w
    b = lib.pgg_moe_combine_bwd
    b.argtypes = [P, P, P, P, P, P, I64, I32, I64, P]
    assert b(g, g, g, g, g, g + 2, 8, 4, 64, None) == 3               # dw


def test_stall_hook_validation_without_gpu(lib):
    # the test hook rejects a negative stall point and a wait limit outside [100 us, 1 s]
    # before any CUDA call
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f = lib.pgg_test_stalled_fwd
    f.argtypes = [ctypes.c_int, P, P, P, P, P, P, I64, I64, I64, ctypes.c_int, I64, ctypes.c_uint64, P, P]
    g = P(1 << 20)
    assert f(0, g, None, g, None, g, g, 256, 256, 256, 1, -1, 2_000_000, None, None) == 1
    assert f(0, g, None, g, None, g, g, 256, 256, 256, 1, 0, 50_000, None, None) == 1
    assert f(0, g, None, g, None, g, g, 256, 256, 256, 1, 0, 2_000_000_000, None, None) == 1
