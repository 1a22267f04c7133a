"""GPU MX quantization (row-wise and group-aware column-wise) vs the oracle: bit-exact."""
import os

import numpy as np
import pytest
import torch

from oracle import mx as omx
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mx_blocks.txt")


def _mixed(R, C, seed):
    """bf16 [R, C] with per-row scales over a wide exponent range, zeros, ties and extremes."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, C, generator=g, dtype=torch.float64)
    x *= torch.pow(2.0, torch.randint(-40, 40, (R, 1), generator=g).double())
    x[::7, :5] = 0.0
    x[1::11, 3] = -0.0
    x[2::13, :] *= 1e-30
    t = x.to(torch.bfloat16)
    t[3::17, 0] = torch.tensor(3.0e38, dtype=torch.bfloat16)
    return t


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("R,C", [(1, 32), (37, 96), (512, 1024)])
def test_rowwise_bit_exact(fmt, R, C):
    x = _mixed(R, C, R * 1000 + C)
    codes, scales = pgg.mx_quantize_rowwise(x.to(DEV), fmt)
    rc, rs = omx.mx_quantize_rowwise(util.bits(x), fmt)
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


def test_rowwise_golden_blocks():
    rows = []
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            p = line.split()
            rows.append((p[0], float.fromhex(p[1]), float.fromhex(p[2]), int(p[3], 16), int(p[4], 16)))
    for fmt in ("e4m3", "e2m1"):
        cases = [r for r in rows if r[0] == fmt]
        x = torch.zeros(len(cases), 32, dtype=torch.float64)
        for i, (_, amax, v, _, _) in enumerate(cases):
            x[i, 0], x[i, 1] = amax, v
        codes, scales = pgg.mx_quantize_rowwise(x.to(torch.bfloat16).to(DEV), fmt)
        codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
        if fmt == "e2m1":
            codes = omx.unpack_e2m1(codes)
        for i, (_, amax, v, sc, code) in enumerate(cases):
            assert scales[i, 0] == sc, (fmt, amax, v)
            assert codes[i, 1] == code, (fmt, amax, v, hex(codes[i, 1]))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_rowwise_non_finite_block(fmt):
    x = torch.ones(2, 64, dtype=torch.bfloat16)
    x[0, 5] = float("nan")
    x[1, 40] = float("inf")
    codes, scales = pgg.mx_quantize_rowwise(x.to(DEV), fmt)
    rc, rs = omx.mx_quantize_rowwise(util.bits(x), fmt)
    np.testing.assert_array_equal(scales.cpu().numpy(), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    assert scales[0, 0].item() == 0xFF and scales[1, 1].item() == 0xFF


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("R,C", [(200, 256), (128, 128), (1, 384)])
def test_rowwise_blocked_bit_exact(fmt, R, C):
    # the weight layout: same codes as the row-wise quantizer, scales in 512-byte atoms
    x = _mixed(R, C, R + C)
    codes, scales = pgg.mx_quantize_rowwise_blocked(x.to(DEV), fmt)
    rc, rs = omx.mx_quantize_rowwise(util.bits(x), fmt)
    assert tuple(scales.shape) == (-(-R // 128) * 128, C // 32)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(util.unblock_scales(scales, R, C), rs)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("lens", [[33, 0, 5, 64, 1, 200], [128, 256], [0, 0, 7]])
def test_colwise_bit_exact(fmt, lens):
    lens = np.asarray(lens, dtype=np.int32)
    M, C = int(lens.sum()), 136
    x = _mixed(M, C, int(lens.sum()) + 5)
    M_pad = pgg.mx_pad_rows(M, len(lens)) + 128
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ct, st = pgg.mx_quantize_colwise(x.to(DEV), torch.from_numpy(lens).to(DEV), fmt, M_pad, err=err)
    assert pgg.read_error(err) == 0
    rc, rs = omx.mx_quantize_colwise(util.bits(x), lens, fmt, M_pad, 128)
    assert tuple(st.shape) == (256, M_pad // 32)  # 136 scale rows padded to whole 128-row atoms
    np.testing.assert_array_equal(util.unblock_scales(st, C, M_pad), rs)
    np.testing.assert_array_equal(ct.cpu().numpy(), rc)


def test_colwise_single_group_and_errors():
    x = _mixed(100, 64, 3)
    ct, st = pgg.mx_quantize_colwise(x.to(DEV), None, "e4m3", 128)
    rc, rs = omx.mx_quantize_colwise(util.bits(x), [100], "e4m3", 128, 128)
    np.testing.assert_array_equal(ct.cpu().numpy(), rc)
    np.testing.assert_array_equal(util.unblock_scales(st, 64, 128), rs)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    # two groups of 50 rows need 256 padded columns; 128 is too few
    pgg.mx_quantize_colwise(x.to(DEV), torch.tensor([50, 50], dtype=torch.int32, device=DEV),
                            "e4m3", 128, err=err)
    assert pgg.read_error(err) == 18
    err.zero_()
    pgg.mx_quantize_colwise(x.to(DEV), torch.tensor([60, 30], dtype=torch.int32, device=DEV), "e4m3", 256, err=err)
    assert pgg.read_error(err) == 16


def test_rowwise_full_size_activation_sample():
    # DeepSeek-shaped layer activation X [24576, 4096]: GPU quantizes the whole tensor,
    # the oracle checks a seeded sample of 256 rows
    w = wl.DSV4_MXFP8
    M = 24576
    X = wl.gen_matrix(wl.KEY_X, M, w.hidden, 1.0, w.seed, device=DEV)
    codes, scales = pgg.mx_quantize_rowwise(X, "e4m3")
    rows = np.sort(np.random.default_rng(0).choice(M, 256, replace=False))
    ref_c, ref_s = omx.mx_quantize_rowwise(util.bits(X[rows]), "e4m3")
    np.testing.assert_array_equal(codes[rows].cpu().numpy(), ref_c)
    np.testing.assert_array_equal(scales[rows].cpu().numpy(), ref_s)
