"""GPU block-scaled (MX) grouped GEMM vs the oracle.

Both sides start from the same bf16 tensors: the GPU quantizes them with its
own kernels, the oracle with its own code (the two agree bit for bit, which
test_parity_mx_quant checks), and the oracle's reference is the fp64 grouped
GEMM of its dequantized operands.  Bound per element:
|gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref).
"""
import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from oracle import mx as omx
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"
FMTS = ["e4m3", "e2m1"]


def _bf16(key, rows, cols, std, seed):
    return util.gen(key, rows, cols, std, seed)


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("lens,N,K", [([40, 0, 157], 256, 256), ([129, 1, 300, 0, 77], 384, 512), ([5], 128, 128)])
def test_mx_fwd(fmt, lens, N, K):
    lens = np.asarray(lens, dtype=np.int32)
    G, M = len(lens), int(lens.sum())
    X, W = _bf16(wl.KEY_X, M, K, 1.0, 31), _bf16(wl.KEY_W1, G * N, K, 0.5, 31)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W.to(DEV), fmt)
    err = _err()
    Y = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, torch.from_numpy(lens).to(DEV), M, N, K, err=err)
    assert pgg.read_error(err) == 0
    oA, oSA = omx.mx_quantize_rowwise(util.bits(X), fmt)
    oB, oSB = omx.mx_quantize_rowwise(util.bits(W), fmt)
    util.assert_close(Y, omx.mx_grouped_gemm_fwd(fmt, oA, oSA, oB, oSB, lens, G), f"mx fwd {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("lens,N,K", [([40, 0, 157], 256, 256), ([129, 1, 300, 0, 77], 384, 320)])
def test_mx_dgrad(fmt, lens, N, K):
    lens = np.asarray(lens, dtype=np.int32)
    G, M = len(lens), int(lens.sum())
    dY, W = _bf16(wl.KEY_DY, M, N, 1.0, 32), _bf16(wl.KEY_W1, G * N, K, 0.5, 32)
    A, SA = pgg.mx_quantize_rowwise(dY.to(DEV), fmt)
    wl_ = torch.full((G,), N, dtype=torch.int32, device=DEV)
    Bt, SBt = pgg.mx_quantize_colwise(W.to(DEV), wl_, fmt, G * N)
    err = _err()
    dX = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, A, SA, Bt, SBt, torch.from_numpy(lens).to(DEV), M, N, K, err=err)
    assert pgg.read_error(err) == 0
    oA, oSA = omx.mx_quantize_rowwise(util.bits(dY), fmt)
    oBt, oSBt = omx.mx_quantize_colwise(util.bits(W), [N] * G, fmt, G * N)
    util.assert_close(dX, omx.mx_grouped_gemm_dgrad(fmt, oA, oSA, oBt, oSBt, lens, G), f"mx dgrad {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("lens,N,K", [([40, 0, 157], 256, 256), ([129, 1, 300, 0, 77], 200, 320)])
def test_mx_wgrad(fmt, lens, N, K):
    lens = np.asarray(lens, dtype=np.int32)
    G, M = len(lens), int(lens.sum())
    X, dY = _bf16(wl.KEY_X, M, K, 1.0, 33), _bf16(wl.KEY_DY, M, N, 1.0, 33)
    gl = torch.from_numpy(lens).to(DEV)
    M_pad = pgg.mx_pad_rows(M, G)
    At, SAt = pgg.mx_quantize_colwise(dY.to(DEV), gl, fmt, M_pad)
    Bt, SBt = pgg.mx_quantize_colwise(X.to(DEV), gl, fmt, M_pad)
    err = _err()
    dW = pgg.mx_grouped_gemm(pgg.MODE_WGRAD, fmt, At, SAt, Bt, SBt, gl, M, N, K, M_pad=M_pad, err=err)
    assert pgg.read_error(err) == 0
    oAt, oSAt = omx.mx_quantize_colwise(util.bits(dY), lens, fmt, M_pad)
    oBt, oSBt = omx.mx_quantize_colwise(util.bits(X), lens, fmt, M_pad)
    ref = omx.mx_grouped_gemm_wgrad(fmt, oAt, oSAt, oBt, oSBt, lens)
    util.assert_close(dW, ref, f"mx wgrad {fmt}")
    for g in np.nonzero(lens == 0)[0]:
        assert torch.count_nonzero(dW[g]).item() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_swiglu_fwd_bwd(fmt):
    lens = np.array([70, 0, 190], dtype=np.int32)
    G, M, I, K = 3, 260, 192, 256
    X, W1 = _bf16(wl.KEY_X, M, K, 1.0, 34), _bf16(wl.KEY_W1, G * 2 * I, K, 0.1, 34)
    gl = torch.from_numpy(lens).to(DEV)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W1.to(DEV), fmt)
    H = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=DEV)
    err = _err()
    Aout = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, 2 * I, K, out2=H,
                               epilogue=pgg.EPI_SWIGLU, err=err)
    oA, oSA = omx.mx_quantize_rowwise(util.bits(X), fmt)
    oB, oSB = omx.mx_quantize_rowwise(util.bits(W1), fmt)
    refA, refH = omx.mx_grouped_fc1_swiglu(fmt, oA, oSA, oB, oSB, lens, G)
    util.assert_close(H, refH, f"mx fc1 H {fmt}")
    util.assert_close(Aout, refA, f"mx fc1 A {fmt}")
    # FC2 dgrad + SwiGLU backward with a synthetic saved H
    Hd = 256
    dY = _bf16(wl.KEY_DY, M, Hd, 1.0, 35)
    W2 = _bf16(wl.KEY_W2, G * Hd, I, 0.1, 35)
    Hs = _bf16(wl.KEY_H, M, 2 * I, 1.0, 35)
    Ad, SAd = pgg.mx_quantize_rowwise(dY.to(DEV), fmt)
    Bt, SBt = pgg.mx_quantize_colwise(W2.to(DEV), torch.full((G,), Hd, dtype=torch.int32, device=DEV), fmt, G * Hd)
    dH = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, Ad, SAd, Bt, SBt, gl, M, Hd, I, H=Hs.to(DEV),
                             epilogue=pgg.EPI_SWIGLU, err=err)
    assert pgg.read_error(err) == 0
    oAd, oSAd = omx.mx_quantize_rowwise(util.bits(dY), fmt)
    oBt, oSBt = omx.mx_quantize_colwise(util.bits(W2), [Hd] * G, fmt, G * Hd)
    ref = omx.mx_grouped_fc2_dgrad_swiglu_bwd(fmt, oAd, oSAd, oBt, oSBt, util.f64(Hs), lens, G)
    util.assert_close(dH, ref, f"mx fc2 dgrad swiglu bwd {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_swiglu_clamped(fmt):
    limit = 0.75
    lens = np.array([70, 0, 190], dtype=np.int32)
    G, M, I, K = 3, 260, 256, 256
    X, W1 = _bf16(wl.KEY_X, M, K, 1.0, 39), _bf16(wl.KEY_W1, G * 2 * I, K, 0.1, 39)
    gl = torch.from_numpy(lens).to(DEV)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W1.to(DEV), fmt)
    H = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=DEV)
    err = _err()
    Aout = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, 2 * I, K, out2=H,
                               epilogue=pgg.EPI_SWIGLU, err=err, swiglu_limit=limit)
    oA, oSA = omx.mx_quantize_rowwise(util.bits(X), fmt)
    oB, oSB = omx.mx_quantize_rowwise(util.bits(W1), fmt)
    refA, refH = omx.mx_grouped_fc1_swiglu(fmt, oA, oSA, oB, oSB, lens, G, limit)
    util.assert_close(H, refH, f"clamped mx fc1 H {fmt}")
    util.assert_close(Aout, refA, f"clamped mx fc1 A {fmt}")
    Hd = 256
    dY, W2, Hs = _bf16(wl.KEY_DY, M, Hd, 1.0, 40), _bf16(wl.KEY_W2, G * Hd, I, 0.1, 40), _bf16(wl.KEY_H, M, 2 * I, 1.0, 40)
    Ad, SAd = pgg.mx_quantize_rowwise(dY.to(DEV), fmt)
    Bt, SBt = pgg.mx_quantize_colwise(W2.to(DEV), torch.full((G,), Hd, dtype=torch.int32, device=DEV), fmt, G * Hd)
    dH = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, Ad, SAd, Bt, SBt, gl, M, Hd, I, H=Hs.to(DEV),
                             epilogue=pgg.EPI_SWIGLU, err=err, swiglu_limit=limit)
    assert pgg.read_error(err) == 0
    oAd, oSAd = omx.mx_quantize_rowwise(util.bits(dY), fmt)
    oBt, oSBt = omx.mx_quantize_colwise(util.bits(W2), [Hd] * G, fmt, G * Hd)
    ref = omx.mx_grouped_fc2_dgrad_swiglu_bwd(fmt, oAd, oSAd, oBt, oSBt, util.f64(Hs), lens, G, limit)
    util.assert_close(dH, ref, f"clamped mx fc2 dgrad swiglu bwd {fmt}")


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_lossless_operands_exact(fmt):
    # operands on the MX grid with power-of-two-friendly values: the block-scaled GEMM must
    # match the fp64 GEMM of the original values to fp32 accumulation accuracy
    rng = np.random.default_rng(36)
    grid = omx._grid(fmt)
    G, N, K = 2, 128, 256
    lens = np.array([64, 90], dtype=np.int32)
    M = int(lens.sum())

    def grid_tensor(rows, cols):
        codes = rng.integers(0, len(grid), size=(rows, cols))
        codes[:, ::32] = len(grid) - 1
        E = np.repeat(rng.integers(-3, 3, size=(rows, cols // 32)), 32, axis=1)
        v = grid[codes] * np.ldexp(1.0, E) * np.where(rng.random((rows, cols)) < 0.5, -1, 1)
        return torch.tensor(v, dtype=torch.float64).to(torch.bfloat16), v

    X, x = grid_tensor(M, K)
    W, w = grid_tensor(G * N, K)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W.to(DEV), fmt)
    Y = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, torch.from_numpy(lens).to(DEV), M, N, K)
    ref = og.grouped_gemm_fwd(x, w.reshape(G, N, K), lens)
    util.assert_close(Y, ref, f"mx lossless {fmt}")


def test_mx_pad_overflow_and_bad_lens():
    fmt = "e4m3"
    G, N, K = 2, 128, 128
    lens = torch.tensor([100, 100], dtype=torch.int32, device=DEV)
    M = 200
    z = torch.zeros((N, 128), dtype=torch.uint8, device=DEV)
    zs = torch.zeros((N, 4), dtype=torch.uint8, device=DEV)
    err = _err()
    # 2 groups of 100 rows need 256 padded columns; M_pad 128 is too small
    pgg.mx_grouped_gemm(pgg.MODE_WGRAD, fmt, z, zs, z, zs, lens, M, N, K, M_pad=128, err=err)
    assert pgg.read_error(err) == 18
    err.zero_()
    A = torch.zeros((M, K), dtype=torch.uint8, device=DEV)
    SA = torch.zeros((M, K // 32), dtype=torch.uint8, device=DEV)
    B = torch.zeros((G * N, K), dtype=torch.uint8, device=DEV)
    SB = torch.zeros((G * N, K // 32), dtype=torch.uint8, device=DEV)
    pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, torch.tensor([100, 99], dtype=torch.int32, device=DEV),
                        M, N, K, err=err)
    assert pgg.read_error(err) == 16


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_fused_quantized_outputs(fmt):
    # the SwiGLU epilogues' fused MX outputs equal the row-wise quantizer applied to the
    # bf16 tensor they stored (the quantizer itself is bit-exact against the oracle)
    lens = np.array([70, 0, 190], dtype=np.int32)
    G, M, I, K = 3, 260, 192, 256
    X, W1 = _bf16(wl.KEY_X, M, K, 1.0, 37), _bf16(wl.KEY_W1, G * 2 * I, K, 0.1, 37)
    gl = torch.from_numpy(lens).to(DEV)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W1.to(DEV), fmt)
    cb = I if fmt == "e4m3" else I // 2
    qc = torch.empty((M, cb), dtype=torch.uint8, device=DEV)
    qs = torch.empty((M, I // 32), dtype=torch.uint8, device=DEV)
    Aout = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, 2 * I, K, epilogue=pgg.EPI_SWIGLU,
                               out_q=(qc, qs))
    rc, rs = pgg.mx_quantize_rowwise(Aout, fmt)
    assert torch.equal(qc, rc) and torch.equal(qs, rs)
    Hd = 256
    dY, W2, Hs = _bf16(wl.KEY_DY, M, Hd, 1.0, 38), _bf16(wl.KEY_W2, G * Hd, I, 0.1, 38), _bf16(wl.KEY_H, M, 2 * I, 1.0, 38)
    Ad, SAd = pgg.mx_quantize_rowwise(dY.to(DEV), fmt)
    Bt, SBt = pgg.mx_quantize_colwise(W2.to(DEV), torch.full((G,), Hd, dtype=torch.int32, device=DEV), fmt, G * Hd)
    qc2 = torch.empty((M, 2 * cb), dtype=torch.uint8, device=DEV)
    qs2 = torch.empty((M, 2 * I // 32), dtype=torch.uint8, device=DEV)
    dH = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, Ad, SAd, Bt, SBt, gl, M, Hd, I, H=Hs.to(DEV),
                             epilogue=pgg.EPI_SWIGLU, out_q=(qc2, qs2))
    rc2, rs2 = pgg.mx_quantize_rowwise(dH, fmt)
    assert torch.equal(qc2, rc2) and torch.equal(qs2, rs2)
    # fused outputs exist only for the SwiGLU epilogues
    with pytest.raises(pgg.PggError):
        pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, 2 * I, K, out_q=(qc, qs))


@pytest.mark.parametrize("fmt", FMTS)
def test_mx_fwd_dgrad_max_groups(fmt):
    # 1024 groups (the most the kernels scan): their shared-memory group tables leave the
    # plain-store kernels one pipeline stage fewer than at a few hundred groups
    rng = np.random.default_rng(71)
    G, N, K = 1024, 128, 128
    lens = np.where(rng.random(G) < 0.1, rng.integers(1, 40, G), 0).astype(np.int32)
    M = int(lens.sum())
    gl = torch.from_numpy(lens).to(DEV)
    X, W = _bf16(wl.KEY_X, M, K, 1.0, 71), _bf16(wl.KEY_W1, G * N, K, 0.5, 71)
    dY = _bf16(wl.KEY_DY, M, N, 1.0, 71)
    A, SA = pgg.mx_quantize_rowwise(X.to(DEV), fmt)
    B, SB = pgg.mx_quantize_rowwise_blocked(W.to(DEV), fmt)
    err = _err()
    Y = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, N, K, err=err)
    dA, dSA = pgg.mx_quantize_rowwise(dY.to(DEV), fmt)
    Bt, SBt = pgg.mx_quantize_colwise(W.to(DEV), torch.full((G,), N, dtype=torch.int32, device=DEV), fmt, G * N)
    dX = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, dA, dSA, Bt, SBt, gl, M, N, K, err=err)
    assert pgg.read_error(err) == 0
    oA, oSA = omx.mx_quantize_rowwise(util.bits(X), fmt)
    oB, oSB = omx.mx_quantize_rowwise(util.bits(W), fmt)
    util.assert_close(Y, omx.mx_grouped_gemm_fwd(fmt, oA, oSA, oB, oSB, lens, G), f"mx fwd {fmt}, G = 1024")
    odA, odSA = omx.mx_quantize_rowwise(util.bits(dY), fmt)
    oBt, oSBt = omx.mx_quantize_colwise(util.bits(W), [N] * G, fmt, G * N)
    util.assert_close(dX, omx.mx_grouped_gemm_dgrad(fmt, odA, odSA, oBt, oSBt, lens, G), f"mx dgrad {fmt}, G = 1024")
