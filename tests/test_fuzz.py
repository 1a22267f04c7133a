"""Randomised shapes against the fp64 oracle (seeded, so every failure reproduces).

Each case draws G <= 64 groups whose lengths mix the boundary values around the
128-row tile and the 32-row MX block (0, 1, 31, 33, 127, 129, ...) with random
ones, and N, K as random multiples of 32 (of 128 where an MX operand is K-major
along that axis).  BF16 fwd / dgrad / wgrad, the MX GEMMs in e4m3 and e2m1 and
the FP8 tensor-wise GEMMs are compared element by element at
|gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref); empty-group weight gradients must be
exactly zero."""
import numpy as np
import pytest
import torch

from oracle import fp8 as of8
from oracle import grouped_gemm as og
from oracle import mx as omx
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"
EDGE_LENS = (0, 1, 31, 32, 33, 127, 128, 129, 255, 257)


def _case(seed, max_rows=6000, nonempty=True):
    rng = np.random.Generator(np.random.PCG64(seed))
    G = int(rng.integers(1, 65))
    pick = rng.random(G) < 0.6
    lens = np.where(pick, rng.choice(EDGE_LENS, size=G), rng.integers(0, 300, size=G)).astype(np.int32)
    while lens.sum() > max_rows:                       # keep the oracle fast: shrink the longest group
        lens[np.argmax(lens)] //= 2
    if nonempty and lens.sum() == 0:                   # the quantizers take a non-empty batch
        lens[-1] = 33
    return rng, lens


def _mult(rng, lo, hi, m):
    return int(rng.integers(lo // m, hi // m + 1)) * m


def _empty_groups_zero(dW, lens):
    for g in np.nonzero(lens == 0)[0]:
        assert torch.count_nonzero(dW[g]).item() == 0, f"empty group {g}: dW not zero"


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_bf16(seed):
    rng, lens = _case(100 + seed, nonempty=False)
    G, M = len(lens), int(lens.sum())
    N, K = _mult(rng, 32, 640, 32), _mult(rng, 32, 640, 32)
    X = util.gen(wl.KEY_X, max(M, 1), K, 1.0, seed)[:M]
    W = util.gen(wl.KEY_W1, G * N, K, 0.5, seed).view(G, N, K)
    dY = util.gen(wl.KEY_DY, max(M, 1), N, 1.0, seed)[:M]
    gl = torch.from_numpy(lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Xd, Wd, dYd = X.contiguous().to(DEV), W.to(DEV), dY.contiguous().to(DEV)
    Y = pgg.grouped_gemm_fwd(Xd, Wd, gl, err=err)
    dX = pgg.grouped_gemm_dgrad(dYd, Wd, gl, err=err)
    dW = pgg.grouped_gemm_wgrad(Xd, dYd, gl, err=err)
    assert pgg.read_error(err) == 0
    x, w, dy = util.f64(X), util.f64(W), util.f64(dY)
    what = f"seed {seed} G={G} M={M} N={N} K={K}"
    util.assert_close(Y, og.grouped_gemm_fwd(x, w, lens), f"{what} fwd")
    util.assert_close(dX, og.grouped_gemm_dgrad(dy, w, lens), f"{what} dgrad")
    util.assert_close(dW, og.grouped_gemm_wgrad(x, dy, lens), f"{what} wgrad")
    _empty_groups_zero(dW, lens)


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
@pytest.mark.parametrize("seed", range(5))
def test_fuzz_mx(fmt, seed):
    rng, lens = _case(200 + seed)
    G, M = len(lens), int(lens.sum())
    N, K = _mult(rng, 128, 512, 128), _mult(rng, 128, 512, 128)  # fwd: K-major K; dgrad: N
    Kw, Nw = _mult(rng, 32, 480, 32), _mult(rng, 32, 480, 32)    # wgrad output [G, Nw, Kw]
    gl = torch.from_numpy(lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    what = f"{fmt} seed {seed} G={G} M={M}"
    b = util.bits
    # fwd: X [M, K] row-wise, W [G*N, K] row-wise (blocked scales)
    X = util.gen(wl.KEY_X, max(M, 1), K, 1.0, seed)[:M].contiguous()
    W = util.gen(wl.KEY_W1, G * N, K, 0.5, seed)
    Y = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, *pgg.mx_quantize_rowwise(X.to(DEV), fmt),
                            *pgg.mx_quantize_rowwise_blocked(W.to(DEV), fmt), gl, M, N, K, err=err)
    ref = omx.mx_grouped_gemm_fwd(fmt, *omx.mx_quantize_rowwise(b(X), fmt), *omx.mx_quantize_rowwise(b(W), fmt),
                                  lens, G)
    util.assert_close(Y, ref, f"{what} fwd N={N} K={K}")
    # dgrad: dY [M, N] row-wise along N; W quantized along N, stored [K, G*N]
    dY = util.gen(wl.KEY_DY, max(M, 1), N, 1.0, seed)[:M].contiguous()
    wlen = torch.full((G,), N, dtype=torch.int32, device=DEV)
    dX = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, *pgg.mx_quantize_rowwise(dY.to(DEV), fmt),
                             *pgg.mx_quantize_colwise(W.to(DEV), wlen, fmt, G * N), gl, M, N, K, err=err)
    ref = omx.mx_grouped_gemm_dgrad(fmt, *omx.mx_quantize_rowwise(b(dY), fmt),
                                    *omx.mx_quantize_colwise(b(W), [N] * G, fmt, G * N), lens, G)
    util.assert_close(dX, ref, f"{what} dgrad N={N} K={K}")
    # wgrad: column-wise dY [M, Nw] and X [M, Kw]
    Mp = pgg.mx_pad_rows(M, G)
    dYw = util.gen(wl.KEY_DY, max(M, 1), Nw, 1.0, seed + 50)[:M].contiguous()
    Xw = util.gen(wl.KEY_X, max(M, 1), Kw, 1.0, seed + 50)[:M].contiguous()
    dW = pgg.mx_grouped_gemm(pgg.MODE_WGRAD, fmt, *pgg.mx_quantize_colwise(dYw.to(DEV), gl, fmt, Mp, err=err),
                             *pgg.mx_quantize_colwise(Xw.to(DEV), gl, fmt, Mp, err=err), gl, M, Nw, Kw, M_pad=Mp,
                             err=err)
    ref = omx.mx_grouped_gemm_wgrad(fmt, *omx.mx_quantize_colwise(b(dYw), lens, fmt, Mp),
                                    *omx.mx_quantize_colwise(b(Xw), lens, fmt, Mp), lens)
    assert pgg.read_error(err) == 0
    util.assert_close(dW, ref, f"{what} wgrad N={Nw} K={Kw}")
    _empty_groups_zero(dW, lens)


@pytest.mark.parametrize("seed", range(4))
def test_fuzz_fp8(seed):
    rng, lens = _case(300 + seed)
    G, M = len(lens), int(lens.sum())
    # the FP8 GEMM takes the MX operand layouts: K-major K (fwd) and N (dgrad) in whole
    # 128-element k-blocks; the wgrad output [G, Nw, Kw] is free in multiples of 32
    N, K = _mult(rng, 128, 512, 128), _mult(rng, 128, 512, 128)
    Nw, Kw = _mult(rng, 32, 480, 32), _mult(rng, 32, 480, 32)
    gl = torch.from_numpy(lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    X = util.gen(wl.KEY_X, max(M, 1), K, 1.0, seed)[:M].contiguous()
    W = util.gen(wl.KEY_W1, G * N, K, 0.5, seed)
    dY = util.gen(wl.KEY_DY, max(M, 1), N, 1.0, seed)[:M].contiguous()
    Xw = util.gen(wl.KEY_X, max(M, 1), Kw, 1.0, seed + 50)[:M].contiguous()
    dYw = util.gen(wl.KEY_DY, max(M, 1), Nw, 1.0, seed + 50)[:M].contiguous()
    Xd, Wd, dYd, Xwd, dYwd = X.to(DEV), W.to(DEV), dY.to(DEV), Xw.to(DEV), dYw.to(DEV)
    Mp = pgg.mx_pad_rows(M, G)
    sx, sw, sd = (pgg.fp8_tensor_scale(t) if t.numel() else None for t in (Xd, Wd, dYd))
    what = f"fp8 seed {seed} G={G} M={M} N={N} K={K}"
    g = pgg.fp8_grouped_gemm
    x, w, dy = util.f64(X), util.f64(W), util.f64(dY)
    s_w = of8.fp8_tensor_scale(w)
    wq, _ = of8.fp8_quantize_tensorwise(w, scale=s_w)
    if M:
        s_x, s_d = of8.fp8_tensor_scale(x), of8.fp8_tensor_scale(dy)
        xq, _ = of8.fp8_quantize_tensorwise(x, scale=s_x)
        dq, _ = of8.fp8_quantize_tensorwise(dy, scale=s_d)
        Y = g(pgg.MODE_FWD, pgg.fp8_quantize_rowwise(Xd, sx), sx, pgg.fp8_quantize_rowwise(Wd, sw), sw, gl, M, N, K,
              err=err)
        util.assert_close(Y, of8.fp8_grouped_gemm_fwd(xq, s_x, wq, s_w, lens, G), f"{what} fwd")
        wt = pgg.fp8_quantize_colwise(Wd, torch.full((G,), N, dtype=torch.int32, device=DEV), sw, G * N)
        dX = g(pgg.MODE_DGRAD, pgg.fp8_quantize_rowwise(dYd, sd), sd, wt, sw, gl, M, N, K, err=err)
        util.assert_close(dX, of8.fp8_grouped_gemm_dgrad(dq, s_d, wq, s_w, lens, G), f"{what} dgrad")
        sxw, sdw = pgg.fp8_tensor_scale(Xwd), pgg.fp8_tensor_scale(dYwd)
        dW = g(pgg.MODE_WGRAD, pgg.fp8_quantize_colwise(dYwd, gl, sdw, Mp, err=err), sdw,
               pgg.fp8_quantize_colwise(Xwd, gl, sxw, Mp, err=err), sxw, gl, M, Nw, Kw, M_pad=Mp, err=err)
        assert pgg.read_error(err) == 0
        xw, dyw = util.f64(Xw), util.f64(dYw)
        s_xw, s_dw = of8.fp8_tensor_scale(xw), of8.fp8_tensor_scale(dyw)
        xwq, _ = of8.fp8_quantize_tensorwise(xw, scale=s_xw)
        dwq, _ = of8.fp8_quantize_tensorwise(dyw, scale=s_dw)
        util.assert_close(dW, of8.fp8_grouped_gemm_wgrad(xwq, s_xw, dwq, s_dw, lens), f"{what} wgrad Nw={Nw} Kw={Kw}")
        _empty_groups_zero(dW, lens)
