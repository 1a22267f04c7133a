"""Bitwise run-to-run reproducibility of every kernel family.

Each output tile is owned by one CTA and reduced in a fixed order (no float
atomics), and the fp32 main_grad accumulation adds each element exactly once
per call, so two runs on the same inputs must agree bit for bit: the block-
scaled (MX) and FP8 tensor-wise GEMMs in every mode, the fused SwiGLU
epilogues with their fused MX outputs, the fp32 accumulate, the quantizers
and the MoE combine and its backward."""
import numpy as np
import pytest
import torch

from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = [pytest.mark.gpu, pytest.mark.deterministic]
DEV = "cuda"
LENS = [100, 0, 300, 57, 1, 129]


def _twice(fn):
    a = fn()
    b = fn()
    torch.cuda.synchronize()
    return a, b


def _same(a, b, what):
    a = a if isinstance(a, (tuple, list)) else (a,)
    b = b if isinstance(b, (tuple, list)) else (b,)
    for i, (x, y) in enumerate(zip(a, b)):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), f"{what}: output {i} differs between runs"


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_mx_gemms_bitwise(fmt):
    lens = np.asarray(LENS, dtype=np.int32)
    G, M, N, K, I = len(lens), int(lens.sum()), 256, 384, 128
    gl = torch.from_numpy(lens).to(DEV)
    X = util.gen(wl.KEY_X, M, K, 1.0, 41, device=DEV)
    dY = util.gen(wl.KEY_DY, M, N, 1.0, 41, device=DEV)
    W = util.gen(wl.KEY_W1, G * N, K, 0.5, 41, device=DEV)
    W1 = util.gen(wl.KEY_W1, G * 2 * I, K, 0.5, 42, device=DEV)
    H = util.gen(wl.KEY_H, M, 2 * I, 1.0, 42, device=DEV)
    dYi = util.gen(wl.KEY_DY, M, N, 1.0, 43, device=DEV)
    W2 = util.gen(wl.KEY_W2, G * N, I, 0.5, 43, device=DEV)
    Mp = pgg.mx_pad_rows(M, G)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Xq = pgg.mx_quantize_rowwise(X, fmt)
    Wq = pgg.mx_quantize_rowwise_blocked(W, fmt)
    W1q = pgg.mx_quantize_rowwise_blocked(W1, fmt)
    dYq = pgg.mx_quantize_rowwise(dYi, fmt)
    W2t = pgg.mx_quantize_colwise(W2, torch.full((G,), N, dtype=torch.int32, device=DEV), fmt, G * N)
    Wt = pgg.mx_quantize_colwise(W, torch.full((G,), N, dtype=torch.int32, device=DEV), fmt, G * N)
    dYr = pgg.mx_quantize_rowwise(dY, fmt)
    cb = (lambda c: c) if fmt == "e4m3" else (lambda c: c // 2)

    def run():
        out = {}
        out["q_row"] = pgg.mx_quantize_rowwise(X, fmt)
        out["q_col"] = pgg.mx_quantize_colwise(X, gl, fmt, Mp, err=err)
        out["fwd"] = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, *Xq, *Wq, gl, M, N, K, err=err)
        out["dgrad"] = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, *dYr, *Wt, gl, M, N, K, err=err)
        dYc = pgg.mx_quantize_colwise(dY, gl, fmt, Mp, err=err)
        out["wgrad"] = pgg.mx_grouped_gemm(pgg.MODE_WGRAD, fmt, *dYc, *out["q_col"], gl, M, N, K, M_pad=Mp, err=err)
        Aq = (torch.empty((M, cb(I)), dtype=torch.uint8, device=DEV), torch.empty((M, I // 32), dtype=torch.uint8,
                                                                                     device=DEV))
        A = torch.empty((M, I), dtype=torch.bfloat16, device=DEV)
        Hs = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=DEV)
        pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, *Xq, *W1q, gl, M, 2 * I, K, out=A, out2=Hs, epilogue=pgg.EPI_SWIGLU,
                            err=err, out_q=Aq)
        out["swiglu"] = (A, Hs, *Aq)
        dHq = (torch.empty((M, cb(2 * I)), dtype=torch.uint8, device=DEV),
               torch.empty((M, 2 * I // 32), dtype=torch.uint8, device=DEV))
        dH = pgg.mx_grouped_gemm(pgg.MODE_DGRAD, fmt, *dYq, *W2t, gl, M, N, I, H=H, epilogue=pgg.EPI_SWIGLU,
                                 err=err, out_q=dHq)
        out["swiglu_bwd"] = (dH, *dHq)
        return out

    a, b = _twice(run)
    assert pgg.read_error(err) == 0
    for k in a:
        _same(a[k], b[k], f"mx {fmt} {k}")


def test_fp32_accumulate_bitwise():
    lens = np.asarray(LENS, dtype=np.int32)
    G, M, N, K = len(lens), int(lens.sum()), 192, 320
    gl = torch.from_numpy(lens).to(DEV)
    X = util.gen(wl.KEY_X, M, K, 1.0, 44, device=DEV)
    dY = util.gen(wl.KEY_DY, M, N, 1.0, 44, device=DEV)
    base = util.gen(wl.KEY_W1, G * N, K, 3.0, 44, device=DEV).float().view(G, N, K)

    def run():
        acc = base.clone()
        for _ in range(3):  # repeated accumulation into the same main_grad
            pgg.grouped_gemm_wgrad_accumulate(X, dY, gl, acc)
        return acc

    a, b = _twice(run)
    _same(a, b, "fp32 accumulate")


def test_fp8_gemms_bitwise():
    lens = np.asarray(LENS, dtype=np.int32)
    G, M, N, K = len(lens), int(lens.sum()), 256, 256
    gl = torch.from_numpy(lens).to(DEV)
    X = util.gen(wl.KEY_X, M, K, 1.0, 45, device=DEV)
    dY = util.gen(wl.KEY_DY, M, N, 1.0, 45, device=DEV)
    W = util.gen(wl.KEY_W1, G * N, K, 0.5, 45, device=DEV)
    Mp = pgg.mx_pad_rows(M, G)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def run():
        sx, sd, sw = pgg.fp8_tensor_scale(X), pgg.fp8_tensor_scale(dY), pgg.fp8_tensor_scale(W)
        xq, dq, wq = pgg.fp8_quantize_rowwise(X, sx), pgg.fp8_quantize_rowwise(dY, sd), pgg.fp8_quantize_rowwise(W, sw)
        wt = pgg.fp8_quantize_colwise(W, torch.full((G,), N, dtype=torch.int32, device=DEV), sw, G * N)
        xc, dc = pgg.fp8_quantize_colwise(X, gl, sx, Mp, err=err), pgg.fp8_quantize_colwise(dY, gl, sd, Mp, err=err)
        g = pgg.fp8_grouped_gemm
        y = g(pgg.MODE_FWD, xq, sx, wq, sw, gl, M, N, K, err=err)
        dx = g(pgg.MODE_DGRAD, dq, sd, wt, sw, gl, M, N, K, err=err)
        dw = g(pgg.MODE_WGRAD, dc, sd, xc, sx, gl, M, N, K, M_pad=Mp, err=err)
        return (sx, sd, sw, xq, dq, wq, wt, xc, dc, y, dx, dw)

    a, b = _twice(run)
    assert pgg.read_error(err) == 0
    _same(a, b, "fp8")


def test_combine_bitwise():
    rng = np.random.Generator(np.random.PCG64(46))
    T, k, E, H = 777, 6, 64, 520
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    X = util.gen(wl.KEY_X, T, H, 1.0, 46, device=DEV)
    Xs, _, pos = pgg.moe_permute(torch.from_numpy(ids).to(DEV), X, E)
    w = torch.from_numpy(rng.random((T, k)).astype(np.float32)).to(DEV)
    dOut = util.gen(wl.KEY_DY, T, H, 1.0, 46, device=DEV)

    def run():
        out = pgg.moe_combine(Xs, pos, w)
        dYs, dw = pgg.moe_combine_bwd(dOut, Xs, pos, w)
        return (out, dYs, dw)

    a, b = _twice(run)
    _same(a, b, "combine")
