"""Full-size parity of the block-scaled (MX) expert layer in the launch configuration
bench.py times (all experts, full shapes), step-isolated: every call gets generator
inputs (synthetic A, H, dH in place of the previous call's output).  The GPU quantizes
with its own kernels; the oracle quantizes the same bf16 values of whole sampled experts
itself and compares each call's output against the fp64 GEMM of its dequantized
operands at |gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref)."""
import numpy as np
import pytest
import torch

import precision_grouped_gemm_gb300 as pgg
from oracle import mx as omx
from precision_grouped_gemm_gb300 import workloads as wl
from precision_grouped_gemm_gb300.layer import MxLayerBuffers, build_layer_inputs, expert_inputs_cpu
import util

pytestmark = pytest.mark.gpu
DEV = "cuda"
SYN_STD = {"A": 0.5, "H": 1.25, "dH": 0.25}


def _syn(w, key, rows, cols, std, row0=0, device="cpu"):
    return wl.gen_matrix(key, rows, cols, std, w.seed, device=device, row0=row0)


@pytest.mark.parametrize("w", [wl.DSV4_MXFP8, wl.ZIPF_MXFP4], ids=lambda w: w.name)
def test_mx_layer_full_size_isolated(w):
    f = w.fmt
    lens, row_token, b = build_layer_inputs(w, torch.device(DEV), allocate=False)
    M, G, Hd, I = int(lens.sum()), len(lens), w.hidden, w.inter
    mb = MxLayerBuffers.build(f, b.X, b.W1, b.W2, b.dY, b.group_lens)
    del b
    torch.cuda.empty_cache()
    u, gl, err, Mp = mb.bufs, mb.group_lens, mb.bufs["err"], mb.M_pad
    As = _syn(w, wl.KEY_A, M, I, SYN_STD["A"], device=DEV)
    Hs = _syn(w, wl.KEY_H, M, 2 * I, SYN_STD["H"], device=DEV)
    dHs = _syn(w, wl.KEY_DH, M, 2 * I, SYN_STD["dH"], device=DEV)
    mg = pgg.mx_grouped_gemm
    # the six GEMMs of the layer step, each on generator inputs quantized by the GPU
    pgg.mx_quantize_rowwise(mb.X, f, *u["Xq"])
    mg(pgg.MODE_FWD, f, *u["Xq"], *mb.W1q, gl, M, 2 * I, Hd, out=u["A"], out2=u["H"], epilogue=pgg.EPI_SWIGLU,
       err=err)
    Aq = pgg.mx_quantize_rowwise(As, f)
    Y = mg(pgg.MODE_FWD, f, *Aq, *mb.W2q, gl, M, Hd, I, err=err)
    pgg.mx_quantize_rowwise(mb.dY, f, *u["dYq"])
    dH = mg(pgg.MODE_DGRAD, f, *u["dYq"], *mb.W2t, gl, M, Hd, I, H=Hs, epilogue=pgg.EPI_SWIGLU, err=err)
    dYc = pgg.mx_quantize_colwise(mb.dY, gl, f, Mp, err=err)
    Ac = pgg.mx_quantize_colwise(As, gl, f, Mp, err=err)
    dW2 = mg(pgg.MODE_WGRAD, f, *dYc, *Ac, gl, M, Hd, I, M_pad=Mp, err=err)
    dHq = pgg.mx_quantize_rowwise(dHs, f)
    dX = mg(pgg.MODE_DGRAD, f, *dHq, *mb.W1t, gl, M, 2 * I, Hd, err=err)
    dHc = pgg.mx_quantize_colwise(dHs, gl, f, Mp, err=err)
    Xc = pgg.mx_quantize_colwise(mb.X, gl, f, Mp, err=err)
    dW1 = mg(pgg.MODE_WGRAD, f, *dHc, *Xc, gl, M, 2 * I, Hd, M_pad=Mp, err=err)
    assert pgg.read_error(err) == 0
    nz = np.nonzero(lens)[0]
    experts = (int(nz[0]), int(nz[np.argmax(lens[nz])]), int(nz[np.argmin(lens[nz])]))
    one = lambda n: np.array([n], dtype=np.int32)
    for e in experts:
        X, W1, W2, dY, (r0, r1) = expert_inputs_cpu(w, lens, row_token, e)
        n = r1 - r0
        a = _syn(w, wl.KEY_A, n, I, SYN_STD["A"], row0=r0)
        h = _syn(w, wl.KEY_H, n, 2 * I, SYN_STD["H"], row0=r0)
        dh = _syn(w, wl.KEY_DH, n, 2 * I, SYN_STD["dH"], row0=r0)
        B = util.bits
        xq = omx.mx_quantize_rowwise(B(X), f)
        w1q = omx.mx_quantize_rowwise(B(W1), f)
        refA, refH = omx.mx_grouped_fc1_swiglu(f, *xq, *w1q, one(n), 1)
        util.assert_close(u["H"][r0:r1], refH, f"expert {e} fc1 H")
        util.assert_close(u["A"][r0:r1], refA, f"expert {e} fc1 A")
        aq, w2q = omx.mx_quantize_rowwise(B(a), f), omx.mx_quantize_rowwise(B(W2), f)
        util.assert_close(Y[r0:r1], omx.mx_grouped_gemm_fwd(f, *aq, *w2q, one(n), 1), f"expert {e} fc2 fwd")
        dyq = omx.mx_quantize_rowwise(B(dY), f)
        w2t = omx.mx_quantize_colwise(B(W2), [Hd], f, Hd)
        ref = omx.mx_grouped_fc2_dgrad_swiglu_bwd(f, *dyq, *w2t, util.f64(h), one(n), 1)
        util.assert_close(dH[r0:r1], ref, f"expert {e} fc2 dgrad+swiglu'")
        mp = -(-n // 128) * 128
        dyc, ac = omx.mx_quantize_colwise(B(dY), [n], f, mp), omx.mx_quantize_colwise(B(a), [n], f, mp)
        util.assert_close(dW2[e], omx.mx_grouped_gemm_wgrad(f, *dyc, *ac, one(n))[0], f"expert {e} fc2 wgrad")
        dhq, w1t = omx.mx_quantize_rowwise(B(dh), f), omx.mx_quantize_colwise(B(W1), [2 * I], f, 2 * I)
        util.assert_close(dX[r0:r1], omx.mx_grouped_gemm_dgrad(f, *dhq, *w1t, one(n), 1), f"expert {e} fc1 dgrad")
        dhc, xc = omx.mx_quantize_colwise(B(dh), [n], f, mp), omx.mx_quantize_colwise(B(X), [n], f, mp)
        util.assert_close(dW1[e], omx.mx_grouped_gemm_wgrad(f, *dhc, *xc, one(n))[0], f"expert {e} fc1 wgrad")
