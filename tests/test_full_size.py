"""Full-size parity in the benchmark's launch configuration.

The six launches of one expert-layer step run on the complete workload (all
experts, full shapes, the same kernels and grids bench.py times); the fp64
oracle then recomputes whole experts from the generator's values -- never from
a GPU result -- and every element of those experts' outputs is compared.

* isolated: each call gets its own generator inputs (synthetic A, H, dH in
  place of the previous call's output), so every call is checked on exactly
  the operands it consumed, at |gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref).
* chained: the real step (FC1 output feeds FC2, ...).  The GPU hands A, H and
  dH to the next call in bf16, the oracle rounds its own fp64 values of those
  tensors, and the two roundings can land one bf16 ulp apart (at most 2^-7
  relative) where the tensor core's fp32 sum and the fp64 sum straddle a
  rounding midpoint.  Each downstream output is checked at the stated bound
  plus that ulp propagated to first order: 2^-7 (|P| . |Q|) for a GEMM whose
  operand P is a bf16 intermediate, and 2^-7 (|dA phi(g)| |u| + |dA u phi'(g)|
  |g|), 2^-7 |dA phi(g)| |g| for the SwiGLU backward's two halves, with
  phi = d silu / dg.  The direct FC1 outputs get the plain stated bound.
"""
import numpy as np
import pytest
import torch

import precision_grouped_gemm_gb300 as pgg
from oracle import grouped_gemm as og
from precision_grouped_gemm_gb300 import workloads as wl
from precision_grouped_gemm_gb300.layer import build_layer_inputs, expert_inputs_cpu, expert_layer_step
import util

pytestmark = pytest.mark.gpu
DEV = "cuda"
SYN_STD = {"A": 0.5, "H": 1.25, "dH": 0.25}


def _synthetic(w, key, rows, cols, std, row0=0, device="cpu"):
    return wl.gen_matrix(key, rows, cols, std, w.seed, device=device, row0=row0)


def _experts(w, lens):
    nz = np.nonzero(lens)[0]
    if w is wl.DSV4_BF16:
        return (0, 97, 255)
    return (int(nz[np.argmax(lens[nz])]), int(nz[np.argmin(lens[nz])]))


@pytest.mark.parametrize("w", [wl.DSV4_BF16, wl.GPTOSS_BF16], ids=lambda w: w.name)
def test_layer_full_size_isolated(w):
    lens, row_token, b = build_layer_inputs(w, torch.device(DEV))
    M, I, Hd = int(lens.sum()), w.inter, w.hidden
    As = _synthetic(w, wl.KEY_A, M, I, SYN_STD["A"], device=DEV)
    Hs = _synthetic(w, wl.KEY_H, M, 2 * I, SYN_STD["H"], device=DEV)
    dHs = _synthetic(w, wl.KEY_DH, M, 2 * I, SYN_STD["dH"], device=DEV)
    gl, err = b.group_lens, b.err
    pgg.grouped_fc1_swiglu(b.X, b.W1, gl, A=b.A, H=b.H, err=err)
    pgg.grouped_gemm_fwd(As, b.W2, gl, Y=b.Y, err=err)
    pgg.grouped_fc2_dgrad_swiglu_bwd(b.dY, b.W2, Hs, gl, dH=b.dH, err=err)
    pgg.grouped_gemm_wgrad(As, b.dY, gl, dW=b.dW2, err=err)
    pgg.grouped_gemm_dgrad(dHs, b.W1, gl, dX=b.dX, err=err)
    pgg.grouped_gemm_wgrad(b.X, dHs, gl, dW=b.dW1, err=err)
    assert pgg.read_error(err) == 0
    for e in _experts(w, lens):
        X, W1, W2, dY, (r0, r1) = expert_inputs_cpu(w, lens, row_token, e)
        n = r1 - r0
        one = np.array([n], dtype=np.int32)
        x, w1, w2, dy = util.f64(X), util.f64(W1)[None], util.f64(W2)[None], util.f64(dY)
        a = util.f64(_synthetic(w, wl.KEY_A, n, I, SYN_STD["A"], row0=r0))
        h = util.f64(_synthetic(w, wl.KEY_H, n, 2 * I, SYN_STD["H"], row0=r0))
        dh = util.f64(_synthetic(w, wl.KEY_DH, n, 2 * I, SYN_STD["dH"], row0=r0))
        refA, refH = og.grouped_fc1_swiglu(x, w1, one)
        util.assert_close(b.H[r0:r1], refH, f"expert {e} fc1 H")
        util.assert_close(b.A[r0:r1], refA, f"expert {e} fc1 A")
        util.assert_close(b.Y[r0:r1], og.grouped_gemm_fwd(a, w2, one), f"expert {e} fc2 fwd")
        util.assert_close(b.dH[r0:r1], og.grouped_fc2_dgrad_swiglu_bwd(dy, w2, h, one), f"expert {e} fc2 dgrad+swiglu'")
        util.assert_close(b.dW2[e], og.grouped_gemm_wgrad(a, dy, one)[0], f"expert {e} fc2 wgrad")
        util.assert_close(b.dX[r0:r1], og.grouped_gemm_dgrad(dh, w1, one), f"expert {e} fc1 dgrad")
        util.assert_close(b.dW1[e], og.grouped_gemm_wgrad(x, dh, one)[0], f"expert {e} fc1 wgrad")
    for e in np.nonzero(lens == 0)[0]:
        assert torch.count_nonzero(b.dW1[e]).item() == 0 and torch.count_nonzero(b.dW2[e]).item() == 0


@pytest.mark.parametrize("w", [wl.DSV4_BF16, wl.GPTOSS_BF16], ids=lambda w: w.name)
def test_layer_full_size_chained(w):
    lens, row_token, b = build_layer_inputs(w, torch.device(DEV))
    expert_layer_step(b)
    torch.cuda.synchronize()
    assert pgg.read_error(b.err) == 0
    for e in _experts(w, lens):
        X, W1, W2, dY, (r0, r1) = expert_inputs_cpu(w, lens, row_token, e)
        assert torch.equal(b.X[r0:r1].cpu().view(torch.int16), X.view(torch.int16))
        one = np.array([r1 - r0], dtype=np.int32)
        x, w1, w2, dy = util.f64(X), util.f64(W1)[None], util.f64(W2)[None], util.f64(dY)
        ref = og.expert_layer_chain(x, w1, w2, dy, one)
        util.assert_close(b.H[r0:r1], ref["H"], f"expert {e} H")
        util.assert_close(b.A[r0:r1], ref["A"], f"expert {e} A")
        ulp = 2.0 ** -7
        A16, H16, dH16 = (og.round_bf16(ref[k]) for k in ("A", "H", "dH"))
        ab = np.abs
        ex = {"Y": ulp * og.grouped_gemm_fwd(ab(A16), ab(w2), one),
              "dW2": ulp * og.grouped_gemm_wgrad(ab(A16), ab(dy), one)[0],
              "dX": ulp * og.grouped_gemm_dgrad(ab(dH16), ab(w1), one),
              "dW1": ulp * og.grouped_gemm_wgrad(ab(x), ab(dH16), one)[0]}
        dA = og.grouped_gemm_dgrad(dy, w2, one)
        g, u = H16[:, :w.inter], H16[:, w.inter:]
        sg = og.sigmoid(g)
        phi = sg * (1 + g * (1 - sg))
        dphi = sg * (1 - sg) * (2 + g * (1 - 2 * sg))
        ex["dH"] = ulp * np.concatenate([ab(dA * phi) * ab(u) + ab(dA * u * dphi) * ab(g),
                                         ab(dA * phi) * ab(g)], axis=1)
        for name, got in (("Y", b.Y[r0:r1]), ("dH", b.dH[r0:r1]), ("dX", b.dX[r0:r1]),
                          ("dW2", b.dW2[e]), ("dW1", b.dW1[e])):
            r = ref[name][0] if name.startswith("dW") else ref[name]
            util.assert_close(got, r, f"expert {e} {name} (chained)", extra=ex[name])
    for e in np.nonzero(lens == 0)[0]:
        assert torch.count_nonzero(b.dW1[e]).item() == 0 and torch.count_nonzero(b.dW2[e]).item() == 0
