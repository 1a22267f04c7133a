"""GPU wgrad accumulation into an fp32 main_grad (dW_f32[g] += dY_g^T X_g) vs the oracle."""
import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _f32(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("lens,N,K", [([0, 1, 129, 300, 37], 320, 200), ([100, 0, 57], 256, 256),
                                      ([600, 0, 431], 320, 256),
                                      ([257], 264, 72), ([64, 65, 0, 3], 128, 96)])
def test_wgrad_accumulate(lens, N, K):
    lens = np.asarray(lens, dtype=np.int32)
    G, M = len(lens), int(lens.sum())
    X, dY = util.gen(wl.KEY_X, M, K, 1.0, 41), util.gen(wl.KEY_DY, M, N, 1.0, 41)
    dW0 = wl.gen_f32(wl.KEY_W2, torch.arange(G * N), K, 3.0, 41).view(G, N, K).contiguous()
    gl = torch.from_numpy(lens).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    acc = dW0.to(DEV)
    pgg.grouped_gemm_wgrad_accumulate(X.to(DEV), dY.to(DEV), gl, acc, err=err)
    assert pgg.read_error(err) == 0
    x, dy, w0 = util.f64(X), util.f64(dY), dW0.double().numpy()
    ref = og.grouped_gemm_wgrad_accumulate(w0, x, dy, lens)
    util.assert_close(acc, ref, "wgrad accumulate")
    for g in np.nonzero(lens == 0)[0]:
        assert torch.equal(acc[g].cpu(), dW0[g]), "an empty group must leave main_grad unchanged"
    # a second call adds the same gradient again (micro-batch accumulation), deterministically
    acc2 = dW0.to(DEV)
    for _ in range(2):
        pgg.grouped_gemm_wgrad_accumulate(X.to(DEV), dY.to(DEV), gl, acc2)
    pgg.grouped_gemm_wgrad_accumulate(X.to(DEV), dY.to(DEV), gl, acc)
    assert torch.equal(acc, acc2)
    util.assert_close(acc2, ref + og.grouped_gemm_wgrad(x, dy, lens), "wgrad accumulate x2")


def test_wgrad_accumulate_full_size_sample():
    # FC1 wgrad of the DeepSeek-shaped layer accumulated into an fp32 [256, 4096, 4096] buffer
    from precision_grouped_gemm_gb300.layer import build_layer_inputs, expert_inputs_cpu
    w = wl.DSV4_BF16
    lens, row_token, b = build_layer_inputs(w, torch.device(DEV), allocate=False)
    G, Hd, I = len(lens), w.hidden, w.inter
    dHs = wl.gen_matrix(wl.KEY_DH, int(lens.sum()), 2 * I, 0.25, w.seed, device=DEV)
    acc = torch.full((G, 2 * I, Hd), 0.5, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pgg.grouped_gemm_wgrad_accumulate(b.X, dHs, b.group_lens, acc, err=err)
    assert pgg.read_error(err) == 0
    for e in (0, 131, 255):
        X, _, _, _, (r0, r1) = expert_inputs_cpu(w, lens, row_token, e)
        dh = util.f64(wl.gen_matrix(wl.KEY_DH, r1 - r0, 2 * I, 0.25, w.seed, row0=r0))
        ref = 0.5 + og.grouped_gemm_wgrad(util.f64(X), dh, np.array([r1 - r0], dtype=np.int32))[0]
        util.assert_close(acc[e], ref, f"expert {e} fc1 wgrad accumulate")
