"""Full-size parity in the benchmark's launch configuration.

The whole expert layer (six launches) runs on the complete workload exactly as
bench.py times it; the fp64 oracle then recomputes whole experts -- chained
from the generator's X, W1, W2 and dY, never from a GPU result -- and every
output row/slice of those experts is compared element by element.
"""
import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from precision_grouped_gemm_gb300 import workloads as wl
from precision_grouped_gemm_gb300.layer import build_layer_inputs, expert_inputs_cpu, expert_layer_step
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_expert(w, lens, row_token, buf, e):
    X, W1, W2, dY, (a, b) = expert_inputs_cpu(w, lens, row_token, e)
    one = np.array([b - a], dtype=np.int32)
    x, w1, w2, dy = util.f64(X), util.f64(W1)[None], util.f64(W2)[None], util.f64(dY)
    A, H = og.grouped_fc1_swiglu(x, w1, one)
    Y = og.grouped_gemm_fwd(A, w2, one)
    dH = og.grouped_fc2_dgrad_swiglu_bwd(dy, w2, H, one)
    dW2 = og.grouped_gemm_wgrad(A, dy, one)[0]
    dX = og.grouped_gemm_dgrad(dH, w1, one)
    dW1 = og.grouped_gemm_wgrad(x, dH, one)[0]
    # the GPU's inputs for this expert are the same generator values
    assert torch.equal(buf.X[a:b].cpu().view(torch.int16), X.view(torch.int16))
    util.assert_close(buf.H[a:b], H, f"expert {e} H")
    util.assert_close(buf.A[a:b], A, f"expert {e} A")
    util.assert_close(buf.Y[a:b], Y, f"expert {e} Y")
    util.assert_close(buf.dH[a:b], dH, f"expert {e} dH")
    util.assert_close(buf.dX[a:b], dX, f"expert {e} dX")
    util.assert_close(buf.dW2[e], dW2, f"expert {e} dW2")
    util.assert_close(buf.dW1[e], dW1, f"expert {e} dW1")


@pytest.mark.parametrize("w,experts", [(wl.DSV4_BF16, (0, 97, 255)), (wl.GPTOSS_BF16, None)])
def test_layer_full_size(w, experts):
    lens, row_token, buf = build_layer_inputs(w, torch.device(DEV))
    expert_layer_step(buf)
    torch.cuda.synchronize()
    assert pgg.read_error(buf.err) == 0
    if experts is None:  # the largest and smallest non-empty experts
        nz = np.nonzero(lens)[0]
        experts = (int(nz[np.argmax(lens[nz])]), int(nz[np.argmin(lens[nz])]))
    for e in experts:
        _check_expert(w, lens, row_token, buf, e)
    for e in np.nonzero(lens == 0)[0]:
        assert torch.count_nonzero(buf.dW1[e]).item() == 0
        assert torch.count_nonzero(buf.dW2[e]).item() == 0
    del buf
    torch.cuda.empty_cache()
