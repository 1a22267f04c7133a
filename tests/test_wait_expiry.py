"""The bounded-wait failure path, run on purpose without faulting or hanging the GPU.

pgg_test_stalled_fwd runs the forward grouped GEMM with a short wait limit and
tells each CTA's load producer to stop before a given k-block: nothing ever
arrives on that stage's barrier, so the MMA and epilogue waits behind it run
out.  The kernel must then raise its abort flag, drain what it issued, free its
tensor memory and exit, writing PGG_ERR_TIMEOUT to the error word within a few
wait limits.  The context stays usable: a normal call on the same stream right
after it must pass parity against the oracle."""
import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from oracle import mx as omx
from precision_grouped_gemm_gb300 import _binding
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"
PGG_ERR_TIMEOUT = 17
WAIT_NS = 2_000_000  # 2 ms


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("fmt", [0, "e4m3", "e2m1"], ids=["bf16", "e4m3", "e2m1"])
@pytest.mark.parametrize("stall_at", [0, 3])
def test_stalled_pipeline_times_out_and_the_next_call_passes(fmt, stall_at):
    L = _binding.lib()
    lens = np.asarray([100, 0, 157, 300], dtype=np.int32)
    # K = 1024: 16 (BF16), 8 (e4m3) and 4 (e2m1) k-blocks per tile, so every CTA's producer
    # reaches k-block 3 (each CTA gets at least one tile)
    G, M, N, K = len(lens), int(lens.sum()), 256, 1024
    gl = torch.from_numpy(lens).to(DEV)
    X, W = util.gen(wl.KEY_X, M, K, 1.0, 61), util.gen(wl.KEY_W1, G * N, K, 0.5, 61)
    Xd, Wd = X.to(DEV), W.to(DEV)
    if fmt == 0:
        A, SA, B, SB = Xd, None, Wd, None
        f = 0
    else:
        A, SA = pgg.mx_quantize_rowwise(Xd, fmt)
        B, SB = pgg.mx_quantize_rowwise_blocked(Wd, fmt)
        f = _binding._FMT[fmt]
    out = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = L.pgg_test_stalled_fwd(f, _p(A), _p(SA), _p(B), _p(SB), _p(gl), _p(out), M, N, K, G, stall_at, WAIT_NS,
                                _p(err), _stream())
    assert st == 0
    code = pgg.read_error(err)                       # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert code == PGG_ERR_TIMEOUT, f"error word {code}"
    assert elapsed < 1.0, f"the stalled launch took {elapsed:.3f} s to unwind"
    # the same stream, right after: a normal launch of the same GEMM must be correct
    err.zero_()
    if fmt == 0:
        Y = pgg.grouped_gemm_fwd(Xd, Wd.view(G, N, K), gl, err=err)
        ref = og.grouped_gemm_fwd(util.f64(X), util.f64(W).reshape(G, N, K), lens)
    else:
        Y = pgg.mx_grouped_gemm(pgg.MODE_FWD, fmt, A, SA, B, SB, gl, M, N, K, err=err)
        ref = omx.mx_grouped_gemm_fwd(fmt, *omx.mx_quantize_rowwise(util.bits(X), fmt),
                                      *omx.mx_quantize_rowwise(util.bits(W), fmt), lens, G)
    assert pgg.read_error(err) == 0
    util.assert_close(Y, ref, f"forward after a stalled launch ({fmt})")
