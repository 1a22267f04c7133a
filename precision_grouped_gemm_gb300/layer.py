"""One MoE expert layer, forward + backward, as six grouped-GEMM calls.

The expert path GEMM1 -> SwiGLU -> GEMM2 with w1 [g, 2I, H] ("gate + up") and
w2 [g, H, I], and a backward that emits dW2 then dW1 ("Enabling
DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with Primus", section
"MegaMoE: fusing communication into the grouped GEMM"):

    1  FC1 fwd + SwiGLU     A, H = swiglu(X . W1_g^T)          [M, I], [M, 2I]
    2  FC2 fwd              Y    = A . W2_g^T                   [M, H]
    3  FC2 dgrad + SwiGLU'  dH   = swiglu_bwd(dY . W2_g, H)     [M, 2I]
    4  FC2 wgrad            dW2  = dY_g^T . A_g                 [G, H, I]
    5  FC1 dgrad            dX   = dH . W1_g                    [M, H]
    6  FC1 wgrad            dW1  = dH_g^T . X_g                 [G, 2I, H]

Every call is one kernel launch of libpgg.so on the current stream.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import _binding as B
from . import workloads as wl

STEP_NAMES = ("fc1_fwd_swiglu", "fc2_fwd", "fc2_dgrad_swiglu_bwd", "fc2_wgrad", "fc1_dgrad",
              "fc1_wgrad")


@dataclasses.dataclass
class ExpertLayerBuffers:
    X: torch.Tensor        # [M, H] bf16, rows sorted by expert
    W1: torch.Tensor       # [G, 2I, H] bf16
    W2: torch.Tensor       # [G, H, I] bf16
    dY: torch.Tensor       # [M, H] bf16, gradient of the layer output
    group_lens: torch.Tensor  # [G] int32
    A: torch.Tensor = None
    H: torch.Tensor = None
    Y: torch.Tensor = None
    dH: torch.Tensor = None
    dX: torch.Tensor = None
    dW1: torch.Tensor = None
    dW2: torch.Tensor = None
    err: torch.Tensor = None

    def allocate(self):
        M, Hd = self.X.shape
        G, I2, _ = self.W1.shape
        I = I2 // 2
        dev, bf = self.X.device, torch.bfloat16
        self.A = torch.empty((M, I), dtype=bf, device=dev)
        self.H = torch.empty((M, I2), dtype=bf, device=dev)
        self.Y = torch.empty((M, Hd), dtype=bf, device=dev)
        self.dH = torch.empty((M, I2), dtype=bf, device=dev)
        self.dX = torch.empty((M, Hd), dtype=bf, device=dev)
        self.dW1 = torch.empty((G, I2, Hd), dtype=bf, device=dev)
        self.dW2 = torch.empty((G, Hd, I), dtype=bf, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        return self


def expert_layer_step(b: ExpertLayerBuffers, between=None):
    """Run the six calls; `between(i)` (optional) is called before call i and after the last."""
    gl, err = b.group_lens, b.err
    calls = (
        lambda: B.grouped_fc1_swiglu(b.X, b.W1, gl, A=b.A, H=b.H, err=err),
        lambda: B.grouped_gemm_fwd(b.A, b.W2, gl, Y=b.Y, err=err),
        lambda: B.grouped_fc2_dgrad_swiglu_bwd(b.dY, b.W2, b.H, gl, dH=b.dH, err=err),
        lambda: B.grouped_gemm_wgrad(b.A, b.dY, gl, dW=b.dW2, err=err),
        lambda: B.grouped_gemm_dgrad(b.dH, b.W1, gl, dX=b.dX, err=err),
        lambda: B.grouped_gemm_wgrad(b.X, b.dH, gl, dW=b.dW1, err=err),
    )
    for i, c in enumerate(calls):
        if between:
            between(i)
        c()
    if between:
        between(len(calls))


def layer_work(M: int, G: int, Hd: int, I: int) -> dict:
    """Algorithmic flops and HBM bytes of each call (each tensor moved once; bf16)."""
    e = 2
    W1b, W2b = G * 2 * I * Hd * e, G * Hd * I * e
    X, A, H, Y = M * Hd * e, M * I * e, M * 2 * I * e, M * Hd * e
    lens = 4 * G
    f1, f2 = 2.0 * M * 2 * I * Hd, 2.0 * M * Hd * I
    return {
        "fc1_fwd_swiglu": (f1, X + W1b + A + H + lens),
        "fc2_fwd": (f2, A + W2b + Y + lens),
        "fc2_dgrad_swiglu_bwd": (f2, Y + W2b + H + H + lens),
        "fc2_wgrad": (f2, A + Y + W2b + lens),
        "fc1_dgrad": (f1, H + W1b + X + lens),
        "fc1_wgrad": (f1, X + H + W1b + lens),
    }


def build_layer_inputs(w, device, cap: int = 0):
    """Seeded inputs of workload `w` on `device` (only the first `cap` experts when cap > 0).

    X rows are the generated token activations gathered in expert-sorted row order;
    W1, W2 and dY come straight from the counter-based generator."""
    lens, row_token = w.group_lens()
    if cap:
        lens = lens[:cap].copy()
        row_token = row_token[:int(lens.sum())]
    M, G, Hd, I = int(lens.sum()), len(lens), w.hidden, w.inter
    rt = torch.from_numpy(row_token).to(device)
    xtok = wl.gen_matrix(wl.KEY_X, w.tokens, Hd, 1.0, w.seed, device=device)
    X = xtok[rt].contiguous()
    del xtok
    W1 = wl.gen_matrix(wl.KEY_W1, G * 2 * I, Hd, w.w_std, w.seed, device=device).view(G, 2 * I, Hd)
    W2 = wl.gen_matrix(wl.KEY_W2, G * Hd, I, w.w_std, w.seed, device=device).view(G, Hd, I)
    dY = wl.gen_matrix(wl.KEY_DY, M, Hd, 1.0, w.seed, device=device)
    gl = torch.from_numpy(np.ascontiguousarray(lens)).to(device)
    return lens, row_token, ExpertLayerBuffers(X, W1, W2, dY, gl).allocate()


def expert_inputs_cpu(w, lens, row_token, e: int):
    """The same generator values for expert e alone, on the CPU (bf16 tensors)."""
    off = np.concatenate([[0], np.cumsum(lens)])
    a, b = int(off[e]), int(off[e + 1])
    X = wl.gen_bf16(wl.KEY_X, torch.from_numpy(row_token[a:b]), w.hidden, 1.0, w.seed)
    W1 = wl.gen_matrix(wl.KEY_W1, 2 * w.inter, w.hidden, w.w_std, w.seed, row0=e * 2 * w.inter)
    W2 = wl.gen_matrix(wl.KEY_W2, w.hidden, w.inter, w.w_std, w.seed, row0=e * w.hidden)
    dY = wl.gen_matrix(wl.KEY_DY, b - a, w.hidden, 1.0, w.seed, row0=a)
    return X, W1, W2, dY, (a, b)
