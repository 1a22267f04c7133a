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

    def clone_empty(self):
        """An independent buffer set of the same shapes (inputs uninitialised)."""
        e = lambda t: torch.empty_like(t)
        return ExpertLayerBuffers(e(self.X), e(self.W1), e(self.W2), e(self.dY),
                                  self.group_lens.clone()).allocate()

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


def build_layer_inputs(w, device, cap: int = 0, allocate: bool = True):
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
    b = ExpertLayerBuffers(X, W1, W2, dY, gl)
    return lens, row_token, (b.allocate() if allocate else b)


def expert_inputs_cpu(w, lens, row_token, e: int):
    """The same generator values for expert e alone, on the CPU (bf16 tensors)."""
    off = np.concatenate([[0], np.cumsum(lens)])
    a, b = int(off[e]), int(off[e + 1])
    X = wl.gen_bf16(wl.KEY_X, torch.from_numpy(row_token[a:b]), w.hidden, 1.0, w.seed)
    W1 = wl.gen_matrix(wl.KEY_W1, 2 * w.inter, w.hidden, w.w_std, w.seed, row0=e * 2 * w.inter)
    W2 = wl.gen_matrix(wl.KEY_W2, w.hidden, w.inter, w.w_std, w.seed, row0=e * w.hidden)
    dY = wl.gen_matrix(wl.KEY_DY, b - a, w.hidden, 1.0, w.seed, row0=a)
    return X, W1, W2, dY, (a, b)


# ----------------------------------------------------------------------------
# MX (MXFP8 / MXFP4) expert layer
# ----------------------------------------------------------------------------

MX_STEP_NAMES = ("q_x_row", "fc1_fwd_swiglu", "fc2_fwd", "q_dy_row", "fc2_dgrad_swiglu_bwd", "q_dy_col",
                 "q_a_col", "fc2_wgrad", "fc1_dgrad", "q_dh_col", "q_x_col", "fc1_wgrad")


@dataclasses.dataclass
class MxLayerBuffers:
    """Block-scaled expert layer: bf16 activations, MX weights quantized once (the caller's
    weight cache), and the MX activation / gradient operands each step re-quantizes."""
    fmt: str
    X: torch.Tensor
    dY: torch.Tensor
    group_lens: torch.Tensor
    W1q: tuple = None      # row-wise  [G*2I, H], blocked scales (fc1 fwd, blocks along H)
    W1t: tuple = None      # column-wise [H, G*2I] (fc1 dgrad, blocks along 2I)
    W2q: tuple = None      # row-wise  [G*H, I], blocked scales (fc2 fwd, blocks along I)
    W2t: tuple = None      # column-wise [I, G*H]  (fc2 dgrad, blocks along H)
    M_pad: int = 0
    bufs: dict = None

    def clone_empty(self):
        """An independent buffer set of the same shapes (inputs and weight caches uninitialised)."""
        e = lambda t: torch.empty_like(t)
        c = MxLayerBuffers(self.fmt, e(self.X), e(self.dY), self.group_lens.clone())
        c.W1q, c.W1t = tuple(map(e, self.W1q)), tuple(map(e, self.W1t))
        c.W2q, c.W2t = tuple(map(e, self.W2q)), tuple(map(e, self.W2t))
        c.M_pad = self.M_pad
        c.bufs = {k: (tuple(map(e, v)) if isinstance(v, tuple) else e(v)) for k, v in self.bufs.items()}
        c.bufs["err"].zero_()
        return c

    @staticmethod
    def build(fmt, X, W1, W2, dY, group_lens, host_lens=None):
        """Quantize the weights (outside any timed region) and allocate every step buffer.

        host_lens (optional, numpy): the group lengths as the host knows them after
        routing; the column-wise operands then take exactly sum(round_up(len, 128))
        padded columns instead of the worst case for M rows in G groups."""
        G, I2, Hd = W1.shape
        I = I2 // 2
        M = X.shape[0]
        dev = X.device
        b = MxLayerBuffers(fmt, X, dY, group_lens)
        W1f, W2f = W1.reshape(G * I2, Hd), W2.reshape(G * Hd, I)
        b.W1q = B.mx_quantize_rowwise_blocked(W1f, fmt)
        b.W1t = B.mx_quantize_colwise(W1f, torch.full((G,), I2, dtype=torch.int32, device=dev), fmt, G * I2)
        b.W2q = B.mx_quantize_rowwise_blocked(W2f, fmt)
        b.W2t = B.mx_quantize_colwise(W2f, torch.full((G,), Hd, dtype=torch.int32, device=dev), fmt, G * Hd)
        if host_lens is not None:
            b.M_pad = max(B.PAD, int(sum(-(-int(n) // B.PAD) * B.PAD for n in host_lens)))
        else:
            b.M_pad = B.mx_pad_rows(M, G)
        cb = (lambda c: c) if fmt == "e4m3" else (lambda c: c // 2)
        u8, bf = torch.uint8, torch.bfloat16
        Mp = b.M_pad
        e = lambda *s: torch.empty(s, dtype=u8, device=dev)
        r128 = lambda n: -(-n // 128) * 128  # blocked column-wise scales: rows padded to 128
        b.bufs = {
            "Xq": (e(M, cb(Hd)), e(M, Hd // 32)), "A": torch.empty((M, I), dtype=bf, device=dev),
            "H": torch.empty((M, I2), dtype=bf, device=dev), "Aq": (e(M, cb(I)), e(M, I // 32)),
            "Y": torch.empty((M, Hd), dtype=bf, device=dev), "dYq": (e(M, cb(Hd)), e(M, Hd // 32)),
            "dH": torch.empty((M, I2), dtype=bf, device=dev), "dYc": (e(Hd, cb(Mp)), e(r128(Hd), Mp // 32)),
            "Ac": (e(I, cb(Mp)), e(r128(I), Mp // 32)), "dW2": torch.empty((G, Hd, I), dtype=bf, device=dev),
            "dHq": (e(M, cb(I2)), e(M, I2 // 32)), "dX": torch.empty((M, Hd), dtype=bf, device=dev),
            "dHc": (e(I2, cb(Mp)), e(r128(I2), Mp // 32)), "Xc": (e(Hd, cb(Mp)), e(r128(Hd), Mp // 32)),
            "dW1": torch.empty((G, I2, Hd), dtype=bf, device=dev),
            "err": torch.zeros(1, dtype=torch.int32, device=dev),
        }
        return b


def mx_layer_step(b: MxLayerBuffers, between=None):
    """One MX expert-layer fwd + bwd: 6 activation quantizations and 6 block-scaled GEMMs; the
    FC1 and FC2-dgrad epilogues emit A and dH already MX-quantized for the next GEMM."""
    f, gl, u = b.fmt, b.group_lens, b.bufs
    err, Mp = u["err"], b.M_pad
    M, Hd = b.X.shape
    I = u["A"].shape[1]
    G = gl.numel()
    calls = (
        lambda: B.mx_quantize_rowwise(b.X, f, *u["Xq"]),
        lambda: B.mx_grouped_gemm(B.MODE_FWD, f, *u["Xq"], *b.W1q, gl, M, 2 * I, Hd, out=u["A"], out2=u["H"],
                                  epilogue=B.EPI_SWIGLU, err=err, out_q=u["Aq"]),
        lambda: B.mx_grouped_gemm(B.MODE_FWD, f, *u["Aq"], *b.W2q, gl, M, Hd, I, out=u["Y"], err=err),
        lambda: B.mx_quantize_rowwise(b.dY, f, *u["dYq"]),
        lambda: B.mx_grouped_gemm(B.MODE_DGRAD, f, *u["dYq"], *b.W2t, gl, M, Hd, I, out=u["dH"], H=u["H"],
                                  epilogue=B.EPI_SWIGLU, err=err, out_q=u["dHq"]),
        lambda: B.mx_quantize_colwise(b.dY, gl, f, Mp, *u["dYc"], err=err),
        lambda: B.mx_quantize_colwise(u["A"], gl, f, Mp, *u["Ac"], err=err),
        lambda: B.mx_grouped_gemm(B.MODE_WGRAD, f, *u["dYc"], *u["Ac"], gl, M, Hd, I, out=u["dW2"], M_pad=Mp,
                                  err=err),
        lambda: B.mx_grouped_gemm(B.MODE_DGRAD, f, *u["dHq"], *b.W1t, gl, M, 2 * I, Hd, out=u["dX"], err=err),
        lambda: B.mx_quantize_colwise(u["dH"], gl, f, Mp, *u["dHc"], err=err),
        lambda: B.mx_quantize_colwise(b.X, gl, f, Mp, *u["Xc"], err=err),
        lambda: B.mx_grouped_gemm(B.MODE_WGRAD, f, *u["dHc"], *u["Xc"], gl, M, 2 * I, Hd, out=u["dW1"],
                                  M_pad=Mp, err=err),
    )
    assert len(calls) == len(MX_STEP_NAMES) and G > 0
    for i, c in enumerate(calls):
        if between:
            between(i)
        c()
    if between:
        between(len(calls))


def mx_layer_work(fmt: str, M: int, G: int, Hd: int, I: int, M_pad: int) -> dict:
    """Algorithmic flops and bytes of each MX-layer call (codes at 1 or 0.5 B/element,
    scales at 1/32 B/element, bf16 activations and outputs at 2 B/element).  The column-wise
    operands count their M real rows, not the M_pad columns of their padded layout: padding
    the kernels read or write is not algorithmic work (M_pad is kept in the signature for
    callers that size buffers with it)."""
    c = 1.0 if fmt == "e4m3" else 0.5
    q = c + 1.0 / 32                          # bytes per quantized element (codes + scale)
    f1, f2 = 2.0 * M * 2 * I * Hd, 2.0 * M * Hd * I
    W1, W2 = G * 2 * I * Hd, G * Hd * I       # elements
    lens = 4 * G
    return {
        "q_x_row": (0.0, M * Hd * (2 + q)),
        "fc1_fwd_swiglu": (f1, M * Hd * q + W1 * q + M * I * (2 + q) + M * 2 * I * 2 + lens),
        "fc2_fwd": (f2, M * I * q + W2 * q + M * Hd * 2 + lens),
        "q_dy_row": (0.0, M * Hd * (2 + q)),
        "fc2_dgrad_swiglu_bwd": (f2, M * Hd * q + W2 * q + M * 2 * I * 2 + M * 2 * I * (2 + q) + lens),
        "q_dy_col": (0.0, M * Hd * 2 + Hd * M * q + lens),
        "q_a_col": (0.0, M * I * 2 + I * M * q + lens),
        "fc2_wgrad": (f2, (Hd + I) * M * q + W2 * 2 + lens),
        "fc1_dgrad": (f1, M * 2 * I * q + W1 * q + M * Hd * 2 + lens),
        "q_dh_col": (0.0, M * 2 * I * 2 + 2 * I * M * q + lens),
        "q_x_col": (0.0, M * Hd * 2 + Hd * M * q + lens),
        "fc1_wgrad": (f1, (2 * I + Hd) * M * q + W1 * 2 + lens),
    }


# ----------------------------------------------------------------------------
# FP8 tensor-wise (current scaling) expert layer
# ----------------------------------------------------------------------------

FP8_STEP_NAMES = ("s_x", "q_x_row", "fc1_fwd_swiglu", "s_a", "q_a_row", "fc2_fwd", "s_dy", "q_dy_row",
                  "fc2_dgrad_swiglu_bwd", "q_dy_col", "q_a_col", "fc2_wgrad", "s_dh", "q_dh_row", "fc1_dgrad",
                  "q_dh_col", "q_x_col", "fc1_wgrad")


@dataclasses.dataclass
class Fp8LayerBuffers:
    """FP8 tensor-wise expert layer: bf16 activations; the weights quantized once with their
    own tensor scales (the caller's weight cache); every activation and gradient operand
    re-scaled (amax of the whole tensor) and re-quantized each step, as current scaling
    requires."""
    X: torch.Tensor
    dY: torch.Tensor
    group_lens: torch.Tensor
    W1q: torch.Tensor = None   # row-wise codes [G*2I, H] (fc1 fwd)
    W1t: torch.Tensor = None   # column-wise codes [H, G*2I] (fc1 dgrad)
    s_w1: torch.Tensor = None  # {s, amax} of W1
    W2q: torch.Tensor = None   # row-wise codes [G*H, I] (fc2 fwd)
    W2t: torch.Tensor = None   # column-wise codes [I, G*H] (fc2 dgrad)
    s_w2: torch.Tensor = None
    M_pad: int = 0
    bufs: dict = None

    def clone_empty(self):
        """An independent buffer set of the same shapes (inputs and weight caches uninitialised)."""
        e = lambda t: torch.empty_like(t)
        c = Fp8LayerBuffers(e(self.X), e(self.dY), self.group_lens.clone())
        c.W1q, c.W1t, c.s_w1 = e(self.W1q), e(self.W1t), e(self.s_w1)
        c.W2q, c.W2t, c.s_w2 = e(self.W2q), e(self.W2t), e(self.s_w2)
        c.M_pad = self.M_pad
        c.bufs = {k: e(v) for k, v in self.bufs.items()}
        c.bufs["err"].zero_()
        return c

    @staticmethod
    def build(X, W1, W2, dY, group_lens, host_lens=None):
        """Quantize the weights (outside any timed region) and allocate every step buffer;
        host_lens as MxLayerBuffers.build."""
        G, I2, Hd = W1.shape
        I = I2 // 2
        M = X.shape[0]
        dev = X.device
        b = Fp8LayerBuffers(X, dY, group_lens)
        W1f, W2f = W1.reshape(G * I2, Hd), W2.reshape(G * Hd, I)
        b.s_w1 = B.fp8_tensor_scale(W1f)
        b.W1q = B.fp8_quantize_rowwise(W1f, b.s_w1)
        b.W1t = B.fp8_quantize_colwise(W1f, torch.full((G,), I2, dtype=torch.int32, device=dev), b.s_w1, G * I2)
        b.s_w2 = B.fp8_tensor_scale(W2f)
        b.W2q = B.fp8_quantize_rowwise(W2f, b.s_w2)
        b.W2t = B.fp8_quantize_colwise(W2f, torch.full((G,), Hd, dtype=torch.int32, device=dev), b.s_w2, G * Hd)
        if host_lens is not None:
            b.M_pad = max(B.PAD, int(sum(-(-int(n) // B.PAD) * B.PAD for n in host_lens)))
        else:
            b.M_pad = B.mx_pad_rows(M, G)
        Mp = b.M_pad
        u8, bf, f32 = torch.uint8, torch.bfloat16, torch.float32
        e = lambda *s: torch.empty(s, dtype=u8, device=dev)
        t = lambda *s: torch.empty(s, dtype=bf, device=dev)
        sc = lambda: torch.empty(2, dtype=f32, device=dev)
        b.bufs = {
            "sx": sc(), "Xq": e(M, Hd), "A": t(M, I), "H": t(M, I2), "sa": sc(), "Aq": e(M, I), "Y": t(M, Hd),
            "sdy": sc(), "dYq": e(M, Hd), "dH": t(M, I2), "dYc": e(Hd, Mp), "Ac": e(I, Mp), "dW2": t(G, Hd, I),
            "sdh": sc(), "dHq": e(M, I2), "dX": t(M, Hd), "dHc": e(I2, Mp), "Xc": e(Hd, Mp), "dW1": t(G, I2, Hd),
            "err": torch.zeros(1, dtype=torch.int32, device=dev),
        }
        return b


def fp8_layer_step(b: Fp8LayerBuffers, between=None):
    """One FP8 tensor-wise expert-layer fwd + bwd: 4 tensor scales, 8 quantizations and 6 grouped
    GEMMs (FC1 and FC2-dgrad with the SwiGLU and its backward in the epilogue)."""
    u, gl = b.bufs, b.group_lens
    err, Mp = u["err"], b.M_pad
    M, Hd = b.X.shape
    I = u["A"].shape[1]
    G = gl.numel()
    g = B.fp8_grouped_gemm
    calls = (
        lambda: B.fp8_tensor_scale(b.X, u["sx"]),
        lambda: B.fp8_quantize_rowwise(b.X, u["sx"], u["Xq"]),
        lambda: g(B.MODE_FWD, u["Xq"], u["sx"], b.W1q, b.s_w1, gl, M, 2 * I, Hd, out=u["A"], out2=u["H"],
                  epilogue=B.EPI_SWIGLU, err=err),
        lambda: B.fp8_tensor_scale(u["A"], u["sa"]),
        lambda: B.fp8_quantize_rowwise(u["A"], u["sa"], u["Aq"]),
        lambda: g(B.MODE_FWD, u["Aq"], u["sa"], b.W2q, b.s_w2, gl, M, Hd, I, out=u["Y"], err=err),
        lambda: B.fp8_tensor_scale(b.dY, u["sdy"]),
        lambda: B.fp8_quantize_rowwise(b.dY, u["sdy"], u["dYq"]),
        lambda: g(B.MODE_DGRAD, u["dYq"], u["sdy"], b.W2t, b.s_w2, gl, M, Hd, I, out=u["dH"], H=u["H"],
                  epilogue=B.EPI_SWIGLU, err=err),
        lambda: B.fp8_quantize_colwise(b.dY, gl, u["sdy"], Mp, u["dYc"], err=err),
        lambda: B.fp8_quantize_colwise(u["A"], gl, u["sa"], Mp, u["Ac"], err=err),
        lambda: g(B.MODE_WGRAD, u["dYc"], u["sdy"], u["Ac"], u["sa"], gl, M, Hd, I, out=u["dW2"], M_pad=Mp,
                  err=err),
        lambda: B.fp8_tensor_scale(u["dH"], u["sdh"]),
        lambda: B.fp8_quantize_rowwise(u["dH"], u["sdh"], u["dHq"]),
        lambda: g(B.MODE_DGRAD, u["dHq"], u["sdh"], b.W1t, b.s_w1, gl, M, 2 * I, Hd, out=u["dX"], err=err),
        lambda: B.fp8_quantize_colwise(u["dH"], gl, u["sdh"], Mp, u["dHc"], err=err),
        lambda: B.fp8_quantize_colwise(b.X, gl, u["sx"], Mp, u["Xc"], err=err),
        lambda: g(B.MODE_WGRAD, u["dHc"], u["sdh"], u["Xc"], u["sx"], gl, M, 2 * I, Hd, out=u["dW1"], M_pad=Mp,
                  err=err),
    )
    assert len(calls) == len(FP8_STEP_NAMES) and G > 0
    for i, c in enumerate(calls):
        if between:
            between(i)
        c()
    if between:
        between(len(calls))


def fp8_layer_work(M: int, G: int, Hd: int, I: int, M_pad: int) -> dict:
    """Algorithmic flops and bytes of each FP8-layer call: codes at 1 B per element, bf16
    activations and outputs at 2; a tensor scale reads its tensor once.  Column-wise operands
    count their M real rows (padding is not algorithmic work)."""
    f1, f2 = 2.0 * M * 2 * I * Hd, 2.0 * M * Hd * I
    W1, W2 = G * 2 * I * Hd, G * Hd * I       # elements
    lens = 4 * G
    return {
        "s_x": (0.0, M * Hd * 2),
        "q_x_row": (0.0, M * Hd * 3),
        "fc1_fwd_swiglu": (f1, M * Hd + W1 + M * I * 2 + M * 2 * I * 2 + lens),
        "s_a": (0.0, M * I * 2),
        "q_a_row": (0.0, M * I * 3),
        "fc2_fwd": (f2, M * I + W2 + M * Hd * 2 + lens),
        "s_dy": (0.0, M * Hd * 2),
        "q_dy_row": (0.0, M * Hd * 3),
        "fc2_dgrad_swiglu_bwd": (f2, M * Hd + W2 + M * 2 * I * 2 + M * 2 * I * 2 + lens),
        "q_dy_col": (0.0, M * Hd * 2 + Hd * M + lens),
        "q_a_col": (0.0, M * I * 2 + I * M + lens),
        "fc2_wgrad": (f2, (Hd + I) * M + W2 * 2 + lens),
        "s_dh": (0.0, M * 2 * I * 2),
        "q_dh_row": (0.0, M * 2 * I * 3),
        "fc1_dgrad": (f1, M * 2 * I + W1 + M * Hd * 2 + lens),
        "q_dh_col": (0.0, M * 2 * I * 2 + 2 * I * M + lens),
        "q_x_col": (0.0, M * Hd * 2 + Hd * M + lens),
        "fc1_wgrad": (f1, (2 * I + Hd) * M + W1 * 2 + lens),
    }
