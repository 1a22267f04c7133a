"""fp64 oracle: grouped GEMM forward / dgrad / wgrad and the SwiGLU epilogues.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The problem statement this follows:

* "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with Primus",
  section "Expert parallelism: DeepEP and the grouped GEMM": every local expert
  multiplies its own (different) number of tokens by its own weights, and the
  grouped GEMM runs all of them as one kernel over a ragged batch.
* Same page, section "MegaMoE: fusing communication into the grouped GEMM":
  the expert weights are w1 [g, 2I, H] ("gate + up") and w2 [g, H, I]; the
  expert path is GEMM1 -> SwiGLU -> GEMM2, and the backward emits dW2 and dW1.
* "[Megatron-LM] feat: add grouped gemm fp4 support ... Pull Request #891",
  review comments: the per-expert token counts (m_splits) come from routing and
  are bounded by the token count.

Shapes (G groups, M = sum(group_lens)); rows of group g are
[off_g, off_g + len_g), off_0 = 0, off_{g+1} = off_g + len_g:

    fwd    Y[M, N]   : Y_g  = X_g  . W_g^T          X [M, K], W [G, N, K]
    dgrad  dX[M, K]  : dX_g = dY_g . W_g            dY [M, N]
    wgrad  dW[G,N,K] : dW_g = dY_g^T . X_g          (len_g = 0  =>  dW_g = 0)

Readings where the pages are silent (each also listed in the design notes):

* SwiGLU layout: rows 0..I-1 of w1 are the gate, rows I..2I-1 the up
  projection ("gate + up", gate first); A = silu(gate) * up, unclamped.
* SwiGLU backward: the plain derivative of A = g * sigmoid(g) * u.

All arithmetic is fp64.  A library matmul (numpy) is one step per group; there
is no blocking or reordering beyond the per-group definition.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp64 values (bf16 is the top half of fp32)."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def group_offsets(group_lens, M: int) -> np.ndarray:
    """off[0..G]: exclusive prefix sum of group_lens; checks len >= 0 and sum == M."""
    lens = np.asarray(group_lens, dtype=np.int64)
    if np.any(lens < 0):
        raise ValueError("negative group length")
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    if off[-1] != M:
        raise ValueError(f"sum(group_lens)={off[-1]} != M={M}")
    return off


def grouped_gemm_fwd(X: np.ndarray, W: np.ndarray, group_lens) -> np.ndarray:
    """Y_g = X_g . W_g^T for every group; X [M,K], W [G,N,K] (fp64) -> Y [M,N]."""
    M, K = X.shape
    G, N, K2 = W.shape
    assert K == K2 and len(group_lens) == G
    off = group_offsets(group_lens, M)
    Y = np.zeros((M, N), dtype=np.float64)
    for g in range(G):
        a, b = off[g], off[g + 1]
        if b > a:
            Y[a:b] = X[a:b] @ W[g].T
    return Y


def grouped_gemm_dgrad(dY: np.ndarray, W: np.ndarray, group_lens) -> np.ndarray:
    """dX_g = dY_g . W_g for every group; dY [M,N], W [G,N,K] -> dX [M,K]."""
    M, N = dY.shape
    G, N2, K = W.shape
    assert N == N2 and len(group_lens) == G
    off = group_offsets(group_lens, M)
    dX = np.zeros((M, K), dtype=np.float64)
    for g in range(G):
        a, b = off[g], off[g + 1]
        if b > a:
            dX[a:b] = dY[a:b] @ W[g]
    return dX


def grouped_gemm_wgrad(X: np.ndarray, dY: np.ndarray, group_lens) -> np.ndarray:
    """dW_g = dY_g^T . X_g, reduced over the group's own rows; empty group -> 0."""
    M, K = X.shape
    M2, N = dY.shape
    assert M == M2
    G = len(group_lens)
    off = group_offsets(group_lens, M)
    dW = np.zeros((G, N, K), dtype=np.float64)
    for g in range(G):
        a, b = off[g], off[g + 1]
        if b > a:
            dW[g] = dY[a:b].T @ X[a:b]
    return dW


def grouped_gemm_wgrad_accumulate(dW0: np.ndarray, X: np.ndarray, dY: np.ndarray, group_lens) -> np.ndarray:
    """main_grad accumulation: dW0[g] + dY_g^T . X_g (the weight-gradient bridge of
    Pull Request #891, "Changes": the gradient is always added into weight.main_grad)."""
    return np.asarray(dW0, dtype=np.float64) + grouped_gemm_wgrad(X, dY, group_lens)


def sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def _clamp_gate_up(g: np.ndarray, u: np.ndarray, limit):
    """The swiglu_limit clamp ("Enabling DeepSeek-V4-Flash ...", model-config table names the
    knob without a formula; read here as gate <- min(gate, L), up <- clip(up, -L, L)).
    Returns the clamped values and the masks where each clamp is inactive (boundaries
    included), which is where the gradient passes."""
    if limit is None or limit <= 0:
        return g, u, np.ones_like(g, dtype=bool), np.ones_like(u, dtype=bool)
    return np.minimum(g, limit), np.clip(u, -limit, limit), g <= limit, np.abs(u) <= limit


def swiglu_fwd(H: np.ndarray, limit=None) -> np.ndarray:
    """A = silu(gate) * up with gate = H[:, :I], up = H[:, I:] (H [M, 2I]); with a limit L > 0
    the gate and up are clamped first (see _clamp_gate_up)."""
    I = H.shape[1] // 2
    g, u, _, _ = _clamp_gate_up(H[:, :I], H[:, I:], limit)
    return g * sigmoid(g) * u


def swiglu_bwd(dA: np.ndarray, H: np.ndarray, limit=None) -> np.ndarray:
    """dH = [dA*u*sigma(g)*(1 + g*(1-sigma(g))) | dA*g*sigma(g)] (derivative of swiglu_fwd),
    on the clamped g, u and zero where a clamp is active."""
    I = H.shape[1] // 2
    g, u, mg, mu = _clamp_gate_up(H[:, :I], H[:, I:], limit)
    s = sigmoid(g)
    dgate = np.where(mg, dA * u * s * (1.0 + g * (1.0 - s)), 0.0)
    dup = np.where(mu, dA * g * s, 0.0)
    return np.concatenate([dgate, dup], axis=1)


def grouped_fc1_swiglu(X: np.ndarray, W1: np.ndarray, group_lens, limit=None):
    """FC1 with SwiGLU folded in: H = grouped fwd(X, W1) [M, 2I]; A = swiglu(H) [M, I]."""
    H = grouped_gemm_fwd(X, W1, group_lens)
    return swiglu_fwd(H, limit), H


def grouped_fc2_dgrad_swiglu_bwd(dY: np.ndarray, W2: np.ndarray, H: np.ndarray, group_lens, limit=None):
    """FC2 dgrad followed by the SwiGLU backward: dA = dgrad(dY, W2); dH = swiglu_bwd(dA, H)."""
    dA = grouped_gemm_dgrad(dY, W2, group_lens)
    return swiglu_bwd(dA, H, limit)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even (8 significant bits,
    normal exponent floor -126, subnormal quantum 2^-133); returns fp64."""
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                       # |x| = f * 2^e, f in [0.5, 1)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)  # quantum of x's bf16 binade
    return np.rint(x / q) * q                # rint: round half to even


def expert_layer_chain(X, W1, W2, dY, group_lens):
    """The expert layer fwd + bwd as the library's six calls compute it.

    A, H = FC1+SwiGLU(X); Y = FC2(A); dH = SwiGLU'(dY . W2_g, H); dW2 = dY_g^T A_g;
    dX = dH . W1_g; dW1 = dH_g^T X_g.  The tensors that one call hands to the next
    (A, H, dH) are stored in bf16 by the library, so the downstream calls here
    consume their bf16 roundings; every returned array is the unrounded fp64
    result of its own call."""
    Hf = grouped_gemm_fwd(X, W1, group_lens)
    Af = swiglu_fwd(Hf)
    A, H = round_bf16(Af), round_bf16(Hf)
    Y = grouped_gemm_fwd(A, W2, group_lens)
    dHf = grouped_fc2_dgrad_swiglu_bwd(dY, W2, H, group_lens)
    dH = round_bf16(dHf)
    return {"A": Af, "H": Hf, "Y": Y, "dH": dHf,
            "dW2": grouped_gemm_wgrad(A, dY, group_lens),
            "dX": grouped_gemm_dgrad(dH, W1, group_lens),
            "dW1": grouped_gemm_wgrad(X, dH, group_lens)}


def rms(x: np.ndarray) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def within_tol(got: np.ndarray, ref: np.ndarray, rel: float = 1e-2, abs_rms: float = 1e-2):
    """Per element |got - ref| <= rel*|ref| + abs_rms*rms(ref); returns (ok, worst ratio)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = rel * np.abs(ref) + abs_rms * rms(ref)
    err = np.abs(got - ref)
    if err.size == 0:
        return True, 0.0
    bad = ~(err <= bound)  # NaN counts as bad
    ratio = float(np.max(np.where(bound > 0, err / np.maximum(bound, 1e-300), np.where(err > 0, np.inf, 0.0))))
    return (not bool(bad.any())), ratio
