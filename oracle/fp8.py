"""fp64 oracle: FP8 (e4m3) tensor-wise current-scaling grouped GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"[Megatron-LM] feat: add grouped gemm fp4 support ... Pull Request #891",
"Changes" and review: the FP8 grouped GEMM (`grouped_gemm_fp8`) runs under
current scaling, under which a cached transposed weight must not be reused; the
"Primus-Turbo" README lists the FP8 grouped GEMM.  The pages give no formula;
this oracle takes the usual per-tensor current scaling as the plainest reading:

* amax = max |x| over the tensor's finite values;
* scale s = 448 / amax in fp32 (s = 1 when amax is 0), 448 being e4m3's
  largest finite value, so the tensor's largest element maps to +-448; a
  quotient that overflows fp32 (amax below 448 / 2^128, a subnormal amax) is
  clamped to the largest finite fp32, so that s stays finite and 0 * s = 0;
* code = e4m3 round-to-nearest-even of x * s, saturating at +-448, sign of zero
  kept; NaN gives the NaN code 0x7F (with its sign), +-Inf saturates.  x * s is
  formed in fp32: the product decides an integer code, so it is taken in the
  precision a kernel uses;
* dequantized value = decode(code) / s;
* the grouped GEMMs reduce decoded codes in fp64 and divide by s_A * s_B;
* the column-wise (wgrad) operand is the same codes transposed into the
  group-padded layout of the MX column-wise operand: group g's rows become
  columns poff_g .. poff_g + len_g - 1 of [C, M_pad], poff the prefix sum of
  round_up(len, 128), and pad columns hold code 0 (one tensor scale, so no
  per-block scales exist).
"""
from __future__ import annotations

import numpy as np

from . import grouped_gemm as og
from . import mx as omx

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def fp8_tensor_scale(x: np.ndarray) -> np.float32:
    """fp32 scale 448 / amax over the finite values of x (1 when amax is 0)."""
    v = np.asarray(x, dtype=np.float64)
    fin = np.isfinite(v)
    amax = float(np.max(np.abs(v[fin]))) if fin.any() else 0.0
    if amax == 0.0:
        return np.float32(1.0)
    with np.errstate(over="ignore"):
        s = np.float32(E4M3_MAX) / np.float32(amax)
    return s if np.isfinite(s) else np.float32(np.finfo(np.float32).max)


def fp8_quantize_tensorwise(x: np.ndarray, scale=None):
    """fp64 / bf16-valued x -> (e4m3 codes u8, fp32 scale); scale None computes it."""
    v = np.asarray(x, dtype=np.float64)
    s = fp8_tensor_scale(v) if scale is None else np.float32(scale)
    with np.errstate(invalid="ignore", over="ignore"):
        prod = (v.astype(np.float32) * s).astype(np.float64)  # fp32 product, RNE
    codes = omx.round_to_grid("e4m3", np.where(np.isnan(prod), 0.0, prod))
    nan = np.isnan(v)
    codes = np.where(nan, NAN_CODE | np.where(np.signbit(v), 0x80, 0), codes).astype(np.uint8)
    return codes, s


def fp8_dequantize(codes: np.ndarray, scale) -> np.ndarray:
    return omx.decode_e4m3(codes) / float(np.float32(scale))


def fp8_grouped_gemm_fwd(A, sA, B, sB, group_lens, G: int):
    """out_g = deq(A)_g . deq(B)_g^T; A [M, K] codes, B [G*N, K] codes."""
    b = omx.decode_e4m3(B)
    return og.grouped_gemm_fwd(omx.decode_e4m3(A), b.reshape(G, -1, b.shape[1]), group_lens) / (
        float(np.float32(sA)) * float(np.float32(sB)))


def fp8_grouped_gemm_dgrad(dY, sdY, W, sW, group_lens, G: int):
    """out_g = deq(dY)_g . deq(W)_g; dY [M, N] codes, W [G*N, K] codes."""
    w = omx.decode_e4m3(W)
    return og.grouped_gemm_dgrad(omx.decode_e4m3(dY), w.reshape(G, -1, w.shape[1]), group_lens) / (
        float(np.float32(sdY)) * float(np.float32(sW)))


def fp8_grouped_gemm_wgrad(X, sX, dY, sdY, group_lens):
    """out[g] = deq(dY)_g^T . deq(X)_g; X [M, K], dY [M, N] codes (one scale per tensor)."""
    return og.grouped_gemm_wgrad(omx.decode_e4m3(X), omx.decode_e4m3(dY), group_lens) / (
        float(np.float32(sX)) * float(np.float32(sdY)))


def fp8_quantize_colwise(x: np.ndarray, group_lens, M_pad: int, scale=None, P: int = 128):
    """fp64 / bf16-valued x [M, C] -> (codes_t [C, M_pad] u8, fp32 scale): group g's row i
    goes to column poff_g + i, pad columns are code 0; scale None computes it over x."""
    v = np.asarray(x, dtype=np.float64)
    M, C = v.shape
    codes, s = fp8_quantize_tensorwise(v, scale)
    off = og.group_offsets(group_lens, M)
    poff = omx.padded_offsets(group_lens, P)
    assert M_pad % P == 0 and poff[-1] <= M_pad
    codes_t = np.zeros((C, M_pad), dtype=np.uint8)
    for g in range(len(group_lens)):
        n = int(off[g + 1] - off[g])
        codes_t[:, poff[g]:poff[g] + n] = codes[off[g]:off[g + 1]].T
    return codes_t, s


def fp8_grouped_fc1_swiglu(X, sX, W1, sW1, group_lens, G: int, limit=None):
    """(A, H): FC1 on FP8 operands (X [M, K], W1 [G*2I, K] codes) with SwiGLU folded in;
    H = (code products) / (s_X s_W1), A = swiglu(H) (clamped when limit is given)."""
    H = fp8_grouped_gemm_fwd(X, sX, W1, sW1, group_lens, G)
    return og.swiglu_fwd(H, limit), H


def fp8_grouped_fc2_dgrad_swiglu_bwd(dY, sdY, W2, sW2, H, group_lens, G: int, limit=None):
    """dH: FC2 dgrad on FP8 operands (dY [M, N], W2 [G*N, K] codes) followed by the SwiGLU
    backward against the saved fp64 / bf16-valued H [M, 2K]."""
    dA = fp8_grouped_gemm_dgrad(dY, sdY, W2, sW2, group_lens, G)
    return og.swiglu_bwd(dA, H, limit)
