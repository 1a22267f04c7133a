"""fp64 oracle: MX (microscaling) formats, quantization and the block-scaled grouped GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the formats but do not define them:

* "Primus-Turbo" README, "What's New" and "Component Details": GroupedGEMM in
  BF16, FP8, MXFP8 and MXFP4; MXFP4 GEMM and grouped GEMM stacks;
* "[Megatron-LM] feat: add grouped gemm fp4 support ... Pull Request #891",
  "Changes": MXFP4 weights are built as float4_e2m1fn_x2 buffers and sent to
  grouped_gemm_fp4; the quant config must be an MXFP4 recipe.

Reading (the public definition of "MX", OCP Microscaling Formats v1.0):

* element formats: e4m3 (bias 7, no infinities, S.1111.111 = NaN, max 448,
  subnormal step 2^-9) and e2m1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6; sign in
  bit 3); scale format E8M0: 2^(code-127), code 0xFF = NaN;
* one scale per block of 32 consecutive elements along the reduction axis;
* shared exponent E = floor(log2(amax)) - emax_elem, clamped to [-127, 127],
  with emax_elem = 8 (e4m3) or 2 (e2m1); amax = 0 gives E = -127 (code 0x00);
* element code = round-to-nearest-even(v * 2^-E) on the element grid,
  saturated to the largest finite magnitude; the sign of zero is kept;
* a block holding a NaN or an infinity gets scale 0xFF and all-zero codes;
* e2m1 packing: element 2j in the low nibble, element 2j+1 in the high nibble.

Group-aware column-wise quantization (for the wgrad operands) is a reading of
its own: blocks run down the rows of one group only, starting at the group's
first row; each group's rows are stored in a region of round_up(len_g, P)
columns of the transposed output, tail positions hold code 0 and whole-pad
blocks scale 0x00.  P is the padding granule (128 in the library).

The block-scaled grouped GEMM is: dequantize both operands exactly in fp64,
then the fp64 grouped GEMM of grouped_gemm.py.
"""
from __future__ import annotations

import numpy as np

from .grouped_gemm import (bf16_to_f64, group_offsets, grouped_gemm_dgrad,
                           grouped_gemm_fwd, swiglu_bwd, swiglu_fwd)

FORMATS = ("e4m3", "e2m1")
EMAX = {"e4m3": 8, "e2m1": 2}
BLOCK = 32


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def decode_e8m0(code) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64)
    out = np.ldexp(1.0, c - 127)
    return np.where(c == 0xFF, np.nan, out)


def decode_e4m3(code) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m.astype(np.float64), -9),
                   np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def decode_e2m1(code) -> np.ndarray:
    c = np.asarray(code, dtype=np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + m / 2.0, e - 1))
    return sign * mag


def decode(fmt: str, code) -> np.ndarray:
    return decode_e4m3(code) if fmt == "e4m3" else decode_e2m1(code)


def _grid(fmt: str) -> np.ndarray:
    """Non-negative finite magnitudes in code order (code i has magnitude grid[i])."""
    n = 0x7F if fmt == "e4m3" else 0x8  # e4m3 0x7F is NaN; e2m1 has 8 magnitudes
    return decode(fmt, np.arange(n))


def sign_bit(fmt: str) -> int:
    return 0x80 if fmt == "e4m3" else 0x8


# ---------------------------------------------------------------------------
# element rounding and block quantization
# ---------------------------------------------------------------------------

def round_to_grid(fmt: str, v: np.ndarray) -> np.ndarray:
    """Codes of round-to-nearest-even(v) on the element grid, saturating; sign of zero kept."""
    grid = _grid(fmt)
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    top = len(grid) - 1
    lo = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    even = np.where(lo % 2 == 0, lo, hi)
    code = np.where(d_lo < d_hi, lo, np.where(d_lo > d_hi, hi, even))
    code = np.where(a >= grid[top], top, code)
    return (code | np.where(np.signbit(v), sign_bit(fmt), 0)).astype(np.uint8)


def quantize_blocks(fmt: str, blocks: np.ndarray, valid=None):
    """MX-quantize fp64 blocks [..., 32] -> (scale codes [...], element codes [..., 32]).

    `valid` (bool, same shape) marks real elements; others must be 0 and are
    excluded from amax (they only occur in padded column-wise tails).
    """
    blocks = np.asarray(blocks, dtype=np.float64)
    if valid is None:
        valid = np.ones(blocks.shape, dtype=bool)
    vals = np.where(valid, blocks, 0.0)
    finite = np.all(np.isfinite(vals), axis=-1)
    amax = np.max(np.abs(np.where(np.isfinite(vals), vals, 0.0)), axis=-1)
    _, ex = np.frexp(amax)                 # amax = f * 2^ex, f in [0.5, 1)
    flog2 = np.where(amax > 0, ex - 1, -1000)  # floor(log2(amax)); -inf for 0
    E = np.clip(flog2 - EMAX[fmt], -127, 127)
    scaled = np.ldexp(vals, -E[..., None])
    codes = round_to_grid(fmt, scaled)
    codes = np.where(valid, codes, 0).astype(np.uint8)
    scale = (E + 127).astype(np.int64)
    scale = np.where(finite, scale, 0xFF).astype(np.uint8)
    codes = np.where(finite[..., None], codes, 0).astype(np.uint8)
    return scale, codes


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[..., 2n] nibble codes -> [..., n] bytes: element 2j low nibble, 2j+1 high nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def mx_quantize_rowwise(bits: np.ndarray, fmt: str):
    """bf16 bits [R, C] -> (codes [R, C] u8 or packed [R, C/2], scales [R, C/32]); blocks along C."""
    R, C = bits.shape
    assert C % BLOCK == 0
    v = bf16_to_f64(bits).reshape(R, C // BLOCK, BLOCK)
    scale, codes = quantize_blocks(fmt, v)
    codes = codes.reshape(R, C)
    if fmt == "e2m1":
        codes = pack_e2m1(codes)
    return codes, scale


def padded_offsets(group_lens, P: int) -> np.ndarray:
    """poff[0..G]: exclusive prefix sum of round_up(len_g, P)."""
    lens = np.asarray(group_lens, dtype=np.int64)
    padded = -(-lens // P) * P
    poff = np.zeros(len(lens) + 1, dtype=np.int64)
    poff[1:] = np.cumsum(padded)
    return poff


def mx_quantize_colwise(bits: np.ndarray, group_lens, fmt: str, M_pad: int, P: int = 128):
    """bf16 bits [M, C] -> transposed (codes_t [C, M_pad] or packed [C, M_pad/2], scales_t [C, M_pad/32]).

    Blocks of 32 run down the rows of one group, aligned to the group's first row.
    """
    M, C = bits.shape
    off = group_offsets(group_lens, M)
    poff = padded_offsets(group_lens, P)
    assert M_pad % P == 0 and poff[-1] <= M_pad
    v = bf16_to_f64(bits)
    codes_t = np.zeros((C, M_pad), dtype=np.uint8)
    scales_t = np.zeros((C, M_pad // BLOCK), dtype=np.uint8)
    for g in range(len(group_lens)):
        n = int(off[g + 1] - off[g])
        if n == 0:
            continue
        nb = -(-n // BLOCK)
        blk = np.zeros((C, nb * BLOCK), dtype=np.float64)
        blk[:, :n] = v[off[g]:off[g + 1]].T
        valid = np.zeros_like(blk, dtype=bool)
        valid[:, :n] = True
        s, c = quantize_blocks(fmt, blk.reshape(C, nb, BLOCK), valid.reshape(C, nb, BLOCK))
        p0 = int(poff[g])
        codes_t[:, p0:p0 + nb * BLOCK] = c.reshape(C, nb * BLOCK)
        scales_t[:, p0 // BLOCK:p0 // BLOCK + nb] = s
    if fmt == "e2m1":
        codes_t = pack_e2m1(codes_t)
    return codes_t, scales_t


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, fmt: str) -> np.ndarray:
    """Row-major codes [R, C] (packed [R, C/2] for e2m1) with scales [R, C/32] -> fp64 [R, C]."""
    c = unpack_e2m1(codes) if fmt == "e2m1" else np.asarray(codes)
    R, C = c.shape
    vals = decode(fmt, c).reshape(R, C // BLOCK, BLOCK)
    return (vals * decode_e8m0(scales)[..., None]).reshape(R, C)


# ---------------------------------------------------------------------------
# block-scaled grouped GEMM = dequantize, then the fp64 grouped GEMM
# ---------------------------------------------------------------------------

def mx_grouped_gemm_fwd(fmt, A, SA, B, SB, group_lens, G: int):
    """Y_g = deq(A)_g . deq(B)_g^T; A [M, K] rowwise codes, B [G*N, K] rowwise codes."""
    a = mx_dequantize(A, SA, fmt)
    b = mx_dequantize(B, SB, fmt)
    return grouped_gemm_fwd(a, b.reshape(G, -1, a.shape[1]), group_lens)


def mx_grouped_gemm_dgrad(fmt, A, SA, Bt, SBt, group_lens, G: int):
    """dX_g = deq(dY)_g . W_g with A = dY codes [M, N] (blocks along N) and
    Bt = W quantized along N, stored transposed as [K, G*N] (blocks along N)."""
    a = mx_dequantize(A, SA, fmt)             # [M, N]
    bt = mx_dequantize(Bt, SBt, fmt)          # [K, G*N]
    K = bt.shape[0]
    N = a.shape[1]
    W = bt.T.reshape(G, N, K)
    return grouped_gemm_dgrad(a, W, group_lens)


def mx_grouped_gemm_wgrad(fmt, At, SAt, Bt, SBt, group_lens, P: int = 128):
    """dW_g = sum over group g's padded region of deq(At)[:, r] deq(Bt)[:, r]^T.

    At = dY column-wise codes [N, M_pad], Bt = X column-wise codes [K, M_pad]."""
    at = mx_dequantize(At, SAt, fmt)          # [N, M_pad]
    bt = mx_dequantize(Bt, SBt, fmt)          # [K, M_pad]
    poff = padded_offsets(group_lens, P)
    G = len(group_lens)
    dW = np.zeros((G, at.shape[0], bt.shape[0]), dtype=np.float64)
    for g in range(G):
        a, b = poff[g], poff[g + 1]
        if b > a:
            dW[g] = at[:, a:b] @ bt[:, a:b].T
    return dW


def mx_grouped_fc1_swiglu(fmt, A, SA, B, SB, group_lens, G: int, limit=None):
    H = mx_grouped_gemm_fwd(fmt, A, SA, B, SB, group_lens, G)
    return swiglu_fwd(H, limit), H


def mx_grouped_fc2_dgrad_swiglu_bwd(fmt, A, SA, Bt, SBt, H, group_lens, G: int, limit=None):
    dA = mx_grouped_gemm_dgrad(fmt, A, SA, Bt, SBt, group_lens, G)
    return swiglu_bwd(dA, H, limit)
