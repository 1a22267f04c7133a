"""Pins for the fp64 CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something other than itself: brute-force
loop nests written here, closed forms, adjoint identities, hand-derived MX
values (tests/golden/mx_blocks.txt), torch's own float8 decoders and casts, and
lossless round trips.  A plausible slip in the oracle (a transposed operand, a
dropped group, a wrong offset, a wrong sign, a wrong rounding tie) fails at
least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from oracle import mx as omx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_lens(rng, G, M, zeros=1):
    cuts = np.sort(rng.integers(0, M + 1, size=G - 1))
    lens = np.diff(np.concatenate([[0], cuts, [M]])).astype(np.int32)
    for g in rng.choice(G, size=min(zeros, G), replace=False):
        lens[(g + 1) % G] += lens[g]
        lens[g] = 0
    return lens


# ---------------------------------------------------------------------------
# grouped GEMM: brute force, identities, closed forms
# ---------------------------------------------------------------------------

def _brute(X, W, dY, lens):
    """Pure-Python loops, token by token: which group owns row r is found by walking lens."""
    M, K = X.shape
    G, N, _ = W.shape
    owner = []
    for g, n in enumerate(lens):
        owner += [g] * int(n)
    Y = [[0.0] * N for _ in range(M)]
    dX = [[0.0] * K for _ in range(M)]
    dW = [[[0.0] * K for _ in range(N)] for _ in range(G)]
    for r in range(M):
        g = owner[r]
        for n in range(N):
            for k in range(K):
                Y[r][n] += float(X[r, k]) * float(W[g, n, k])
                dX[r][k] += float(dY[r, n]) * float(W[g, n, k])
                dW[g][n][k] += float(dY[r, n]) * float(X[r, k])
    return np.array(Y), np.array(dX), np.array(dW)


@pytest.mark.parametrize("seed", range(6))
def test_grouped_gemm_vs_brute_force(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.integers(1, 6))
    M = int(rng.integers(0, 17))
    N = int(rng.integers(1, 7))
    K = int(rng.integers(1, 7))
    lens = _rand_lens(rng, G, M, zeros=1 if G > 1 else 0)
    X = rng.standard_normal((M, K))
    W = rng.standard_normal((G, N, K))
    dY = rng.standard_normal((M, N))
    Yb, dXb, dWb = _brute(X, W, dY, lens)
    np.testing.assert_allclose(og.grouped_gemm_fwd(X, W, lens), Yb.reshape(M, N), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(og.grouped_gemm_dgrad(dY, W, lens), dXb.reshape(M, K), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(og.grouped_gemm_wgrad(X, dY, lens), dWb.reshape(G, N, K), rtol=1e-12, atol=1e-12)


def test_adjoint_identity():
    # <fwd(X,W), dY> = <X, dgrad(dY,W)> = <W, wgrad(X,dY)>: all three are the same trilinear form
    rng = np.random.default_rng(7)
    G, M, N, K = 6, 200, 48, 40
    lens = _rand_lens(rng, G, M, zeros=2)
    X, W, dY = rng.standard_normal((M, K)), rng.standard_normal((G, N, K)), rng.standard_normal((M, N))
    a = np.sum(og.grouped_gemm_fwd(X, W, lens) * dY)
    b = np.sum(X * og.grouped_gemm_dgrad(dY, W, lens))
    c = np.sum(W * og.grouped_gemm_wgrad(X, dY, lens))
    assert abs(a - b) < 1e-9 * (1 + abs(a)) and abs(a - c) < 1e-9 * (1 + abs(a))


def test_groups_concatenate():
    rng = np.random.default_rng(8)
    G, M, N, K = 5, 90, 12, 10
    lens = _rand_lens(rng, G, M, zeros=1)
    X, W, dY = rng.standard_normal((M, K)), rng.standard_normal((G, N, K)), rng.standard_normal((M, N))
    Y, dX, dW = og.grouped_gemm_fwd(X, W, lens), og.grouped_gemm_dgrad(dY, W, lens), og.grouped_gemm_wgrad(X, dY, lens)
    off = np.concatenate([[0], np.cumsum(lens)])
    for g in range(G):
        a, b = off[g], off[g + 1]
        one = np.array([b - a], dtype=np.int32)
        np.testing.assert_array_equal(og.grouped_gemm_fwd(X[a:b], W[g:g + 1], one), Y[a:b])
        np.testing.assert_array_equal(og.grouped_gemm_dgrad(dY[a:b], W[g:g + 1], one), dX[a:b])
        np.testing.assert_array_equal(og.grouped_gemm_wgrad(X[a:b], dY[a:b], one)[0], dW[g])


def test_one_hot_picks_weight_entries():
    # X rows one-hot at k_r: Y[r, n] = W[g(r), n, k_r]; dY one-hot at n_r: dX[r, k] = W[g(r), n_r, k]
    rng = np.random.default_rng(9)
    G, N, K = 3, 5, 4
    lens = np.array([2, 0, 3], dtype=np.int32)
    owner = [0, 0, 2, 2, 2]
    M = 5
    W = rng.standard_normal((G, N, K))
    kr = rng.integers(0, K, size=M)
    nr = rng.integers(0, N, size=M)
    X = np.zeros((M, K)); X[np.arange(M), kr] = 1.0
    dY = np.zeros((M, N)); dY[np.arange(M), nr] = 1.0
    Y = og.grouped_gemm_fwd(X, W, lens)
    dX = og.grouped_gemm_dgrad(dY, W, lens)
    for r in range(M):
        np.testing.assert_array_equal(Y[r], W[owner[r], :, kr[r]])
        np.testing.assert_array_equal(dX[r], W[owner[r], nr[r], :])
    dW = og.grouped_gemm_wgrad(X, dY, lens)
    assert np.all(dW[1] == 0.0)
    expect = np.zeros((N, K))
    for r in (2, 3, 4):
        expect[nr[r], kr[r]] += 1.0
    np.testing.assert_array_equal(dW[2], expect)


def test_empty_groups_and_validation():
    X = np.ones((3, 2)); dY = np.ones((3, 4))
    dW = og.grouped_gemm_wgrad(X, dY, [0, 3, 0])
    assert np.all(dW[0] == 0) and np.all(dW[2] == 0) and np.all(dW[1] == 3.0)
    with pytest.raises(ValueError):
        og.group_offsets([2, -1, 2], 3)
    with pytest.raises(ValueError):
        og.group_offsets([2, 2], 3)
    assert og.grouped_gemm_fwd(np.zeros((0, 2)), np.ones((2, 4, 2)), [0, 0]).shape == (0, 4)


def test_bf16_decode_exact():
    vals = np.array([1.0, -2.5, 3.140625, 0.0, -0.0, 2.0 ** -133, 65280.0 * 2 ** 112], dtype=np.float64)
    bits = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(og.bf16_to_f64(bits), vals)


# ---------------------------------------------------------------------------
# SwiGLU forward / backward
# ---------------------------------------------------------------------------

def test_swiglu_closed_forms():
    H = np.array([[0.0, 1.0, 5.0, 7.0],      # gate 0 -> A = 0
                  [1.0, 30.0, 2.0, 3.0],      # A = silu(1)*2, silu(30)*3 ~ 30*3
                  [-1.0, -40.0, 4.0, 1.0]])   # silu(-1)*4; silu(-40) ~ -40*e^-40
    A = og.swiglu_fwd(H)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert A[0, 0] == 0.0 and A[0, 1] == pytest.approx(silu1 * 7.0, rel=1e-15)
    assert A[1, 0] == pytest.approx(silu1 * 2.0, rel=1e-15)
    assert A[1, 1] == pytest.approx(90.0, rel=1e-12)
    assert A[2, 0] == pytest.approx(-1.0 / (1.0 + math.e) * 4.0, rel=1e-15)
    assert abs(A[2, 1]) < 1e-15


def test_swiglu_bwd_finite_difference():
    rng = np.random.default_rng(11)
    H = rng.standard_normal((4, 6)) * 2
    dA = rng.standard_normal((4, 3))
    dH = og.swiglu_bwd(dA, H)
    eps = 1e-6
    num = np.zeros_like(H)
    for i in range(H.shape[0]):
        for j in range(H.shape[1]):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, j] += eps; Hm[i, j] -= eps
            num[i, j] = np.sum(dA * (og.swiglu_fwd(Hp) - og.swiglu_fwd(Hm))) / (2 * eps)
    np.testing.assert_allclose(dH, num, rtol=1e-7, atol=1e-8)


def test_clamped_swiglu_closed_forms_and_special_cases():
    # limit L: gate -> min(gate, L), up -> clip(up, -L, L) before silu(gate) * up
    L = 2.0
    H = np.array([[5.0, -1.0, 7.0, 0.5],      # gate 5 -> 2; up 7 -> 2 | gate -1, up 0.5 untouched
                  [1.0, -30.0, -9.0, 3.0]])   # up -9 -> -2 | gate -30 (below: no clamp), up 3 -> 2
    A = og.swiglu_fwd(H, L)
    silu = lambda x: x / (1.0 + math.exp(-x))
    assert A[0, 0] == pytest.approx(silu(2.0) * 2.0, rel=1e-15)
    assert A[0, 1] == pytest.approx(silu(-1.0) * 0.5, rel=1e-15)
    assert A[1, 0] == pytest.approx(silu(1.0) * -2.0, rel=1e-15)
    assert A[1, 1] == pytest.approx(silu(-30.0) * 2.0, rel=1e-15)
    # no limit (None or 0) and a limit above every value both reduce to the plain SwiGLU
    rng = np.random.default_rng(21)
    Hr = rng.standard_normal((5, 8))
    for lim in (None, 0.0, 1e9):
        np.testing.assert_array_equal(og.swiglu_fwd(Hr, lim), og.swiglu_fwd(Hr))
        np.testing.assert_array_equal(og.swiglu_bwd(Hr[:, :4], Hr, lim), og.swiglu_bwd(Hr[:, :4], Hr))
    # clamped entries get no gradient; unclamped ones match the plain derivative at the clamped values
    dA = np.ones((2, 2))
    dH = og.swiglu_bwd(dA, H, L)
    assert dH[0, 0] == 0.0 and dH[0, 2] == 0.0      # gate 5 > L, up 7 > L
    assert dH[1, 2] == 0.0 and dH[1, 3] == 0.0      # up -9 < -L, up 3 > L
    s1 = 1.0 / (1.0 + math.exp(1.0))                # sigma(-1)
    assert dH[0, 1] == pytest.approx(0.5 * s1 * (1.0 - 1.0 * (1.0 - s1)), rel=1e-14)


def test_clamped_swiglu_bwd_finite_difference():
    # away from the clamp boundaries the clamped backward is the derivative of the clamped forward
    rng = np.random.default_rng(22)
    L = 1.5
    H = rng.standard_normal((6, 8)) * 2
    H[np.abs(np.abs(H) - L) < 0.05] += 0.2   # keep every entry clear of a kink
    dA = rng.standard_normal((6, 4))
    dH = og.swiglu_bwd(dA, H, L)
    eps = 1e-6
    num = np.zeros_like(H)
    for i in range(H.shape[0]):
        for j in range(H.shape[1]):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, j] += eps; Hm[i, j] -= eps
            num[i, j] = np.sum(dA * (og.swiglu_fwd(Hp, L) - og.swiglu_fwd(Hm, L))) / (2 * eps)
    np.testing.assert_allclose(dH, num, rtol=1e-7, atol=1e-8)
    assert (dH == 0).any() and (dH != 0).any()


def test_fc1_fc2_compositions():
    rng = np.random.default_rng(12)
    G, M, I, K = 3, 20, 4, 6
    lens = np.array([7, 0, 13], dtype=np.int32)
    X, W1 = rng.standard_normal((M, K)), rng.standard_normal((G, 2 * I, K))
    A, H = og.grouped_fc1_swiglu(X, W1, lens)
    Yb, _, _ = _brute(X, W1, np.zeros((M, 2 * I)), lens)
    np.testing.assert_allclose(H, Yb, rtol=1e-12, atol=1e-12)
    g, u = Yb[:, :I], Yb[:, I:]
    np.testing.assert_allclose(A, g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12)
    W2 = rng.standard_normal((G, K, I))
    dY = rng.standard_normal((M, K))
    dH = og.grouped_fc2_dgrad_swiglu_bwd(dY, W2, H, lens)
    # chain rule through a perturbation: d/dt <dY, fwd(swiglu(H + t V), W2)> = <dH, V>
    V = rng.standard_normal(H.shape)
    f = lambda t: np.sum(dY * og.grouped_gemm_fwd(og.swiglu_fwd(H + t * V), W2, lens))
    num = (f(1e-6) - f(-1e-6)) / 2e-6
    assert np.sum(dH * V) == pytest.approx(num, rel=1e-6)


def test_within_tol():
    ref = np.array([1.0, -1.0, 0.0, 100.0])
    assert og.within_tol(ref, ref)[0]
    assert not og.within_tol(ref + np.array([0, 0, 0, 2.0]), ref)[0]
    assert not og.within_tol(np.array([np.nan, -1, 0, 100]), ref)[0]


# ---------------------------------------------------------------------------
# MX formats
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = omx.decode_e4m3(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_e8m0_decode_matches_torch():
    codes = np.arange(255, dtype=np.uint8)  # 0xFF is NaN in both
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    np.testing.assert_array_equal(omx.decode_e8m0(codes), ref)
    assert np.isnan(omx.decode_e8m0(0xFF))


def test_e2m1_decode_table():
    table = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    np.testing.assert_array_equal(omx.decode_e2m1(np.arange(8)), table)
    np.testing.assert_array_equal(omx.decode_e2m1(np.arange(8, 16)), [-v for v in table])


def _golden_cases():
    cases = []
    with open(os.path.join(GOLDEN, "mx_blocks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            p = line.split()
            cases.append((p[0], float.fromhex(p[1]), float.fromhex(p[2]), int(p[3], 16), int(p[4], 16)))
    return cases


@pytest.mark.parametrize("case", _golden_cases())
def test_mx_golden_blocks(case):
    fmt, amax, v, scale, code = case
    blk = np.zeros((1, 32))
    blk[0, 0], blk[0, 1] = amax, v
    s, c = omx.quantize_blocks(fmt, blk)
    assert int(s[0]) == scale
    assert int(c[0, 1]) == code


def test_e4m3_rounding_matches_torch_cast_in_range():
    rng = np.random.default_rng(13)
    v = rng.uniform(-440, 440, size=20000)
    v = np.concatenate([v, rng.uniform(-2.0 ** -6, 2.0 ** -6, size=5000)])
    # include exact ties: midpoints between consecutive grid values
    grid = omx.decode_e4m3(np.arange(0x7E))
    mids = (grid[:-1] + np.diff(grid) / 2)
    v = np.concatenate([v, mids, -mids])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(omx.round_to_grid("e4m3", v), ref)


def test_mx_roundtrip_and_idempotence():
    rng = np.random.default_rng(14)
    for fmt in omx.FORMATS:
        grid = omx._grid(fmt)
        # values already on a block's grid: code * 2^E with the block's amax setting E
        E = rng.integers(-20, 20, size=(64, 1))
        codes = rng.integers(0, len(grid), size=(64, 32))
        codes[:, 0] = len(grid) - 1  # amax = top of the grid, so the rule picks this E back
        vals = grid[codes] * np.ldexp(1.0, E + 0) * np.where(rng.random((64, 32)) < 0.5, -1, 1)
        # rule: floor(log2(amax)) - emax = E + floor(log2(grid max)) - emax = E
        s, c = omx.quantize_blocks(fmt, vals)
        np.testing.assert_array_equal(s.astype(np.int64) - 127, E[:, 0])
        deq = omx.decode(fmt, c) * omx.decode_e8m0(s)[:, None]
        np.testing.assert_array_equal(deq, vals)
        s2, c2 = omx.quantize_blocks(fmt, deq)
        np.testing.assert_array_equal(s2, s)
        np.testing.assert_array_equal(c2, c)


def test_mx_monotone_and_top_binade():
    rng = np.random.default_rng(15)
    for fmt in omx.FORMATS:
        v = np.sort(rng.uniform(0, 3, size=4000))
        c = omx.round_to_grid(fmt, v)
        assert np.all(np.diff(omx.decode(fmt, c)) >= 0)
        blocks = rng.standard_normal((200, 32)) * np.ldexp(1.0, rng.integers(-30, 30, size=(200, 1)))
        s, _ = omx.quantize_blocks(fmt, blocks)
        scaled_amax = np.max(np.abs(blocks), axis=1) * omx.decode_e8m0(s) ** -1
        assert np.all(scaled_amax >= 2.0 ** omx.EMAX[fmt]) and np.all(scaled_amax < 2.0 ** (omx.EMAX[fmt] + 1))


def test_e2m1_pack_order():
    codes = np.array([[0x1, 0x2, 0x7, 0x8]], dtype=np.uint8)
    packed = omx.pack_e2m1(codes)
    np.testing.assert_array_equal(packed, [[0x21, 0x87]])
    np.testing.assert_array_equal(omx.unpack_e2m1(packed), codes)


def _bf16_bits(a):
    return torch.tensor(a, dtype=torch.float64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_colwise_equals_rowwise_of_group_slices():
    # colwise on [M, C] == rowwise on each group's transposed, zero-padded slice
    rng = np.random.default_rng(16)
    lens = np.array([33, 0, 5, 64, 1], dtype=np.int32)
    M, C = int(lens.sum()), 8
    bits = _bf16_bits(rng.standard_normal((M, C)) * 3)
    P = 128
    M_pad = 4 * P + P
    for fmt in omx.FORMATS:
        ct, st = omx.mx_quantize_colwise(bits, lens, fmt, M_pad, P)
        if fmt == "e2m1":
            ct = omx.unpack_e2m1(ct)
        off = 0
        poff = 0
        for n in lens:
            n = int(n)
            if n:
                nb = -(-n // 32)
                sl = np.zeros((C, nb * 32), dtype=np.uint16)
                sl[:, :n] = bits[off:off + n].T
                rc, rs = omx.mx_quantize_rowwise(sl, fmt)
                if fmt == "e2m1":
                    rc = omx.unpack_e2m1(rc)
                np.testing.assert_array_equal(ct[:, poff:poff + n], rc[:, :n])
                assert np.all(ct[:, poff + n:poff + -(-n // P) * P] == 0)
                np.testing.assert_array_equal(st[:, poff // 32:poff // 32 + nb], rs)
            off += n
            poff += -(-n // P) * P
        assert np.all(ct[:, poff:] == 0) and np.all(st[:, poff // 32:] == 0)


def _grid_operand(rng, fmt, rows, cols, shift=0):
    """bf16 bits of values that MX-quantize losslessly (block amax on the grid top); block
    exponents are drawn from [shift - 4, shift + 4)."""
    grid = omx._grid(fmt)
    codes = rng.integers(0, len(grid), size=(rows, cols))
    codes[:, ::32] = len(grid) - 1
    E = rng.integers(shift - 4, shift + 4, size=(rows, cols // 32)).repeat(32, axis=1)
    vals = grid[codes] * np.ldexp(1.0, E) * np.where(rng.random((rows, cols)) < 0.5, -1, 1)
    return _bf16_bits(vals), vals


@pytest.mark.parametrize("fmt", omx.FORMATS)
def test_mx_grouped_gemm_lossless_equals_fp64(fmt):
    # operands on the MX grid quantize exactly, so the block-scaled GEMM must equal the fp64 one
    rng = np.random.default_rng(17)
    G, N, K = 3, 64, 96
    lens = np.array([40, 0, 57], dtype=np.int32)
    M = int(lens.sum())
    xb, X = _grid_operand(rng, fmt, M, K)
    wb, W = _grid_operand(rng, fmt, G * N, K)
    A, SA = omx.mx_quantize_rowwise(xb, fmt)
    B, SB = omx.mx_quantize_rowwise(wb, fmt)
    Y = omx.mx_grouped_gemm_fwd(fmt, A, SA, B, SB, lens, G)
    np.testing.assert_array_equal(Y, og.grouped_gemm_fwd(X, W.reshape(G, N, K), lens))
    # dgrad: dY [M, N] rowwise; W quantized along N, stored [K, G*N]
    dyb, dY = _grid_operand(rng, fmt, M, N)
    wtb, Wt = _grid_operand(rng, fmt, K, G * N)
    Ad, SAd = omx.mx_quantize_rowwise(dyb, fmt)
    Bt, SBt = omx.mx_quantize_rowwise(wtb, fmt)
    dX = omx.mx_grouped_gemm_dgrad(fmt, Ad, SAd, Bt, SBt, lens, G)
    np.testing.assert_array_equal(dX, og.grouped_gemm_dgrad(dY, Wt.T.reshape(G, N, K), lens))
    # wgrad: column-wise (group-aligned) operands; lossless when each group block is on the grid
    P = 128
    M_pad = 3 * P
    dyc_b, dYc = _colwise_grid(rng, fmt, lens, N)
    xc_b, Xc = _colwise_grid(rng, fmt, lens, K)
    At, SAt = omx.mx_quantize_colwise(dyc_b, lens, fmt, M_pad, P)
    Bt2, SBt2 = omx.mx_quantize_colwise(xc_b, lens, fmt, M_pad, P)
    dW = omx.mx_grouped_gemm_wgrad(fmt, At, SAt, Bt2, SBt2, lens, P)
    np.testing.assert_array_equal(dW, og.grouped_gemm_wgrad(Xc, dYc, lens))


def _brute_swiglu_rows(Hrows, I, limit):
    """A = silu(gate) * up row by row with plain loops and math.exp; the clamp written out."""
    out = []
    for h in Hrows:
        row = []
        for j in range(I):
            g, u = float(h[j]), float(h[I + j])
            if limit:
                g, u = min(g, limit), max(-limit, min(u, limit))
            row.append(g / (1.0 + math.exp(-g)) * u)
        out.append(row)
    return np.array(out).reshape(len(Hrows), I)


def _brute_swiglu_bwd_rows(dArows, Hrows, I, limit):
    """dH row by row: d/dgate and d/dup of silu(gate) * up, zero where a clamp is active."""
    out = []
    for da_r, h in zip(dArows, Hrows):
        dg_row, du_row = [], []
        for j in range(I):
            g, u, da = float(h[j]), float(h[I + j]), float(da_r[j])
            pg = pu = True
            if limit:
                pg, pu = g <= limit, abs(u) <= limit
                g, u = min(g, limit), max(-limit, min(u, limit))
            s = 1.0 / (1.0 + math.exp(-g))
            dg_row.append(da * u * (s + g * s * (1.0 - s)) if pg else 0.0)
            du_row.append(da * g * s if pu else 0.0)
        out.append(dg_row + du_row)
    return np.array(out).reshape(len(Hrows), 2 * I)


@pytest.mark.parametrize("fmt", omx.FORMATS)
def test_mx_swiglu_gemms_lossless_operands(fmt):
    # operands on the MX grid quantize exactly, so the MX FC1+SwiGLU and FC2-dgrad+SwiGLU'
    # compositions must equal (1) brute-force loops over the original values and (2) the
    # BF16-path oracle on those values; with and without a clamp that is active somewhere,
    # so a limit that is not passed on, a swapped H, or a mis-shaped weight stack all fail
    rng = np.random.default_rng(35)
    G, I, K, Hd = 3, 3, 64, 32
    lens = np.array([5, 0, 7], dtype=np.int32)
    M = int(lens.sum())
    owner = [0] * 5 + [2] * 7
    # grid values times a power of two stay on the grid (only the block exponent moves);
    # the shift keeps |H| in the range where the SwiGLU is not saturated
    shift = -12 if fmt == "e4m3" else -6
    xb, X = _grid_operand(rng, fmt, M, K, shift)
    wb, W1 = _grid_operand(rng, fmt, G * 2 * I, K, shift)
    A, SA = omx.mx_quantize_rowwise(xb, fmt)
    B, SB = omx.mx_quantize_rowwise(wb, fmt)
    W1g = W1.reshape(G, 2 * I, K)
    Hb = np.array([[sum(X[r, k] * W1g[owner[r], n, k] for k in range(K)) for n in range(2 * I)]
                   for r in range(M)])
    gate_max = float(np.max(Hb[:, :I]))
    results = {}
    for limit in (None, 0.5 * gate_max):
        Am, Hm = omx.mx_grouped_fc1_swiglu(fmt, A, SA, B, SB, lens, G, limit)
        np.testing.assert_allclose(Hm, Hb, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(Am, _brute_swiglu_rows(Hb, I, limit), rtol=1e-12, atol=1e-12)
        rA, rH = og.grouped_fc1_swiglu(X, W1g, lens, limit)
        np.testing.assert_allclose(Am, rA, rtol=1e-13, atol=1e-13)
        results[limit] = Am
    assert not np.allclose(results[None], results[0.5 * gate_max])  # the clamp is active somewhere
    # FC2 dgrad + SwiGLU': dY [M, Hd] row-wise along Hd; W2 quantized along Hd, stored [I, G*Hd]
    dyb, dY = _grid_operand(rng, fmt, M, Hd, shift)
    wtb, Wt = _grid_operand(rng, fmt, I, G * Hd, shift)
    Ad, SAd = omx.mx_quantize_rowwise(dyb, fmt)
    Bt, SBt = omx.mx_quantize_rowwise(wtb, fmt)
    W2g = Wt.T.reshape(G, Hd, I)
    Hs = rng.standard_normal((M, 2 * I)) * 1.5
    dA = np.array([[sum(dY[r, n] * W2g[owner[r], n, j] for n in range(Hd)) for j in range(I)] for r in range(M)])
    grads = {}
    for limit in (None, 0.75):
        dH = omx.mx_grouped_fc2_dgrad_swiglu_bwd(fmt, Ad, SAd, Bt, SBt, Hs, lens, G, limit)
        np.testing.assert_allclose(dH, _brute_swiglu_bwd_rows(dA, Hs, I, limit), rtol=1e-12, atol=1e-12)
        ref = og.grouped_fc2_dgrad_swiglu_bwd(dY, W2g, Hs, lens, limit)
        np.testing.assert_allclose(dH, ref, rtol=1e-13, atol=1e-13)
        grads[limit] = dH
    assert (grads[0.75] == 0).any() and not np.allclose(grads[None], grads[0.75])
    # a different H changes the result: the composition consumes the H it is given
    dH_other = omx.mx_grouped_fc2_dgrad_swiglu_bwd(fmt, Ad, SAd, Bt, SBt, Hs[:, ::-1].copy(), lens, G)
    assert not np.allclose(dH_other, grads[None])


def _colwise_grid(rng, fmt, lens, C):
    grid = omx._grid(fmt)
    parts_b, parts = [], []
    for n in lens:
        n = int(n)
        if not n:
            continue
        codes = rng.integers(0, len(grid), size=(n, C))
        codes[::32, :] = len(grid) - 1  # first row of each 32-row block holds the grid top
        E = np.repeat(rng.integers(-4, 4, size=(-(-n // 32), C)), 32, axis=0)[:n]
        v = grid[codes] * np.ldexp(1.0, E) * np.where(rng.random((n, C)) < 0.5, -1, 1)
        parts.append(v)
    vals = np.concatenate(parts, axis=0)
    return _bf16_bits(vals), vals


def test_round_bf16_matches_torch_cast():
    # fp32 inputs make torch's fp32 -> bf16 cast a single RNE rounding, the same rule
    rng = np.random.default_rng(21)
    v = (rng.standard_normal(50000) * np.ldexp(1.0, rng.integers(-140, 120, 50000))).astype(np.float32)
    # exact ties: bf16 midpoints (9 significant bits with the last one set)
    m = rng.integers(256, 512, 5000) * 2 + 1
    ties = np.ldexp(m.astype(np.float64), rng.integers(-120, 100, 5000)).astype(np.float32)
    v = np.concatenate([v, ties, -ties, np.float32([0.0, -0.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134])])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(og.round_bf16(v.astype(np.float64)), ref)


def test_layer_chain_matches_step_by_step():
    rng = np.random.default_rng(22)
    lens = np.array([9, 0, 14], dtype=np.int32)
    M, Hd, I = 23, 16, 8
    X, dY = rng.standard_normal((M, Hd)), rng.standard_normal((M, Hd))
    W1, W2 = rng.standard_normal((3, 2 * I, Hd)) * 0.3, rng.standard_normal((3, Hd, I)) * 0.3
    out = og.expert_layer_chain(X, W1, W2, dY, lens)
    Yb, _, _ = _brute(X, W1, np.zeros((M, 2 * I)), lens)
    np.testing.assert_allclose(out["H"], Yb, rtol=1e-12, atol=1e-12)
    g, u = Yb[:, :I], Yb[:, I:]
    np.testing.assert_allclose(out["A"], g / (1 + np.exp(-g)) * u, rtol=1e-12, atol=1e-12)
    # downstream calls consume the bf16 roundings of A, H and dH
    A16, H16 = og.round_bf16(out["A"]), og.round_bf16(out["H"])
    Y2, _, dW2 = _brute(A16, W2, dY, lens)
    np.testing.assert_allclose(out["Y"], Y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dW2"], dW2, rtol=1e-12, atol=1e-12)
    _, dA, _ = _brute(np.zeros((M, I)), W2, dY, lens)
    np.testing.assert_allclose(out["dH"], og.swiglu_bwd(dA, H16), rtol=1e-12, atol=1e-12)
    dH16 = og.round_bf16(out["dH"])
    _, dXb, dW1b = _brute(X, W1, dH16, lens)
    np.testing.assert_allclose(out["dX"], dXb, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["dW1"], dW1b, rtol=1e-12, atol=1e-12)


def test_wgrad_accumulate_adds_to_main_grad():
    rng = np.random.default_rng(23)
    lens = np.array([3, 0, 5], dtype=np.int32)
    X, dY = rng.standard_normal((8, 4)), rng.standard_normal((8, 6))
    dW0 = rng.standard_normal((3, 6, 4))
    out = og.grouped_gemm_wgrad_accumulate(dW0, X, dY, lens)
    _, _, dWb = _brute(X, np.zeros((3, 6, 4)), dY, lens)
    np.testing.assert_allclose(out, dW0 + dWb, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(out[1], dW0[1])  # empty group: main_grad unchanged


# ---------------------------------------------------------------------------
# MoE glue: permute / combine
# ---------------------------------------------------------------------------

from oracle import moe_glue as omg  # noqa: E402


def _topk_ids(rng, T, E, k):
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])


def test_permute_is_stable_expert_sort():
    rng = np.random.default_rng(24)
    T, E, k = 37, 9, 3
    ids = _topk_ids(rng, T, E, k)
    pos, lens, row_token = omg.permute(ids, E)
    assert sorted(pos.reshape(-1).tolist()) == list(range(T * k))  # a bijection onto the rows
    np.testing.assert_array_equal(lens, np.bincount(ids.reshape(-1), minlength=E))
    # brute force: walk experts, then tokens, assigning rows in order
    r = 0
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    assert pos[t, j] == r and row_token[r] == t
                    r += 1
    X = rng.standard_normal((T, 5))
    Xs = omg.permute_rows(X, pos)
    np.testing.assert_array_equal(Xs, X[row_token])


def test_permute_reproduces_the_workload_layout():
    # the generator builds each workload's expert-sorted rows (group_lens, row_token) with its own
    # lexsort; the oracle permute of the same top-k ids must give exactly that layout
    from precision_grouped_gemm_gb300 import workloads as wl
    for w in (wl.DSV4_BF16, wl.GPTOSS_BF16):
        lens, row_token = w.group_lens()
        pos, glens, rtok = omg.permute(w.topk_ids(), w.experts)
        np.testing.assert_array_equal(glens, lens)
        np.testing.assert_array_equal(rtok, row_token)


def test_combine_and_backward():
    rng = np.random.default_rng(25)
    T, E, k, H = 20, 6, 2, 7
    ids = _topk_ids(rng, T, E, k)
    pos, lens, row_token = omg.permute(ids, E)
    Ys = rng.standard_normal((T * k, H))
    w = rng.random((T, k))
    out = omg.combine(Ys, pos, w)
    for t in range(T):
        np.testing.assert_allclose(out[t], sum(w[t, j] * Ys[pos[t, j]] for j in range(k)), rtol=1e-12)
    # one-hot weights pick a row; unit weights of the permute round trip give k * X
    X = rng.standard_normal((T, H))
    np.testing.assert_allclose(omg.combine(omg.permute_rows(X, pos), pos), k * X, rtol=1e-12)
    dOut = rng.standard_normal((T, H))
    dYs, dw = omg.combine_bwd(dOut, Ys, pos, w)
    # adjoint in Ys: <combine(Ys), dOut> = <Ys, dYs>; derivative in w by finite differences
    assert np.sum(out * dOut) == pytest.approx(np.sum(Ys * dYs), rel=1e-12)
    eps = 1e-6
    for t, j in [(0, 0), (7, 1), (19, 0)]:
        wp, wm = w.copy(), w.copy()
        wp[t, j] += eps; wm[t, j] -= eps
        num = (np.sum(omg.combine(Ys, pos, wp) * dOut) - np.sum(omg.combine(Ys, pos, wm) * dOut)) / (2 * eps)
        assert dw[t, j] == pytest.approx(num, rel=1e-6)
    with pytest.raises(ValueError):
        omg.permute(np.array([[0, E]]), E)


# ---------------------------------------------------------------------------
# FP8 (e4m3) tensor-wise current scaling
# ---------------------------------------------------------------------------
from oracle import fp8 as of8  # noqa: E402


def test_fp8_tensorwise_hand_values():
    # amax 2 -> s = 224: 1 -> 224 = 1.75 * 2^7 (0x76), -2 -> -448 (0xFE), 0.5 -> 112 (0x6E), 0 -> 0
    codes, s = of8.fp8_quantize_tensorwise(np.array([1.0, -2.0, 0.5, 0.0, -0.0]))
    assert s == np.float32(224.0)
    assert codes.tolist() == [0x76, 0xFE, 0x6E, 0x00, 0x80]
    np.testing.assert_array_equal(of8.fp8_dequantize(codes, s), [1.0, -2.0, 0.5, 0.0, -0.0])
    # an all-zero tensor keeps scale 1
    z, sz = of8.fp8_quantize_tensorwise(np.zeros(5))
    assert sz == np.float32(1.0) and not z.any()


def test_fp8_tensorwise_amax_maps_to_448_and_ties_round_to_even():
    rng = np.random.default_rng(31)
    x = rng.standard_normal(1000) * 3.0
    codes, s = of8.fp8_quantize_tensorwise(x)
    i = int(np.argmax(np.abs(x)))
    assert codes[i] & 0x7F == 0x7E                      # |448|
    assert np.all(np.abs(omx.decode_e4m3(codes)) <= 448.0)
    # a power-of-two scale makes x * s exact: 1.0625 lies halfway between 1.0 and 1.125 -> 1.0
    # (even mantissa); 1.1875 halfway between 1.125 and 1.25 -> 1.25
    c, _ = of8.fp8_quantize_tensorwise(np.array([1.0625, 1.1875, 448.0 / 64]), scale=64.0)
    assert omx.decode_e4m3(c).tolist() == [64.0 * 1.0, 64.0 * 1.25, 448.0]


def test_fp8_tensorwise_monotone_and_non_finite():
    x = np.linspace(-5, 5, 2001)
    codes, _ = of8.fp8_quantize_tensorwise(x)
    assert np.all(np.diff(omx.decode_e4m3(codes)) >= 0)
    c, s = of8.fp8_quantize_tensorwise(np.array([1.0, np.nan, np.inf, -np.inf, -4.0]))
    assert s == np.float32(448.0 / 4.0)                 # amax over the finite values
    assert c[1] & 0x7F == 0x7F and c[2] == 0x7E and c[3] == 0xFE and c[4] == 0xFE


def test_fp8_grouped_gemms_lossless_operands():
    # operands on the e4m3 grid times 2^-3 with amax 448 * 2^-3: s = 8 exactly, quantization
    # is lossless, so the FP8 GEMMs equal the fp64 GEMMs of the original values (brute force)
    rng = np.random.default_rng(32)
    grid = omx.decode_e4m3(np.arange(0x7F))

    def on_grid(shape):
        v = grid[rng.integers(0, len(grid), size=shape)] * np.where(rng.random(shape) < 0.5, -1, 1) / 8.0
        v.flat[0] = 448.0 / 8.0
        return v

    G, N, K = 3, 5, 7
    lens = np.array([4, 0, 6], dtype=np.int32)
    M = int(lens.sum())
    X, W, dY = on_grid((M, K)), on_grid((G * N, K)), on_grid((M, N))
    (cx, sx), (cw, sw), (cd, sd) = (of8.fp8_quantize_tensorwise(t) for t in (X, W, dY))
    assert sx == sw == sd == np.float32(8.0)
    off = np.concatenate([[0], np.cumsum(lens)])
    Y = of8.fp8_grouped_gemm_fwd(cx, sx, cw, sw, lens, G)
    dX = of8.fp8_grouped_gemm_dgrad(cd, sd, cw, sw, lens, G)
    dW = of8.fp8_grouped_gemm_wgrad(cx, sx, cd, sd, lens)
    Wg = W.reshape(G, N, K)
    for g in range(G):
        for r in range(off[g], off[g + 1]):
            for n in range(N):
                assert Y[r, n] == pytest.approx(sum(X[r, k] * Wg[g, n, k] for k in range(K)), abs=1e-12)
            for k in range(K):
                assert dX[r, k] == pytest.approx(sum(dY[r, n] * Wg[g, n, k] for n in range(N)), abs=1e-12)
        for n in range(N):
            for k in range(K):
                ref = sum(dY[r, n] * X[r, k] for r in range(off[g], off[g + 1]))
                assert dW[g, n, k] == pytest.approx(ref, abs=1e-12)
    assert not dW[1].any()


def test_fp8_tensorwise_scale_overflow_is_clamped():
    # amax = 2^-133 (the smallest bf16 subnormal): 448 / amax overflows fp32, so s is the largest
    # finite fp32, (2 - 2^-23) 2^127; x * s = (2 - 2^-23) 2^-6 rounds up to 2^-5 (code 0x10)
    tiny = 2.0 ** -133
    codes, s = of8.fp8_quantize_tensorwise(np.array([tiny, 0.0, -tiny]))
    assert s == np.finfo(np.float32).max
    assert codes.tolist() == [0x10, 0x00, 0x90]
    # amax = 2^-119 still gives a finite quotient, 448 * 2^119 = 1.75 * 2^127: no clamp
    c2, s2 = of8.fp8_quantize_tensorwise(np.array([2.0 ** -119]))
    assert s2 == np.float32(1.75 * 2.0 ** 127) and c2.tolist() == [0x7E]


def test_fp8_colwise_is_the_group_padded_transpose():
    # brute force on a tiny ragged case: every code of the column-wise operand is the row-wise
    # code of the same element (one tensor scale), pad columns are 0, and the scale is shared
    rng = np.random.default_rng(33)
    lens = np.array([5, 0, 130, 1], dtype=np.int32)
    M, C = int(lens.sum()), 6
    x = rng.standard_normal((M, C))
    codes, s = of8.fp8_quantize_tensorwise(x)
    M_pad = 512
    ct, sc = of8.fp8_quantize_colwise(x, lens, M_pad)
    assert sc == s and ct.shape == (C, M_pad)
    poff = [0, 128, 128, 384, 512]
    off = [0, 5, 5, 135, 136]
    used = np.zeros(M_pad, dtype=bool)
    for g in range(len(lens)):
        for i in range(int(lens[g])):
            used[poff[g] + i] = True
            for c in range(C):
                assert ct[c, poff[g] + i] == codes[off[g] + i, c]
    assert not ct[:, ~used].any()


def test_fp8_swiglu_gemms_lossless_operands():
    # lossless FP8 operands (e4m3 grid values times 2^-6, amax 7: s = 64) make the FP8 SwiGLU
    # GEMMs equal the fp64 BF16-path oracle on the original values, clamp included
    rng = np.random.default_rng(34)
    grid = omx.decode_e4m3(np.arange(0x7F))

    def on_grid(shape):
        v = grid[rng.integers(0, len(grid), size=shape)] * np.where(rng.random(shape) < 0.5, -1, 1) / 64.0
        v.flat[0] = 448.0 / 64.0
        return v

    G, I, K = 2, 3, 5
    lens = np.array([3, 4], dtype=np.int32)
    M = int(lens.sum())
    X, W1 = on_grid((M, K)), on_grid((G * 2 * I, K))
    (cx, sx), (cw, sw) = of8.fp8_quantize_tensorwise(X), of8.fp8_quantize_tensorwise(W1)
    assert sx == sw == np.float32(64.0)
    for limit in (None, 7.0):
        A, H = of8.fp8_grouped_fc1_swiglu(cx, sx, cw, sw, lens, G, limit)
        rA, rH = og.grouped_fc1_swiglu(X, W1.reshape(G, 2 * I, K), lens, limit)
        np.testing.assert_allclose(H, rH, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(A, rA, rtol=1e-13, atol=1e-13)
    dY, W2 = on_grid((M, 4)), on_grid((G * 4, I))
    (cd, sd), (cw2, sw2) = of8.fp8_quantize_tensorwise(dY), of8.fp8_quantize_tensorwise(W2)
    Hs = rng.standard_normal((M, 2 * I))
    dH = of8.fp8_grouped_fc2_dgrad_swiglu_bwd(cd, sd, cw2, sw2, Hs, lens, G, 0.5)
    ref = og.grouped_fc2_dgrad_swiglu_bwd(dY, W2.reshape(G, 4, I), Hs, lens, 0.5)
    np.testing.assert_allclose(dH, ref, rtol=1e-13, atol=1e-13)
    assert (dH == 0).any()                  # the clamp at 0.5 zeroes some gradients
