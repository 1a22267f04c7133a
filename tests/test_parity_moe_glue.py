"""GPU MoE glue (permute / combine / combine backward) vs the oracle.

Positions and group_lens are integers: bit-exact.  The permuted rows are
copies: bit-exact.  The combine and its backward round to bf16 (dw stays fp32):
the stated bf16 bound."""
import numpy as np
import pytest
import torch

from oracle import grouped_gemm as og
from oracle import moe_glue as mg
from precision_grouped_gemm_gb300 import workloads as wl
import util

pgg = pytest.importorskip("precision_grouped_gemm_gb300")
pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ids(T, k, E, seed, distinct=True, skew=0.0):
    """Seeded [T, k] expert ids: distinct per token (top-k) or drawn with repeats; skew > 0
    concentrates tokens on low expert ids (leaves high ones empty)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    p = (np.arange(1, E + 1, dtype=np.float64)) ** -skew
    p /= p.sum()
    if distinct:
        keys = np.log(p)[None, :] - np.log(-np.log(rng.random((T, E))))
        return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    return rng.choice(E, size=(T, k), p=p).astype(np.int32)


def _weights(T, k, seed):
    return wl.gen_f32(wl.KEY_LOGITS, torch.arange(T), k, 1.0, seed + 7).abs().contiguous()


def _check_permute(ids, E, H, seed):
    T, k = ids.shape
    X = util.gen(wl.KEY_X, T, H, 1.0, seed) if H else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    Xs, lens, pos = pgg.moe_permute(torch.from_numpy(ids).to(DEV), None if X is None else X.to(DEV), E, err=err)
    assert pgg.read_error(err) == 0
    rpos, rlens, _ = mg.permute(ids, E)
    np.testing.assert_array_equal(lens.cpu().numpy(), rlens)
    np.testing.assert_array_equal(pos.cpu().numpy(), rpos)
    if X is not None:
        np.testing.assert_array_equal(util.bits(Xs), mg.permute_rows(util.bits(X), rpos))
    return X, pos, rpos


@pytest.mark.parametrize("T,k,E,H,distinct,skew", [
    (100, 3, 7, 72, True, 0.0),        # ragged last chunk (100 = 3 x 32 + 4), H not a multiple of 256
    (257, 6, 64, 520, True, 1.2),      # skewed: high experts empty
    (64, 1, 4, 8, True, 0.0),          # top-1, minimal H
    (33, 4, 5, 64, False, 0.0),        # repeated experts within a token
    (1, 8, 16, 128, True, 0.0),        # a single token
    (500, 32, 1024, 16, True, 0.5),    # the largest k and E
    (96, 2, 3, 0, True, 0.0),          # routing only (no rows)
])
def test_permute(T, k, E, H, distinct, skew):
    _check_permute(_ids(T, k, E, T + E, distinct, skew), E, H, T)


def test_permute_empty_batch():
    ids = torch.empty((0, 4), dtype=torch.int32, device=DEV)
    lens = torch.full((9,), 77, dtype=torch.int32, device=DEV)
    pgg.moe_permute(ids, torch.empty((0, 64), dtype=torch.bfloat16, device=DEV), 9, group_lens=lens)
    assert torch.equal(lens.cpu(), torch.zeros(9, dtype=torch.int32))


def test_permute_bad_expert_id_is_flagged():
    ids = _ids(70, 4, 8, 3)
    ids[40, 2] = 8                                   # out of range: flagged, not counted, not copied
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    X = util.gen(wl.KEY_X, 70, 32, 1.0, 3).to(DEV)
    _, lens, pos = pgg.moe_permute(torch.from_numpy(ids).to(DEV), X, 8, err=err)
    assert pgg.read_error(err) == 19
    assert int(lens.sum()) == 70 * 4 - 1
    p = pos.cpu().numpy()
    assert p[40, 2] == -1
    good = p[p >= 0]
    np.testing.assert_array_equal(np.sort(good), np.arange(70 * 4 - 1))


def test_permute_matches_workload_layout():
    # the DeepSeek-shaped routing: permute gives the layer's group_lens and row order
    w = wl.DSV4_BF16
    lens, row_token = w.group_lens()
    ids = w.topk_ids().astype(np.int32)
    X = util.gen(wl.KEY_X, w.tokens, w.hidden, 1.0, w.seed).to(DEV)
    Xs, glens, pos = pgg.moe_permute(torch.from_numpy(ids).to(DEV), X, w.experts)
    np.testing.assert_array_equal(glens.cpu().numpy(), lens)
    rpos, _, rtok = mg.permute(ids, w.experts)
    np.testing.assert_array_equal(pos.cpu().numpy(), rpos)
    np.testing.assert_array_equal(rtok, row_token)
    rows = np.random.Generator(np.random.PCG64(5)).choice(len(row_token), 64, replace=False)
    for r in rows:
        assert torch.equal(Xs[r], X[int(row_token[r])]), f"row {r}"


@pytest.mark.parametrize("T,k,H,weighted", [(100, 3, 72, True), (257, 6, 520, True), (64, 1, 8, False),
                                            (33, 4, 4096, True)])
def test_combine_and_backward(T, k, H, weighted):
    E = 11
    ids = _ids(T, k, E, T * 3, distinct=k <= E)
    rpos, _, _ = mg.permute(ids, E)
    R = T * k
    Ys = util.gen(wl.KEY_H, R, H, 1.0, T)
    dOut = util.gen(wl.KEY_DY, T, H, 1.0, T)
    w = _weights(T, k, T) if weighted else None
    pos = torch.from_numpy(rpos.astype(np.int32)).to(DEV)
    out = pgg.moe_combine(Ys.to(DEV), pos, None if w is None else w.to(DEV))
    ys = util.f64(Ys)
    ref = mg.combine(ys, rpos, None if w is None else w.double().numpy())
    util.assert_close(out, ref, "combine")
    wb = w if w is not None else torch.ones((T, k), dtype=torch.float32)
    dYs, dw = pgg.moe_combine_bwd(dOut.to(DEV), Ys.to(DEV), pos, wb.to(DEV))
    rdYs, rdw = mg.combine_bwd(util.f64(dOut), ys, rpos, wb.double().numpy())
    util.assert_close(dYs, rdYs, "combine bwd dYs")
    util.assert_close(dw, rdw, "combine bwd dw")
    # deterministic: a second call gives the same bits
    dYs2, dw2 = pgg.moe_combine_bwd(dOut.to(DEV), Ys.to(DEV), pos, wb.to(DEV))
    assert torch.equal(dYs, dYs2) and torch.equal(dw, dw2)


def test_combine_skips_dropped_entries():
    T, k, H = 40, 2, 64
    rpos, _, _ = mg.permute(_ids(T, k, 5, 1), 5)
    p = rpos.astype(np.int32).copy()
    p[7, 1] = -1
    Ys = util.gen(wl.KEY_H, T * k, H, 1.0, 2)
    out = pgg.moe_combine(Ys.to(DEV), torch.from_numpy(p).to(DEV))
    ys = util.f64(Ys)
    ref = ys[rpos[:, 0]] + ys[rpos[:, 1]]
    ref[7] = ys[rpos[7, 0]]
    util.assert_close(out, ref, "combine with a dropped entry")


def test_permute_gemm_combine_chain():
    # route -> permute -> grouped GEMM forward -> weighted combine, against the oracle composition
    T, k, E, K, N = 300, 4, 9, 256, 192
    ids = _ids(T, k, E, 9, skew=0.8)
    X = util.gen(wl.KEY_X, T, K, 1.0, 9)
    W = util.gen(wl.KEY_W1, E * N, K, 0.05, 9).view(E, N, K)
    w = _weights(T, k, 9)
    Xs, lens, pos = pgg.moe_permute(torch.from_numpy(ids).to(DEV), X.to(DEV), E)
    Ys = pgg.grouped_gemm_fwd(Xs, W.to(DEV), lens)
    out = pgg.moe_combine(Ys, pos, w.to(DEV))
    rpos, rlens, _ = mg.permute(ids, E)
    xs = mg.permute_rows(util.f64(X), rpos)
    ys = og.grouped_gemm_fwd(xs, util.f64(W), rlens)
    # Ys is rounded to bf16 before the combine: allow its propagated rounding
    extra = 2.0 ** -8 * mg.combine(np.abs(ys), rpos, w.double().numpy())
    util.assert_close(out, mg.combine(ys, rpos, w.double().numpy()), "permute-gemm-combine", extra=extra)


def test_combine_full_size_sample():
    # the DeepSeek-shaped routing at full size: 4096 tokens, top-6 of 256 experts, hidden 4096;
    # sampled tokens checked against the oracle, combine and its backward
    w = wl.DSV4_BF16
    T, k, E, H = w.tokens, w.topk, w.experts, w.hidden
    rpos, _, _ = mg.permute(w.topk_ids(), E)
    pos = torch.from_numpy(rpos.astype(np.int32)).to(DEV)
    Ys = wl.gen_matrix(wl.KEY_H, T * k, H, 1.0, w.seed, device=DEV)
    dOut = wl.gen_matrix(wl.KEY_DY, T, H, 1.0, w.seed, device=DEV)
    wts = _weights(T, k, w.seed).to(DEV)
    out = pgg.moe_combine(Ys, pos, wts)
    dYs, dw = pgg.moe_combine_bwd(dOut, Ys, pos, wts)
    torch.cuda.synchronize()
    toks = np.random.Generator(np.random.PCG64(6)).choice(T, 48, replace=False)
    for t in toks:
        rows = rpos[t]
        ys = util.f64(Ys[torch.from_numpy(rows.astype(np.int64)).to(DEV)])
        wt = wts[t].double().cpu().numpy()
        util.assert_close(out[t], mg.combine(ys, np.arange(k)[None, :], wt[None, :])[0], f"combine token {t}")
        g = util.f64(dOut[t:t + 1])
        rdys, rdw = mg.combine_bwd(g, ys, np.arange(k)[None, :], wt[None, :])
        util.assert_close(dYs[torch.from_numpy(rows.astype(np.int64)).to(DEV)], rdys, f"combine bwd dYs token {t}")
        util.assert_close(dw[t], rdw[0], f"combine bwd dw token {t}")
