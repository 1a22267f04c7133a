"""fp64 / integer oracle: the single-GPU MoE glue around the grouped GEMM.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs with Primus",
section "Expert parallelism: DeepEP and the grouped GEMM": the token dispatch
permutes tokens into the layout the grouped GEMM wants (rows sorted by expert)
and the combine brings the results back; section "MegaMoE": the second grouped
GEMM is followed by the combine and the weighted reduce.  Without the
communication (one GPU) that is:

* permute: token t's j-th routed expert e = ids[t, j] gets row pos[t, j] of the
  expert-sorted batch; rows are ordered by expert, then by token (a stable
  sort of the flattened (t, j) entries by expert); group_lens[e] = number of
  entries routed to e; Xs[pos[t, j]] = X[t];
* combine: out[t] = sum_j w[t, j] * Ys[pos[t, j]] (w = 1 when no weights);
* combine backward: dYs[pos[t, j]] = w[t, j] * dOut[t] and
  dw[t, j] = <dOut[t], Ys[pos[t, j]]>;
* permute backward: dX[t] = sum_j dXs[pos[t, j]] (the combine with w = 1).
"""
from __future__ import annotations

import numpy as np


def permute(ids: np.ndarray, E: int):
    """ids [T, k] int -> (pos [T, k] int64, group_lens [E] int64, row_token [T*k] int64)."""
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    if np.any(ids < 0) or np.any(ids >= E):
        raise ValueError("expert id out of range")
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")  # entries by expert; ties keep (t, j) order
    pos = np.empty(T * k, dtype=np.int64)
    pos[order] = np.arange(T * k)
    lens = np.bincount(flat, minlength=E).astype(np.int64)
    row_token = order // k
    return pos.reshape(T, k), lens, row_token


def permute_rows(X: np.ndarray, pos: np.ndarray) -> np.ndarray:
    T, k = pos.shape
    Xs = np.zeros((T * k, X.shape[1]), dtype=X.dtype)
    for t in range(T):
        for j in range(k):
            Xs[pos[t, j]] = X[t]
    return Xs


def combine(Ys: np.ndarray, pos: np.ndarray, w=None) -> np.ndarray:
    T, k = pos.shape
    Ys = np.asarray(Ys, dtype=np.float64)
    out = np.zeros((T, Ys.shape[1]), dtype=np.float64)
    for j in range(k):
        wj = 1.0 if w is None else np.asarray(w, dtype=np.float64)[:, j:j + 1]
        out += wj * Ys[pos[:, j]]
    return out


def combine_bwd(dOut: np.ndarray, Ys: np.ndarray, pos: np.ndarray, w: np.ndarray):
    """-> (dYs [T*k, H], dw [T, k])."""
    T, k = pos.shape
    dOut = np.asarray(dOut, dtype=np.float64)
    Ys = np.asarray(Ys, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dYs = np.zeros((T * k, dOut.shape[1]), dtype=np.float64)
    dw = np.zeros((T, k), dtype=np.float64)
    for j in range(k):
        dYs[pos[:, j]] = w[:, j:j + 1] * dOut
        dw[:, j] = np.sum(dOut * Ys[pos[:, j]], axis=1)
    return dYs, dw
