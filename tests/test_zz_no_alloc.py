"""pgg_moe_permute_noalloc (fixed module scratch, no caller workspace) against
pgg_moe_permute (caller workspace), both called through the C ABI, and against
the oracle's stable expert sort (positions, group_lens and the gathered rows,
bit for bit).

The file name sorts last so that it runs after every other test: it must pass
both alone and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_glue as omg
from precision_grouped_gemm_gb300 import _binding
from precision_grouped_gemm_gb300 import workloads as wl
import util

PGG_ERR_TOO_LARGE = 6
MAX_WS_INTS = 1 << 20
DEV = "cuda"


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ids(T, k, E, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    keys = -np.log(-np.log(rng.random((T, E))))
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def test_noalloc_rejects_beyond_its_scratch():
    # validation happens before any CUDA call, so this also runs without a GPU
    L = _binding.lib()
    g = ctypes.c_void_p(1 << 20)
    T, E = 32 * (MAX_WS_INTS // 1024) + 1, 1024          # ceil(T / 32) * E = MAX + 1024
    assert L.pgg_moe_permute_noalloc(g, g, T, 4, 64, E, g, g, g, None, None) == PGG_ERR_TOO_LARGE
    assert b"scratch" in L.pgg_status_string(PGG_ERR_TOO_LARGE)


def _permute_both(ids_np, E, H, seed):
    L = _binding.lib()
    T, k = ids_np.shape
    ids = torch.from_numpy(ids_np).to(DEV)
    X = util.gen(wl.KEY_X, T, H, 1.0, seed).to(DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the workspace entry point: its own scratch table from the caller
    ws = torch.empty(max(1, L.pgg_moe_permute_workspace_size(T, E) // 4), dtype=torch.int32, device=DEV)
    Xs_ref = torch.zeros((T * k, H), dtype=torch.bfloat16, device=DEV)
    lens_ref = torch.zeros(E, dtype=torch.int32, device=DEV)
    pos_ref = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    err = torch.zeros(2, dtype=torch.int32, device=DEV)
    assert L.pgg_moe_permute(_p(ids), _p(X), T, k, H, E, _p(Xs_ref), _p(lens_ref), _p(pos_ref), _p(ws),
                             ws.numel() * 4, _p(err[:1]), stream) == 0
    outs = []
    for _ in range(2):                                    # two calls in a row reuse the same scratch
        Xs = torch.full((T * k, H), 7.0, dtype=torch.bfloat16, device=DEV)
        lens = torch.full((E,), -1, dtype=torch.int32, device=DEV)
        pos = torch.full((T, k), -5, dtype=torch.int32, device=DEV)
        assert L.pgg_moe_permute_noalloc(_p(ids), _p(X), T, k, H, E, _p(Xs), _p(lens), _p(pos),
                                         _p(err[1:]), stream) == 0
        outs.append((Xs, lens, pos))
    torch.cuda.synchronize()
    assert err.cpu().tolist() == [0, 0]
    M = int(lens_ref.sum())
    o_pos, o_lens, o_row_token = omg.permute(ids_np, E)
    Xb = util.bits(X)
    for Xs, lens, pos in outs:
        assert torch.equal(lens, lens_ref)
        assert torch.equal(pos, pos_ref)
        assert torch.equal(Xs[:M], Xs_ref[:M])
        np.testing.assert_array_equal(lens.cpu().numpy(), o_lens)
        np.testing.assert_array_equal(pos.cpu().numpy(), o_pos)
        np.testing.assert_array_equal(util.bits(Xs[:M]), Xb[o_row_token])


@pytest.mark.gpu
@pytest.mark.parametrize("T,k,E,H", [(100, 3, 7, 72), (4096, 6, 256, 4096), (2049, 8, 1024, 16)])
def test_noalloc_matches_workspace_permute(T, k, E, H):
    assert (T + 31) // 32 * E <= MAX_WS_INTS
    _permute_both(_ids(T, k, E, T + k), E, H, T)


@pytest.mark.gpu
def test_noalloc_at_its_capacity():
    # ceil(T / 32) * E == the stated maximum exactly
    E = 256
    T = 32 * (MAX_WS_INTS // E)
    ids = np.random.Generator(np.random.PCG64(3)).integers(0, E, size=(T, 2), dtype=np.int32)
    _permute_both(ids, E, 8, 3)
