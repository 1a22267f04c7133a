"""Shared helpers for the tests: seeded inputs, bf16 <-> numpy, tolerance check."""
import numpy as np
import torch

from oracle import grouped_gemm as og
from precision_grouped_gemm_gb300 import workloads as wl


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> exact fp64 values, decoded by the oracle's own decoder."""
    return og.bf16_to_f64(bits(t))


def gen(key, nrows, cols, std=1.0, seed=0, device="cpu", row0=0):
    return wl.gen_matrix(key, nrows, cols, std, seed, device=device, row0=row0)


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str = "", rel: float = 1e-2, abs_rms: float = 1e-2,
                 extra=None):
    """|got - ref| <= rel |ref| + abs_rms rms(ref) [+ extra] per element (bf16 output vs fp64 oracle).

    The default (1e-2, 1e-2) is the stated bound for bf16 outputs; `extra` is an
    optional per-element allowance (the propagated rounding of a bf16 intermediate)."""
    g = f64(got) if got.dtype == torch.bfloat16 else got.detach().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64).reshape(g.shape)
    if extra is None:
        ok, ratio = og.within_tol(g, ref, rel, abs_rms)
    else:
        bound = rel * np.abs(ref) + abs_rms * og.rms(ref) + np.asarray(extra).reshape(g.shape)
        err = np.abs(g - ref)
        ok = bool(np.all(err <= bound))
        ratio = float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0
    if not ok:
        bound = rel * np.abs(ref) + abs_rms * og.rms(ref) + (0 if extra is None else np.asarray(extra).reshape(g.shape))
        i = np.unravel_index(np.argmax(np.abs(g - ref) / np.maximum(bound, 1e-300)), g.shape)
        raise AssertionError(f"{what}: tolerance exceeded, worst err/bound = {ratio:.3g} at {i}: "
                             f"got {g[i]!r} ref {ref[i]!r} bound {bound[i]:.3g} rms {og.rms(ref):.3g}")
    return ratio


def _blocked_index(C: int, M_pad: int) -> np.ndarray:
    """Byte position in the blocked scale layout of column-wise scale (row r, 32-block j):
    atom (r // 128, j // 4) at ((r // 128) * M_pad / 128 + j // 4) * 512, and inside it
    byte 16 (m % 32) + 4 (m // 32) + j % 4 with m = r % 128."""
    r = np.arange(C)[:, None]
    j = np.arange(M_pad // 32)[None, :]
    m = r % 128
    return ((r // 128) * (M_pad // 128) + j // 4) * 512 + 16 * (m % 32) + 4 * (m // 32) + j % 4


def block_scales(s: np.ndarray, M_pad: int) -> np.ndarray:
    """Row-major column-wise scales [C, M_pad/32] -> the blocked layout [round_up(C,128), M_pad/32]."""
    C = s.shape[0]
    out = np.zeros(-(-C // 128) * 128 * (M_pad // 32), dtype=np.uint8)
    out[_blocked_index(C, M_pad)] = s
    return out.reshape(-1, M_pad // 32)


def unblock_scales(b, C: int, M_pad: int) -> np.ndarray:
    """The blocked layout (any shape, tensor or array) -> row-major [C, M_pad/32]; also
    checks that the rows past C are zero."""
    flat = (b.detach().cpu().numpy() if isinstance(b, torch.Tensor) else np.asarray(b)).reshape(-1)
    idx = _blocked_index(C, M_pad)
    pad = np.ones(flat.size, dtype=bool)
    pad[idx.reshape(-1)] = False
    assert not flat[pad].any(), "blocked scales: rows past C must hold scale 0"
    return flat[idx]
