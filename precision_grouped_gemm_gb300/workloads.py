"""Seeded synthetic inputs for the MoE expert grouped GEMM.

This module is the one piece shared by the CUDA path's callers (tests, bench)
and the CPU oracle's callers.  It holds none of the grouped GEMM's arithmetic:
it only draws numbers and routes tokens to experts.

Value generator
---------------
Every tensor element is a pure function of (tensor key, row, column), so any
slice of a multi-GB tensor can be regenerated on its own, on the CPU or on the
GPU, with bit-identical results.  The generator is integer-only up to one final
fp32 multiply and one fp32 -> bf16 round-to-nearest-even:

    mix32(x)  = the "lowbias32" integer hash (xor-shift 16, * 0x7feb352d,
                xor-shift 15, * 0x846ca68b, xor-shift 16), all mod 2^32
    base(r)   = mix32(mix32(key) ^ r)
    h1, h2    = mix32(base(r) ^ mix32(2c)), mix32(base(r) ^ mix32(2c + 1))
    s         = sum of the four 16-bit halves of h1 and h2        (0..262140)
    value     = fp32(s - 131070) * fp32(std / 37837.23)           (one rounding)

s is an Irwin-Hall(4) sum of uniform 16-bit integers, so `value` is close to
N(0, std^2) (variance exact, tails truncated at about 3.46 std).  The same code
runs on a CPU or CUDA torch device; integer ops and a single IEEE fp32 multiply
give the same bits on both.

Routing
-------
Token -> expert choice is made on the host (the group_lens vector is an input
of the grouped GEMM, not part of it):

* softmax top-k: logits from the generator; the top-k of softmax are the top-k
  logits; ties go to the lower expert index (stable sort);
* Zipf: top-k without replacement with p_e proportional to (e+1)^-s, drawn by
  Gumbel-top-k from a numpy PCG64 stream.

Rows are sorted by expert, tokens ascending within an expert, so the
activation of row r is the activation of token `row_token[r]`.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

MASK32 = 0xFFFFFFFF
_IH4_SD = 37837.23  # standard deviation of the sum of four uniform 16-bit integers

# tensor keys: distinct integers per logical tensor
KEY_X, KEY_W1, KEY_W2, KEY_DY, KEY_DA, KEY_H, KEY_LOGITS = 11, 12, 13, 14, 15, 16, 17
KEY_A, KEY_DH = 18, 19


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2^32 for x in [0, 2^32) held in int64, without int64 overflow
    lo = (x * (c & 0xFFFF)) & MASK32
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & MASK32


def mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def gen_f32(key: int, rows: torch.Tensor, cols: int, std: float, seed: int = 0) -> torch.Tensor:
    """fp32 [len(rows), cols] values of tensor `key` at the given row ids."""
    dev = rows.device
    k = mix32(torch.tensor([(key * 1000003 + seed) & MASK32], dtype=torch.int64, device=dev))
    base = mix32(k ^ (rows.to(torch.int64) & MASK32)).view(-1, 1)
    c = torch.arange(cols, dtype=torch.int64, device=dev)
    c1 = mix32(2 * c).view(1, -1)
    c2 = mix32(2 * c + 1).view(1, -1)
    h1 = mix32(base ^ c1)
    h2 = mix32(base ^ c2)
    s = (h1 & 0xFFFF) + (h1 >> 16) + (h2 & 0xFFFF) + (h2 >> 16)
    scale = torch.tensor(std / _IH4_SD, dtype=torch.float32, device=dev)
    return (s - 131070).to(torch.float32) * scale


def gen_bf16(key: int, rows: torch.Tensor, cols: int, std: float, seed: int = 0) -> torch.Tensor:
    return gen_f32(key, rows, cols, std, seed).to(torch.bfloat16)


def gen_matrix(key: int, nrows: int, cols: int, std: float, seed: int = 0,
               device="cpu", row0: int = 0, chunk_rows: int = 1 << 14) -> torch.Tensor:
    """bf16 [nrows, cols] rows row0..row0+nrows-1 of tensor `key`, built in chunks."""
    out = torch.empty((nrows, cols), dtype=torch.bfloat16, device=device)
    for r in range(0, nrows, chunk_rows):
        n = min(chunk_rows, nrows - r)
        rows = torch.arange(row0 + r, row0 + r + n, dtype=torch.int64, device=device)
        out[r:r + n] = gen_bf16(key, rows, cols, std, seed)
    return out


# ----------------------------------------------------------------------------
# routing -> group_lens
# ----------------------------------------------------------------------------

def topk_softmax(T: int, E: int, k: int, seed: int, blocked=()) -> np.ndarray:
    """Top-k expert ids [T, k] of softmax over generator logits [T, E], best first."""
    logits = gen_f32(KEY_LOGITS, torch.arange(T), E, 1.0, seed).numpy().astype(np.float64)
    for e in blocked:
        logits[:, e] = -np.inf
    # stable sort on -logit: equal logits keep ascending expert order
    return np.argsort(-logits, axis=1, kind="stable")[:, :k]


def topk_zipf(T: int, E: int, k: int, s: float, seed: int) -> np.ndarray:
    """Top-k ids [T, k] without replacement, p_e ~ (e+1)^-s, by Gumbel-top-k (numpy PCG64)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    u = rng.random((T, E))
    keys = logp[None, :] - np.log(-np.log(u))
    return np.argsort(-keys, axis=1, kind="stable")[:, :k]


def route_softmax_topk(T: int, E: int, k: int, seed: int, blocked=()) -> tuple[np.ndarray, np.ndarray]:
    """Softmax top-k routing; returns (group_lens[E], row_token[M])."""
    return _rows_from_choice(topk_softmax(T, E, k, seed, blocked), T, E)


def route_zipf(T: int, E: int, k: int, s: float, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """Zipf top-k routing; returns (group_lens[E], row_token[M])."""
    return _rows_from_choice(topk_zipf(T, E, k, s, seed), T, E)


def _rows_from_choice(order: np.ndarray, T: int, E: int):
    tok = np.repeat(np.arange(T), order.shape[1])
    exp = order.reshape(-1)
    perm = np.lexsort((tok, exp))  # by expert, then token
    row_token = tok[perm].astype(np.int64)
    group_lens = np.bincount(exp, minlength=E).astype(np.int32)
    return group_lens, row_token


def lens_tiny(seed: int, G: int = 4, M: int = 512) -> np.ndarray:
    """Multinomial(M, uniform over G-1 groups); group (seed % G) is forced empty."""
    rng = np.random.Generator(np.random.PCG64(seed))
    draw = rng.multinomial(M, [1.0 / (G - 1)] * (G - 1))
    zero = seed % G
    lens = np.zeros(G, dtype=np.int32)
    lens[[g for g in range(G) if g != zero]] = draw
    return lens


# ----------------------------------------------------------------------------
# the workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    fmt: str            # "bf16", "e4m3", "e2m1" (MX block scales) or "fp8" (e4m3, one scale per tensor)
    hidden: int         # K of FC1, N of FC2
    inter: int          # I (FC1 produces 2I = gate | up)
    experts: int
    tokens: int
    topk: int
    seed: int
    routing: str        # "tiny", "softmax", "zipf"
    blocked: tuple = ()
    zipf_s: float = 0.0
    w_std: float = 0.02
    swiglu: bool = True

    def group_lens(self) -> tuple[np.ndarray, np.ndarray]:
        if self.routing == "tiny":
            lens = lens_tiny(self.seed, self.experts, self.tokens)
            return lens, np.arange(int(lens.sum()), dtype=np.int64)
        if self.routing == "softmax":
            return route_softmax_topk(self.tokens, self.experts, self.topk, self.seed, self.blocked)
        if self.routing == "zipf":
            return route_zipf(self.tokens, self.experts, self.topk, self.zipf_s, self.seed)
        raise ValueError(self.routing)

    def topk_ids(self) -> np.ndarray:
        """The routing's expert ids [tokens, topk] (group_lens / row_token are their stable sort)."""
        if self.routing == "softmax":
            return topk_softmax(self.tokens, self.experts, self.topk, self.seed, self.blocked)
        if self.routing == "zipf":
            return topk_zipf(self.tokens, self.experts, self.topk, self.zipf_s, self.seed)
        raise ValueError(f"routing {self.routing!r} has no top-k ids")


def _gptoss_blocked(seed: int, E: int = 32) -> tuple:
    rng = np.random.Generator(np.random.PCG64(seed))
    return tuple(int(e) for e in sorted(rng.choice(E, size=2, replace=False)))


# tiny: one grouped GEMM with K=256, N=512 (no SwiGLU layer); "inter" is N/2
TINY = Workload("tiny_bf16_g4_k256_n512_m512", "bf16", hidden=256, inter=256, experts=4,
                tokens=512, topk=1, seed=0, routing="tiny", w_std=1.0, swiglu=False)
DSV4_BF16 = Workload("dsv4flash_moe_bf16_h4096_e256_top6_t4096_i2048", "bf16", 4096, 2048,
                     256, 4096, 6, seed=1, routing="softmax")
DSV4_MXFP8 = Workload("dsv4flash_moe_mxfp8_h4096_e256_top6_t4096_i2048", "e4m3", 4096, 2048,
                      256, 4096, 6, seed=1, routing="softmax")
GPTOSS_BF16 = Workload("gptoss20b_moe_bf16_h2880_e32_top4_t8192_i2880", "bf16", 2880, 2880,
                       32, 8192, 4, seed=3, routing="softmax", blocked=_gptoss_blocked(3))
ZIPF_MXFP4 = Workload("zipf_moe_mxfp4_h4096_e256_top8_t16384_i2048", "e2m1", 4096, 2048,
                      256, 16384, 8, seed=4, routing="zipf", zipf_s=1.2)
# the DeepSeek-shaped layer in FP8 with one current-scaling scale per tensor
DSV4_FP8 = Workload("dsv4flash_moe_fp8_h4096_e256_top6_t4096_i2048", "fp8", 4096, 2048,
                    256, 4096, 6, seed=1, routing="softmax")

WORKLOADS = {w.name: w for w in (TINY, DSV4_BF16, DSV4_MXFP8, GPTOSS_BF16, ZIPF_MXFP4, DSV4_FP8)}


def layer_flops(lens: np.ndarray, hidden: int, inter: int) -> dict:
    """Algorithmic flops of one MoE expert layer, fwd + dgrad + wgrad, 2*M*N*K each."""
    M = int(lens.sum())
    fc1 = 2.0 * M * (2 * inter) * hidden
    fc2 = 2.0 * M * hidden * inter
    return {"fc1": fc1, "fc2": fc2, "total": 3.0 * (fc1 + fc2)}


def ragged_ok(lens: np.ndarray, tile: int = 128) -> bool:
    nz = lens[lens > 0]
    return bool(np.all(nz % tile != 0))


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


