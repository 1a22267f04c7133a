"""CPU oracle for the variable-size MoE expert grouped GEMM.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package;
only tests, the smoke check and the benchmark's CPU-baseline leg may call it.

A plain, slow, obviously correct fp64 restatement of what the pages define:

* grouped_gemm.py -- group offsets, forward, dgrad, variable-K wgrad, SwiGLU
  forward/backward and the fused FC1 / FC2-dgrad compositions;
* mx.py -- E8M0 / e4m3 / e2m1 decode, MX block quantization (row- and
  group-aware column-wise), dequantization, and the block-scaled grouped GEMM
  as "dequantize, then the fp64 grouped GEMM";
* moe_glue.py -- the single-GPU token permute / combine around the grouped
  GEMM and their backward passes;
* fp8.py -- e4m3 tensor-wise current scaling and the FP8 grouped GEMMs.

It shares no code with the CUDA path and imports nothing from it.  Inputs are
bf16 bit patterns (numpy uint16) or MX byte codes; everything is computed in
fp64.  Every function is pinned by a `-m "not gpu"` test against brute force,
closed forms, invariants or hand-derived format values.
"""
from . import fp8, grouped_gemm, moe_glue, mx  # noqa: F401
