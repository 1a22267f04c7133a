"""GB300-native MoE expert grouped GEMM (sm_103a tcgen05 kernels behind a C ABI).

The Python functions below carry the C entry points' names (without the
`pgg_` prefix) and only marshal arguments: torch tensors supply device
pointers, the current CUDA stream is passed through, and a non-zero status
raises PggError.  Every step of the computation runs in libpgg.so's kernels;
there is no fallback path.
"""
from ._binding import (PggError, PAD, FMT_E4M3, FMT_E2M1, MODE_FWD, MODE_DGRAD, MODE_WGRAD,
                       EPI_NONE, EPI_SWIGLU, lib, library_path, init, version, read_error,
                       grouped_gemm_fwd, grouped_gemm_dgrad, grouped_gemm_wgrad,
                       grouped_gemm_wgrad_accumulate,
                       grouped_fc1_swiglu, grouped_fc2_dgrad_swiglu_bwd,
                       mx_quantize_rowwise, mx_quantize_rowwise_blocked, mx_quantize_colwise, mx_grouped_gemm,
                       mx_pad_rows,
                       fp8_tensor_scale, fp8_quantize_rowwise, fp8_quantize_colwise, fp8_workspace_size,
                       fp8_grouped_gemm,
                       moe_permute_workspace_size, moe_permute, moe_combine, moe_combine_bwd)

__all__ = [
    "PggError", "PAD", "FMT_E4M3", "FMT_E2M1", "MODE_FWD", "MODE_DGRAD", "MODE_WGRAD",
    "EPI_NONE", "EPI_SWIGLU", "lib", "library_path", "init", "version", "read_error",
    "grouped_gemm_fwd", "grouped_gemm_dgrad", "grouped_gemm_wgrad", "grouped_gemm_wgrad_accumulate",
    "grouped_fc1_swiglu",
    "grouped_fc2_dgrad_swiglu_bwd", "mx_quantize_rowwise", "mx_quantize_rowwise_blocked", "mx_quantize_colwise",
    "mx_grouped_gemm", "mx_pad_rows", "fp8_tensor_scale", "fp8_quantize_rowwise", "fp8_quantize_colwise",
    "fp8_workspace_size", "fp8_grouped_gemm", "moe_permute_workspace_size", "moe_permute", "moe_combine",
    "moe_combine_bwd",
]
