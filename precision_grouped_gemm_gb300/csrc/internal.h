// Internal host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pgg.h"

namespace pgg {

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  size_t smem_optin = 0;
};

// Returns PGG_OK and fills `info` for the current device (initialising it on first use).
int current_device(DeviceInfo* info);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
// dims/strides in elements/bytes as the driver expects; rank 2 to 5.
int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle);

int cuda_status(cudaError_t e);

// Output map of a wgrad dW [G, N, K] bf16: the 4-D view {64, N, K/64, G} with
// `atoms` 32 x 64 atoms per store when K % 64 == 0 and the driver accepts it
// (*four_d = 1), else the 3-D {K, N, G} view with 32 x 64 boxes.
int encode_wgrad_out(CUtensorMap* map, void* out, int64_t N, int64_t K, int G, int atoms, int* four_d);

// Reduce-add map of an fp32 wgrad accumulator [G, N, K]: the 4-D view {32, N, K/32, G}
// (*four_d = 1) when K % 32 == 0 and accepted, else the 3-D view {K, N, G}.
int encode_wgrad_accum_f32(CUtensorMap* map, void* out, int64_t N, int64_t K, int G, int* four_d);

// BF16 grouped GEMM family (gemm_bf16.cu)
struct Bf16Call {
  int mode;      // 0 fwd, 1 dgrad, 2 wgrad
  int epi;       // 0 store, 1 swiglu fwd, 2 swiglu bwd, 3 fp32 accumulate (wgrad)
  const void* a; // fwd: X; dgrad: dY; wgrad: dY
  const void* b; // fwd/dgrad: W; wgrad: X
  const int32_t* group_lens;
  void* out;
  void* out2;
  const void* aux;
  int64_t M, N, K;  // fwd: Y[M,N]=X[M,K]W^T; dgrad: dX[M,K]=dY[M,N]W; wgrad: dW[G,N,K]
  int64_t I;        // SwiGLU width
  int G;
  int32_t* err;
  cudaStream_t stream;
  float limit = 0.0f;  // SwiGLU clamp limit (0: none)
  unsigned long long wait_ns = 0;  // pipeline wait limit (0: the kernels' default)
  long long stall_at = -1;         // test hook: producer stops before this k-block (-1: never)
};
int launch_bf16(const Bf16Call& c);

// MX quantize (mx_quant.cu)
int launch_mx_quantize_rowwise(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                               uint8_t* scales, cudaStream_t s);
int launch_mx_quantize_rowwise_blocked(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                                       uint8_t* scales, cudaStream_t s);
int launch_mx_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens,
                               int G, int fmt, uint8_t* codes_t, uint8_t* scales_t,
                               int64_t M_pad, int32_t* err, cudaStream_t s);

// Block-scaled grouped GEMM (gemm_mx.cu)
struct MxCall {
  int mode, fmt, epi;
  const uint8_t *A, *SA, *B, *SB;
  const void* H;
  const int32_t* group_lens;
  void* out;
  void* out2;
  uint8_t* q_codes;   // fused row-wise MX output of `out` (SwiGLU epilogues) or nullptr
  uint8_t* q_scales;
  int64_t M, N, K, M_pad;
  int G;
  int32_t* err;
  cudaStream_t stream;
  float limit = 0.0f;  // SwiGLU clamp limit (0: none)
  // FP8 tensor-wise operands (e4m3, plain FP8 MMAs): device fp32 scales s_A, s_B; SA, SB unused
  const float* ts_a = nullptr;
  const float* ts_b = nullptr;
  unsigned long long wait_ns = 0;  // pipeline wait limit (0: the kernels' default)
  long long stall_at = -1;         // test hook: producer stops before this k-block (-1: never)
};
int launch_mx_gemm(const MxCall& c);


// FP8 tensor-wise current scaling (mx_quant.cu): amax_scale = device float[2] {s, amax}
int launch_fp8_tensor_scale(const void* in, int64_t n, float* amax_scale, cudaStream_t s);
int launch_fp8_quantize_rowwise(const void* in, int64_t n, const float* amax_scale, uint8_t* codes,
                                cudaStream_t s);
int launch_fp8_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens, int G,
                                const float* amax_scale, uint8_t* codes_t, int64_t M_pad, int32_t* err,
                                cudaStream_t s);

// MoE glue (moe_glue.cu)
size_t moe_permute_ws_bytes(int64_t T, int E);
int launch_moe_permute(const int32_t* ids, const void* X, int64_t T, int k, int64_t H, int E, void* Xs,
                       int32_t* group_lens, int32_t* pos, int32_t* ws, int32_t* err, cudaStream_t s);
int launch_moe_combine(const void* Ys, const int32_t* pos, const float* w, int64_t T, int k, int64_t H,
                       void* out, cudaStream_t s);
int launch_moe_combine_bwd(const void* dOut, const void* Ys, const int32_t* pos, const float* w, int64_t T, int k,
                           int64_t H, void* dYs, float* dw, cudaStream_t s);

}  // namespace pgg
