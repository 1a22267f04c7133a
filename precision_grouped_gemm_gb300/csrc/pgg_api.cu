// C ABI of the library: argument validation, device checks, tensor-map
// encoding and dispatch to the kernel launchers.  No entry point allocates
// memory or synchronises (except pgg_read_error, which exists to synchronise).
#include <cstring>
#include <mutex>

#include "internal.h"
#include "sched.cuh"

namespace pgg {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PGG_OK : PGG_ERR_CUDA; }

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int init_device(int device) {
  if (device < 0 || device >= kMaxDevices) return PGG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[device];
  if (d.device == device) return PGG_OK;
  cudaDeviceProp p;
  if (cudaGetDeviceProperties(&p, device) != cudaSuccess) return PGG_ERR_CUDA;
  if (!(p.major == 10 && p.minor == 3)) return PGG_ERR_UNSUPPORTED;
  d.sms = p.multiProcessorCount;
  d.cc_major = p.major;
  d.cc_minor = p.minor;
  d.smem_optin = p.sharedMemPerBlockOptin;
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return PGG_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  d.device = device;
  return PGG_OK;
}
}  // namespace

int current_device(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PGG_ERR_CUDA;
  int st = init_device(dev);
  if (st != PGG_OK) return st;
  *info = g_dev[dev];
  return PGG_OK;
}

int encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle) {
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  CUresult r = g_encode(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PGG_OK : PGG_ERR_INVALID_ARG;
}

int encode_wgrad_out(CUtensorMap* map, void* out, int64_t N, int64_t K, int G, int atoms, int* four_d) {
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (K % 64 == 0) {
    // 4-D view {64, N, K/64, G}: one bulk store moves `atoms` 32-row x 64-column atoms
    uint64_t d[4] = {64, (uint64_t)N, (uint64_t)(K / 64), (uint64_t)G};
    uint64_t s[3] = {(uint64_t)K * 2, 128, (uint64_t)(N * K * 2)};
    uint32_t b[4] = {64, 32, (uint32_t)atoms, 1};
    if (encode_tmap(map, bf, 4, out, d, s, b, sw) == PGG_OK) {
      *four_d = 1;
      return PGG_OK;
    }
  }
  // 3-D view {K, N, G}: stores of 32 x 64 boxes
  uint64_t d[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G};
  uint64_t s[2] = {(uint64_t)K * 2, (uint64_t)(N * K * 2)};
  uint32_t b[3] = {64, 32, 1};
  *four_d = 0;
  return encode_tmap(map, bf, 3, out, d, s, b, sw);
}

int encode_wgrad_accum_f32(CUtensorMap* map, void* out, int64_t N, int64_t K, int G, int* four_d) {
  const auto f32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  if (K % 32 == 0) {
    // 4-D view {32, N, K/32, G}: one reduce-add covers 32 rows x 64 fp32 columns
    uint64_t d[4] = {32, (uint64_t)N, (uint64_t)(K / 32), (uint64_t)G};
    uint64_t s[3] = {(uint64_t)K * 4, 128, (uint64_t)(N * K * 4)};
    uint32_t b[4] = {32, 32, 2, 1};
    if (encode_tmap(map, f32, 4, out, d, s, b, sw) == PGG_OK) {
      *four_d = 1;
      return PGG_OK;
    }
  }
  uint64_t d[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G};
  uint64_t s[2] = {(uint64_t)K * 4, (uint64_t)(N * K * 4)};
  uint32_t b[3] = {32, 32, 1};
  *four_d = 0;
  return encode_tmap(map, f32, 3, out, d, s, b, sw);
}

}  // namespace pgg

using namespace pgg;

namespace {
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
constexpr int64_t kMaxRows = (int64_t)1 << 31;

int check_common(int64_t M, int G, const int32_t* lens) {
  if (G < 1 || G > kMaxGroups) return PGG_ERR_INVALID_ARG;
  if (M < 0 || M >= kMaxRows) return PGG_ERR_INVALID_ARG;
  if (!lens) return PGG_ERR_INVALID_ARG;
  if (!aligned4(lens)) return PGG_ERR_ALIGNMENT;
  return PGG_OK;
}

int check_dim(int64_t x, int mult) {
  if (x < mult || x >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (x % mult) return PGG_ERR_ALIGNMENT;
  return PGG_OK;
}
}  // namespace

static int mx_gemm_impl(int mode, int fmt, int epilogue, const uint8_t* A, const uint8_t* SA,
                        const uint8_t* B, const uint8_t* SB, const void* H,
                        const int32_t* group_lens, void* out, void* out2, uint8_t* out_codes,
                        uint8_t* out_scales, int64_t M, int64_t N, int64_t K, int G, int64_t M_pad,
                        float limit, int32_t* err, void* stream, const float* ts_a = nullptr,
                        const float* ts_b = nullptr, unsigned long long wait_ns = 0, long long stall_at = -1) {
  int st;
  if (mode < 0 || mode > 2) return PGG_ERR_INVALID_ARG;
  if (fmt != PGG_FMT_E4M3 && fmt != PGG_FMT_E2M1) return PGG_ERR_INVALID_ARG;
  if (epilogue != PGG_EPI_NONE && epilogue != PGG_EPI_SWIGLU) return PGG_ERR_INVALID_ARG;
  if (epilogue == PGG_EPI_SWIGLU && mode == PGG_MODE_WGRAD) return PGG_ERR_INVALID_ARG;
  if ((st = check_common(M, G, group_lens))) return st;
  const bool block_scaled = ts_a == nullptr;  // else FP8 tensor-wise: no scale factors
  if (!A || !B || !out || (block_scaled && (!SA || !SB))) return PGG_ERR_INVALID_ARG;
  if (mode == PGG_MODE_DGRAD && epilogue == PGG_EPI_SWIGLU && !H) return PGG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out) || (out2 && !aligned16(out2)) ||
      (H && !aligned16(H)))
    return PGG_ERR_ALIGNMENT;
  // blocked scale atoms (SB always, wgrad SA) are fetched by 16-byte-aligned bulk copies,
  // row-major scales (fwd / dgrad SA) by 4-byte copies
  if (block_scaled && ((mode == PGG_MODE_WGRAD && !aligned16(SA)) || !aligned4(SA) || !aligned16(SB)))
    return PGG_ERR_ALIGNMENT;
  if (err && !aligned4(err)) return PGG_ERR_ALIGNMENT;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (mode == PGG_MODE_FWD && (K % 128 || (epilogue == PGG_EPI_SWIGLU && N % 16)))
    return PGG_ERR_ALIGNMENT;
  if (mode == PGG_MODE_DGRAD && N % 128) return PGG_ERR_ALIGNMENT;
  if (mode == PGG_MODE_WGRAD && (M_pad <= 0 || M_pad % PGG_MX_PAD || M_pad >= kMaxRows))
    return PGG_ERR_ALIGNMENT;
  if ((out_codes != nullptr) != (out_scales != nullptr)) return PGG_ERR_INVALID_ARG;
  if (out_codes) {
    // fused row-wise MX output of `out`: SwiGLU epilogues only, whole 32-column blocks
    const int64_t w = mode == PGG_MODE_FWD ? N / 2 : K;
    if (epilogue != PGG_EPI_SWIGLU) return PGG_ERR_INVALID_ARG;
    if (w % 32) return PGG_ERR_ALIGNMENT;
    if (!aligned16(out_codes)) return PGG_ERR_ALIGNMENT;
  }
  if (M == 0 && mode != PGG_MODE_WGRAD) return PGG_OK;
  MxCall c{mode, fmt, epilogue, A, SA, B, SB, H, group_lens, out, out2, out_codes, out_scales,
           M, N, K, M_pad, G, err, as_stream(stream)};
  c.limit = limit;
  c.ts_a = ts_a;
  c.ts_b = ts_b;
  c.wait_ns = wait_ns;
  c.stall_at = stall_at;
  return launch_mx_gemm(c);
}

extern "C" {

int pgg_version(void) { return 101; }

int pgg_init(int device) {
  if (cudaSetDevice(device) != cudaSuccess) return PGG_ERR_CUDA;
  DeviceInfo d;
  return current_device(&d);
}

const char* pgg_status_string(int s) {
  switch (s) {
    case PGG_OK: return "ok";
    case PGG_ERR_INVALID_ARG: return "invalid argument";
    case PGG_ERR_UNSUPPORTED: return "unsupported device or shape";
    case PGG_ERR_ALIGNMENT: return "misaligned pointer or dimension";
    case PGG_ERR_NOT_INITIALIZED: return "not initialized";
    case PGG_ERR_CUDA: return "CUDA runtime error";
    case PGG_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of a no-alloc entry point";
    case PGG_ERR_BAD_GROUP_LENS: return "bad group_lens (negative length or sum != M)";
    case PGG_ERR_TIMEOUT: return "bounded pipeline wait expired";
    case PGG_ERR_PAD_OVERFLOW: return "padded column-wise layout exceeds M_pad";
    case PGG_ERR_BAD_EXPERT: return "expert id out of range";
    default: return "unknown status";
  }
}

int pgg_read_error(const int32_t* err_dev, int32_t* host_out, void* stream) {
  if (!err_dev || !host_out) return PGG_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(host_out, err_dev, sizeof(int32_t), cudaMemcpyDeviceToHost,
                      as_stream(stream)) != cudaSuccess)
    return PGG_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(as_stream(stream)));
}

int pgg_grouped_gemm_fwd(const void* X, const void* W, const int32_t* group_lens, void* Y,
                         int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream) {
  int st;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (M == 0) return PGG_OK;
  if (!X || !W || !Y) return PGG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W) || !aligned16(Y)) return PGG_ERR_ALIGNMENT;
  Bf16Call c{0, 0, X, W, group_lens, Y, nullptr, nullptr, M, N, K, 0, G, err, as_stream(stream)};
  return launch_bf16(c);
}

int pgg_grouped_gemm_dgrad(const void* dY, const void* W, const int32_t* group_lens, void* dX,
                           int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream) {
  int st;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (M == 0) return PGG_OK;
  if (!dY || !W || !dX) return PGG_ERR_INVALID_ARG;
  if (!aligned16(dY) || !aligned16(W) || !aligned16(dX)) return PGG_ERR_ALIGNMENT;
  Bf16Call c{1, 0, dY, W, group_lens, dX, nullptr, nullptr, M, N, K, 0, G, err, as_stream(stream)};
  return launch_bf16(c);
}

int pgg_grouped_gemm_wgrad(const void* X, const void* dY, const int32_t* group_lens, void* dW,
                           int64_t M, int64_t N, int64_t K, int G, int32_t* err, void* stream) {
  int st;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (!dW || !aligned16(dW)) return dW ? PGG_ERR_ALIGNMENT : PGG_ERR_INVALID_ARG;
  if (M == 0) {  // every group is empty: dW = 0
    return cuda_status(cudaMemsetAsync(dW, 0, (size_t)G * N * K * 2, as_stream(stream)));
  }
  if (!X || !dY) return PGG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(dY)) return PGG_ERR_ALIGNMENT;
  Bf16Call c{2, 0, dY, X, group_lens, dW, nullptr, nullptr, M, N, K, 0, G, err, as_stream(stream)};
  return launch_bf16(c);
}

int pgg_grouped_gemm_wgrad_accumulate(const void* X, const void* dY, const int32_t* group_lens,
                                      float* dW_f32, int64_t M, int64_t N, int64_t K, int G, int32_t* err,
                                      void* stream) {
  int st;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (!dW_f32) return PGG_ERR_INVALID_ARG;
  if (!aligned16(dW_f32)) return PGG_ERR_ALIGNMENT;
  if (M == 0) return PGG_OK;  // every group is empty: nothing to add
  if (!X || !dY) return PGG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(dY)) return PGG_ERR_ALIGNMENT;
  Bf16Call c{2, 3, dY, X, group_lens, dW_f32, nullptr, nullptr, M, N, K, 0, G, err, as_stream(stream)};
  return launch_bf16(c);
}

int pgg_grouped_fc1_swiglu(const void* X, const void* W1, const int32_t* group_lens, void* A,
                           void* H, int64_t M, int64_t I, int64_t K, int G, int32_t* err,
                           void* stream) {
  return pgg_grouped_fc1_swiglu_clamped(X, W1, group_lens, A, H, M, I, K, G, 0.0f, err, stream);
}

int pgg_grouped_fc1_swiglu_clamped(const void* X, const void* W1, const int32_t* group_lens, void* A,
                                   void* H, int64_t M, int64_t I, int64_t K, int G, float swiglu_limit,
                                   int32_t* err, void* stream) {
  int st;
  if (!(swiglu_limit >= 0.0f) || swiglu_limit > 3.0e38f) return PGG_ERR_INVALID_ARG;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(I, 8)) || (st = check_dim(K, 8))) return st;
  if (M == 0) return PGG_OK;
  if (!X || !W1 || !A) return PGG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(W1) || !aligned16(A) || (H && !aligned16(H)))
    return PGG_ERR_ALIGNMENT;
  Bf16Call c{0, 1, X, W1, group_lens, A, H, nullptr, M, 2 * I, K, I, G, err, as_stream(stream)};
  c.limit = swiglu_limit;
  return launch_bf16(c);
}

int pgg_grouped_fc2_dgrad_swiglu_bwd(const void* dY, const void* W2, const void* H,
                                     const int32_t* group_lens, void* dH, int64_t M, int64_t Hd,
                                     int64_t I, int G, int32_t* err, void* stream) {
  return pgg_grouped_fc2_dgrad_swiglu_bwd_clamped(dY, W2, H, group_lens, dH, M, Hd, I, G, 0.0f, err, stream);
}

int pgg_grouped_fc2_dgrad_swiglu_bwd_clamped(const void* dY, const void* W2, const void* H,
                                             const int32_t* group_lens, void* dH, int64_t M, int64_t Hd,
                                             int64_t I, int G, float swiglu_limit, int32_t* err,
                                             void* stream) {
  int st;
  if (!(swiglu_limit >= 0.0f) || swiglu_limit > 3.0e38f) return PGG_ERR_INVALID_ARG;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(Hd, 8)) || (st = check_dim(I, 8))) return st;
  if (M == 0) return PGG_OK;
  if (!dY || !W2 || !H || !dH) return PGG_ERR_INVALID_ARG;
  if (!aligned16(dY) || !aligned16(W2) || !aligned16(H) || !aligned16(dH))
    return PGG_ERR_ALIGNMENT;
  Bf16Call c{1, 2, dY, W2, group_lens, dH, nullptr, H, M, Hd, I, I, G, err, as_stream(stream)};
  c.limit = swiglu_limit;
  return launch_bf16(c);
}

int pgg_mx_quantize_rowwise(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                            uint8_t* scales, void* stream) {
  if (!in || !codes || !scales) return PGG_ERR_INVALID_ARG;
  if (fmt != PGG_FMT_E4M3 && fmt != PGG_FMT_E2M1) return PGG_ERR_INVALID_ARG;
  if (R < 0 || R >= kMaxRows || C <= 0 || C >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (C % 32) return PGG_ERR_ALIGNMENT;
  if (!aligned16(in) || !aligned16(codes) || !aligned16(scales)) return PGG_ERR_ALIGNMENT;
  if (R == 0) return PGG_OK;
  return launch_mx_quantize_rowwise(in, R, C, fmt, codes, scales, as_stream(stream));
}

int pgg_mx_quantize_rowwise_blocked(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                                    uint8_t* scales, void* stream) {
  if (!in || !codes || !scales) return PGG_ERR_INVALID_ARG;
  if (fmt != PGG_FMT_E4M3 && fmt != PGG_FMT_E2M1) return PGG_ERR_INVALID_ARG;
  if (R < 0 || R >= kMaxRows || C <= 0 || C >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (C % 128) return PGG_ERR_ALIGNMENT;
  if (!aligned16(in) || !aligned16(codes) || !aligned16(scales)) return PGG_ERR_ALIGNMENT;
  if (R == 0) return PGG_OK;
  return launch_mx_quantize_rowwise_blocked(in, R, C, fmt, codes, scales, as_stream(stream));
}

int pgg_mx_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens,
                            int G, int fmt, uint8_t* codes_t, uint8_t* scales_t, int64_t M_pad,
                            int32_t* err, void* stream) {
  if (!in || !codes_t || !scales_t) return PGG_ERR_INVALID_ARG;
  if (fmt != PGG_FMT_E4M3 && fmt != PGG_FMT_E2M1) return PGG_ERR_INVALID_ARG;
  if (group_lens ? (G < 1 || G > kMaxGroups) : (G != 1 && G != 0)) return PGG_ERR_INVALID_ARG;
  if (M < 0 || M >= kMaxRows || C <= 0 || C >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (M_pad <= 0 || M_pad >= kMaxRows || M_pad % PGG_MX_PAD) return PGG_ERR_ALIGNMENT;
  if (C % 8) return PGG_ERR_ALIGNMENT;
  if (!aligned16(in) || !aligned16(codes_t) || !aligned16(scales_t)) return PGG_ERR_ALIGNMENT;
  return launch_mx_quantize_colwise(in, M, C, group_lens, group_lens ? G : 1, fmt, codes_t,
                                    scales_t, M_pad, err, as_stream(stream));
}

int pgg_mx_grouped_gemm(int mode, int fmt, int epilogue, const uint8_t* A, const uint8_t* SA,
                        const uint8_t* B, const uint8_t* SB, const void* H,
                        const int32_t* group_lens, void* out, void* out2, uint8_t* out_codes,
                        uint8_t* out_scales, int64_t M, int64_t N, int64_t K, int G, int64_t M_pad,
                        int32_t* err, void* stream) {
  return mx_gemm_impl(mode, fmt, epilogue, A, SA, B, SB, H, group_lens, out, out2, out_codes, out_scales, M, N,
                      K, G, M_pad, 0.0f, err, stream);
}

int pgg_mx_grouped_gemm_clamped(int mode, int fmt, const uint8_t* A, const uint8_t* SA, const uint8_t* B,
                                const uint8_t* SB, const void* H, const int32_t* group_lens, void* out,
                                void* out2, uint8_t* out_codes, uint8_t* out_scales, int64_t M, int64_t N,
                                int64_t K, int G, float swiglu_limit, int32_t* err, void* stream) {
  if (mode != PGG_MODE_FWD && mode != PGG_MODE_DGRAD) return PGG_ERR_INVALID_ARG;
  if (!(swiglu_limit >= 0.0f) || swiglu_limit > 3.0e38f) return PGG_ERR_INVALID_ARG;
  return mx_gemm_impl(mode, fmt, PGG_EPI_SWIGLU, A, SA, B, SB, H, group_lens, out, out2, out_codes, out_scales,
                      M, N, K, G, 0, swiglu_limit, err, stream);
}

int pgg_fp8_tensor_scale(const void* in, int64_t n, float* amax_scale, void* stream) {
  if (!amax_scale || (n > 0 && !in)) return PGG_ERR_INVALID_ARG;
  if (n < 0 || n >= ((int64_t)1 << 40)) return PGG_ERR_INVALID_ARG;
  if (n % 8) return PGG_ERR_ALIGNMENT;
  if ((n > 0 && !aligned16(in)) || !aligned16(amax_scale)) return PGG_ERR_ALIGNMENT;
  return launch_fp8_tensor_scale(in, n, amax_scale, as_stream(stream));
}

int pgg_fp8_quantize_rowwise(const void* in, int64_t R, int64_t C, const float* amax_scale, uint8_t* codes,
                             void* stream) {
  if (!in || !amax_scale || !codes) return PGG_ERR_INVALID_ARG;
  if (R < 0 || R >= kMaxRows || C <= 0 || C >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (C % 8) return PGG_ERR_ALIGNMENT;
  if (!aligned16(in) || !aligned16(codes) || !aligned16(amax_scale)) return PGG_ERR_ALIGNMENT;
  if (R == 0) return PGG_OK;
  return launch_fp8_quantize_rowwise(in, R * C, amax_scale, codes, as_stream(stream));
}

int pgg_fp8_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens, int G,
                             const float* amax_scale, uint8_t* codes_t, int64_t M_pad, int32_t* err,
                             void* stream) {
  // M == 0 (every group empty) is valid without an input: all M_pad columns get code 0
  if ((M > 0 && !in) || !amax_scale || !codes_t) return PGG_ERR_INVALID_ARG;
  if (group_lens ? (G < 1 || G > kMaxGroups) : (G != 1 && G != 0)) return PGG_ERR_INVALID_ARG;
  if (M < 0 || M >= kMaxRows || C <= 0 || C >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
  if (M_pad <= 0 || M_pad >= kMaxRows || M_pad % PGG_MX_PAD) return PGG_ERR_ALIGNMENT;
  if (C % 8) return PGG_ERR_ALIGNMENT;
  if ((M > 0 && !aligned16(in)) || !aligned16(codes_t) || !aligned16(amax_scale)) return PGG_ERR_ALIGNMENT;
  if ((group_lens && !aligned4(group_lens)) || (err && !aligned4(err))) return PGG_ERR_ALIGNMENT;
  return launch_fp8_quantize_colwise(in, M, C, group_lens, group_lens ? G : 1, amax_scale, codes_t, M_pad, err,
                                     as_stream(stream));
}

size_t pgg_fp8_workspace_size(int64_t N, int64_t K, int G, int64_t M_pad) {
  (void)N; (void)K; (void)G; (void)M_pad;
  return 0;  // the plain FP8 MMAs read no scale factors: no scratch
}

int pgg_fp8_grouped_gemm(int mode, int epilogue, const uint8_t* A, const float* scale_a, const uint8_t* B,
                         const float* scale_b, const void* H, const int32_t* group_lens, void* out, void* out2,
                         int64_t M, int64_t N, int64_t K, int G, int64_t M_pad, float swiglu_limit, void* ws,
                         size_t ws_bytes, int32_t* err, void* stream) {
  (void)ws; (void)ws_bytes;  // reserved: no scratch is needed
  if (!scale_a || !scale_b) return PGG_ERR_INVALID_ARG;
  if (!aligned4(scale_a) || !aligned4(scale_b)) return PGG_ERR_ALIGNMENT;
  if (!(swiglu_limit >= 0.0f) || swiglu_limit > 3.0e38f) return PGG_ERR_INVALID_ARG;
  if (swiglu_limit > 0.0f && epilogue != PGG_EPI_SWIGLU) return PGG_ERR_INVALID_ARG;
  if (N < 0 || K < 0 || M_pad < 0 || G < 1 || G > kMaxGroups) return PGG_ERR_INVALID_ARG;
  return mx_gemm_impl(mode, PGG_FMT_E4M3, epilogue, A, nullptr, B, nullptr, H, group_lens, out, out2, nullptr,
                      nullptr, M, N, K, G, M_pad, swiglu_limit, err, stream, scale_a, scale_b);
}

size_t pgg_moe_permute_workspace_size(int64_t T, int E) {
  if (T < 0 || E < 1) return 0;
  return moe_permute_ws_bytes(T, E);
}

int pgg_moe_permute(const int32_t* topk_ids, const void* X, int64_t T, int k, int64_t H, int E,
                    void* Xs, int32_t* group_lens, int32_t* pos, void* ws, size_t ws_bytes,
                    int32_t* err, void* stream) {
  if (k < 1 || k > 32 || E < 1 || E > kMaxGroups || T < 0 || T * k >= kMaxRows) return PGG_ERR_INVALID_ARG;
  if (!group_lens) return PGG_ERR_INVALID_ARG;
  if (X) {
    int st = check_dim(H, 8);
    if (st) return st;
    if (!Xs) return PGG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Xs)) return PGG_ERR_ALIGNMENT;
  }
  if (T > 0) {
    if (!topk_ids || !pos || !ws) return PGG_ERR_INVALID_ARG;
    if (ws_bytes < moe_permute_ws_bytes(T, E)) return PGG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 3u) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
        (reinterpret_cast<uintptr_t>(pos) & 3u))
      return PGG_ERR_ALIGNMENT;
  }
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  return launch_moe_permute(topk_ids, X, T, k, H, E, Xs, group_lens, pos, static_cast<int32_t*>(ws), err,
                            as_stream(stream));
}

int pgg_moe_combine(const void* Ys, const int32_t* pos, const float* w, void* out, int64_t T, int k,
                    int64_t H, void* stream) {
  if (k < 1 || k > 32 || T < 0 || T * k >= kMaxRows) return PGG_ERR_INVALID_ARG;
  int st = check_dim(H, 8);
  if (st) return st;
  if (T == 0) return PGG_OK;
  if (!Ys || !pos || !out) return PGG_ERR_INVALID_ARG;
  if (!aligned16(Ys) || !aligned16(out) || !aligned4(pos) || (w && !aligned4(w))) return PGG_ERR_ALIGNMENT;
  return launch_moe_combine(Ys, pos, w, T, k, H, out, as_stream(stream));
}

int pgg_moe_combine_bwd(const void* dOut, const void* Ys, const int32_t* pos, const float* w,
                        void* dYs, float* dw, int64_t T, int k, int64_t H, void* stream) {
  if (k < 1 || k > 32 || T < 0 || T * k >= kMaxRows) return PGG_ERR_INVALID_ARG;
  int st = check_dim(H, 8);
  if (st) return st;
  if (T == 0) return PGG_OK;
  if (!dOut || !Ys || !pos || !w || !dYs || !dw) return PGG_ERR_INVALID_ARG;
  if (!aligned16(dOut) || !aligned16(Ys) || !aligned16(dYs) || !aligned4(pos) || !aligned4(w) || !aligned4(dw))
    return PGG_ERR_ALIGNMENT;
  return launch_moe_combine_bwd(dOut, Ys, pos, w, T, k, H, dYs, dw, as_stream(stream));
}

int pgg_test_stalled_fwd(int fmt, const void* A, const uint8_t* SA, const void* B, const uint8_t* SB,
                         const int32_t* group_lens, void* out, int64_t M, int64_t N, int64_t K, int G,
                         int64_t stall_at, uint64_t wait_ns, int32_t* err, void* stream) {
  if (stall_at < 0 || wait_ns < 100000ull || wait_ns > 1000000000ull) return PGG_ERR_INVALID_ARG;
  if (fmt != 0)
    return mx_gemm_impl(PGG_MODE_FWD, fmt, PGG_EPI_NONE, static_cast<const uint8_t*>(A), SA,
                        static_cast<const uint8_t*>(B), SB, nullptr, group_lens, out, nullptr, nullptr, nullptr, M, N,
                        K, G, 0, 0.0f, err, stream, nullptr, nullptr, wait_ns, stall_at);
  int st;
  if ((st = check_common(M, G, group_lens))) return st;
  if ((st = check_dim(N, 8)) || (st = check_dim(K, 8))) return st;
  if (M == 0) return PGG_OK;
  if (!A || !B || !out) return PGG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return PGG_ERR_ALIGNMENT;
  if (err && !aligned4(err)) return PGG_ERR_ALIGNMENT;
  Bf16Call c{0, 0, A, B, group_lens, out, nullptr, nullptr, M, N, K, 0, G, err, as_stream(stream)};
  c.wait_ns = wait_ns;
  c.stall_at = stall_at;
  return launch_bf16(c);
}

}  // extern "C"
