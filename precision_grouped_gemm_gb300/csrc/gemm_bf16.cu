// Host launchers of the BF16 grouped GEMM family (see gemm_bf16.cuh).
#include <algorithm>

#include "gemm_bf16.cuh"
#include "internal.h"

namespace pgg {
namespace {

constexpr int kBN = 256;

// stages: fwd/dgrad stream W through 4 x 48 KB (BK 64).  The wgrad store keeps a
// 32 KB staging ring and runs 7 x 24 KB (BK 32) or 4 x 48 KB (BK 64; 3 when the group
// tables of a large G leave no room); the fp32 accumulate keeps 64 KB and runs 6 x 24 KB
// or 3 x 48 KB.
template <int MODE, int EPI, int BK>
constexpr int stages() {
  return MODE != kWgrad ? 4 : (EPI == kEpiAccumF32 ? (BK == 32 ? 6 : 3) : (BK == 32 ? 7 : 4));
}

template <int MODE, int EPI, int BK, int S>
int run_s(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& args,
          int grid, cudaStream_t s) {
  using L = GemmSmem<kBN, BK, S, epi_bytes<MODE, EPI>()>;
  auto kern = grouped_gemm_bf16_kernel<MODE, EPI, kBN, S, BK>;
  const size_t smem = L::bytes(args.G);
  static size_t attr_bytes = 0;  // per instantiation: raised to the largest G seen
  if (smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e == cudaErrorInvalidValue ? PGG_ERR_UNSUPPORTED : cuda_status(e);
    attr_bytes = smem;
  }
  kern<<<grid, kGemmThreads, smem, s>>>(ta, tb, tc, args);
  return cuda_status(cudaGetLastError());
}

template <int MODE, int EPI, int BK = 64>
int run(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const GemmArgs& args,
        int grid, cudaStream_t s) {
  constexpr int S = stages<MODE, EPI, BK>();
  if constexpr (MODE == kWgrad && EPI != kEpiAccumF32 && BK == 64) {
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != PGG_OK) return st;
    using L = GemmSmem<kBN, BK, S, epi_bytes<MODE, EPI>()>;
    if (L::bytes(args.G) > dev.smem_optin) return run_s<MODE, EPI, BK, S - 1>(ta, tb, tc, args, grid, s);
  }
  return run_s<MODE, EPI, BK, S>(ta, tb, tc, args, grid, s);
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

}  // namespace

int launch_bf16(const Bf16Call& c) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  const uint32_t sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap ta, tb, tc;
  GemmArgs a{};
  a.group_lens = c.group_lens;
  a.G = c.G;
  a.M = c.M;
  a.out = c.out;
  a.out2 = c.out2;
  a.aux = c.aux;
  a.err = c.err;
  a.I = (int)c.I;
  a.swiglu_limit = c.limit;
  a.wait_ns = c.wait_ns;
  a.stall_at = c.stall_at;
  int tiles_ub = 0;
  int wbk = 64;

  if (c.mode == 0) {  // forward (optionally FC1 + SwiGLU): B = W [G, Nw, K]
    const int64_t Nw = c.epi == 1 ? 2 * c.I : c.N;
    uint64_t da[2] = {(uint64_t)c.K, (uint64_t)c.M}, sa[1] = {(uint64_t)c.K * 2};
    uint32_t ba[2] = {64, 128};
    uint64_t db[3] = {(uint64_t)c.K, (uint64_t)Nw, (uint64_t)c.G};
    uint64_t sb[2] = {(uint64_t)c.K * 2, (uint64_t)(Nw * c.K * 2)};
    uint32_t bb[3] = {64, c.epi == 1 ? (uint32_t)(kBN / 2) : (uint32_t)kBN, 1};
    if ((st = encode_tmap(&ta, bf, 2, c.a, da, sa, ba, (CUtensorMapSwizzle)sw))) return st;
    if ((st = encode_tmap(&tb, bf, 3, c.b, db, sb, bb, (CUtensorMapSwizzle)sw))) return st;
    a.out_cols = (int)(c.epi == 1 ? c.I : c.N);
    a.red = (int)c.K;
    const int tcw = c.epi == 1 ? kBN / 2 : kBN;
    tiles_ub = (ceil_div(c.M, kBM) + c.G) * ceil_div(a.out_cols, tcw);
  } else if (c.mode == 1) {  // dgrad (optionally FC2 dgrad + SwiGLU bwd): A = dY [M, N]
    uint64_t da[2] = {(uint64_t)c.N, (uint64_t)c.M}, sa[1] = {(uint64_t)c.N * 2};
    uint32_t ba[2] = {64, 128};
    if ((st = encode_tmap(&ta, bf, 2, c.a, da, sa, ba, (CUtensorMapSwizzle)sw))) return st;
    a.b_multi = 0;
    if (c.K % 64 == 0) {  // W as {64, N, K/64, G}: all BN/64 k-atoms of a k-block in one load
      uint64_t d4[4] = {64, (uint64_t)c.N, (uint64_t)(c.K / 64), (uint64_t)c.G};
      uint64_t s4[3] = {(uint64_t)c.K * 2, 128, (uint64_t)(c.N * c.K * 2)};
      uint32_t b4[4] = {64, 64, (uint32_t)(kBN / 64), 1};
      a.b_multi = encode_tmap(&tb, bf, 4, c.b, d4, s4, b4, (CUtensorMapSwizzle)sw) == PGG_OK;
    }
    if (!a.b_multi) {
      uint64_t db[3] = {(uint64_t)c.K, (uint64_t)c.N, (uint64_t)c.G};
      uint64_t sb[2] = {(uint64_t)c.K * 2, (uint64_t)(c.N * c.K * 2)};
      uint32_t bb[3] = {64, 64, 1};
      if ((st = encode_tmap(&tb, bf, 3, c.b, db, sb, bb, (CUtensorMapSwizzle)sw))) return st;
    }
    a.out_cols = (int)c.K;
    a.red = (int)c.N;
    tiles_ub = (ceil_div(c.M, kBM) + c.G) * ceil_div(c.K, kBN);
  } else {  // wgrad: A = dY [M, N] MN-major, B = X [M, K] MN-major
    wbk = (c.M <= 256 * (int64_t)c.G) ? 32 : 64;  // short groups: smaller, deeper k-blocks
    // operands as atom views {64, M, cols/64} (one load per k-block) when cols % 64 == 0,
    // else 64-column boxes
    auto enc = [&](CUtensorMap* m, const void* base, int64_t cols, uint32_t atoms, int* multi) {
      *multi = 0;
      if (cols % 64 == 0) {
        uint64_t d3[3] = {64, (uint64_t)c.M, (uint64_t)(cols / 64)}, s3[2] = {(uint64_t)cols * 2, 128};
        uint32_t b3[3] = {64, (uint32_t)wbk, atoms};
        if (encode_tmap(m, bf, 3, base, d3, s3, b3, (CUtensorMapSwizzle)sw) == PGG_OK) {
          *multi = 1;
          return (int)PGG_OK;
        }
      }
      uint64_t d2[2] = {(uint64_t)cols, (uint64_t)c.M}, s2[1] = {(uint64_t)cols * 2};
      uint32_t b2[2] = {64, (uint32_t)wbk};
      return encode_tmap(m, bf, 2, base, d2, s2, b2, (CUtensorMapSwizzle)sw);
    };
    if ((st = enc(&ta, c.a, c.N, kBM / 64, &a.a_multi))) return st;
    if ((st = enc(&tb, c.b, c.K, kBN / 64, &a.b_multi))) return st;
    if (c.epi == 3) st = encode_wgrad_accum_f32(&tc, c.out, c.N, c.K, c.G, &a.c4d);
    else st = encode_wgrad_out(&tc, c.out, c.N, c.K, c.G, kWgradStoreAtoms, &a.c4d);
    if (st) return st;
    a.out_cols = (int)c.K;
    a.wg_rows = (int)c.N;
    a.nct = FastDiv((uint32_t)ceil_div(c.K, kBN));
    tiles_ub = c.G * ceil_div(c.N, kBM) * ceil_div(c.K, kBN);
  }
  if (c.mode != 2) tc = ta;  // unused outside wgrad
  const int grid = std::max(1, std::min(dev.sms, tiles_ub));
  if (c.mode == 0 && c.epi == 0) return run<kFwd, kEpiStore>(ta, tb, tc, a, grid, c.stream);
  if (c.mode == 0 && c.epi == 1) return run<kFwd, kEpiSwiGLU>(ta, tb, tc, a, grid, c.stream);
  if (c.mode == 1 && c.epi == 0) return run<kDgrad, kEpiStore>(ta, tb, tc, a, grid, c.stream);
  if (c.mode == 1 && c.epi == 2) return run<kDgrad, kEpiSwiGLUBwd>(ta, tb, tc, a, grid, c.stream);
  if (c.mode == 2 && c.epi == 0)
    return wbk == 32 ? run<kWgrad, kEpiStore, 32>(ta, tb, tc, a, grid, c.stream)
                     : run<kWgrad, kEpiStore, 64>(ta, tb, tc, a, grid, c.stream);
  if (c.mode == 2 && c.epi == 3)
    return wbk == 32 ? run<kWgrad, kEpiAccumF32, 32>(ta, tb, tc, a, grid, c.stream)
                     : run<kWgrad, kEpiAccumF32, 64>(ta, tb, tc, a, grid, c.stream);
  return PGG_ERR_INVALID_ARG;
}

}  // namespace pgg
