// MX (microscaling) quantization kernels: bf16 -> e4m3 or e2m1 codes with one
// E8M0 scale per 32-element block (the MXFP8 / MXFP4 operands of the
// block-scaled grouped GEMM; "Primus-Turbo" README, "What's New"; Pull Request
// #891, "Changes": MXFP4 weights as float4_e2m1fn_x2 buffers).
//
// Rule (OCP Microscaling v1.0): amax = max |v| over the block; E =
// clamp(floor(log2 amax) - emax, -127, 127), emax 8 (e4m3) / 2 (e2m1); scale
// code E + 127; code = RNE(v * 2^-E) saturated to the largest finite value,
// sign of zero kept; a block holding NaN or Inf gets scale 0xFF and zero codes.
// For bf16 inputs floor(log2 amax) is the exponent field minus 127 (zero and
// subnormal amax clamp to E = -127), and v * 2^-E is exact in fp32 for every
// value that can round to a non-zero code, so the conversion instruction's
// single rounding is the rule's rounding.
#include <algorithm>

#include "internal.h"
#include "mx_codec.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace pgg {
namespace {

// ------------------------------------------------------------------ row-wise
// The tensor is a flat run of 32-element blocks (C % 32 == 0), so block i's
// scale is scales[i] and its codes start at byte 32 i (e4m3) or 16 i (e2m1).
// Four lanes own one block: each loads 8 bf16 (16 B, fully coalesced across the
// warp), the block amax is a 2-step xor shuffle, each lane writes 8 (e4m3) or
// 4 (e2m1) bytes and lane%4 == 0 writes the scale byte.
// BLOCKED: scales go to the atom layout of the block-scaled MMA instead of row-major
// [R, C/32] (the weight operand of the forward GEMM; C % 128 == 0): block j of row r
// at ((r / 128) * C / 128 + j / 4) * 512 + 16 (r % 32) + 4 ((r % 128) / 32) + j % 4.
// One 16-byte chunk i (8 bf16 of block i / 4); every lane of the warp calls it (shuffles).
template <int FMT, bool BLOCKED>
__device__ __forceinline__ void rowwise_chunk(const uint4& v, int64_t i, bool live, uint8_t* __restrict__ codes,
                                              uint8_t* __restrict__ scales, uint32_t row_blocks) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t am = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) am = max(am, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
  if (!live) return;
  uint32_t sc;
  float mult;
  const bool fin = block_scale<FMT>(am, sc, mult);
  float f[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = bf16_lo(w[j]) * mult;
    f[2 * j + 1] = bf16_hi(w[j]) * mult;
  }
  if (FMT == kE4M3) {
    uint2 o;
    o.x = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
    o.y = cvt_e4m3x2(f[4], f[5]) | (cvt_e4m3x2(f[6], f[7]) << 16);
    if (!fin) o = make_uint2(0, 0);
    reinterpret_cast<uint2*>(codes)[i] = o;
  } else {
    uint32_t o = cvt_e2m1x2(f[0], f[1]) | (cvt_e2m1x2(f[2], f[3]) << 8) |
                 (cvt_e2m1x2(f[4], f[5]) << 16) | (cvt_e2m1x2(f[6], f[7]) << 24);
    if (!fin) o = 0;
    reinterpret_cast<uint32_t*>(codes)[i] = o;
  }
  if ((threadIdx.x & 3) == 0) {
    const int64_t b = i >> 2;  // block index = r * row_blocks + j
    if (BLOCKED) {
      const int64_t r = b / row_blocks;
      const uint32_t j = (uint32_t)(b - r * row_blocks), m = (uint32_t)(r & 127);
      scales[(((r >> 7) * (row_blocks >> 2) + (j >> 2)) << 9) + 16 * (m & 31) + 4 * (m >> 5) + (j & 3)] =
          (uint8_t)sc;
    } else {
      scales[b] = (uint8_t)sc;
    }
  }
}

// Two chunks per thread per iteration (i and i + stride), both loads issued first.
template <int FMT, bool BLOCKED = false>
__global__ void __launch_bounds__(256) mx_quant_rowwise_kernel(const uint4* __restrict__ in,
                                                               uint8_t* __restrict__ codes,
                                                               uint8_t* __restrict__ scales,
                                                               int64_t n_chunks, uint32_t row_blocks) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int lane = threadIdx.x & 31;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i - lane < n_chunks; i += 2 * stride) {
    const int64_t i2 = i + stride;
    const bool live = i < n_chunks, live2 = i2 < n_chunks;
    const uint4 v = live ? __ldg(in + i) : make_uint4(0, 0, 0, 0);
    const uint4 v2 = live2 ? __ldg(in + i2) : make_uint4(0, 0, 0, 0);
    rowwise_chunk<FMT, BLOCKED>(v, i, live, codes, scales, row_blocks);
    if (i2 - lane < n_chunks) rowwise_chunk<FMT, BLOCKED>(v2, i2, live2, codes, scales, row_blocks);  // warp-uniform
  }
}

// ------------------------------------------------------------------ column-wise
// Output column space [0, M_pad) is cut into 32-wide blocks; block j holds
// rows off_g + 32 b .. of group g for j = pb_g + b with pb_g the prefix of
// round_up(len_g, 128) / 32, or nothing (pad) -- every output byte is written
// once.  One warp handles one 128-wide k-block p (blocks j = 4 p .. 4 p + 3, one
// scale atom; it never straddles groups, whose spans are padded to 128) x 64 input
// columns: for each block, lane l reads columns c0 + 2l, c0 + 2l + 1 of the
// block's rows (32 coalesced 128-byte row loads), takes each column's amax and
// converts the column's 32 codes.  The loads of block q + 1 are issued before block
// q is converted, so 64 row loads per warp are in flight.  The codes collect in
// the warp's shared-memory stage (64 columns x 128 codes) and leave as whole
// output-row segments -- 128 bytes e4m3 / 64 bytes e2m1 per column, written by 8 /
// 4 lanes at once -- instead of 16- or 32-byte pieces per lane (partial sectors).
// The column's four scales of the k-block leave together as one 32-bit store.
// Work items run with p fastest.
//
// Scales go to the blocked layout the block-scaled MMA reads: for every 128-row
// block rb of the C rows and every 128-column k-block p of [0, M_pad), one 512-byte
// atom at ((rb * M_pad / 128) + p) * 512 in which row r = 128 rb + m, 32-block
// j = 4 p + q sits at byte 16 (m % 32) + 4 (m / 32) + q.  Rows past C up to the
// next multiple of 128 get scale 0.
constexpr int kColSlab = 64;
constexpr int kColThreads = 256;

// Shared-memory bytes of one warp's code stage, and of the kernel for G groups (the two
// [G + 1] scan tables, rounded up to 16 bytes, then eight stages).
template <int FMT>
__host__ __device__ constexpr int col_stage_bytes() { return kColSlab * (FMT == kE4M3 ? 128 : 64); }
// The MXFP8 codes (32 bytes per column and block: whole sectors) go straight to the output; the
// stage pays for e2m1 (16-byte pieces) and for the FP8 tensor-wise pass (timed: MXFP8 column-wise
// 0.068 ms direct vs 0.074 ms staged on the DeepSeek-shaped layer, FP8 0.080 vs 0.066 ms).
template <int FMT, bool TENSOR>
__host__ __device__ constexpr bool col_staged() { return FMT == kE2M1 || TENSOR; }
template <int FMT, bool TENSOR = false>
__host__ __device__ constexpr size_t col_smem_bytes(int G) {
  return ((8 * (size_t)(G + 1) + 15) & ~(size_t)15) +
         (col_staged<FMT, TENSOR>() ? (kColThreads / 32) * (size_t)col_stage_bytes<FMT>() : 0);
}

// Byte offset in a warp's stage of 16-byte chunk ch of stage column k (its codes
// 16 ch .. 16 ch + 15, e4m3 bytes or e2m1 pairs): the stage is a run of 128-byte rows
// whose chunks are permuted by ((k / 2) % 8), so that both the lane-per-column writes
// and the row-segment reads spread over all banks.
template <int FMT>
__device__ __forceinline__ uint32_t col_stage_off(int k, int ch) {
  const uint32_t lin = (uint32_t)k * (FMT == kE4M3 ? 128u : 64u) + 16u * ch;
  return (lin & ~127u) | ((((lin >> 4) & 7u) ^ ((k >> 1) & 7u)) << 4);
}

// Byte offset of row r's four scales of k-block p in the blocked layout.
__device__ __forceinline__ int64_t blocked_atom_word(int r, int p, int64_t M_pad) {
  const int m = r & 127;
  return (((int64_t)(r >> 7) * (M_pad >> 7) + p) << 9) + 16 * (m & 31) + 4 * (m >> 5);
}

// Quantize column `half` of the packed bf16 pairs v (zero past `valid`): its 32 codes
// land in o (32 bytes e4m3 / 16 bytes e2m1, o[1] unused for e2m1); returns the scale
// byte (0 when the block holds no rows).  TENSOR (FP8 tensor-wise, e4m3): the
// multiplier is the tensor scale ts for every block and no scale byte exists (a
// non-finite element converts on its own).
template <int FMT, bool TENSOR = false>
__device__ __forceinline__ uint32_t colwise_codes(const uint32_t (&v)[32], int half, int valid, uint4 (&o)[2],
                                                  float ts = 0.0f) {
  uint32_t sc = 0;
  float mult = 0.0f;
  bool keep;
  if constexpr (TENSOR) {
    mult = ts;
    keep = valid > 0;
  } else {
    uint32_t m[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) m[r] = max((v[2 * r] >> (16 * half)) & 0x7FFFu, (v[2 * r + 1] >> (16 * half)) & 0x7FFFu);
#pragma unroll
    for (int d = 8; d >= 1; d >>= 1)
#pragma unroll
      for (int r = 0; r < d; ++r) m[r] = max(m[r], m[r + d]);
    const bool fin = valid > 0 ? block_scale<FMT>(m[0], sc, mult) : true;
    keep = valid > 0 && fin;
  }
  uint32_t* ow = reinterpret_cast<uint32_t*>(o);
  if (FMT == kE4M3) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) f[e] = keep ? __uint_as_float((v[4 * k + e] >> (16 * half)) << 16) * mult : 0.0f;
      ow[k] = cvt_e4m3x2(f[0], f[1]) | (cvt_e4m3x2(f[2], f[3]) << 16);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = keep ? __uint_as_float((v[8 * k + e] >> (16 * half)) << 16) * mult : 0.0f;
      ow[k] = cvt_e2m1x2(f[0], f[1]) | (cvt_e2m1x2(f[2], f[3]) << 8) | (cvt_e2m1x2(f[4], f[5]) << 16) |
              (cvt_e2m1x2(f[6], f[7]) << 24);
    }
  }
  return valid > 0 ? sc : 0u;
}

// Rows 32 q .. 32 q + 31 of the k-block's group rows (zero past `valid`), columns c, c + 1
// as packed bf16 pairs.
__device__ __forceinline__ void col_load32(const __nv_bfloat16* __restrict__ in, int64_t row0, int C, int c,
                                           int valid, uint32_t (&v)[32]) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(in + row0 * C + c);
#pragma unroll
  for (int r = 0; r < 32; ++r) v[r] = r < valid ? __ldg(src + (int64_t)r * (C / 2)) : 0u;
}

// TENSOR: FP8 tensor-wise codes (multiplier amax_scale[0] for every element), no scales.
template <int FMT, bool TENSOR = false>
__global__ void __launch_bounds__(kColThreads) mx_quant_colwise_kernel(
    const __nv_bfloat16* __restrict__ in, int64_t M, int C, const int32_t* __restrict__ lens,
    int G, uint8_t* __restrict__ codes_t, uint8_t* __restrict__ scales_t, int64_t M_pad,
    int32_t* err, const float* __restrict__ amax_scale = nullptr) {
  static_assert(!TENSOR || FMT == kE4M3, "tensor-wise scaling is e4m3");
  constexpr int kCB = FMT == kE4M3 ? 128 : 64;  // code bytes of one column in one k-block
  extern __shared__ __align__(16) int32_t s_dyn[];
  int32_t* s_off = s_dyn;             // [G+1] row offsets
  int32_t* s_blk = s_dyn + (G + 1);   // [G+1] prefix of 32-blocks in the padded layout
  __shared__ int s_bad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* stg = reinterpret_cast<uint8_t*>(s_dyn) + ((8 * (size_t)(G + 1) + 15) & ~(size_t)15) +
                 (size_t)warp * col_stage_bytes<FMT>();
  if (warp == 0) {
    bool bad;
    if (lens) {
      TileCount tc;
      tc.bm = PGG_MX_PAD;
      tc.per_row_tile = PGG_MX_PAD / 32;
      bad = scan_groups(lens, G, M, tc, s_off, s_blk, nullptr, 0, lane);
    } else {
      if (lane == 0) {
        s_off[0] = 0; s_off[1] = (int32_t)M;
        s_blk[0] = 0; s_blk[1] = (int32_t)(((M + PGG_MX_PAD - 1) / PGG_MX_PAD) * (PGG_MX_PAD / 32));
      }
      bad = false;
      __syncwarp();
    }
    if (lane == 0) {
      int code = bad ? kErrBadGroupLens : ((int64_t)s_blk[G] * 32 > M_pad ? kErrPadOverflow : 0);
      s_bad = code;
      if (code && blockIdx.x == 0) set_error(err, code);
    }
  }
  __syncthreads();
  if (s_bad) return;
  const float ts = TENSOR ? __ldg(amax_scale) : 0.0f;
  const int nkb = (int)(M_pad / 128);  // k-blocks (scale atoms) along the padded axis
  const int C128 = (C + 127) & ~127;   // scale rows, padded to whole atoms
  const int nslab = C128 / kColSlab;
  const int64_t total = (int64_t)nkb * nslab;
  const int used = s_blk[G];
  const int64_t nwarps = (int64_t)gridDim.x * (kColThreads / 32);
  for (int64_t t = (int64_t)blockIdx.x * (kColThreads / 32) + warp; t < total; t += nwarps) {
    const int p = (int)(t % nkb);
    const int c0 = (int)(t / nkb) * kColSlab;  // the warp's first column
    const int c = c0 + 2 * lane;               // this lane's two columns
    if (c0 >= C) {  // a slab of pad rows of the last atom: scale 0, no codes
      if (!TENSOR && c < C128) {
        *reinterpret_cast<uint32_t*>(scales_t + blocked_atom_word(c, p, M_pad)) = 0u;
        *reinterpret_cast<uint32_t*>(scales_t + blocked_atom_word(c + 1, p, M_pad)) = 0u;
      }
      continue;
    }
    const bool live = c < C;  // columns past C (warp-divergent only in the last slab): zero codes, scale 0
    int len = 0, b0 = 0;
    int64_t grow0 = 0;
    if (4 * p < used) {
      const int g = find_group(s_blk, G, 4 * p);
      b0 = 4 * p - s_blk[g];
      len = s_off[g + 1] - s_off[g];
      grow0 = s_off[g];
    }
    if (!live) len = 0;
    uint32_t sc0 = 0, sc1 = 0;
    uint32_t v[32], nv[32];
    col_load32(in, grow0 + 32 * b0, C, c, min(32, max(0, len - 32 * b0)), nv);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      const int valid = min(32, max(0, len - 32 * (b0 + q)));
#pragma unroll
      for (int r = 0; r < 32; ++r) v[r] = nv[r];
      if (q < 3) col_load32(in, grow0 + 32 * (b0 + q + 1), C, c, min(32, max(0, len - 32 * (b0 + q + 1))), nv);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint4 o[2];
        const uint32_t sc = colwise_codes<FMT, TENSOR>(v, h, valid, o, ts);
        if (h == 0) sc0 |= sc << (8 * q); else sc1 |= sc << (8 * q);
        const int k = 2 * lane + h;
        if constexpr (!col_staged<FMT, TENSOR>()) {  // e4m3: the column's 32 codes of block 4 p + q
          if (c + h < C) {
            uint4* dst = reinterpret_cast<uint4*>(codes_t + (int64_t)(c + h) * M_pad + (int64_t)p * kCB + 32 * q);
            dst[0] = o[0];
            dst[1] = o[1];
          }
        } else if (FMT == kE4M3) {
          *reinterpret_cast<uint4*>(stg + col_stage_off<FMT>(k, 2 * q)) = o[0];
          *reinterpret_cast<uint4*>(stg + col_stage_off<FMT>(k, 2 * q + 1)) = o[1];
        } else {
          *reinterpret_cast<uint4*>(stg + col_stage_off<FMT>(k, q)) = o[0];
        }
      }
    }
    if constexpr (col_staged<FMT, TENSOR>()) {
      __syncwarp();
      // write-out: column k's kCB code bytes of this k-block are one contiguous stretch of
      // output row c0 + k; kCB / 16 lanes per column, 32 * 16 / kCB columns per instruction
      constexpr int kLpc = kCB / 16;
      const int ch = lane % kLpc;
#pragma unroll
      for (int i = 0; i < kColSlab * kLpc / 32; ++i) {
        const int k = i * (32 / kLpc) + lane / kLpc;
        const uint4 x = *reinterpret_cast<const uint4*>(stg + col_stage_off<FMT>(k, ch));
        if (c0 + k < C)
          *reinterpret_cast<uint4*>(codes_t + (int64_t)(c0 + k) * (FMT == kE4M3 ? M_pad : M_pad / 2) +
                                    (int64_t)p * kCB + 16 * ch) = x;
      }
      __syncwarp();
    }
    if (!TENSOR && c < C128) {
      *reinterpret_cast<uint32_t*>(scales_t + blocked_atom_word(c, p, M_pad)) = sc0;
      *reinterpret_cast<uint32_t*>(scales_t + blocked_atom_word(c + 1, p, M_pad)) = sc1;
    }
  }
}

// ------------------------------------------------------------------ FP8 tensor-wise
// Current scaling ("[Megatron-LM] feat: add grouped gemm fp4 support ... Pull Request
// #891", review: the FP8 grouped GEMM under current scaling): amax over the tensor's
// finite values, s = 448 / amax in fp32 (1 for amax 0; a quotient that overflows fp32
// is clamped to the largest finite fp32), codes = e4m3 RNE of the fp32 product x s,
// saturating.  amax_scale is a device float[2] = {s, amax}; while the amax kernel runs,
// word 1 holds the largest finite bf16 magnitude as bits (their integer order is the
// values' order), one atomicMax per block after a shared-memory reduction.
// {s, amax} of a bf16 tensor in one pass.  amax_scale = {0, 0} on entry (the launcher's
// memset): word 1 collects the integer max of the finite bf16 magnitude bits (one atomicMax
// per block) and word 0 counts finished blocks; the last block to finish turns the max into
// the fp32 pair {s = 448 / amax, amax}.  Each thread keeps kAmaxUnroll 16-byte loads in
// flight per iteration.
constexpr int kAmaxUnroll = 4;

__device__ __forceinline__ uint32_t amax_bits8(uint4 v, uint32_t am) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = w[j] & 0x7FFFu, hi = (w[j] >> 16) & 0x7FFFu;
    if (lo < 0x7F80u) am = max(am, lo);  // Inf / NaN excluded
    if (hi < 0x7F80u) am = max(am, hi);
  }
  return am;
}

__global__ void __launch_bounds__(256) fp8_amax_scale_kernel(const uint4* __restrict__ in, int64_t n_chunks,
                                                             float* __restrict__ amax_scale) {
  __shared__ uint32_t s_max[256 / 32];
  __shared__ bool s_last;
  uint32_t* words = reinterpret_cast<uint32_t*>(amax_scale);
  uint32_t am = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * stride < n_chunks; i += kAmaxUnroll * stride) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = __ldg(in + i + u * stride);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) am = amax_bits8(v[u], am);
  }
  for (; i < n_chunks; i += stride) am = amax_bits8(__ldg(in + i), am);
  am = __reduce_max_sync(0xffffffffu, am);
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = am;
  __syncthreads();
  if (threadIdx.x < 32) {
    am = threadIdx.x < (blockDim.x >> 5) ? s_max[threadIdx.x] : 0u;
    am = __reduce_max_sync(0xffffffffu, am);
    if (threadIdx.x == 0) {
      if (am != 0u) atomicMax(words + 1, am);
      __threadfence();  // this block's max is visible before its arrival is counted
      s_last = atomicAdd(words, 1u) == gridDim.x - 1;
    }
  }
  __syncthreads();
  if (s_last && threadIdx.x == 0) {
    __threadfence();
    const uint32_t bits = atomicMax(words + 1, 0u);  // the final max (an atomic read)
    const float amax = __uint_as_float(bits << 16);
    float sc = 1.0f;
    if (bits != 0u) {
      const float fmax = __uint_as_float(0x7F7FFFFFu);
      sc = __fdiv_rn(448.0f, amax);
      if (!(sc <= fmax)) sc = fmax;
    }
    amax_scale[0] = sc;
    amax_scale[1] = amax;
  }
}

// codes[i] = e4m3(x[i] s), eight elements (one 16-byte load, one 8-byte store) per chunk
__global__ void __launch_bounds__(256) fp8_quant_rowwise_kernel(const uint4* __restrict__ in,
                                                                uint2* __restrict__ codes, int64_t n_chunks,
                                                                const float* __restrict__ amax_scale) {
  const float s = __ldg(amax_scale);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks; i += stride) {
    const uint4 v = __ldg(in + i);
    uint2 o;
    o.x = cvt_e4m3x2(bf16_lo(v.x) * s, bf16_hi(v.x) * s) | (cvt_e4m3x2(bf16_lo(v.y) * s, bf16_hi(v.y) * s) << 16);
    o.y = cvt_e4m3x2(bf16_lo(v.z) * s, bf16_hi(v.z) * s) | (cvt_e4m3x2(bf16_lo(v.w) * s, bf16_hi(v.w) * s) << 16);
    codes[i] = o;
  }
}

int stream_grid(int64_t n_chunks) {
  DeviceInfo dev;
  if (current_device(&dev) != PGG_OK) return 0;
  const int64_t want = (n_chunks + 255) / 256;
  return (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sms * 8));
}

}  // namespace

int launch_mx_quantize_rowwise(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                               uint8_t* scales, cudaStream_t s) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  const int64_t n_chunks = R * C / 8;
  const int threads = 256;
  const int64_t want = (n_chunks + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sms * 8));
  const uint32_t rb = (uint32_t)(C / 32);
  if (fmt == PGG_FMT_E4M3)
    mx_quant_rowwise_kernel<kE4M3><<<grid, threads, 0, s>>>(static_cast<const uint4*>(in), codes,
                                                             scales, n_chunks, rb);
  else
    mx_quant_rowwise_kernel<kE2M1><<<grid, threads, 0, s>>>(static_cast<const uint4*>(in), codes,
                                                             scales, n_chunks, rb);
  return cuda_status(cudaGetLastError());
}

int launch_mx_quantize_rowwise_blocked(const void* in, int64_t R, int64_t C, int fmt, uint8_t* codes,
                                       uint8_t* scales, cudaStream_t s) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  if (R % 128) {  // rows past R in the last 128-row block hold scale 0
    const size_t atoms = (size_t)(C / 128);
    cudaError_t e = cudaMemsetAsync(scales + (size_t)(R / 128) * atoms * 512, 0, atoms * 512, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  const int64_t n_chunks = R * C / 8;
  const int threads = 256;
  const int64_t want = (n_chunks + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sms * 8));
  const uint32_t rb = (uint32_t)(C / 32);
  if (fmt == PGG_FMT_E4M3)
    mx_quant_rowwise_kernel<kE4M3, true><<<grid, threads, 0, s>>>(static_cast<const uint4*>(in), codes,
                                                                   scales, n_chunks, rb);
  else
    mx_quant_rowwise_kernel<kE2M1, true><<<grid, threads, 0, s>>>(static_cast<const uint4*>(in), codes,
                                                                   scales, n_chunks, rb);
  return cuda_status(cudaGetLastError());
}

int launch_mx_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens,
                               int G, int fmt, uint8_t* codes_t, uint8_t* scales_t,
                               int64_t M_pad, int32_t* err, cudaStream_t s) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  const int64_t total = (M_pad / 128) * (((C + 127) / 128 * 128) / kColSlab);  // warp work items
  const bool e4 = fmt == PGG_FMT_E4M3;
  const size_t smem = e4 ? col_smem_bytes<kE4M3>(G) : col_smem_bytes<kE2M1>(G);
  auto kern = e4 ? mx_quant_colwise_kernel<kE4M3> : mx_quant_colwise_kernel<kE2M1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int per_sm = 0;  // resident CTAs per SM: the grid-stride loop runs one wave of them
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kColThreads, smem);
  if (e != cudaSuccess) return cuda_status(e);
  const int64_t want = (total + kColThreads / 32 - 1) / (kColThreads / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sms * std::max(per_sm, 1)));
  kern<<<grid, kColThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(in), M, (int)C, group_lens, G, codes_t,
                                       scales_t, M_pad, err, nullptr);
  return cuda_status(cudaGetLastError());
}

int launch_fp8_tensor_scale(const void* in, int64_t n, float* amax_scale, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax_scale, 0, 2 * sizeof(float), s);
  if (e != cudaSuccess) return cuda_status(e);
  // n == 0 runs one block over nothing: amax 0, s = 1
  const int grid = n > 0 ? stream_grid(n / 8) : 1;
  if (grid == 0) return PGG_ERR_CUDA;
  fp8_amax_scale_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(in), n / 8, amax_scale);
  return cuda_status(cudaGetLastError());
}

int launch_fp8_quantize_rowwise(const void* in, int64_t n, const float* amax_scale, uint8_t* codes,
                                cudaStream_t s) {
  const int grid = stream_grid(n / 8);
  if (grid == 0) return PGG_ERR_CUDA;
  fp8_quant_rowwise_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(in), reinterpret_cast<uint2*>(codes),
                                                n / 8, amax_scale);
  return cuda_status(cudaGetLastError());
}

int launch_fp8_quantize_colwise(const void* in, int64_t M, int64_t C, const int32_t* group_lens, int G,
                                const float* amax_scale, uint8_t* codes_t, int64_t M_pad, int32_t* err,
                                cudaStream_t s) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  const int64_t total = (M_pad / 128) * (((C + 127) / 128 * 128) / kColSlab);  // warp work items
  const size_t smem = col_smem_bytes<kE4M3, true>(G);
  auto kern = mx_quant_colwise_kernel<kE4M3, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_status(e);
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kColThreads, smem);
  if (e != cudaSuccess) return cuda_status(e);
  const int64_t want = (total + kColThreads / 32 - 1) / (kColThreads / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)dev.sms * std::max(per_sm, 1)));
  kern<<<grid, kColThreads, smem, s>>>(static_cast<const __nv_bfloat16*>(in), M, (int)C, group_lens, G, codes_t,
                                       nullptr, M_pad, err, amax_scale);
  return cuda_status(cudaGetLastError());
}

}  // namespace pgg
