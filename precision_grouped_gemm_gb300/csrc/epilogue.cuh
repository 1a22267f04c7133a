// Epilogues shared by the grouped GEMM kernels: drain one accumulator tile
// from TMEM (tcgen05.ld, 32 lanes x 32 fp32 columns per load) and write bf16.
//
// Thread (warp quarter q, lane) owns accumulator row q*32 + lane; `tb` is the
// TMEM address of that warp's lane quarter at the tile's first column.
#pragma once
#include "mx_codec.cuh"
#include "ptx.cuh"

namespace pgg {

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile WaitCtl* ctl) {
  bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// silu(x) = x sigmoid(x) with the fast exponential and division intrinsics: a few
// ulp of fp32, far inside the bf16 output's rounding, and short enough not to hold
// up the producer and MMA warps that share issue slots with the epilogue warps.
__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Store 32 consecutive fp32 values of one row as bf16 at dst[0..31], columns
// limited to ncols (<= 32).  16-byte vector stores when the chunk is whole.
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float* v, int ncols) {
  if (ncols >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]);
      w.y = pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]);
      w.z = pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]);
      w.w = pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]);
      d4[q] = w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < ncols) dst[j] = __float2bfloat16_rn(v[j]);
  }
}

__device__ __forceinline__ void load_row32(const __nv_bfloat16* src, float* v, int ncols) {
  if (ncols >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w = __ldg(s4 + q);
      v[q * 8 + 0] = bf16_lo(w.x); v[q * 8 + 1] = bf16_hi(w.x);
      v[q * 8 + 2] = bf16_lo(w.y); v[q * 8 + 3] = bf16_hi(w.y);
      v[q * 8 + 4] = bf16_lo(w.z); v[q * 8 + 5] = bf16_hi(w.z);
      v[q * 8 + 6] = bf16_lo(w.w); v[q * 8 + 7] = bf16_hi(w.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = j < ncols ? __bfloat162float(src[j]) : 0.0f;
  }
}

// Plain store: row `dst_row` (already offset to this thread's output row),
// accumulator columns 0..BN-1 -> output columns col0.., bounded by ncols.
// SCALED: every accumulator is multiplied by alpha first (per-tensor operand scales).
template <int BN, bool SCALED = false>
__device__ __forceinline__ void epi_store(uint32_t tb, __nv_bfloat16* dst_row, bool row_ok, int col0,
                                          int ncols, float alpha = 1.0f) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t rv[32];
    tmem_ld32(tb + c * 32, rv);
    tmem_ld_wait();
    const int c0 = col0 + c * 32;
    if (row_ok && c0 < ncols) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        v[j] = __uint_as_float(rv[j]);
        if constexpr (SCALED) v[j] *= alpha;
      }
      store_row32(dst_row + c0, v, min(32, ncols - c0));
    }
  }
}

// bf16 bit patterns of 32 fp32 values (round to nearest even, as store_row32).
__device__ __forceinline__ void bf16_bits32(const float* v, uint32_t (&b)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) b[j] = __bfloat16_as_ushort(__float2bfloat16_rn(v[j]));
}

// Optional fused MX output (QF = kE4M3 / kE2M1): the 32 bf16 values just stored at
// columns c0..c0+31 of row `grow` of a [rows, ld] tensor form one row-wise MX block;
// its codes and scale go to codes[grow, c0 ..] / scales[grow, c0 / 32] exactly as
// the row-wise quantize kernel would write them for the stored tensor.
template <int QF>
__device__ __forceinline__ void mx_emit(const float* v, uint8_t* codes, uint8_t* scales, size_t grow, int ld,
                                        int c0) {
  uint32_t b[32];
  bf16_bits32(v, b);
  const size_t cb = QF == kE4M3 ? (size_t)ld : (size_t)ld / 2;  // code bytes per row
  const uint32_t sc = quantize_block32<QF>(b, codes + grow * cb + (QF == kE4M3 ? c0 : c0 / 2));
  scales[grow * (size_t)(ld / 32) + c0 / 32] = (uint8_t)sc;
}

// FC1 SwiGLU: accumulator columns [0, BN/2) are gate columns col0.., [BN/2, BN)
// the matching up columns.  A[row, col0 + c] = silu(gate) * up (fp32), and the
// pre-activation H[row, col0 + c] = gate, H[row, I + col0 + c] = up when H != null.
// QF != 0 and qcodes != null: A is also emitted MX-quantized (row-wise, I % 32 == 0).
// limit > 0 clamps first: gate <- min(gate, limit), up <- clamp(up, -limit, limit); H
// keeps the values before the clamp.  SCALED: gate and up are the accumulators times alpha.
template <int BN, int QF = 0, bool SCALED = false>
__device__ __forceinline__ void epi_swiglu(uint32_t tb, __nv_bfloat16* A, __nv_bfloat16* H, size_t grow,
                                           bool row_ok, int col0, int I, uint8_t* qcodes = nullptr,
                                           uint8_t* qscales = nullptr, float limit = 0.0f, float alpha = 1.0f) {
#pragma unroll 1
  for (int c = 0; c < BN / 64; ++c) {
    uint32_t rg[32], ru[32];
    tmem_ld32(tb + c * 32, rg);
    tmem_ld32(tb + BN / 2 + c * 32, ru);
    tmem_ld_wait();
    const int c0 = col0 + c * 32;
    if (row_ok && c0 < I) {
      float g[32], u[32], a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        g[j] = __uint_as_float(rg[j]);
        u[j] = __uint_as_float(ru[j]);
        if constexpr (SCALED) {
          g[j] *= alpha;
          u[j] *= alpha;
        }
        const float gc = limit > 0.0f ? fminf(g[j], limit) : g[j];
        const float uc = limit > 0.0f ? fminf(fmaxf(u[j], -limit), limit) : u[j];
        a[j] = silu_f(gc) * uc;
      }
      const int nc = min(32, I - c0);
      store_row32(A + grow * I + c0, a, nc);
      if (QF != 0 && qcodes) mx_emit<QF == 0 ? 1 : QF>(a, qcodes, qscales, grow, I, c0);
      if (H) {
        store_row32(H + grow * (2 * (size_t)I) + c0, g, nc);
        store_row32(H + grow * (2 * (size_t)I) + I + c0, u, nc);
      }
    }
  }
}

// FC2 dgrad + SwiGLU backward: accumulator = dA[row, col0 ..]; with g, u from
// the saved H: dH[:, c] = dA u s (1 + g (1 - s)), dH[:, I + c] = dA g s, s = sigmoid(g).
// QF != 0 and qcodes != null: dH [rows, 2I] is also emitted MX-quantized (row-wise).
// The saved H is read a chunk ahead of its use (raw bf16 words in registers), so the
// load latency overlaps the previous chunk's arithmetic; epi_swiglu_bwd_prefetch,
// called before the accumulator wait, has already pulled the tile's H into L2.
template <int BN>
__device__ __forceinline__ void epi_swiglu_bwd_prefetch(const __nv_bfloat16* H, size_t grow, bool row_ok,
                                                        int col0, int I) {
  if (!row_ok) return;
  const __nv_bfloat16* g = H + grow * (2 * (size_t)I) + col0;
  const int n = min(BN, I - col0);  // columns of this tile in each half
  if (n <= 0) return;
#pragma unroll 1
  for (int b = 0; b < n * 2; b += 128) {  // 128-byte lines of the gate and up segments
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(g) + b));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(g + I) + b));
  }
}

// 32 bf16 of a row (ncols < 32: the tail, zero-filled) as raw words.
__device__ __forceinline__ void load_raw32(const __nv_bfloat16* src, uint4 (&w)[4], int ncols) {
  if (ncols >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = __ldg(s4 + q);
  } else {
    const uint16_t* s16 = reinterpret_cast<const uint16_t*>(src);
    uint32_t* ww = reinterpret_cast<uint32_t*>(w);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t lo = 2 * j < ncols ? s16[2 * j] : 0u, hi = 2 * j + 1 < ncols ? s16[2 * j + 1] : 0u;
      ww[j] = lo | (hi << 16);
    }
  }
}

// limit > 0: the forward's clamp is applied to the saved g, u again, and the gradient
// is zero where a clamp was active (g > limit, |u| > limit).  SCALED: dA is the
// accumulator times alpha.
template <int BN, int QF = 0, bool SCALED = false>
__device__ __forceinline__ void epi_swiglu_bwd(uint32_t tb, __nv_bfloat16* dH, const __nv_bfloat16* H,
                                               size_t grow, bool row_ok, int col0, int I,
                                               uint8_t* qcodes = nullptr, uint8_t* qscales = nullptr,
                                               float limit = 0.0f, float alpha = 1.0f) {
  const __nv_bfloat16* hrow = H + grow * (2 * (size_t)I);
  uint4 ng[4], nu[4];  // the next chunk's gate / up words
  if (row_ok && col0 < I) {
    load_raw32(hrow + col0, ng, I - col0);
    load_raw32(hrow + I + col0, nu, I - col0);
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int c0 = col0 + c * 32;
    uint4 wg[4], wu[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      wg[q] = ng[q];
      wu[q] = nu[q];
    }
    if (row_ok && c0 + 32 < I && c + 1 < BN / 32) {
      load_raw32(hrow + c0 + 32, ng, I - c0 - 32);
      load_raw32(hrow + I + c0 + 32, nu, I - c0 - 32);
    }
    uint32_t rd[32];
    tmem_ld32(tb + c * 32, rd);
    tmem_ld_wait();
    if (row_ok && c0 < I) {
      const int nc = min(32, I - c0);
      const uint32_t* pg = reinterpret_cast<const uint32_t*>(wg);
      const uint32_t* pu = reinterpret_cast<const uint32_t*>(wu);
      float dg[32], du[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float hg = (j & 1) ? bf16_hi(pg[j >> 1]) : bf16_lo(pg[j >> 1]);
        float hu = (j & 1) ? bf16_hi(pu[j >> 1]) : bf16_lo(pu[j >> 1]);
        const float da = SCALED ? __uint_as_float(rd[j]) * alpha : __uint_as_float(rd[j]);
        bool pass_g = true, pass_u = true;
        if (limit > 0.0f) {
          pass_g = hg <= limit;
          pass_u = fabsf(hu) <= limit;
          hg = fminf(hg, limit);
          hu = fminf(fmaxf(hu, -limit), limit);
        }
        const float s = __fdividef(1.0f, 1.0f + __expf(-hg));
        dg[j] = pass_g ? da * hu * s * (1.0f + hg * (1.0f - s)) : 0.0f;
        du[j] = pass_u ? da * hg * s : 0.0f;
      }
      store_row32(dH + grow * (2 * (size_t)I) + c0, dg, nc);
      store_row32(dH + grow * (2 * (size_t)I) + I + c0, du, nc);
      if (QF != 0 && qcodes) {
        mx_emit<QF == 0 ? 1 : QF>(dg, qcodes, qscales, grow, 2 * I, c0);
        mx_emit<QF == 0 ? 1 : QF>(du, qcodes, qscales, grow, 2 * I, I + c0);
      }
    }
  }
}

// Full-tile store through shared memory and TMA: this warp's 32 rows go out as
// 32 x 64 bf16 boxes (4 KB, 128B-swizzled) staged in two alternating buffers
// at `stg`, written by bulk tensor stores of the 3-D map {cols, rows, G} at
// (col0 + 64 c, row0, g) that clip at the tensor bounds.  zero: write zeros
// without touching TMEM.  A box starting past rows_total / cols_total is
// skipped (warp-uniform), keeping one committed store per used buffer.
// SCALED: values are multiplied by alpha before the bf16 rounding.
template <int BN, bool SCALED = false>
__device__ __forceinline__ void epi_tma_store_rows(uint32_t tb, bool zero, uint8_t* stg, int& nstore,
                                                   const CUtensorMap* tmC, int row0, int col0, int g,
                                                   int rows_total, int cols_total, int lane,
                                                   float alpha = 1.0f) {
#pragma unroll 1
  for (int c = 0; c < BN / 64; ++c) {
    if (row0 >= rows_total || col0 + c * 64 >= cols_total) continue;
    uint32_t ra[32], rb[32];
    if (!zero) {
      tmem_ld32(tb + c * 64, ra);
      tmem_ld32(tb + c * 64 + 32, rb);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) { ra[j] = 0u; rb[j] = 0u; }
    }
    if constexpr (SCALED) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        ra[j] = __float_as_uint(__uint_as_float(ra[j]) * alpha);
        rb[j] = __float_as_uint(__uint_as_float(rb[j]) * alpha);
      }
    }
    uint8_t* sb = stg + (nstore & 1) * 4096;
    if (lane == 0) bulk_wait_read<1>();  // the store that last read this buffer is done
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t* v = j < 4 ? &ra[j * 8] : &rb[(j - 4) * 8];
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
      w.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
      w.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
      w.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
      *reinterpret_cast<uint4*>(sb + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmC, smem_u32(sb), col0 + c * 64, row0, g);
      bulk_commit();
    }
    ++nstore;
  }
}

// Store through the 4-D view {64, rows, cols/64, G} of the output (cols a
// multiple of 64): this warp's 32 rows x BN columns are staged as BN/64 atoms of
// 32 x 64 bf16 (4 KB each, 128B-swizzled) in its `stg` buffer and leave in
// BN/64/SA bulk tensor stores of SA atoms each, at (0, row0, col0 / 64 + s SA, g),
// clipped at the bounds, one bulk group per store.  The atoms cycle through RING
// slots of `stg` (RING a multiple of SA): before a slot is rewritten only the
// store that last read it -- RING/SA groups back -- has to be done reading, so
// with RING/SA > 1 stores drain while the next atoms are filled.  Stores that
// start past `cols_total` are skipped but still commit an (empty) group, which
// keeps that count exact.  SCALED: values are multiplied by alpha before the bf16 rounding.
template <int BN, int SA, int RING = BN / 64, bool SCALED = false>
__device__ __forceinline__ void epi_tma_store_tile(uint32_t tb, bool zero, uint8_t* stg,
                                                   const CUtensorMap* tmC4, int row0, int col0, int g,
                                                   int rows_total, int cols_total, int lane,
                                                   float alpha = 1.0f) {
  static_assert(SA >= 1 && (BN / 64) % SA == 0 && RING % SA == 0, "atoms per store");
  constexpr int NS = BN / 64 / SA;
  constexpr int NW = RING / SA;  // stores sharing the ring
  if (row0 >= rows_total) return;  // nothing of this warp's rows exists (warp-uniform)
#pragma unroll 1
  for (int st = 0; st < NS; ++st) {
#pragma unroll 1
    for (int i = 0; i < SA; ++i) {
      const int a = st * SA + i;
      uint32_t v[64];
      if (!zero) {
        tmem_ld64(tb + a * 64, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = 0u;
      }
      if constexpr (SCALED) {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
      }
      if (i == 0) {
        if (lane == 0) bulk_wait_read<NW - 1>();  // the store that last read these slots
        __syncwarp();
      }
      uint8_t* sb = stg + (a % RING) * 4096;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 w;
        w.x = pack_bf16x2(__uint_as_float(v[j * 8 + 0]), __uint_as_float(v[j * 8 + 1]));
        w.y = pack_bf16x2(__uint_as_float(v[j * 8 + 2]), __uint_as_float(v[j * 8 + 3]));
        w.z = pack_bf16x2(__uint_as_float(v[j * 8 + 4]), __uint_as_float(v[j * 8 + 5]));
        w.w = pack_bf16x2(__uint_as_float(v[j * 8 + 6]), __uint_as_float(v[j * 8 + 7]));
        *reinterpret_cast<uint4*>(sb + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (col0 + st * SA * 64 < cols_total)
        tma_store_4d(tmC4, smem_u32(stg + ((st * SA) % RING) * 4096), 0, row0, col0 / 64 + st * SA, g);
      bulk_commit();
    }
  }
}

// fp32 accumulate: this warp's 32 rows x BN columns are added to an fp32 output
// with bulk tensor reduce-adds, 64 columns at a time.  Each 64-column piece is
// staged as two 32 x 32 fp32 atoms (4 KB each, 128B-swizzled) in one of two
// alternating 8 KB halves of `stg` and leaves with one reduce-add of the 4-D
// view {32, rows, cols/32, G} at (0, row0, (col0 + 64 p) / 32, g) (r4d), or two
// of the 3-D view {cols, rows, G} (cols not a multiple of 32).  Every element
// gets exactly one add per call, so the result is deterministic.
template <int BN>
__device__ __forceinline__ void epi_tma_reduce_f32(uint32_t tb, uint8_t* stg, int& nstore,
                                                   const CUtensorMap* tmC, int row0, int col0, int g,
                                                   int rows_total, int cols_total, bool r4d, int lane) {
  if (row0 >= rows_total) return;
#pragma unroll 1
  for (int p = 0; p < BN / 64; ++p) {
    const int c0 = col0 + p * 64;
    if (c0 >= cols_total) break;
    uint32_t v[64];
    tmem_ld64(tb + p * 64, v);
    tmem_ld_wait();
    uint8_t* sb = stg + (nstore & 1) * 8192;
    if (lane == 0) bulk_wait_read<1>();  // the reduce that last read this half is done
    __syncwarp();
#pragma unroll
    for (int a = 0; a < 2; ++a) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint4 w = make_uint4(v[a * 32 + j * 4 + 0], v[a * 32 + j * 4 + 1], v[a * 32 + j * 4 + 2],
                             v[a * 32 + j * 4 + 3]);
        *reinterpret_cast<uint4*>(sb + a * 4096 + lane * 128 + ((j ^ (lane & 7)) << 4)) = w;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (r4d) {
        tma_reduce_add_4d(tmC, smem_u32(sb), 0, row0, c0 / 32, g);
      } else {
        tma_reduce_add_3d(tmC, smem_u32(sb), c0, row0, g);
        if (c0 + 32 < cols_total) tma_reduce_add_3d(tmC, smem_u32(sb) + 4096, c0 + 32, row0, g);
      }
      bulk_commit();
    }
    ++nstore;
  }
}

}  // namespace pgg
