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

// ---------------------------------------------------------------- warp-transposed row I/O
// In the fwd / dgrad epilogues each lane owns one accumulator row, so a plain 16-byte-per-
// lane access touches 32 rows at once: 32 L1 wavefronts per instruction.  Staged through
// the warp's 2 KB buffer, each global access instead covers 8 rows x 64 contiguous bytes.
// (Per-role clock64 timing of the MXFP4 FC2 dgrad + SwiGLU backward: leaving out its dH
// stores halved the kernel, leaving out its H loads cut it by a fifth.)
// The buffer holds 32 rows x 64 bytes; 16-byte chunk j of row r sits at
// r * 64 + 16 (j ^ ((r >> 1) & 3)), so that both the row-wise accesses (lane = row) and
// the transposed ones (8 rows x 4 chunks per instruction) spread over all banks.
__device__ __forceinline__ uint32_t stg_off(int r, int j) { return r * 64 + ((j ^ ((r >> 1) & 3)) << 4); }

// Lane `lane` holds row `lane`'s 32 bf16 values packed in w[16]; rows [0, nrows) of the
// warp's 32 and columns [0, ncols) (a multiple of 8) are stored at dst (row 0, column 0;
// row stride ld elements).  Warp-collective: every lane calls it with the same arguments
// except w.
__device__ __forceinline__ void store_rows32_t(uint8_t* stg, const uint32_t (&w)[16], __nv_bfloat16* dst,
                                               size_t ld, int nrows, int ncols, int lane) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(stg + stg_off(lane, j)) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  __syncwarp();
  const int J = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int R = 8 * i + (lane >> 2);
    const uint4 v = *reinterpret_cast<const uint4*>(stg + stg_off(R, J));
    if (R < nrows && 8 * J < ncols) *reinterpret_cast<uint4*>(dst + (size_t)R * ld + 8 * J) = v;
  }
  __syncwarp();
}

// Global half of the transposed load: lane `lane` fetches 16 bytes (columns 8 J .. 8 J + 7,
// J = lane % 4) of rows 8 i + lane / 4, i = 0..3, of a 32-row x 32-column bf16 chunk at src;
// rows past nrows and columns past ncols read as 0.
__device__ __forceinline__ void load_rows32_issue(const __nv_bfloat16* src, size_t ld, int nrows, int ncols,
                                                  uint4 (&v)[4], int lane) {
  const int J = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int R = 8 * i + (lane >> 2);
    v[i] = (R < nrows && 8 * J < ncols) ? __ldg(reinterpret_cast<const uint4*>(src + (size_t)R * ld + 8 * J))
                                        : make_uint4(0, 0, 0, 0);
  }
}
// Shared half: the fetched chunk, transposed through stg, lands in w[16] as row `lane`.
__device__ __forceinline__ void load_rows32_finish(uint8_t* stg, const uint4 (&v)[4], uint32_t (&w)[16], int lane) {
  const int J = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(stg + stg_off(8 * i + (lane >> 2), J)) = v[i];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 x = *reinterpret_cast<const uint4*>(stg + stg_off(lane, j));
    w[4 * j] = x.x; w[4 * j + 1] = x.y; w[4 * j + 2] = x.z; w[4 * j + 3] = x.w;
  }
  __syncwarp();
}

// 32 fp32 values -> 16 words of bf16 pairs (round to nearest even).
__device__ __forceinline__ void pack32(const float* v, uint32_t (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
}

// Staging bytes per epilogue warp of the fwd / dgrad epilogues: one 2 KB chunk buffer, which
// every transposed load and store reuses in turn (each completes behind a warp barrier).
constexpr int kEpiRowStageBytes = 2048;

// Plain store: the warp's 32 accumulator rows are output rows row0w .. row0w + 31, of which
// the first nrows exist; accumulator columns 0..BN-1 -> output columns col0.., bounded by
// ncols; output row stride ld.  SCALED: every accumulator is multiplied by alpha first
// (per-tensor operand scales).
template <int BN, bool SCALED = false>
__device__ __forceinline__ void epi_store(uint32_t tb, __nv_bfloat16* out, size_t ld, size_t row0w, int nrows,
                                          int col0, int ncols, uint8_t* stg, int lane, float alpha = 1.0f) {
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t rv[32];
    tmem_ld32(tb + c * 32, rv);
    tmem_ld_wait();
    const int c0 = col0 + c * 32;
    if (c0 < ncols) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        v[j] = __uint_as_float(rv[j]);
        if constexpr (SCALED) v[j] *= alpha;
      }
      uint32_t w[16];
      pack32(v, w);
      store_rows32_t(stg, w, out + row0w * ld + c0, ld, nrows, min(32, ncols - c0), lane);
    }
  }
}

// Plain store through a whole-tile stage, so that tensor memory is free before the global
// stores: pass 1 (epi_stage_tile) converts the warp's 32 rows x BN accumulators to bf16 into
// stg (32 rows x 2 BN bytes, 16-byte chunk j of row r at position j ^ (r % 8) of its row);
// the caller then releases the accumulator; pass 2 (epi_store_staged) writes the rows out,
// 8 rows x 64 contiguous bytes per instruction.  SCALED as epi_store.
template <int BN, bool SCALED = false>
__device__ __forceinline__ void epi_stage_tile(uint32_t tb, uint8_t* stg, int lane, float alpha = 1.0f) {
  uint8_t* row = stg + lane * (2 * BN);
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t rv[32];
    tmem_ld32(tb + c * 32, rv);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = __uint_as_float(rv[j]);
      if constexpr (SCALED) v[j] *= alpha;
    }
    uint32_t w[16];
    pack32(v, w);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(row + (((4 * c + k) ^ (lane & 7)) << 4)) =
          make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
  }
}
// Pass 2: NC staged columns starting at stage column s0 (a multiple of 32; the stage's rows hold
// PITCH columns) go to output columns col0 .. of rows row0w ..; columns from ncols on are dropped.
template <int NC, int PITCH = NC>
__device__ __forceinline__ void epi_store_staged(const uint8_t* stg, __nv_bfloat16* out, size_t ld, size_t row0w,
                                                 int nrows, int col0, int ncols, int lane, int s0 = 0) {
  __syncwarp();
  const int J = lane & 3;
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    const int c0 = col0 + c * 32;
    if (c0 >= ncols) break;
    const int nc = min(32, ncols - c0);
    const int ch = s0 / 8 + 4 * c + J;  // 16-byte chunk of the staged row
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int R = 8 * i + (lane >> 2);
      const uint4 x = *reinterpret_cast<const uint4*>(stg + R * (2 * PITCH) + ((ch ^ (R & 7)) << 4));
      if (R < nrows && 8 * J < nc) *reinterpret_cast<uint4*>(out + (row0w + R) * ld + c0 + 8 * J) = x;
    }
  }
  __syncwarp();
}

// Optional fused MX output (QF = kE4M3 / kE2M1): the 32 bf16 values just stored at
// columns c0..c0+31 of row `grow` of a [rows, ld] tensor -- w[16], packed in pairs exactly
// as stored -- form one row-wise MX block; its codes and scale go to codes[grow, c0 ..] /
// scales[grow, c0 / 32] exactly as the row-wise quantize kernel would write them for the
// stored tensor.
template <int QF>
__device__ __forceinline__ void mx_emit(const uint32_t (&w)[16], uint8_t* codes, uint8_t* scales, size_t grow,
                                        int ld, int c0) {
  const size_t cb = QF == kE4M3 ? (size_t)ld : (size_t)ld / 2;  // code bytes per row
  const uint32_t sc = quantize_block32_packed<QF>(w, codes + grow * cb + (QF == kE4M3 ? c0 : c0 / 2));
  scales[grow * (size_t)(ld / 32) + c0 / 32] = (uint8_t)sc;
}

// FC1 SwiGLU: accumulator columns [0, BN/2) are gate columns col0.., [BN/2, BN)
// the matching up columns.  A[row, col0 + c] = silu(gate) * up (fp32), and the
// pre-activation H[row, col0 + c] = gate, H[row, I + col0 + c] = up when H != null.
// QF != 0 and qcodes != null: A is also emitted MX-quantized (row-wise, I % 32 == 0).
// limit > 0 clamps first: gate <- min(gate, limit), up <- clamp(up, -limit, limit); H
// keeps the values before the clamp.  SCALED: gate and up are the accumulators times alpha.
// Rows as epi_store; this thread's own row is grow (row_ok: it exists).  The warp handles the
// 32-column chunks [cb, ce) of each half (all of them by default).
template <int BN, int QF = 0, bool SCALED = false>
__device__ __forceinline__ void epi_swiglu(uint32_t tb, __nv_bfloat16* A, __nv_bfloat16* H, size_t row0w,
                                           int nrows, bool row_ok, size_t grow, int col0, int I, uint8_t* stg,
                                           int lane, uint8_t* qcodes = nullptr, uint8_t* qscales = nullptr,
                                           float limit = 0.0f, float alpha = 1.0f, int cb = 0, int ce = BN / 64) {
#pragma unroll 1
  for (int c = cb; c < ce; ++c) {
    uint32_t rg[32], ru[32];
    tmem_ld32(tb + c * 32, rg);
    tmem_ld32(tb + BN / 2 + c * 32, ru);
    tmem_ld_wait();
    const int c0 = col0 + c * 32;
    if (c0 < I) {
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
      uint32_t w[16];
      pack32(a, w);
      store_rows32_t(stg, w, A + row0w * I + c0, I, nrows, nc, lane);
      if (QF != 0 && qcodes && row_ok) mx_emit<QF == 0 ? 1 : QF>(w, qcodes, qscales, grow, I, c0);
      if (H) {
        const size_t ldh = 2 * (size_t)I;
        pack32(g, w);
        store_rows32_t(stg, w, H + row0w * ldh + c0, ldh, nrows, nc, lane);
        pack32(u, w);
        store_rows32_t(stg, w, H + row0w * ldh + I + c0, ldh, nrows, nc, lane);
      }
    }
  }
}

// FC2 dgrad + SwiGLU backward: accumulator = dA[row, col0 ..]; with g, u from
// the saved H: dH[:, c] = dA u s (1 + g (1 - s)), dH[:, I + c] = dA g s, s = sigmoid(g).
// QF != 0 and qcodes != null: dH [rows, 2I] is also emitted MX-quantized (row-wise).
// Each lane reads its own row of H a chunk ahead of its use (the loads of chunk c + 1 are
// in flight during chunk c's arithmetic and stores); epi_swiglu_bwd_prefetch, called
// before the accumulator wait, has already pulled the tile's H into L2.
template <int BN>
__device__ __forceinline__ void epi_swiglu_bwd_prefetch(const __nv_bfloat16* H, size_t grow, bool row_ok,
                                                        int col0, int I, int cb = 0, int ce = BN / 32) {
  if (!row_ok) return;
  const __nv_bfloat16* g = H + grow * (2 * (size_t)I) + col0 + cb * 32;
  const int n = min(32 * (ce - cb), I - col0 - cb * 32);  // columns of the chunks [cb, ce) in each half
  if (n <= 0) return;
#pragma unroll 1
  for (int b = 0; b < n * 2; b += 128) {  // 128-byte lines of the gate and up segments
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(g) + b));
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(g + I) + b));
  }
}

// limit > 0: the forward's clamp is applied to the saved g, u again, and the gradient
// is zero where a clamp was active (g > limit, |u| > limit).  SCALED: dA is the
// accumulator times alpha.  TSTORE: dH goes out warp-transposed through stg; otherwise each
// lane stores its own row.  (Timed on the full layer steps: transposed stores are faster in
// the BF16 kernel, per-lane stores in the block-scaled one; transposed H loads lost in both.)
// The warp handles the 32-column chunks [cb, ce) of the tile (all of them by default).
// Warp-collective (stg, TSTORE): every lane calls it with the same tile arguments.
__device__ __forceinline__ void ld_row32(const __nv_bfloat16* src, uint4 (&w)[4], int ncols) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    w[q] = 8 * q < ncols ? __ldg(reinterpret_cast<const uint4*>(src) + q) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void st_row32(__nv_bfloat16* dst, const uint32_t (&w)[16], int ncols) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (8 * q < ncols)
      reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}
template <int BN, int QF = 0, bool SCALED = false, bool TSTORE = true>
__device__ __forceinline__ void epi_swiglu_bwd(uint32_t tb, __nv_bfloat16* dH, const __nv_bfloat16* H,
                                               size_t row0w, int nrows, bool row_ok, size_t grow, int col0, int I,
                                               uint8_t* stg, int lane, uint8_t* qcodes = nullptr,
                                               uint8_t* qscales = nullptr, float limit = 0.0f, float alpha = 1.0f,
                                               int cb = 0, int ce = BN / 32) {
  const size_t ldh = 2 * (size_t)I;
  const __nv_bfloat16* hrow = H + grow * ldh;
  uint4 ng[4], nu[4];  // the next chunk's gate / up words of this lane's row
  if (row_ok && col0 + cb * 32 < I) {
    ld_row32(hrow + col0 + cb * 32, ng, I - col0 - cb * 32);
    ld_row32(hrow + I + col0 + cb * 32, nu, I - col0 - cb * 32);
  }
#pragma unroll 1
  for (int c = cb; c < ce; ++c) {
    const int c0 = col0 + c * 32;
    uint32_t hgw[16], huw[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      hgw[4 * q] = ng[q].x; hgw[4 * q + 1] = ng[q].y; hgw[4 * q + 2] = ng[q].z; hgw[4 * q + 3] = ng[q].w;
      huw[4 * q] = nu[q].x; huw[4 * q + 1] = nu[q].y; huw[4 * q + 2] = nu[q].z; huw[4 * q + 3] = nu[q].w;
    }
    if (row_ok && c0 + 32 < I && c + 1 < ce) {
      ld_row32(hrow + c0 + 32, ng, I - c0 - 32);
      ld_row32(hrow + I + c0 + 32, nu, I - c0 - 32);
    }
    uint32_t rd[32];
    tmem_ld32(tb + c * 32, rd);
    tmem_ld_wait();
    if (c0 < I) {
      const int nc = min(32, I - c0);
      float dg[32], du[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float hg = (j & 1) ? bf16_hi(hgw[j >> 1]) : bf16_lo(hgw[j >> 1]);
        float hu = (j & 1) ? bf16_hi(huw[j >> 1]) : bf16_lo(huw[j >> 1]);
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
      uint32_t w[16];
      pack32(dg, w);
      if constexpr (TSTORE) store_rows32_t(stg, w, dH + row0w * ldh + c0, ldh, nrows, nc, lane);
      else if (row_ok) st_row32(dH + grow * ldh + c0, w, nc);
      if (QF != 0 && qcodes && row_ok) mx_emit<QF == 0 ? 1 : QF>(w, qcodes, qscales, grow, 2 * I, c0);
      pack32(du, w);
      if constexpr (TSTORE) store_rows32_t(stg, w, dH + row0w * ldh + I + c0, ldh, nrows, nc, lane);
      else if (row_ok) st_row32(dH + grow * ldh + I + c0, w, nc);
      if (QF != 0 && qcodes && row_ok) mx_emit<QF == 0 ? 1 : QF>(w, qcodes, qscales, grow, 2 * I, I + c0);
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
