// BF16 grouped GEMM on the 5th-generation tensor cores (tcgen05, kind::f16).
//
// Problem ("Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X GPUs
// with Primus", section "Expert parallelism: DeepEP and the grouped GEMM"):
// one kernel runs every expert's GEMM over a ragged, expert-sorted token
// batch.  Three operand arrangements share this kernel:
//
//   kFwd   Y_g  = X_g  . W_g^T   A = X  [M,K] K-major,   B = W [G,N,K] K-major
//   kDgrad dX_g = dY_g . W_g     A = dY [M,N] K-major,   B = W [G,N,K] read MN-major
//   kWgrad dW_g = dY_g^T . X_g   A = dY [M,N] MN-major,  B = X [M,K] MN-major,
//                                reduction over group g's own rows (variable K)
//
// and three epilogues: plain bf16 store, the FC1 SwiGLU (A = silu(gate)*up with
// the optional pre-activation H saved), and the FC2-dgrad SwiGLU backward (dH
// from dA and the saved H) -- the expert path GEMM1 -> SwiGLU -> GEMM2 of the
// same page, section "MegaMoE: fusing communication into the grouped GEMM".
//
// CTA = 6 warps: warp 0 issues TMA loads into a STAGES-deep shared-memory ring,
// warp 1 owns TMEM and issues tcgen05.mma from one lane, warps 2..5 drain the
// double-buffered fp32 accumulator (2 x BN TMEM columns) with tcgen05.ld and
// store bf16 results bounded to the tile's group.  Persistent: one CTA per SM.
#pragma once
#include "epilogue.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace pgg {

constexpr int kBM = 128;          // MMA M (TMEM lanes)
// Reduction rows per pipeline stage (BK): 64 (one 128-byte swizzle atom of bf16) for
// the K-major fwd / dgrad operands.  wgrad runs 32 when groups are short (a few
// hundred rows): twice the stages in the same shared memory keep more of the short
// k-loop in flight (4% faster on the DeepSeek-shaped fc1 wgrad); long reductions
// keep 64 (fewer, larger steps; 10% faster on the GPT-OSS-shaped wgrad).
constexpr int kGemmThreads = 192;
// 64-column atoms per bulk store of a wgrad output tile: one atom per store lets a
// tile's stores drain while the next tile is staged.
constexpr int kWgradStoreAtoms = 1;

struct GemmArgs {
  const int32_t* group_lens;
  int G;
  int64_t M;        // rows of the ragged operand (sum of group_lens)
  int out_cols;     // columns of the accumulator space: fwd N, dgrad K, wgrad K, swiglu I
  int red;          // reduction length for fwd / dgrad (K resp. N)
  int wg_rows;      // wgrad: N (rows of dW_g)
  float swiglu_limit;  // SwiGLU epilogues: clamp limit (0: none)
  int I;            // SwiGLU width (gate/up halves)
  void* out;        // Y, dX, dW, A or dH (bf16)
  void* out2;       // SwiGLU forward: H (bf16 [M, 2I]) or nullptr
  const void* aux;  // SwiGLU backward: saved H (bf16 [M, 2I])
  int32_t* err;     // device error word or nullptr
  FastDiv nct;      // wgrad: column tiles per row tile
  int c4d;          // wgrad: tmC is the 4-D atom view (cols % 64 == 0)
  int a_multi;      // wgrad: tmA is the atom view {64, M, N/64} (one load per k-block)
  int b_multi;      // wgrad / dgrad: tmB is the atom view of X {64, M, K/64} / W {64, N, K/64, G}
  unsigned long long wait_ns;  // pipeline wait limit (0: kWaitTimeoutNs)
  long long stall_at;          // test hook: the producer stops before this k-block (-1: never)
};

// Shared memory: STAGES x (A tile | B tile), the epilogue staging buffers
// (wgrad: 4 warps x 2 x 4 KB, 1024-byte aligned for the 128-byte swizzle), the
// mbarriers and the group scan arrays.
template <int BN, int BK, int STAGES, int EPI_BYTES>
struct GemmSmem {
  static constexpr int kABytes = kBM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kEpiOff = STAGES * kStageBytes;
  static constexpr int kBarOff = kEpiOff + EPI_BYTES;
  static constexpr int kBarBytes = 256;
  static constexpr int kGroupOff = kBarOff + kBarBytes;
  static __host__ __device__ constexpr size_t bytes(int G) {
    return 1024 + (size_t)kGroupOff + 8 * (size_t)(G + 1) + 16;
  }
};

// Epilogue staging bytes: the wgrad store keeps a ring of kWgradRing 4 KB atoms per
// epilogue warp; the fp32 accumulate two 8 KB halves per warp; the fwd / dgrad epilogues
// a 2 KB chunk buffer per warp.
constexpr int kWgradRing = 2;
template <int MODE, int EPI>
__host__ __device__ constexpr int epi_bytes() {
  return MODE != kWgrad ? 4 * kEpiRowStageBytes
                        : (EPI == kEpiAccumF32 ? 4 * 16384 : 4 * kWgradRing * 4096);
}

struct Tile {
  int g, row0, rows, col0, nkb, red0, red_valid;
};

template <int MODE, int EPI, int BN>
__device__ __forceinline__ int tile_cols() {
  return EPI == kEpiSwiGLU ? BN / 2 : BN;
}

template <int MODE, int EPI, int BN, int BK>
__device__ __forceinline__ Tile decode_tile(int t, const GemmArgs& a, const int32_t* s_off,
                                            const int32_t* s_tile, GroupCursor& cur) {
  Tile T;
  cur.at(s_tile, s_off, nullptr, a.G, t);
  const int local = t - cur.t_lo;
  const int off = cur.off, len = cur.len;
  T.g = cur.g;
  if (MODE == kWgrad) {
    // column tiles vary fastest: the CTAs running at one time fill whole rows of dW_g
    const int rt = (int)a.nct.div((uint32_t)local);
    const int ct = local - rt * (int)a.nct.d;
    T.row0 = rt * kBM;
    T.rows = min(kBM, a.wg_rows - T.row0);
    T.col0 = ct * BN;
    T.nkb = (len + BK - 1) / BK;
    T.red0 = off;
    T.red_valid = len;
  } else {
    const int nmt = (len + kBM - 1) / kBM;
    const int mt = local % nmt, ct = local / nmt;
    T.row0 = off + mt * kBM;
    T.rows = min(kBM, len - mt * kBM);
    T.col0 = ct * tile_cols<MODE, EPI, BN>();
    T.nkb = (a.red + BK - 1) / BK;
    T.red0 = 0;
    T.red_valid = a.red;
  }
  return T;
}

template <int MODE, int EPI, int BN, int STAGES, int BK>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  static_assert(BK == 64 || (MODE == kWgrad && BK == 32), "k-block");
  using L = GemmSmem<BN, BK, STAGES, epi_bytes<MODE, EPI>()>;
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(EPI != kEpiSwiGLU || (MODE == kFwd && BN == 256), "SwiGLU fwd tile");
  static_assert(EPI != kEpiSwiGLUBwd || MODE == kDgrad, "SwiGLU bwd tile");
  static_assert(EPI != kEpiAccumF32 || MODE == kWgrad, "fp32 accumulation is a wgrad epilogue");
  constexpr uint32_t kTmemCols = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  constexpr bool kAmn = (MODE == kWgrad);
  constexpr bool kBmn = (MODE != kFwd);
  constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, kAmn, kBmn);
  // barriers, the wait control (16 B), the TMEM address and the bad-lens flag
  static_assert((2 * STAGES + 2 * 2 + 1) * 8 + 24 <= L::kBarBytes, "barrier area");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;                 // [STAGES]
  uint64_t* empty = bars + STAGES;       // [STAGES]
  uint64_t* tfull = bars + 2 * STAGES;   // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;          // [1]
  volatile WaitCtl* s_ctl = reinterpret_cast<volatile WaitCtl*>(drain + 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(const_cast<WaitCtl*>(s_ctl) + 1);
  int* s_bad = reinterpret_cast<int*>(s_tmem + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + L::kGroupOff);
  int32_t* s_tile = s_off + (args.G + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    s_ctl->abort = 0;
    s_ctl->limit_ns = args.wait_ns ? args.wait_ns : kWaitTimeoutNs;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) {
    TileCount tc;
    if (MODE == kWgrad) {
      tc.bm = 0;
      tc.per_row_tile = ((args.wg_rows + kBM - 1) / kBM) * ((args.out_cols + BN - 1) / BN);
    } else {
      constexpr int tcw = EPI == kEpiSwiGLU ? BN / 2 : BN;
      tc.bm = kBM;
      tc.per_row_tile = (args.out_cols + tcw - 1) / tcw;
    }
    bool bad = scan_groups(args.group_lens, args.G, args.M, tc, s_off, s_tile, nullptr, 0, lane);
    if (lane == 0) {
      *s_bad = bad ? 1 : 0;
      if (bad && blockIdx.x == 0) set_error(args.err, kErrBadGroupLens);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *s_tmem;
  const int total_tiles = *s_bad ? 0 : s_tile[args.G];
  const uint32_t smem_a0 = smem_u32(smem);
  const uint32_t smem_b0 = smem_a0 + STAGES * L::kABytes;
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    GroupCursor cur;
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool stalled = false;
    for (int t = blockIdx.x; t < total_tiles && !aborted && !stalled; t += gridDim.x) {
      const Tile T = decode_tile<MODE, EPI, BN, BK>(t, args, s_off, s_tile, cur);
      for (int kb = 0; kb < T.nkb; ++kb) {
        // test hook: stop producing, so that the consumers' waits run out (every load
        // issued so far is consumed, and so complete, before they do)
        if (issued == args.stall_at) { stalled = true; break; }
        if (!warp_wait(smem_u32(&empty[stage]), phase ^ 1u, s_ctl)) { aborted = true; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&full[stage]);
          const uint32_t sa = smem_a0 + stage * L::kABytes;
          const uint32_t sb = smem_b0 + stage * L::kBBytes;
          mbar_arrive_expect_tx(fb, L::kStageBytes);
          const int kr = kb * BK;
          if (MODE == kFwd) {
            tma_load_2d(sa, &tmA, fb, kr, T.row0);
            if (EPI == kEpiSwiGLU) {
              tma_load_3d(sb, &tmB, fb, kr, T.col0, T.g);
              tma_load_3d(sb + (BN / 2) * 128, &tmB, fb, kr, args.I + T.col0, T.g);
            } else {
              tma_load_3d(sb, &tmB, fb, kr, T.col0, T.g);
            }
          } else if (MODE == kDgrad) {
            tma_load_2d(sa, &tmA, fb, kr, T.row0);
            if (args.b_multi) {
              // BN/64 atoms of 64 k-columns x BK n-rows in one copy: smem [atom][row][64]
              tma_load_4d(sb, &tmB, fb, 0, kr, T.col0 / 64, T.g);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_3d(sb + j * BK * 128, &tmB, fb, T.col0 + 64 * j, kr, T.g);
            }
          } else {
            if (args.a_multi) {
              tma_load_3d(sa, &tmA, fb, 0, T.red0 + kr, T.row0 / 64);
            } else {
#pragma unroll
              for (int j = 0; j < kBM / 64; ++j) tma_load_2d(sa + j * BK * 128, &tmA, fb, T.row0 + 64 * j, T.red0 + kr);
            }
            if (args.b_multi) {
              tma_load_3d(sb, &tmB, fb, 0, T.red0 + kr, T.col0 / 64);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * BK * 128, &tmB, fb, T.col0 + 64 * j, T.red0 + kr);
            }
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (aborted && lane == 0) {
      // drain: wait for the loads still in flight before the CTA's smem goes away
      long long n = issued < STAGES ? issued : STAGES;
      int s = stage;
      uint32_t p = phase;
      for (long long i = 0; i < n; ++i) {
        if (--s < 0) { s = STAGES - 1; p ^= 1u; }
        mbar_wait_drain(smem_u32(&full[s]), p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    GroupCursor cur;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    // Descriptors of stage 0's A and B tiles.  The start-address field holds address / 16 in 14
    // bits, which every address of this block fits, so the descriptor of address + d (d a
    // multiple of 16) is the base descriptor + d / 16.
    const uint64_t kDescA = kAmn ? smem_desc(smem_a0, BK * 128, 1024, kSwizzle128B)
                                 : smem_desc(smem_a0, 16, 1024, kSwizzle128B);
    const uint64_t kDescB = kBmn ? smem_desc(smem_b0, BK * 128, 1024, kSwizzle128B)
                                 : smem_desc(smem_b0, 16, 1024, kSwizzle128B);
    for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
      const Tile T = decode_tile<MODE, EPI, BN, BK>(t, args, s_off, s_tile, cur);
      if (T.nkb == 0) continue;  // empty wgrad group: the epilogue writes zeros
      if (!warp_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, s_ctl)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < T.nkb; ++kb) {
        if (!warp_wait(smem_u32(&full[stage]), phase, s_ctl)) { aborted = true; break; }
        tc_fence_after();
        const uint32_t sa = smem_a0 + stage * L::kABytes;
        const uint32_t sb = smem_b0 + stage * L::kBBytes;
        // variable-K tail (wgrad): rows of this k-block past the group's end belong to the
        // next group (or lie past M); they are zeroed in both operands.  (Running only the
        // K=16 steps that hold group rows measured 4% slower on the DeepSeek-shaped fc1
        // wgrad than zeroing the rest of the k-block and running all four.)
        if (MODE == kWgrad) {
          const int valid = T.red_valid - kb * BK;
          if (valid < BK) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            uint8_t* pa = smem + (sa - smem_a0);
            uint8_t* pb = smem + (sb - smem_a0);
            // each atom column is [BK rows][128 B]; lane writes 16-byte chunk (lane & 7)
            // of rows valid + (lane >> 3), +4, ... (the swizzle stays inside a row)
            const int c16 = (lane & 7) * 16;
            for (int row = valid + (lane >> 3); row < BK; row += 4) {
#pragma unroll
              for (int atom = 0; atom < kBM / 64; ++atom)
                *reinterpret_cast<uint4*>(pa + atom * BK * 128 + row * 128 + c16) = z;
#pragma unroll
              for (int atom = 0; atom < BN / 64; ++atom)
                *reinterpret_cast<uint4*>(pb + atom * BK * 128 + row * 128 + c16) = z;
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }
        if (lane == 0) {
          const uint64_t ao = (uint64_t)(sa - smem_a0) >> 4, bo = (uint64_t)(sb - smem_b0) >> 4;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            // K step ks: 16 rows (2048 bytes) further along an MN-major tile, 32 bytes along a K-major one
            const uint64_t ad = kDescA + ao + (kAmn ? 128 * ks : 2 * ks);
            const uint64_t bd = kDescB + bo + (kBmn ? 128 * ks : 2 * ks);
            mma_f16(d_tmem, ad, bd, kIdesc, (kb > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (aborted) break;
      if (lane == 0) mma_commit(smem_u32(&tfull[acc]));
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (aborted && lane == 0) {
      mma_commit(smem_u32(drain));
      mbar_wait_drain(smem_u32(drain), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;              // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;         // accumulator row held by this thread
    int acc = 0;
    uint32_t acc_phase = 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
    GroupCursor cur;
    uint8_t* stg = smem + L::kEpiOff + (warp - 2) * (epi_bytes<MODE, EPI>() / 4);  // this warp's staging
    int nstore = 0;
    for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
      const Tile T = decode_tile<MODE, EPI, BN, BK>(t, args, s_off, s_tile, cur);
      const bool row_ok = r < T.rows;
      if (MODE == kWgrad) {
        const bool zero = T.nkb == 0;  // empty group: dW_g = 0, no accumulator
        if (!zero) {
          if (!warp_wait(smem_u32(&tfull[acc]), acc_phase, s_ctl)) { aborted = true; break; }
          tc_fence_after();
        }
        const uint32_t tb = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
        if (EPI == kEpiAccumF32) {
          // main_grad += dW_g: an empty group adds nothing
          if (!zero)
            epi_tma_reduce_f32<BN>(tb, stg, nstore, &tmC, T.row0 + q * 32, T.col0, T.g, args.wg_rows,
                                   args.out_cols, args.c4d != 0, lane);
        } else if (args.c4d) {
          epi_tma_store_tile<BN, kWgradStoreAtoms, kWgradRing>(tb, zero, stg, &tmC, T.row0 + q * 32, T.col0, T.g, args.wg_rows,
                                 args.out_cols, lane);
        } else {
          epi_tma_store_rows<BN>(tb, zero, stg, nstore, &tmC, T.row0 + q * 32, T.col0, T.g, args.wg_rows,
                                 args.out_cols, lane);
        }
        if (!zero) {
          tc_fence_before();
          mbar_arrive(smem_u32(&tempty[acc]));
          if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        continue;
      }
      const size_t grow = (size_t)T.row0 + r;
      const size_t row0w = (size_t)T.row0 + q * 32;         // the warp's first output row
      const int nrows = max(0, min(32, T.rows - q * 32));    // of which this many exist
      if (EPI == kEpiSwiGLUBwd)  // the saved H of this tile streams into L2 while the MMAs run
        epi_swiglu_bwd_prefetch<BN>(reinterpret_cast<const __nv_bfloat16*>(args.aux), grow, row_ok, T.col0,
                                    args.I);
      if (!warp_wait(smem_u32(&tfull[acc]), acc_phase, s_ctl)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      if (EPI == kEpiSwiGLU) {
        epi_swiglu<BN>(tb, out, reinterpret_cast<__nv_bfloat16*>(args.out2), row0w, nrows, row_ok, grow, T.col0,
                       args.I, stg, lane, nullptr, nullptr, args.swiglu_limit);
      } else if (EPI == kEpiSwiGLUBwd) {
        epi_swiglu_bwd<BN>(tb, out, reinterpret_cast<const __nv_bfloat16*>(args.aux), row0w, nrows, row_ok, grow,
                           T.col0, args.I, stg, lane, nullptr, nullptr, args.swiglu_limit);
      } else {
        epi_store<BN>(tb, out, args.out_cols, row0w, nrows, T.col0, args.out_cols, stg, lane);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  if (MODE == kWgrad && warp >= 2 && lane == 0) bulk_wait<0>();
  if (aborted && lane == 0) set_error(args.err, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace pgg
