// Block-scaled (MX) grouped GEMM on tcgen05: e4m3 x e4m3 (kind::mxf8f6f4,
// scale_vec::1X) and packed e2m1 x e2m1 (kind::mxf4, scale_vec::2X), UE8M0
// scales per 32-element block of the reduction axis, fp32 accumulation in TMEM,
// bf16 output ("Primus-Turbo" README, "What's New": MXFP8 / MXFP4 grouped GEMM;
// Pull Request #891, "Changes": MXFP4 grouped GEMM on float4_e2m1fn_x2 buffers).
//
// Both operands are K-major along the reduction axis (the quantizers write them
// that way), and a k-block is 128 bytes of every row with the 128-byte swizzle:
// 128 e4m3 elements, or 256 packed e2m1 elements.  The producer warp loads codes with
// TMA and blocked scale atoms with bulk copies; row-major scales (activations) are
// gathered by a separate warp with 4-byte cp.async straight into the 512-byte atom the
// MMA wants (row m's 4 scales at byte 16 (m % 32) + 4 (m / 32)); a copier warp (or, in
// the e2m1 SwiGLU backward, the MMA warp itself) copies each atom into TMEM with
// tcgen05.cp (32x128b, replicated to the four lane quarters), and the MMA warp issues
// the block-scaled MMAs selecting scale bytes by ID.
//
//   fwd    out[M, N]    = A[M, K] . B_g[N, K]^T     A = X rows, B = W [G, N, K]
//   dgrad  out[M, K]    = A[M, N] . Bt_g[K, N]^T    Bt = W^T [K, G*N] (blocks along N)
//   wgrad  out[G, N, K] = At_g[N, .] . Bt_g[K, .]^T over group g's padded columns of
//                         the column-wise operands At = dY^T [N, M_pad], Bt = X^T [K, M_pad]
//
// FP8 tensor-wise operands (one fp32 scale s per tensor, codes = e4m3(x s)) run the
// e4m3 instantiations with TS = true: the plain FP8 MMA (kind::f8f6f4, no block scales:
// no scale loads, no scale copies to tensor memory), and the epilogue multiplies the
// accumulator by 1 / (s_A s_B) before the store or the SwiGLU (forward) / SwiGLU
// backward (dgrad).
#include <algorithm>

#include "epilogue.cuh"
#include "internal.h"
#include "mx_codec.cuh"
#include "ptx.cuh"
#include "sched.cuh"

namespace pgg {
namespace {

constexpr int kMxBM = 128, kMxBN = 128;
// Reduction elements per 512-byte scale atom (four 32-element blocks per row); also the
// padding granule of the column-wise layout.
constexpr int kMxAtomK = 128;
// wgrad tiles: e4m3 128 x 128 with three accumulators (128 x 256 with one accumulator --
// TMEM cannot hold two next to the scale factors -- measured 12% slower on the
// DeepSeek-shaped MXFP8 wgrads: the epilogue no longer overlaps the MMA); e2m1 128 x 256
// with one, which halves the scale copies per flop of the long Zipf-routed group k-loops.
constexpr int kMxWgradBNE4M3 = 128;
constexpr int kMxWgradBNE2M1 = 256;
// Forward / dgrad tile width per format.  A block-scaled MMA carries little work
// per instruction (128 x 128 x 64 e2m1 is ~24 ns of tensor time) and the MMA warp
// pays ~45 ns per MMA and ~36 ns per scale copy, so a 128-wide tile is issue-bound;
// 256-wide tiles double the work per MMA and per scale copy, at the price of a
// single TMEM accumulator.  On one GPU: MXFP4 fc2 fwd 1.46 -> 1.07 ms, fc1 dgrad
// 2.62 -> 1.71 ms; MXFP8 fc2 fwd 0.403 -> 0.368 ms, fc1 dgrad 0.762 -> 0.724 ms.
constexpr int kMxFwdBNE4M3 = 256;
constexpr int kMxFwdBNE2M1 = 256;
// The e4m3 FC2 dgrad + SwiGLU backward is the exception: its epilogue (read H, write dH and
// its MX codes) takes about as long as its MMAs, and the single accumulator of a 256-wide tile
// serialises the two; 128-wide tiles with three accumulators overlap them (timed on the
// DeepSeek-shaped layers: MXFP8 0.61 -> 0.55 ms, FP8 tensor-wise 0.54 -> 0.44 ms; the e2m1
// one is slower at 128, 1.61 -> 1.80 ms, and every other fwd / dgrad call at either format).
constexpr int kMxSwiGLUBwdBNE4M3 = 128;
// Tile width of a fwd / dgrad call; swiglu: the call's SwiGLU epilogue flag (a dgrad with it is
// the SwiGLU backward).
__host__ __device__ constexpr int mx_fwd_bn(bool e4m3, int mode, int swiglu) {
  return e4m3 ? (mode == kDgrad && swiglu ? kMxSwiGLUBwdBNE4M3 : kMxFwdBNE4M3) : kMxFwdBNE2M1;
}
constexpr int kMxWgradStoreAtoms = 2;  // 64-column atoms per bulk store of a wgrad tile
// TMEM accumulator buffers of a 128-column tile.  Three let the MMA for tile t+2
// start before the epilogue has drained tile t: a wgrad tile has a single k-block,
// so the accumulator hand-off round trip is as long as the epilogue itself.
constexpr int kMxAccBufs = 3;
// Epilogue warps: 4 (one per TMEM lane quarter), or 8 for the SwiGLU forward, where two warps
// share a lane quarter and split the tile's columns: that epilogue holds the tile's single
// accumulator while it computes and stores three outputs per value, and the next tile's MMAs
// wait for its release.
template <int EPI>
__host__ __device__ constexpr int mx_epi_warps() { return EPI == kEpiSwiGLU ? 8 : 4; }
// Warps: 0 load producer (TMA tiles, bulk scale atoms), 1 MMA issuer, 2 .. 1 + mx_epi_warps
// epilogue; then for the fwd / dgrad of block-scaled operands the scale gatherer, and for every
// block-scaled kernel the scale copier.
// - Gatherer: the row-major scales of the A operand (and of a forward weight tile not on whole
//   atoms) are gathered into the atom layout by 4-byte cp.async copies, which took the producer
//   about as long as its TMA issue (clock64 on the Zipf-routed MXFP4 layer: 273 of 629 ns per
//   k-block), so they run beside it.
// - Copier: moves each stage's scale atoms into that stage's TMEM slot (tcgen05.cp) and commits
//   them to the stage's scale barrier, on which the MMA issuer waits.  A tcgen05.cp costs its
//   issuing thread ~48 ns; issued by the MMA thread, the six of an e2m1 k-block overlapped its
//   four MMAs only partly (413 ns per k-block against 267 ns for the MMAs alone, timed on a
//   GB300 with all SMs busy), and from a second warp they run beside them (290 ns).  On the
//   Zipf-routed MXFP4 layer: fc1 fwd 1.744 -> 1.624 ms, fc1 wgrad 2.207 -> 2.083 ms; MXFP8 SwiGLU
//   backward 0.543 -> 0.503 ms.  The e2m1 SwiGLU backward keeps the copies in the MMA thread:
//   with the copier it measured 1.606 -> 1.660 ms, and 1.615 -> 1.684 ms with the copies of a tile
//   held back until the previous tile's epilogue had released the accumulator.
template <int FMT, int EPI, bool TS>
__host__ __device__ constexpr bool mx_sf_copier() { return !TS && !(FMT == kE2M1 && EPI == kEpiSwiGLUBwd); }
template <int FMT, int MODE, int EPI, bool TS>
__host__ __device__ constexpr int mx_threads() {
  return 32 * (2 + mx_epi_warps<EPI>() + (MODE != kWgrad && !TS ? 1 : 0) + (mx_sf_copier<FMT, EPI, TS>() ? 1 : 0));
}

struct MxArgs {
  const int32_t* group_lens;
  int G;
  int64_t M;
  const uint8_t* SA;      // scale tensors: row-major [rows, red/32], or blocked atoms (see kGatherA/B)
  const uint8_t* SB;
  int64_t sa_ld, sb_ld;   // scale bytes per row (red/32); blocked: 4 x atoms per 128-row block
  int b_bulk;             // fwd: the tile's B rows start on 128-row atoms (whole-atom copies)
  int64_t sb_blocks;      // 128-row blocks of the blocked B scales (atom copies stay inside them)
  float swiglu_limit;     // SwiGLU epilogues: clamp limit (0: none)
  int a_rows, b_rows;     // rows of the A / B scale tensors that exist (zero-filled beyond)
  int out_cols;           // fwd N (or I with SwiGLU), dgrad K, wgrad K
  int red;                // fwd K / dgrad N (elements)
  int wg_rows;            // wgrad N
  int nw;                 // fwd: rows of W per group (N or 2I)
  int I;
  void* out;
  void* out2;
  const void* aux;
  int32_t* err;
  int64_t M_pad;
  uint8_t* q_codes;   // SwiGLU epilogues: row-wise MX codes of `out` (or nullptr)
  uint8_t* q_scales;  // and their scales
  const float* ts_a;  // TS kernels: the operands' per-tensor fp32 scales s_A, s_B
  const float* ts_b;
  FastDiv nct;  // wgrad: column tiles per row tile
  int c4d;      // wgrad: tmC is the 4-D atom view
  unsigned long long wait_ns;  // pipeline wait limit (0: kWaitTimeoutNs)
  long long stall_at;          // test hook: the producer stops before this k-block (-1: never)
};

// A k-block is 128 bytes of each row in both formats: 128 e4m3 elements (four K=32 MMAs,
// one scale atom per 128-row block) or 256 packed e2m1 elements (four K=64 MMAs, two scale
// atoms).  The e2m1 k-block was 128 elements (64-byte rows) before: per k-block the load
// producer issues the same handful of TMA / bulk copies and the MMA warp the same commit
// and loop work whatever the k-block's size, and at 128 elements those fixed costs --
// ~470 ns of producer time and ~290 ns of MMA-warp time per k-block, measured with clock64
// on the Zipf-routed MXFP4 layer -- dwarfed the ~94 ns of tensor work.
template <int FMT>
struct MxCfg {
  static constexpr int kBK = FMT == kE4M3 ? 128 : 256;            // k-block in elements
  static constexpr int kRowBytes = 128;                           // bytes per row per k-block
  static constexpr uint32_t kSwizzle = kSwizzle128B;
  static constexpr uint32_t kSbo = 8 * kRowBytes;                 // 8-row swizzle atom
  static constexpr int kMmas = 4;                                 // MMAs per k-block (32 bytes of K each)
  static constexpr int kSub = kBK / kMxAtomK;                     // scale atoms per 128 rows per k-block
  static constexpr int kPerMma = kBK / kMmas;                     // reduction elements per MMA
  static constexpr uint32_t kElem = FMT == kE4M3 ? 0 : 1;         // idesc element type code
  static constexpr int kTileBytes = 128 * kRowBytes;
};

// The e2m1 fwd / dgrad plain store stages its whole tile and then releases the accumulator before
// the global stores: with one 256-column accumulator the next tile's MMAs wait for that release.
// Zipf MXFP4 fc2 fwd 0.820 -> 0.689 ms, fc1 dgrad 1.384 -> 1.264 ms (the 64 KB stage leaves room for
// 3 pipeline stages, not 4); the HBM-bound e4m3 calls measured 2% slower that way and keep 4 stages.
template <int FMT, int MODE, int EPI>
__host__ __device__ constexpr bool mx_staged_store() { return FMT == kE2M1 && MODE != kWgrad && EPI == kEpiStore; }
// Epilogue staging per epilogue warp: the wgrad store and the staged plain store hold the warp's
// 32 rows x BN bf16; the plain and SwiGLU forward stores a 2 KB chunk buffer; the SwiGLU backward
// (per-lane stores) none.
template <int FMT, int MODE, int EPI, int BN>
constexpr int mx_epi_warp_bytes() {
  return MODE == kWgrad || mx_staged_store<FMT, MODE, EPI>() ? 32 * BN * 2
         : EPI == kEpiSwiGLUBwd                               ? 0
                                                              : kEpiRowStageBytes;
}
template <int FMT, int MODE, int EPI, int BN>
constexpr int mx_epi_bytes() { return mx_epi_warps<EPI>() * mx_epi_warp_bytes<FMT, MODE, EPI, BN>(); }

// BN = 128 (kMxAccBufs accumulators) or 256 (one accumulator: TMEM cannot hold
// two 256-column accumulators next to the scale factors).  SF: the stages hold scale
// atoms (block-scaled operands; not the FP8 tensor-wise ones).
template <int FMT, int BN, int STAGES, int EPI_BYTES, bool SF = true>
struct MxSmem {
  static constexpr int kA = MxCfg<FMT>::kTileBytes;
  static constexpr int kB = MxCfg<FMT>::kRowBytes * BN;
  // kSub SFA atoms, then kSub SFB atoms for each 128 rows of B (512 B each), padded to keep
  // every stage's tiles 1024-byte aligned
  static constexpr int kSFA = MxCfg<FMT>::kSub * 512;
  static constexpr int kSF = SF ? (kSFA * (1 + BN / 128) + 1023) / 1024 * 1024 : 0;
  static constexpr int kStage = kA + kB + kSF;
  static constexpr int kEpiOff = STAGES * kStage;
  static constexpr int kBarOff = kEpiOff + EPI_BYTES;
  static constexpr int kGroupOff = kBarOff + 384;
  static constexpr size_t bytes(int G) { return 1024 + (size_t)kGroupOff + 12 * (size_t)(G + 1) + 16; }
};

struct MxTile {
  int g, row0, rows, col0, nkb, poff, len;
};

// The scale atoms of one stage (descriptor desc_sf: its first atom) into its TMEM slot at sfa_t:
// for each of the nsub sub-blocks that hold data, SFA 4 columns, then SFB 4 columns per 128 rows
// of B (column n / 32 of the sub-block), after the kSub x 4 SFA columns.  SFA_BYTES: the stage's
// SFA atoms, after which each 128-row block of B has its own.
template <int FMT, int BN, int SFA_BYTES>
__device__ __forceinline__ void mx_copy_scales(uint32_t sfa_t, uint64_t desc_sf, int nsub) {
  constexpr int kSub = MxCfg<FMT>::kSub;
  constexpr uint32_t kSfbPer = 4 * (BN / 128);
  const uint32_t sfb_t = sfa_t + 4 * kSub;
#pragma unroll
  for (int sub = 0; sub < kSub; ++sub) {
    if (sub >= nsub) break;
    tmem_cp_32x128b_x4(sfa_t + 4 * sub, desc_sf + (sub * 512 >> 4));
#pragma unroll
    for (int h = 0; h < BN / 128; ++h)
      tmem_cp_32x128b_x4(sfb_t + sub * kSfbPer + 4 * h, desc_sf + ((SFA_BYTES * (1 + h) + sub * 512) >> 4));
  }
}

template <int EPI, int BN>
__device__ __forceinline__ int mx_tile_cols() { return EPI == kEpiSwiGLU ? BN / 2 : BN; }

template <int MODE, int EPI, int BN, int BK>
__device__ __forceinline__ MxTile mx_decode(int t, const MxArgs& a, const int32_t* s_off,
                                            const int32_t* s_tile, const int32_t* s_poff, GroupCursor& cur) {
  MxTile T;
  cur.at(s_tile, s_off, s_poff, a.G, t);
  const int local = t - cur.t_lo;
  const int len = cur.len;
  T.g = cur.g;
  T.poff = cur.poff;
  T.len = len;
  if (MODE == kWgrad) {
    // column tiles vary fastest (whole rows of dW_g written by concurrent CTAs)
    const int rt = (int)a.nct.div((uint32_t)local);
    T.row0 = rt * kMxBM;
    T.rows = min(kMxBM, a.wg_rows - T.row0);
    T.col0 = (local - rt * (int)a.nct.d) * BN;
    T.nkb = (len + BK - 1) / BK;
  } else {
    const int nmt = (len + kMxBM - 1) / kMxBM;
    const int mt = local % nmt;
    T.row0 = cur.off + mt * kMxBM;
    T.rows = min(kMxBM, len - mt * kMxBM);
    T.col0 = (local / nmt) * mx_tile_cols<EPI, BN>();
    T.nkb = (a.red + BK - 1) / BK;
  }
  return T;
}

template <int FMT, int MODE, int EPI, int STAGES, int BN, bool TS = false>
__global__ void __launch_bounds__(mx_threads<FMT, MODE, EPI, TS>(), 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmC, const MxArgs args) {
  using C = MxCfg<FMT>;
  static_assert(BN == 128 || BN == 256, "BN");
  static_assert(!TS || FMT == kE4M3, "per-tensor scales are e4m3");
  using L = MxSmem<FMT, BN, STAGES, mx_epi_bytes<FMT, MODE, EPI, BN>(), !TS>;
  constexpr bool kSF = !TS;                              // block scale factors (else plain FP8 MMAs)
  constexpr int NACC = BN == 256 ? 1 : kMxAccBufs;       // accumulator buffers
  constexpr int kEpiW = mx_epi_warps<EPI>();              // epilogue warps 2 .. 1 + kEpiW
  constexpr bool kHasGather = MODE != kWgrad && !TS;
  constexpr int kGatherWarp = 2 + kEpiW;                  // the scale gatherer, where there is one
  constexpr bool kCopier = mx_sf_copier<FMT, EPI, TS>();  // scale copies by a warp of their own
  constexpr int kCopyWarp = kGatherWarp + (kHasGather ? 1 : 0);  // the scale copier, where there is one
  // With the copier, the scale atoms complete on their own barrier (sfl), issued ahead of the code
  // tiles, so that they reach TMEM while the tiles are in flight: Zipf MXFP4 fc1 dgrad 1.264 ->
  // 1.226 ms, fc2 fwd 0.662 -> 0.635 ms, fc1 wgrad 2.088 -> 2.029 ms.  Not in the SwiGLU forward,
  // whose long epilogue holds the accumulator while the early copies run (1.630 -> 1.658 ms).
  constexpr bool kSplitSF = kCopier && EPI != kEpiSwiGLU;
  constexpr uint32_t kIdesc = TS ? idesc_f8f6f4(0, kMxBM, BN) : idesc_mx(C::kElem, kMxBM, BN);
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kSfCol0 = NACC * BN;                 // scale-factor columns after the accumulators
  // per stage: for each of the kSub scale sub-blocks, SFA 4 columns and SFB 4 per 128 rows
  constexpr uint32_t kSfbPer = 4 * (BN / 128);            // SFB columns of one sub-block
  constexpr uint32_t kSfPer = C::kSub * (4 + kSfbPer);
  static_assert(kSfCol0 + STAGES * kSfPer <= kTmemCols, "TMEM columns");
  // barriers, the wait control (16 B), the TMEM address and the bad-lens code
  static_assert((4 * STAGES + 2 * NACC + 2) * 8 + 24 <= L::kGroupOff - L::kBarOff, "barrier area");
  // Scale factors of an operand are either row-major [rows, K/32] (activations, whose
  // tiles start at ragged group offsets), gathered 4 bytes per row by cp.async into
  // the atom, or in the blocked atom layout (column-wise operands: wgrad A and B,
  // dgrad B; forward weights B), fetched as whole 512-byte atoms by bulk copy.  A
  // forward weight tile whose rows do not start on an atom (N, or I for SwiGLU, not
  // a multiple of 128) is gathered row by row from the blocked layout instead.
  constexpr bool kGatherA = kSF && MODE != kWgrad;
  const bool gather_b = kSF && MODE == kFwd && (!args.b_bulk || (EPI == kEpiSwiGLU && BN < 256));
  // reduction elements of the operands (wgrad: the group's own length, per tile)
  const int red_all = MODE == kWgrad ? 0 : args.red;
  // bytes of one row of the reduction axis of a group's slice of the dgrad B operand
  const int gbytes = FMT == kE4M3 ? args.red : args.red / 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + NACC;
  uint64_t* drain = tempty + NACC;
  uint64_t* sfull = drain + 1;      // a stage's scale atoms are in its TMEM slot
  uint64_t* sfl = sfull + STAGES;   // kSplitSF: a stage's scale atoms have landed in smem
  uint64_t* cdrain = sfl + STAGES;
  volatile WaitCtl* s_ctl = reinterpret_cast<volatile WaitCtl*>(cdrain + 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(const_cast<WaitCtl*>(s_ctl) + 1);
  int* s_bad = reinterpret_cast<int*>(s_tmem + 1);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + L::kGroupOff);
  int32_t* s_tile = s_off + (args.G + 1);
  int32_t* s_poff = s_tile + (args.G + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // expect_tx arrive (+ 32 cp.async arrives of gathered scales, on sfl when split)
      mbar_init(smem_u32(&full[s]), kGatherA && !kSplitSF ? 1 + 32 : 1);
      mbar_init(smem_u32(&sfl[s]), kGatherA ? 1 + 32 : 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 32 * kEpiW);
    }
    mbar_init(smem_u32(drain), 1);
    for (int s = 0; s < STAGES; ++s) mbar_init(smem_u32(&sfull[s]), 1);
    mbar_init(smem_u32(cdrain), 1);
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
      tc.per_row_tile = ((args.wg_rows + kMxBM - 1) / kMxBM) * ((args.out_cols + BN - 1) / BN);
    } else {
      constexpr int tcw = EPI == kEpiSwiGLU ? BN / 2 : BN;
      tc.bm = kMxBM;
      tc.per_row_tile = (args.out_cols + tcw - 1) / tcw;
    }
    bool bad = scan_groups(args.group_lens, args.G, args.M, tc, s_off, s_tile, s_poff, kMxAtomK, lane);
    int code = bad ? kErrBadGroupLens : 0;
    if (!bad && MODE == kWgrad && (int64_t)s_poff[args.G] > args.M_pad) code = kErrPadOverflow;
    if (lane == 0) {
      *s_bad = code;
      if (code && blockIdx.x == 0) set_error(args.err, code);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem_base = *s_tmem;
  const int total_tiles = *s_bad ? 0 : s_tile[args.G];
  const uint32_t smem0 = smem_u32(smem);
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer: TMA codes + bulk scale atoms
    GroupCursor cur;
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool stalled = false;
    for (int t = blockIdx.x; t < total_tiles && !aborted && !stalled; t += gridDim.x) {
      const MxTile T = mx_decode<MODE, EPI, BN, C::kBK>(t, args, s_off, s_tile, s_poff, cur);
      for (int kb = 0; kb < T.nkb; ++kb) {
        // test hook: stop producing, so that the consumers' waits run out (every load
        // issued so far is consumed, and so complete, before they do)
        if (issued == args.stall_at) { stalled = true; break; }
        if (!warp_wait(smem_u32(&empty[stage]), phase ^ 1u, s_ctl)) { aborted = true; break; }
        const uint32_t sa = smem0 + stage * L::kStage;
        const uint32_t sb = sa + L::kA;
        const uint32_t ssf = sb + L::kB;
        const uint32_t fb = smem_u32(&full[stage]);
        const uint32_t sb_bar = kSplitSF ? smem_u32(&sfl[stage]) : fb;  // where the scale atoms complete
        const int kbyte = kb * C::kRowBytes;  // byte offset of this k-block along a row
        // scale sub-blocks (128 reduction elements each) of this k-block that hold data: a
        // k-block past the end of K / N, or past a wgrad group's last row, copies none of them
        const int valid = (MODE == kWgrad ? T.len : red_all) - kb * C::kBK;
        const int nsub = min(C::kSub, (valid + kMxAtomK - 1) / kMxAtomK);
        const int p0 = kb * C::kSub;  // first scale atom of this k-block along the reduction axis
        if (lane == 0) {
          const uint32_t sf_bytes =
              kSF ? 512u * (uint32_t)nsub * ((kGatherA ? 0u : 1u) + (gather_b ? 0u : BN / 128u)) : 0u;
          if (kSplitSF) {
            mbar_arrive_expect_tx(sb_bar, sf_bytes);
            mbar_arrive_expect_tx(fb, L::kA + L::kB);
          } else {
            mbar_arrive_expect_tx(fb, L::kA + L::kB + sf_bytes);
          }
          // blocked scale atoms: ((row block) * atoms-per-row-block + atom along K) * 512; the
          // nsub atoms of a k-block are adjacent, so one bulk copy takes them all
          if (kSF && !kGatherA)
            bulk_load(ssf, args.SA + ((int64_t)(T.row0 >> 7) * (args.sa_ld >> 2) + (T.poff >> 7) + p0) * 512,
                      512u * nsub, sb_bar);
          if (kSF && !gather_b) {
            const int p = MODE == kWgrad ? (T.poff >> 7) + p0 : MODE == kDgrad ? T.g * (args.red >> 7) + p0 : p0;
#pragma unroll
            for (int h = 0; h < BN / 128; ++h) {
              // first B row of this 128-row group: wgrad / dgrad col0 + 128 h; fwd the weight
              // row g * nw + col0 + 128 h, or with SwiGLU the gate (h = 0) / up (h = 1) half
              int64_t r0;
              if (MODE == kFwd)
                r0 = (int64_t)T.g * args.nw + T.col0 +
                     (EPI == kEpiSwiGLU ? (h < BN / 256 ? 128 * h : args.I + 128 * (h - BN / 256)) : 128 * h);
              else
                r0 = T.col0 + 128 * h;
              // a tile's second half may lie past the operand's last row (N or K not a multiple
              // of 256): its scales only feed outputs that are not stored, so the copy reads the
              // last existing atom row instead of running past the buffer
              const int64_t rb = min(r0 >> 7, args.sb_blocks - 1);
              bulk_load(ssf + L::kSFA * (1 + h), args.SB + (rb * (args.sb_ld >> 2) + p) * 512, 512u * nsub, sb_bar);
            }
          }
          if (MODE == kFwd) {
            tma_load_2d(sa, &tmA, fb, kbyte, T.row0);
            if (EPI == kEpiSwiGLU) {
              tma_load_3d(sb, &tmB, fb, kbyte, T.col0, T.g);
              tma_load_3d(sb + (BN / 2) * C::kRowBytes, &tmB, fb, kbyte, args.I + T.col0, T.g);
            } else {
              tma_load_3d(sb, &tmB, fb, kbyte, T.col0, T.g);
            }
          } else if (MODE == kDgrad) {
            tma_load_2d(sa, &tmA, fb, kbyte, T.row0);
            tma_load_2d(sb, &tmB, fb, T.g * gbytes + kbyte, T.col0);
          } else {
            const int pb = (FMT == kE4M3 ? T.poff : T.poff / 2) + kbyte;
            tma_load_2d(sa, &tmA, fb, pb, T.row0);
            tma_load_2d(sb, &tmB, fb, pb, T.col0);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (aborted && lane == 0) {
      long long n = issued < STAGES ? issued : STAGES;
      int s = stage;
      uint32_t p = phase;
      for (long long i = 0; i < n; ++i) {
        if (--s < 0) { s = STAGES - 1; p ^= 1u; }
        mbar_wait_drain(smem_u32(&full[s]), p);
        if (kSplitSF) mbar_wait_drain(smem_u32(&sfl[s]), p);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    GroupCursor cur;
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    // Shared-memory descriptors of stage 0's A and B tiles.  A descriptor's start-address field
    // holds address / 16 in 14 bits, which every address of this block fits, so the descriptor of
    // address + d (d a multiple of 16) is the base descriptor + d / 16 (here and in the copier).
    const uint64_t kDescA = smem_desc(smem0, 16, C::kSbo, C::kSwizzle);
    const uint64_t kDescB = smem_desc(smem0 + L::kA, 16, C::kSbo, C::kSwizzle);
    const uint64_t kDescSf = smem_desc(smem0 + L::kA + L::kB, 0, 128, kSwizzleNone);  // first scale atom
    for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
      const MxTile T = mx_decode<MODE, EPI, BN, C::kBK>(t, args, s_off, s_tile, s_poff, cur);
      if (T.nkb == 0) continue;
      if (!warp_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, s_ctl)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < T.nkb; ++kb) {
        if (!warp_wait(smem_u32(&full[stage]), phase, s_ctl)) { aborted = true; break; }
        if (kCopier && !warp_wait(smem_u32(&sfull[stage]), phase, s_ctl)) { aborted = true; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t so = (uint64_t)(stage * L::kStage) >> 4;  // this stage's descriptor offset
          const uint32_t sfa_t = tmem_base + kSfCol0 + stage * kSfPer;  // kSub x 4 SFA columns
          const uint32_t sfb_t = sfa_t + 4 * C::kSub;                    // kSub x kSfbPer SFB columns
          // MMAs of this k-block that hold data: past the end of K / N (an e2m1 K that is an odd
          // multiple of 128) or past a wgrad group's rows, the k-steps cover only zeros and are
          // skipped (exact); so are their scale copies
          const int valid = (MODE == kWgrad ? T.len : red_all) - kb * C::kBK;
          const int nmma = min(C::kMmas, (valid + C::kPerMma - 1) / C::kPerMma);
          if (kSF && !kCopier) {
            if (kGatherA) fence_proxy_async_smem();  // cp.async-written scales -> async proxy
            mx_copy_scales<FMT, BN, L::kSFA>(sfa_t, kDescSf + so, min(C::kSub, (valid + kMxAtomK - 1) / kMxAtomK));
          }
#pragma unroll
          for (int j = 0; j < C::kMmas; ++j) {
            if (j >= nmma) break;
            const int sub = j / (C::kMmas / C::kSub);  // the scale sub-block this MMA's K-range lies in
            const uint64_t ad = kDescA + so + 2 * j;  // + 32 bytes of K per MMA
            const uint64_t bd = kDescB + so + 2 * j;
            // scale bytes of the MMA's K-range within its atom: e4m3 one 32-block (j), e2m1 the
            // pair of 32-blocks (2 (j % 2), 2 (j % 2) + 1)
            const uint32_t sfid = FMT == kE4M3 ? (uint32_t)j : (uint32_t)(2 * (j % 2));
            const uint32_t id = kIdesc | idesc_sf_ids(sfid, sfid);
            const uint32_t sfa = sfa_t + 4 * sub, sfb = sfb_t + sub * kSfbPer;
            if (TS) mma_f8f6f4(d_tmem, ad, bd, kIdesc, (kb > 0 || j > 0) ? 1u : 0u);
            else if (FMT == kE4M3) mma_mxf8(d_tmem, ad, bd, id, sfa, sfb, (kb > 0 || j > 0) ? 1u : 0u);
            else mma_mxf4(d_tmem, ad, bd, id, sfa, sfb, (kb > 0 || j > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&empty[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (aborted) break;
      if (lane == 0) mma_commit(smem_u32(&tfull[acc]));
      __syncwarp();
      if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
    }
    if (aborted && lane == 0) {
      mma_commit(smem_u32(drain));
      mbar_wait_drain(smem_u32(drain), 0);
    }
  } else if (kCopier && warp == kCopyWarp) {
    // ------------------------------------------------------------ scale copier (block-scaled)
    // the MMA issuer's stage sequence: once a stage's scale atoms have landed (sfl when split: the
    // bulk copies and the gatherer's cp.async copies, issued ahead of the code tiles), they go to the stage's
    // TMEM slot (SFA: 4 columns per sub-block; SFB: 4 per sub-block and 128 rows of B) and a
    // commit arrives on the stage's scale barrier when they are there.  A slot is rewritten only
    // after the stage was refilled, i.e. after the MMAs that read the slot last completed.
    GroupCursor cur;
    int stage = 0;
    uint32_t phase = 0;
    const uint64_t kDescSf = smem_desc(smem0 + L::kA + L::kB, 0, 128, kSwizzleNone);
    for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
      const MxTile T = mx_decode<MODE, EPI, BN, C::kBK>(t, args, s_off, s_tile, s_poff, cur);
      for (int kb = 0; kb < T.nkb; ++kb) {
        if (!warp_wait(smem_u32(kSplitSF ? &sfl[stage] : &full[stage]), phase, s_ctl)) { aborted = true; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint64_t so = (uint64_t)(stage * L::kStage) >> 4;
          // scale sub-blocks of this k-block that hold data (the MMAs past them are skipped)
          const int valid = (MODE == kWgrad ? T.len : red_all) - kb * C::kBK;
          if (kGatherA) fence_proxy_async_smem();  // cp.async-written scales -> async proxy
          mx_copy_scales<FMT, BN, L::kSFA>(tmem_base + kSfCol0 + stage * kSfPer, kDescSf + so,
                                           min(C::kSub, (valid + kMxAtomK - 1) / kMxAtomK));
          mma_commit(smem_u32(&sfull[stage]));
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (aborted && lane == 0) {  // copies nobody waited for complete before TMEM is freed
      mma_commit(smem_u32(cdrain));
      mbar_wait_drain(smem_u32(cdrain), 0);
    }
  } else if (warp == kGatherWarp) {
    // ------------------------------------------------------------ scale gatherer (fwd / dgrad, block-scaled)
    // the producer's tile and k-block sequence; its 32 cp.async arrivals complete each stage's
    // full barrier together with the producer's expect_tx arrival and copies
    if (kGatherA || gather_b) {
      GroupCursor cur;
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool stalled = false;
      for (int t = blockIdx.x; t < total_tiles && !aborted && !stalled; t += gridDim.x) {
        const MxTile T = mx_decode<MODE, EPI, BN, C::kBK>(t, args, s_off, s_tile, s_poff, cur);
        for (int kb = 0; kb < T.nkb; ++kb) {
          if (issued == args.stall_at) { stalled = true; break; }
          if (!warp_wait(smem_u32(&empty[stage]), phase ^ 1u, s_ctl)) { aborted = true; break; }
          const uint32_t ssf = smem0 + stage * L::kStage + L::kA + L::kB;
          const uint32_t fb = smem_u32(&full[stage]);
          const int valid = red_all - kb * C::kBK;
          const int nsub = min(C::kSub, (valid + kMxAtomK - 1) / kMxAtomK);
          const int p0 = kb * C::kSub;
          // gathered scale factors (row-major operands): for scale sub-block s, lane l fetches
          // rows l, l+32, l+64, l+96 of the operand tile (4 bytes = the sub-block's 4 block
          // scales) into word 4 l + i of atom s
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub) {
            if (sub >= nsub) break;
            const int sfa_col = (p0 + sub) * 4;  // byte column of this sub-block in the row-major A scales
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) {
              const int m = lane + 32 * i;
              // A rows: fwd/dgrad token rows
              if (kGatherA && i < 4) {
                const int ar = T.row0 + m;
                const bool aok = ar < args.a_rows;
                cp_async_4(ssf + sub * 512 + (lane * 4 + i) * 4,
                           args.SA + (aok ? (int64_t)ar * args.sa_ld + sfa_col : 0), aok ? 4u : 0u);
              }
              // B rows
              int br;
              bool bok;
              if (MODE == kFwd) {
                constexpr int kHalf = BN / 2;  // SwiGLU: gate rows, then the matching up rows
                const int n = (EPI == kEpiSwiGLU) ? (m < kHalf ? T.col0 + m : args.I + T.col0 + (m - kHalf))
                                                  : T.col0 + m;
                const int lim = (EPI == kEpiSwiGLU) ? (m < kHalf ? args.I : 2 * args.I) : args.nw;
                bok = n < lim && (EPI != kEpiSwiGLU || T.col0 + (m % kHalf) < args.I);
                br = T.g * args.nw + n;
              } else {
                br = T.col0 + m;
                bok = br < args.b_rows;
              }
              // B row m goes to atom (m / 128, sub), word 4 (m % 32) + (m % 128) / 32; the source
              // is row br's 4 bytes of this sub-block in the blocked layout
              if (gather_b)
                cp_async_4(ssf + L::kSFA * (1 + i / 4) + sub * 512 + (lane * 4 + (i % 4)) * 4,
                           args.SB + (bok ? ((((int64_t)br >> 7) * (args.sb_ld >> 2) + p0 + sub) << 9) +
                                                16 * (br & 31) + 4 * ((br >> 5) & 3)
                                          : 0),
                           bok ? 4u : 0u);
            }
          }
          cp_async_arrive_noinc(kSplitSF ? smem_u32(&sfl[stage]) : fb);
          __syncwarp();
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      cp_async_wait_all();  // nothing of this warp's lands after the block exits
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2 .. 1 + kEpiW)
    const int q = warp & 3;                 // TMEM lane quarter
    const int half = (warp - 2) >> 2;       // with 8 epilogue warps: which half of the tile's columns
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(args.out);
    GroupCursor cur;
    uint8_t* stg = smem + L::kEpiOff + (warp - 2) * mx_epi_warp_bytes<FMT, MODE, EPI, BN>();  // this warp's staging
    int nstore = 0;
    float alpha = 1.0f;  // TS: 1 / (s_A s_B), written by the quantizers earlier on the stream
    // The product of two fp32 scales is exact in fp64 and cannot overflow there (each scale is at
    // most FLT_MAX, for a tensor whose amax is tiny); its reciprocal may be an fp32 subnormal.
    if constexpr (TS) alpha = (float)(1.0 / ((double)__ldg(args.ts_a) * (double)__ldg(args.ts_b)));
    for (int t = blockIdx.x; t < total_tiles && !aborted; t += gridDim.x) {
      const MxTile T = mx_decode<MODE, EPI, BN, C::kBK>(t, args, s_off, s_tile, s_poff, cur);
      const bool row_ok = r < T.rows;
      if (MODE == kWgrad) {
        const bool zero = T.nkb == 0;
        if (!zero) {
          if (!warp_wait(smem_u32(&tfull[acc]), acc_phase, s_ctl)) { aborted = true; break; }
          tc_fence_after();
        }
        const uint32_t tbw = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
        if (args.c4d)
          epi_tma_store_tile<BN, kMxWgradStoreAtoms, BN / 64, TS>(tbw, zero, stg, &tmC, T.row0 + q * 32, T.col0,
                                                                 T.g, args.wg_rows, args.out_cols, lane, alpha);
        else
          epi_tma_store_rows<BN, TS>(tbw, zero, stg, nstore, &tmC, T.row0 + q * 32, T.col0, T.g, args.wg_rows,
                                     args.out_cols, lane, alpha);
        if (!zero) {
          tc_fence_before();
          mbar_arrive(smem_u32(&tempty[acc]));
          if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
        }
        continue;
      }
      const size_t grow = (size_t)T.row0 + r;
      const size_t row0w = (size_t)T.row0 + q * 32;         // the warp's first output row
      const int nrows = max(0, min(32, T.rows - q * 32));    // of which this many exist
      // 32-column chunks of this warp: of each SwiGLU half (BN / 64 per half), or of the tile
      constexpr int kChunks = EPI == kEpiSwiGLU ? BN / 64 : BN / 32;
      constexpr int kMine = kChunks * 4 / kEpiW;
      const int cb = half * kMine, ce = cb + kMine;
      if (EPI == kEpiSwiGLUBwd)  // the saved H of this tile streams into L2 while the MMAs run
        epi_swiglu_bwd_prefetch<BN>(reinterpret_cast<const __nv_bfloat16*>(args.aux), grow, row_ok, T.col0,
                                    args.I, cb, ce);
      if (!warp_wait(smem_u32(&tfull[acc]), acc_phase, s_ctl)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t tb = tmem_base + acc * BN + ((uint32_t)(q * 32) << 16);
      if (EPI == kEpiSwiGLU) {
        epi_swiglu<BN, FMT, TS>(tb, out, reinterpret_cast<__nv_bfloat16*>(args.out2), row0w, nrows, row_ok, grow,
                                T.col0, args.I, stg, lane, args.q_codes, args.q_scales, args.swiglu_limit, alpha, cb,
                                ce);
      } else if (EPI == kEpiSwiGLUBwd) {
        epi_swiglu_bwd<BN, FMT, TS, false>(tb, out, reinterpret_cast<const __nv_bfloat16*>(args.aux), row0w, nrows, row_ok,
                                    grow, T.col0, args.I, stg, lane, args.q_codes, args.q_scales, args.swiglu_limit,
                                    alpha, cb, ce);
      } else if constexpr (mx_staged_store<FMT, MODE, EPI>()) {
        epi_stage_tile<BN, TS>(tb, stg, lane, alpha);
        tc_fence_before();
        mbar_arrive(smem_u32(&tempty[acc]));
        if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
        epi_store_staged<BN>(stg, out, args.out_cols, row0w, nrows, T.col0, args.out_cols, lane);
        continue;
      } else {
        epi_store<BN, TS>(tb, out, args.out_cols, row0w, nrows, T.col0, args.out_cols, stg, lane, alpha);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == NACC) { acc = 0; acc_phase ^= 1u; }
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

template <int FMT, int MODE, int EPI, int STAGES, int BN = kMxBN, bool TS = false>
int run_mx(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const MxArgs& a, int grid,
           cudaStream_t s) {
  using L = MxSmem<FMT, BN, STAGES, mx_epi_bytes<FMT, MODE, EPI, BN>(), !TS>;
  auto kern = grouped_gemm_mx_kernel<FMT, MODE, EPI, STAGES, BN, TS>;
  const size_t smem = L::bytes(a.G);
  static size_t attr_bytes = 0;  // per instantiation: raised to the largest G seen
  if (smem > attr_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e == cudaErrorInvalidValue ? PGG_ERR_UNSUPPORTED : cuda_status(e);
    attr_bytes = smem;
  }
  kern<<<grid, mx_threads<FMT, MODE, EPI, TS>(), smem, s>>>(ta, tb, tc, a);
  return cuda_status(cudaGetLastError());
}

// A fwd / dgrad kernel with `S` stages, or S - 1 when the group tables of a large G leave no room
// next to its epilogue staging.
template <int FMT, int MODE, int EPI, int S, int BN, bool TS = false>
int run_mx_fit(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const MxArgs& a, int grid,
               cudaStream_t s) {
  using L = MxSmem<FMT, BN, S, mx_epi_bytes<FMT, MODE, EPI, BN>(), !TS>;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  if (L::bytes(a.G) > dev.smem_optin) return run_mx<FMT, MODE, EPI, S - 1, BN, TS>(ta, tb, tc, a, grid, s);
  return run_mx<FMT, MODE, EPI, S, BN, TS>(ta, tb, tc, a, grid, s);
}

template <int FMT>
int dispatch_mx(int mode, int epi, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                const MxArgs& a, int grid, cudaStream_t s) {
  constexpr int kBN = FMT == kE4M3 ? kMxFwdBNE4M3 : kMxFwdBNE2M1;
  constexpr int kBNb = mx_fwd_bn(FMT == kE4M3, kDgrad, 1);  // the SwiGLU backward's tile width
  // stages for fwd / dgrad: 4 x (16 KB A + 32 KB B + 2 / 3 KB of scale atoms) next to the group tables
  // and the epilogue staging; 6 x (16 KB + 16 KB + 1 KB) for a 128-wide tile
  constexpr int kS = 4, kSb = kBNb == 128 ? 6 : 4;
  constexpr int kSp = mx_staged_store<FMT, kFwd, kEpiStore>() ? 3 : 4;  // a 64 KB tile stage leaves room for 3
  constexpr int kWBN = FMT == kE4M3 ? kMxWgradBNE4M3 : kMxWgradBNE2M1;
  // wgrad keeps 4 x 32 rows x kWBN bf16 of TMA-store staging next to the stages: e4m3 5 x 33 KB
  // + 32 KB, e2m1 3 x 51 KB + 64 KB (2 stages when the group tables of a large G leave no room)
  constexpr int kSw = FMT == kE4M3 ? 5 : 3;
  if (mode == 0 && epi == 0) return run_mx_fit<FMT, kFwd, kEpiStore, kSp, kBN>(ta, tb, tc, a, grid, s);
  if (mode == 0 && epi == 1) return run_mx_fit<FMT, kFwd, kEpiSwiGLU, kS, kBN>(ta, tb, tc, a, grid, s);
  if (mode == 1 && epi == 0) return run_mx_fit<FMT, kDgrad, kEpiStore, kSp, kBN>(ta, tb, tc, a, grid, s);
  if (mode == 1 && epi == 1) return run_mx<FMT, kDgrad, kEpiSwiGLUBwd, kSb, kBNb>(ta, tb, tc, a, grid, s);
  if (mode == 2 && epi == 0) {
    using L = MxSmem<FMT, kWBN, kSw, 4 * 32 * kWBN * 2>;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != PGG_OK) return st;
    if (L::bytes(a.G) > dev.smem_optin) return run_mx<FMT, kWgrad, kEpiStore, kSw - 1, kWBN>(ta, tb, tc, a, grid, s);
    return run_mx<FMT, kWgrad, kEpiStore, kSw, kWBN>(ta, tb, tc, a, grid, s);
  }
  return PGG_ERR_INVALID_ARG;
}

// FP8 tensor-wise operands: the e4m3 tiles, stage counts and epilogues of dispatch_mx.
int dispatch_ts(int mode, int epi, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                const MxArgs& a, int grid, cudaStream_t s) {
  constexpr int kBN = kMxFwdBNE4M3, kWBN = kMxWgradBNE4M3;
  constexpr int kBNb = mx_fwd_bn(true, kDgrad, 1);
  constexpr int kS = 4, kSb = kBNb == 128 ? 6 : 4;
  constexpr int kSp = 4;
  constexpr int kSw = 5;
  if (mode == 0 && epi == 0) return run_mx_fit<kE4M3, kFwd, kEpiStore, kSp, kBN, true>(ta, tb, tc, a, grid, s);
  if (mode == 0 && epi == 1) return run_mx_fit<kE4M3, kFwd, kEpiSwiGLU, kS, kBN, true>(ta, tb, tc, a, grid, s);
  if (mode == 1 && epi == 0) return run_mx_fit<kE4M3, kDgrad, kEpiStore, kSp, kBN, true>(ta, tb, tc, a, grid, s);
  if (mode == 1 && epi == 1) return run_mx<kE4M3, kDgrad, kEpiSwiGLUBwd, kSb, kBNb, true>(ta, tb, tc, a, grid, s);
  if (mode == 2 && epi == 0) return run_mx<kE4M3, kWgrad, kEpiStore, kSw, kWBN, true>(ta, tb, tc, a, grid, s);
  return PGG_ERR_INVALID_ARG;
}

int cdiv(int64_t x, int64_t y) { return (int)((x + y - 1) / y); }

}  // namespace

int launch_mx_gemm(const MxCall& c) {
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  const bool e4 = c.fmt == PGG_FMT_E4M3;
  const uint32_t rb = 128;  // bytes per row per k-block (128 e4m3 or 256 packed e2m1 elements)
  auto bytes = [&](int64_t elems) { return (uint64_t)(e4 ? elems : elems / 2); };
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const auto u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUtensorMap ta, tb, tc;
  MxArgs a{};
  a.group_lens = c.group_lens;
  a.G = c.G;
  a.M = c.M;
  a.SA = c.SA;
  a.SB = c.SB;
  a.out = c.out;
  a.out2 = c.out2;
  a.aux = c.H;
  a.err = c.err;
  a.M_pad = c.M_pad;
  a.q_codes = c.q_codes;
  a.q_scales = c.q_scales;
  a.swiglu_limit = c.limit;
  a.ts_a = c.ts_a;
  a.ts_b = c.ts_b;
  a.wait_ns = c.wait_ns;
  a.stall_at = c.stall_at;
  const bool ts = c.ts_a != nullptr;
  if (ts && (!e4 || !c.ts_b || c.q_codes)) return PGG_ERR_INVALID_ARG;
  const int fbn = mx_fwd_bn(e4, c.mode, c.epi);  // fwd / dgrad tile width
  int tiles_ub;
  if (c.mode == 0) {
    const int64_t N = c.N, K = c.K;
    uint64_t da[2] = {bytes(K), (uint64_t)c.M}, sa[1] = {bytes(K)};
    uint32_t ba[2] = {rb, 128};
    uint64_t db[3] = {bytes(K), (uint64_t)N, (uint64_t)c.G}, sb[2] = {bytes(K), bytes(K) * (uint64_t)N};
    uint32_t bb[3] = {rb, (uint32_t)(c.epi ? fbn / 2 : fbn), 1};
    if ((st = encode_tmap(&ta, u8, 2, c.A, da, sa, ba, sw))) return st;
    if ((st = encode_tmap(&tb, u8, 3, c.B, db, sb, bb, sw))) return st;
    a.sa_ld = a.sb_ld = K / 32;
    // weight scales are blocked: whole-atom copies when every B tile (or SwiGLU half)
    // starts on a 128-row atom
    a.b_bulk = c.epi ? ((fbn / 2) % 128 == 0 && (N / 2) % 128 == 0) : (N % 128 == 0 && fbn % 128 == 0);
    a.sb_blocks = cdiv((int64_t)c.G * N, 128);
    a.a_rows = (int)c.M;
    a.nw = (int)N;
    a.I = (int)(N / 2);
    a.out_cols = (int)(c.epi ? N / 2 : N);
    a.red = (int)K;
    tiles_ub = (cdiv(c.M, kMxBM) + c.G) * cdiv(a.out_cols, c.epi ? fbn / 2 : fbn);
  } else if (c.mode == 1) {
    const int64_t N = c.N, K = c.K;
    uint64_t da[2] = {bytes(N), (uint64_t)c.M}, sa[1] = {bytes(N)};
    uint64_t db[2] = {bytes(N) * (uint64_t)c.G, (uint64_t)K}, sb[1] = {bytes(N) * (uint64_t)c.G};
    uint32_t bx[2] = {rb, 128}, bwide[2] = {rb, (uint32_t)fbn};
    if ((st = encode_tmap(&ta, u8, 2, c.A, da, sa, bx, sw))) return st;
    if ((st = encode_tmap(&tb, u8, 2, c.B, db, sb, bwide, sw))) return st;
    a.sa_ld = N / 32;
    a.sb_ld = c.G * N / 32;
    a.sb_blocks = cdiv(K, 128);
    a.a_rows = (int)c.M;
    a.b_rows = (int)K;
    a.I = (int)K;
    a.out_cols = (int)K;
    a.red = (int)N;
    tiles_ub = (cdiv(c.M, kMxBM) + c.G) * cdiv(K, fbn);
  } else {
    const int64_t N = c.N, K = c.K, Mp = c.M_pad;
    uint64_t da[2] = {bytes(Mp), (uint64_t)N}, sa[1] = {bytes(Mp)};
    uint64_t db[2] = {bytes(Mp), (uint64_t)K}, sb[1] = {bytes(Mp)};
    const int wbn = e4 ? kMxWgradBNE4M3 : kMxWgradBNE2M1;
    uint32_t bx[2] = {rb, 128}, bw[2] = {rb, (uint32_t)wbn};
    if ((st = encode_tmap(&ta, u8, 2, c.A, da, sa, bx, sw))) return st;
    if ((st = encode_tmap(&tb, u8, 2, c.B, db, sb, bw, sw))) return st;
    if ((st = encode_wgrad_out(&tc, c.out, N, K, c.G, kMxWgradStoreAtoms, &a.c4d))) return st;
    a.nct = FastDiv((uint32_t)cdiv(K, wbn));
    a.sa_ld = a.sb_ld = Mp / 32;
    a.sb_blocks = cdiv(K, 128);
    a.a_rows = (int)N;
    a.b_rows = (int)K;
    a.out_cols = (int)K;
    a.wg_rows = (int)N;
    tiles_ub = c.G * cdiv(N, kMxBM) * cdiv(K, wbn);
  }
  if (c.mode != 2) tc = ta;  // unused outside wgrad
  const int grid = std::max(1, std::min(dev.sms, tiles_ub));
  if (ts) {
    a.SA = a.SB = nullptr;  // no block scales
    return dispatch_ts(c.mode, c.epi, ta, tb, tc, a, grid, c.stream);
  }
  return e4 ? dispatch_mx<kE4M3>(c.mode, c.epi, ta, tb, tc, a, grid, c.stream)
            : dispatch_mx<2>(c.mode, c.epi, ta, tb, tc, a, grid, c.stream);
}

}  // namespace pgg
