// In-kernel group scan and persistent tile schedule for the grouped GEMMs.
//
// group_lens (device int32[G], the per-expert token counts produced by
// routing) split the [M, K] activation into G row blocks; block g covers rows
// [off_g, off_g + len_g).  Every CTA scans group_lens into shared memory
// (off[] and the tile prefix tile0[]), so no host synchronisation and no
// padding copy is needed for ragged or empty groups.  Tiles are numbered
// group-major; a CTA walks tiles blockIdx.x, blockIdx.x + gridDim.x, ...
#pragma once
#include <cstdint>

namespace pgg {

constexpr int kMaxGroups = 1024;

// GEMM modes and epilogues shared by the BF16 and block-scaled kernels.
enum GemmMode : int { kFwd = 0, kDgrad = 1, kWgrad = 2 };
enum GemmEpi : int { kEpiStore = 0, kEpiSwiGLU = 1, kEpiSwiGLUBwd = 2, kEpiAccumF32 = 3 };

// Device error-word codes (the public values of pgg_status).
constexpr int kErrBadGroupLens = 16;
constexpr int kErrTimeout = 17;
constexpr int kErrPadOverflow = 18;
constexpr int kErrBadExpert = 19;

// Tiles of one group as a function of its length.
struct TileCount {
  int per_row_tile;     // column tiles (fwd/dgrad) or constant tiles per group (wgrad)
  int bm;               // row tile height for ragged rows (fwd/dgrad); 0 = constant per group
  __device__ __forceinline__ int operator()(int len) const {
    if (bm == 0) return per_row_tile;
    return ((len + bm - 1) / bm) * per_row_tile;
  }
};

// One warp scans group_lens: s_off[0..G], s_tile[0..G] (exclusive prefix sums),
// plus s_poff[0..G] (prefix of round_up(len, pad)) when s_poff != nullptr.
// Returns true (warp-uniform) when some len < 0 or sum(len) != M.
__device__ __forceinline__ bool scan_groups(const int32_t* __restrict__ lens, int G, int64_t M,
                                            TileCount tc, int32_t* s_off, int32_t* s_tile,
                                            int32_t* s_poff, int pad, int lane) {
  const int per = (G + 31) / 32;
  const int lo = min(lane * per, G), hi = min(lo + per, G);
  long long sl = 0, st = 0, sp = 0;
  bool bad = false;
  for (int i = lo; i < hi; ++i) {
    int l = __ldg(lens + i);
    bad |= (l < 0);
    l = max(l, 0);
    sl += l;
    st += tc(l);
    if (pad > 0) sp += (long long)((l + pad - 1) / pad) * pad;
  }
  // inclusive scans across the warp
  long long il = sl, it = st, ip = sp;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    long long vl = __shfl_up_sync(0xffffffffu, il, d);
    long long vt = __shfl_up_sync(0xffffffffu, it, d);
    long long vp = __shfl_up_sync(0xffffffffu, ip, d);
    if (lane >= d) { il += vl; it += vt; ip += vp; }
  }
  long long rl = il - sl, rt = it - st, rp = ip - sp;
  for (int i = lo; i < hi; ++i) {
    int l = max(__ldg(lens + i), 0);
    s_off[i] = (int32_t)rl;
    s_tile[i] = (int32_t)rt;
    if (s_poff) s_poff[i] = (int32_t)rp;
    rl += l;
    rt += tc(l);
    if (pad > 0) rp += (long long)((l + pad - 1) / pad) * pad;
  }
  long long tot_l = __shfl_sync(0xffffffffu, il, 31);
  long long tot_t = __shfl_sync(0xffffffffu, it, 31);
  long long tot_p = __shfl_sync(0xffffffffu, ip, 31);
  if (lane == 0) {
    s_off[G] = (int32_t)min(tot_l, (long long)INT32_MAX);
    s_tile[G] = (int32_t)min(tot_t, (long long)INT32_MAX);
    if (s_poff) s_poff[G] = (int32_t)min(tot_p, (long long)INT32_MAX);
  }
  bad = __any_sync(0xffffffffu, bad) || tot_l != M || tot_t > INT32_MAX;
  return bad;
}

// Division by a divisor fixed for the launch (Granlund-Montgomery: n / d =
// (umulhi(n, m) + n) >> s for 0 <= n < 2^31, with s = ceil(log2 d) and
// m = floor(2^32 (2^s - d) / d) + 1), so per-tile index math needs no divide.
struct FastDiv {
  uint32_t d, m, s;
  __host__ __device__ FastDiv() : d(1), m(0), s(0) {}
  __host__ __device__ explicit FastDiv(uint32_t div) : d(div) {
    s = 0;
    while ((1u << s) < d) ++s;
    m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - d)) / d + 1);
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> s; }
};

// Group owning linear tile t: the largest g with s_tile[g] <= t (empty groups
// have s_tile[g] == s_tile[g+1] and are skipped).
__device__ __forceinline__ int find_group(const int32_t* s_tile, int G, int t) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (s_tile[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The group of a CTA's tiles, tracked as t grows (t, t + gridDim.x, ...): a
// binary search for the first tile, then a short forward walk.
// The group of a role's current tile with its scan values, held in registers.
// A CTA's tiles ascend and almost always stay in one group from one tile to
// the next, so the shared-memory tables are read only when a tile crosses into
// another group: while the pipeline keeps shared memory busy, each dependent
// table read costs hundreds of cycles.
struct GroupCursor {
  int g = -1;
  int t_lo = 0, t_hi = 0;    // tiles [t_lo, t_hi) belong to group g
  int off = 0, len = 0;      // rows [off, off + len) of the ragged operand
  int poff = 0;              // padded column offset (column-wise MX layout), if tracked
  __device__ __forceinline__ void at(const int32_t* s_tile, const int32_t* s_off, const int32_t* s_poff,
                                     int G, int t) {
    if (g >= 0 && t >= t_lo && t < t_hi) return;
    if (g < 0 || t < t_lo) g = find_group(s_tile, G, t);
    while (g + 1 < G && s_tile[g + 1] <= t) ++g;
    t_lo = s_tile[g];
    t_hi = s_tile[g + 1];
    off = s_off[g];
    len = s_off[g + 1] - off;
    if (s_poff) poff = s_poff[g];
  }
};

}  // namespace pgg
