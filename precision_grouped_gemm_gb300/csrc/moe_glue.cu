// Single-GPU MoE glue on either side of the grouped GEMM: the token permute into
// expert-sorted rows (with group_lens) and the weighted combine back, and their
// backward passes.  "Enabling DeepSeek-V4-Flash Training on AMD Instinct MI355X
// GPUs with Primus", section "Expert parallelism: DeepEP and the grouped GEMM"
// (the dispatch lays tokens out the way the grouped GEMM wants them) and section
// "MegaMoE" (the second grouped GEMM is followed by the combine and the weighted
// reduce).  With one GPU there is no communication: what remains is a stable
// counting sort of the (token, choice) entries by expert and two row gathers.
//
// permute, four launches:
//   count   one warp per 32-token chunk counts its entries per expert into the
//           caller's table ws [E, nchunk] int32 (expert-major)
//   scan    one block per expert: ws[e, .] becomes its exclusive prefix over
//           chunks, group_lens[e] its total
//   rank    one warp per chunk: pos[t, j] = (rows of experts < e) + ws[e, c] +
//           (earlier entries of expert e inside the chunk, in (token, choice)
//           order) -- exactly the stable sort's position; the chunk's tokens are
//           walked in order, a token's k choices ranked in parallel across lanes
//   gather  one warp per entry, Xs[pos[t, j]] = X[t] with 16-byte copies
// All integer work is exact, so pos and group_lens are deterministic.
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace pgg {
namespace {

constexpr int kChunk = 32;          // tokens per warp chunk
constexpr int kCountWarps = 8;      // warps per block of the count kernel
constexpr int kRankWarps = 4;       // warps per block of the rank kernel
constexpr int kScanThreads = 256;
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCountWarps * 32) moe_count_kernel(const int32_t* __restrict__ ids,
                                                                     int64_t T, int k, int E, int64_t nchunk,
                                                                     int32_t* __restrict__ ws, int32_t* err) {
  extern __shared__ int32_t s_cnt[];  // [kCountWarps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t c = (int64_t)blockIdx.x * kCountWarps + warp;
  if (c >= nchunk) return;
  int32_t* cnt = s_cnt + warp * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t t = c * kChunk + lane;
  if (t < T) {
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(ids + t * k + j);
      if (e < 0 || e >= E) {
        set_error(err, kErrBadExpert);
        continue;
      }
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncwarp();
  for (int e = lane; e < E; e += 32) ws[(int64_t)e * nchunk + c] = cnt[e];
}

// One block per expert: in-place exclusive scan of ws[e, 0 .. nchunk) and its total.
__global__ void __launch_bounds__(kScanThreads) moe_scan_kernel(int64_t nchunk, int32_t* __restrict__ ws,
                                                                int32_t* __restrict__ group_lens) {
  __shared__ int32_t s_part[kScanThreads];
  const int tid = threadIdx.x;
  int32_t* row = ws + (int64_t)blockIdx.x * nchunk;
  const int64_t per = (nchunk + kScanThreads - 1) / kScanThreads;
  const int64_t lo = min((int64_t)tid * per, nchunk), hi = min(lo + per, nchunk);
  int32_t sum = 0;
  for (int64_t c = lo; c < hi; ++c) sum += row[c];
  s_part[tid] = sum;
  __syncthreads();
  for (int d = 1; d < kScanThreads; d <<= 1) {  // inclusive scan of the partial sums
    const int32_t v = tid >= d ? s_part[tid - d] : 0;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  int32_t run = s_part[tid] - sum;
  for (int64_t c = lo; c < hi; ++c) {
    const int32_t v = row[c];
    row[c] = run;
    run += v;
  }
  if (tid == kScanThreads - 1) group_lens[blockIdx.x] = s_part[tid];
}

// One warp per chunk.  Shared memory: expert offsets [E], then per warp the
// running positions [E] and the chunk's ids [32 * k].
__global__ void __launch_bounds__(kRankWarps * 32) moe_rank_kernel(const int32_t* __restrict__ ids, int64_t T,
                                                                   int k, int E, int64_t nchunk,
                                                                   const int32_t* __restrict__ ws,
                                                                   const int32_t* __restrict__ group_lens,
                                                                   int32_t* __restrict__ pos) {
  extern __shared__ int32_t s_dyn[];
  int32_t* s_off = s_dyn;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* base = s_dyn + E + warp * (E + kChunk * k);
  int32_t* sid = base + E;
  if (warp == 0) {
    // exclusive prefix of group_lens over experts: lane-blocked sums, then a shuffle scan
    const int per = (E + 31) / 32;
    const int lo = min(lane * per, E), hi = min(lo + per, E);
    int32_t s = 0;
    for (int e = lo; e < hi; ++e) s += __ldg(group_lens + e);
    int32_t inc = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += v;
    }
    int32_t run = inc - s;
    for (int e = lo; e < hi; ++e) {
      s_off[e] = run;
      run += __ldg(group_lens + e);
    }
  }
  __syncthreads();
  const int64_t c = (int64_t)blockIdx.x * kRankWarps + warp;
  if (c >= nchunk) return;
  for (int e = lane; e < E; e += 32) base[e] = s_off[e] + __ldg(ws + (int64_t)e * nchunk + c);
  const int64_t t0 = c * kChunk;
  const int n = (int)min((int64_t)kChunk, T - t0) * k;  // entries of this chunk, contiguous in ids
  for (int i = lane; i < n; i += 32) sid[i] = __ldg(ids + t0 * k + i);
  __syncwarp();
  if (lane < k) {
    // tokens in order; lane j takes choice j.  Choices of one token that name the same
    // expert are ordered by j, so positions follow the (token, choice) order: the stable
    // order within each expert.
    const unsigned km = k == 32 ? 0xffffffffu : ((1u << k) - 1u);
    const int nt = n / k;
    for (int i = 0; i < nt; ++i) {
      const int e = sid[i * k + lane];
      const bool ok = e >= 0 && e < E;
      const unsigned peers = __match_any_sync(km, ok ? e : -1);
      const int before = __popc(peers & ((1u << lane) - 1u));
      const int p = ok ? base[e] + before : -1;
      __syncwarp(km);
      if (ok && before == 0) base[e] += __popc(peers);
      __syncwarp(km);
      sid[i * k + lane] = p;
    }
  }
  __syncwarp();
  for (int i = lane; i < n; i += 32) pos[t0 * k + i] = sid[i];
}

// Xs[pos[r]] = X[r / k] for every entry r = t * k + j; one warp per entry, grid-stride.
__global__ void __launch_bounds__(kCopyThreads) moe_gather_kernel(const __nv_bfloat16* __restrict__ X,
                                                                  const int32_t* __restrict__ pos, int64_t R,
                                                                  int k, int64_t H,
                                                                  __nv_bfloat16* __restrict__ Xs) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = (int64_t)gridDim.x * (kCopyThreads / 32);
  const int64_t nvec = H / 8;
  for (int64_t r = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); r < R; r += nwarp) {
    const int32_t p = __ldg(pos + r);
    if (p < 0) continue;
    const uint4* src = reinterpret_cast<const uint4*>(X + (r / k) * H);
    uint4* dst = reinterpret_cast<uint4*>(Xs + (int64_t)p * H);
    int64_t v = lane;
    for (; v + 96 < nvec; v += 128) {  // four independent 16-byte loads in flight per lane
      const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64),
                  d = __ldg(src + v + 96);
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
    for (; v < nvec; v += 32) dst[v] = __ldg(src + v);
  }
}

__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4& y) {
  acc[0] += w * bf16_lo(y.x); acc[1] += w * bf16_hi(y.x);
  acc[2] += w * bf16_lo(y.y); acc[3] += w * bf16_hi(y.y);
  acc[4] += w * bf16_lo(y.z); acc[5] += w * bf16_hi(y.z);
  acc[6] += w * bf16_lo(y.w); acc[7] += w * bf16_hi(y.w);
}

// out[t] = sum_j w[t, j] * Ys[pos[t, j]] (w = 1 when w == nullptr), fp32 accumulation in
// choice order, bf16 output.  One warp per token; lane j < k holds pos / w of choice j.  A lane
// owns kCombineU 16-byte column pieces at once, and the next choice's pieces are loaded while
// the current one is accumulated: up to 2 kCombineU loads in flight per lane.  (With one warp
// per token the DeepSeek-shaped routing gives ~27 warps per SM; two loads in flight per lane
// left the kernel latency-bound at about half the DRAM bandwidth.)
constexpr int kCombineU = 4;
__global__ void __launch_bounds__(kCopyThreads) moe_combine_kernel(const __nv_bfloat16* __restrict__ Ys,
                                                                   const int32_t* __restrict__ pos,
                                                                   const float* __restrict__ w, int64_t T, int k,
                                                                   int64_t H, __nv_bfloat16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = (int64_t)gridDim.x * (kCopyThreads / 32);
  const int64_t nvec = H / 8;
  for (int64_t t = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); t < T; t += nwarp) {
    const int32_t my_p = lane < k ? __ldg(pos + t * k + lane) : -1;
    const float my_w = (lane < k && w) ? __ldg(w + t * k + lane) : 1.0f;
    // warp-uniform trip counts: every lane takes part in the shuffles, only the loads are guarded
    for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kCombineU) {
      float acc[kCombineU][8];
#pragma unroll
      for (int u = 0; u < kCombineU; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[u][e] = 0.0f;
      // nxt: choice j's pieces v0 + lane + 32 u, u < kCombineU (zero when the choice is dropped)
      uint4 nxt[kCombineU];
      int32_t pn = __shfl_sync(0xffffffffu, my_p, 0);
      float wn = __shfl_sync(0xffffffffu, my_w, 0);
#pragma unroll
      for (int u = 0; u < kCombineU; ++u) {
        const int64_t v = v0 + lane + 32 * u;
        nxt[u] = (pn >= 0 && v < nvec) ? __ldg(reinterpret_cast<const uint4*>(Ys + (int64_t)pn * H) + v)
                                       : make_uint4(0, 0, 0, 0);
      }
      for (int j = 0; j < k; ++j) {
        uint4 cur[kCombineU];
#pragma unroll
        for (int u = 0; u < kCombineU; ++u) cur[u] = nxt[u];
        const int32_t pc = pn;
        const float wc = wn;
        if (j + 1 < k) {
          pn = __shfl_sync(0xffffffffu, my_p, (j + 1) & 31);
          wn = __shfl_sync(0xffffffffu, my_w, (j + 1) & 31);
#pragma unroll
          for (int u = 0; u < kCombineU; ++u) {
            const int64_t v = v0 + lane + 32 * u;
            nxt[u] = (pn >= 0 && v < nvec) ? __ldg(reinterpret_cast<const uint4*>(Ys + (int64_t)pn * H) + v)
                                           : make_uint4(0, 0, 0, 0);
          }
        }
        if (pc >= 0) {
#pragma unroll
          for (int u = 0; u < kCombineU; ++u) fma8(acc[u], wc, cur[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kCombineU; ++u) {
        const int64_t v = v0 + lane + 32 * u;
        if (v >= nvec) continue;
        uint4 o;
        o.x = pack_bf16x2(acc[u][0], acc[u][1]);
        o.y = pack_bf16x2(acc[u][2], acc[u][3]);
        o.z = pack_bf16x2(acc[u][4], acc[u][5]);
        o.w = pack_bf16x2(acc[u][6], acc[u][7]);
        reinterpret_cast<uint4*>(out + t * H)[v] = o;
      }
    }
  }
}

// dYs[pos[t, j]] = bf16(w[t, j] * dOut[t]);  dw[t, j] = <dOut[t], Ys[pos[t, j]]> in fp32
// (lane partial sums, then a fixed xor-tree: deterministic).  One warp per token.
__global__ void __launch_bounds__(kCopyThreads) moe_combine_bwd_kernel(
    const __nv_bfloat16* __restrict__ dOut, const __nv_bfloat16* __restrict__ Ys, const int32_t* __restrict__ pos,
    const float* __restrict__ w, int64_t T, int k, int64_t H, __nv_bfloat16* __restrict__ dYs,
    float* __restrict__ dw) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarp = (int64_t)gridDim.x * (kCopyThreads / 32);
  const int64_t nvec = H / 8;
  for (int64_t t = (int64_t)blockIdx.x * (kCopyThreads / 32) + (threadIdx.x >> 5); t < T; t += nwarp) {
    const uint4* g = reinterpret_cast<const uint4*>(dOut + t * H);
    for (int j = 0; j < k; ++j) {
      const int32_t p = __ldg(pos + t * k + j);
      if (p < 0) {
        if (lane == 0) dw[t * k + j] = 0.0f;
        continue;
      }
      const float wj = __ldg(w + t * k + j);
      const uint4* y = reinterpret_cast<const uint4*>(Ys + (int64_t)p * H);
      uint4* d = reinterpret_cast<uint4*>(dYs + (int64_t)p * H);
      float dot = 0.0f;
      // kCombineU pieces per lane at a time (2 kCombineU loads in flight); the lane's partial
      // sum still runs over v = lane, lane + 32, ... in order
      for (int64_t v0 = 0; v0 < nvec; v0 += 32 * kCombineU) {
        uint4 gv[kCombineU], yv[kCombineU];
#pragma unroll
        for (int u = 0; u < kCombineU; ++u) {
          const int64_t v = v0 + lane + 32 * u;
          gv[u] = v < nvec ? __ldg(g + v) : make_uint4(0, 0, 0, 0);
          yv[u] = v < nvec ? __ldg(y + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kCombineU; ++u) {
          const int64_t v = v0 + lane + 32 * u;
          if (v >= nvec) continue;
          const uint32_t ga[4] = {gv[u].x, gv[u].y, gv[u].z, gv[u].w};
          const uint32_t ya[4] = {yv[u].x, yv[u].y, yv[u].z, yv[u].w};
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float g0 = bf16_lo(ga[q]), g1 = bf16_hi(ga[q]);
            dot += g0 * bf16_lo(ya[q]);
            dot += g1 * bf16_hi(ya[q]);
            o[q] = pack_bf16x2(wj * g0, wj * g1);
          }
          d[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      if (lane == 0) dw[t * k + j] = dot;
    }
  }
}

int copy_grid(int64_t warps_needed) {
  DeviceInfo dev;
  if (current_device(&dev) != PGG_OK) return 0;
  const int64_t per_block = kCopyThreads / 32;
  return (int)std::max<int64_t>(1, std::min<int64_t>((warps_needed + per_block - 1) / per_block,
                                                     (int64_t)dev.sms * (2048 / kCopyThreads)));
}

}  // namespace

size_t moe_permute_ws_bytes(int64_t T, int E) {
  return (size_t)((T + kChunk - 1) / kChunk) * (size_t)E * sizeof(int32_t);
}

int launch_moe_permute(const int32_t* ids, const void* X, int64_t T, int k, int64_t H, int E, void* Xs,
                       int32_t* group_lens, int32_t* pos, int32_t* ws, int32_t* err, cudaStream_t s) {
  if (T == 0) return cuda_status(cudaMemsetAsync(group_lens, 0, (size_t)E * sizeof(int32_t), s));
  const int64_t nchunk = (T + kChunk - 1) / kChunk;
  const size_t rank_smem = ((size_t)E + kRankWarps * ((size_t)E + kChunk * k)) * sizeof(int32_t);
  if (rank_smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(moe_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)rank_smem);
    if (e != cudaSuccess) return cuda_status(e);
  }
  moe_count_kernel<<<(unsigned)((nchunk + kCountWarps - 1) / kCountWarps), kCountWarps * 32,
                     (size_t)kCountWarps * E * sizeof(int32_t), s>>>(ids, T, k, E, nchunk, ws, err);
  moe_scan_kernel<<<E, kScanThreads, 0, s>>>(nchunk, ws, group_lens);
  moe_rank_kernel<<<(unsigned)((nchunk + kRankWarps - 1) / kRankWarps), kRankWarps * 32, rank_smem, s>>>(
      ids, T, k, E, nchunk, ws, group_lens, pos);
  if (X) {
    const int blocks = copy_grid(T * k);
    if (blocks == 0) return PGG_ERR_CUDA;
    moe_gather_kernel<<<blocks, kCopyThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(X), pos, T * k, k, H,
                                                      static_cast<__nv_bfloat16*>(Xs));
  }
  return cuda_status(cudaGetLastError());
}

int launch_moe_combine(const void* Ys, const int32_t* pos, const float* w, int64_t T, int k, int64_t H,
                       void* out, cudaStream_t s) {
  if (T == 0) return PGG_OK;
  // one wave of resident blocks (the kernel walks tokens with a grid stride): its registers
  // allow fewer blocks per SM than copy_grid assumes
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_combine_kernel, kCopyThreads, 0);
  if (e != cudaSuccess) return cuda_status(e);
  const int64_t need = (T + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)dev.sms * std::max(per_sm, 1)));
  moe_combine_kernel<<<blocks, kCopyThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(Ys), pos, w, T, k, H,
                                                     static_cast<__nv_bfloat16*>(out));
  return cuda_status(cudaGetLastError());
}

int launch_moe_combine_bwd(const void* dOut, const void* Ys, const int32_t* pos, const float* w, int64_t T, int k,
                           int64_t H, void* dYs, float* dw, cudaStream_t s) {
  if (T == 0) return PGG_OK;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, moe_combine_bwd_kernel, kCopyThreads, 0);
  if (e != cudaSuccess) return cuda_status(e);
  const int64_t need = (T + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)dev.sms * std::max(per_sm, 1)));
  moe_combine_bwd_kernel<<<blocks, kCopyThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(dOut), static_cast<const __nv_bfloat16*>(Ys), pos, w, T, k, H,
      static_cast<__nv_bfloat16*>(dYs), dw);
  return cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------- permute without a caller workspace
//
// Some callers cannot hand the permute a scratch buffer: a C or real-time host
// component with no access to the framework's caching allocator and a fixed
// device-memory budget, or code that must not call cudaMalloc because it
// implicitly synchronises the device in the middle of a pipelined stream
// schedule.  For them the count table lives in a statically sized module
// array instead, and the call allocates nothing.
namespace {

constexpr int64_t kNoAllocScratchInts = PGG_MOE_NOALLOC_MAX_WS_INTS;

// The count table of pgg_moe_permute_noalloc.  In host code this name is only
// a stand-in for the symbol; its device address comes from cudaGetSymbolAddress.
__device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kScratchDevices = 64;

// The cached address of g_permute_scratch per device, with the unique ID of the
// context it was looked up in: a device reset (cudaDeviceReset) destroys that
// context and reloads the module in a new one, whose array may sit elsewhere, so
// an address is reused only while the current context is the one it came from.
struct ScratchSlot {
  unsigned long long ctx_id = 0;
  int32_t* ptr = nullptr;
};
ScratchSlot g_scratch[kScratchDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// ID of the current context, or 0 when no context is current yet (called with g_scratch_mu held).
int current_ctx_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return PGG_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext c = nullptr;
  *id = 0;
  if (g_ctx_get_current(&c) != CUDA_SUCCESS) return PGG_ERR_CUDA;
  if (c && g_ctx_get_id(c, id) != CUDA_SUCCESS) return PGG_ERR_CUDA;
  return PGG_OK;
}

// Device address of g_permute_scratch on `device` (the current device): looked up
// with cudaGetSymbolAddress on the first call in each context and cached.
int scratch_for(int device, int32_t** out) {
  if (device < 0 || device >= kScratchDevices) return PGG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchSlot& slot = g_scratch[device];
  unsigned long long id = 0;
  int st = current_ctx_id(&id);
  if (st != PGG_OK) return st;
  if (!slot.ptr || id == 0 || id != slot.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);  // makes the context current
    if (e != cudaSuccess || p == nullptr) return PGG_ERR_CUDA;
    if ((st = current_ctx_id(&id)) != PGG_OK) return st;
    slot.ptr = static_cast<int32_t*>(p);
    slot.ctx_id = id;
  }
  *out = slot.ptr;
  return PGG_OK;
}

}  // namespace
}  // namespace pgg

extern "C" int pgg_moe_permute_noalloc(const int32_t* topk_ids, const void* X, int64_t T, int k, int64_t H,
                                       int E, void* Xs, int32_t* group_lens, int32_t* pos, int32_t* err,
                                       void* stream) {
  using namespace pgg;
  if (k < 1 || k > 32 || E < 1 || E > kMaxGroups || T < 0 || T * k >= ((int64_t)1 << 31))
    return PGG_ERR_INVALID_ARG;
  if (!group_lens) return PGG_ERR_INVALID_ARG;
  if (X) {
    if (H < 8 || H >= ((int64_t)1 << 30)) return PGG_ERR_INVALID_ARG;
    if (H % 8) return PGG_ERR_ALIGNMENT;
    if (!Xs) return PGG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(Xs) & 15u))
      return PGG_ERR_ALIGNMENT;
  }
  if ((int64_t)moe_permute_ws_bytes(T, E) > kNoAllocScratchInts * (int64_t)sizeof(int32_t))
    return PGG_ERR_TOO_LARGE;
  if (T > 0) {
    if (!topk_ids || !pos) return PGG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(pos) & 3u))
      return PGG_ERR_ALIGNMENT;
  }
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != PGG_OK) return st;
  int32_t* ws = nullptr;
  if ((st = scratch_for(dev.device, &ws)) != PGG_OK) return st;
  // The count kernel writes every table entry that the scan and rank kernels
  // read, so the scratch needs no clearing between calls.
  return launch_moe_permute(topk_ids, X, T, k, H, E, Xs, group_lens, pos, ws, err,
                            reinterpret_cast<cudaStream_t>(stream));
}
