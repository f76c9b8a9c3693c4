// Router and dispatch in one cooperative launch, for layers of up to 16
// experts (the Mixtral-shaped layers): the router of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2 (logits, top-k on the
// device) with the gate of "Colibri：面向MoE模型的高性能C语言推理引擎" §2.1,
// then the dispatch of the first page's §2.3 (per-expert histogram, prefix
// sum, stable permutation, row copy), without a kernel boundary between them.
//
// One block per SM.  Block b owns the tokens [b T / G, (b + 1) T / G) of the
// G blocks (an even share: at decode size 64 tokens spread over 64 blocks):
//   1. the logits and gate of its tokens, 16 at a time (one mma.sync
//      m-tile, the last one of a block possibly partial): the 16 warps split
//      d 16 ways, the partial logits are summed in a fixed order in shared
//      memory, the bias added, one warp per token takes the gate; the block
//      keeps its tokens' ids;
//   2. ranks of its pairs within the block, in (token, slot) order
//      (match-any groups per warp, then a scan over the warps), and its
//      per-expert counts -> chunk[b][e];
//   3. one grid barrier (the cooperative launch keeps every block resident;
//      the wait is bounded by wall time all the same; the barrier words reset
//      themselves, so the launch needs no memset before it);
//   4. every block scans the count rows itself (one warp per expert): expert
//      totals and its own base sum_{b' < b} chunk[b'][e]; block 0 publishes
//      the counts, offsets and 128-row tile maps;
//   5. the global ranks of its pairs (base + in-block rank) into tok and inv,
//      and the copy of its tokens' rows, Xp[row(t, s)] = x[t].  Those rows
//      were read in step 1 a few microseconds earlier, so they come from L2:
//      x crosses HBM once, where the separate router and row-copy kernels
//      read it twice, and the one-block scan kernel between them is gone.
// The results are those of the separate router and dispatch kernels: the same
// logit sums in the same order, the same gate, and ranks in the canonical
// order (expert ascending, then token ascending).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "grid_barrier.cuh"
#include "route_ranks.cuh"
#include "router_common.cuh"

namespace cbmoe {
namespace {

using namespace router_detail;

constexpr int kRdThreads = 512;
constexpr int kRdWarps = kRdThreads / 32;  // each takes 1/16 of d in step 1
constexpr int kUnit = 16;                  // tokens per unit: one m16 tile
constexpr int kMaxExperts = 16;
constexpr int kSegVec = 128;               // 16-byte vectors per copy item
constexpr int kMaxGridRounds = 8;          // blocks of the launch at most 32 kMaxGridRounds
constexpr int kSmemLimit = 160 * 1024;     // dynamic shared memory of a launch at most

// warp-wide exclusive scan of v over lanes
__device__ __forceinline__ int warp_exclusive_scan(int v) {
  const int lane = threadIdx.x % 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x - v;
}

// NT n-tiles of 8 experts (E <= 8 NT); d a multiple of 512.  Dynamic shared
// memory: partial logits [16][16][8 NT] fp32, the block's ids and their
// in-block ranks (then padded rows), [own_max][k] int32 each, and the
// blocks' bases [G][E] int32.
template <int NT>
__global__ void __launch_bounds__(kRdThreads, 1) route_dispatch_kernel(RouterArgs r, DispatchArgs a,
                                                                       int32_t own_max) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  constexpr int EP = NT * 8;
  extern __shared__ __align__(16) unsigned char rd_smem[];
  float* part = reinterpret_cast<float*>(rd_smem);                // [16][16][EP]
  int* s_ids = reinterpret_cast<int*>(part + kRdWarps * kUnit * EP);
  int* s_row = s_ids + own_max * r.k;                              // [own_max][k]
  int* s_pref = s_row + own_max * r.k;                             // [G][E]
  __shared__ int s_cnt[kMaxExperts], s_off[kMaxExperts], s_moff[kMaxExperts];
  __shared__ int s_wcnt[kRdWarps][kMaxExperts];
  __shared__ int s_ok;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, q = lane & 3;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const int T = r.T, E = r.E, k = r.k, d = r.d;
  const int64_t M = static_cast<int64_t>(T) * k;
  const int t_lo = static_cast<int>(static_cast<int64_t>(b) * T / G);
  const int t_hi = static_cast<int>(static_cast<int64_t>(b + 1) * T / G);
  const int own = t_hi - t_lo;

  // 1. logits and gate of the block's tokens, 16 at a time (rows at or past
  // t_hi read as zero)
  const int dslice = d / kRdWarps;
  const int dbeg = warp * dslice;
  for (int tok0 = t_lo; tok0 < t_hi; tok0 += kUnit) {
    float acc[NT][4];
    tile_logits<NT, 8>(r.x, r.wr, t_hi, d, E, tok0, 0, dbeg, dslice, acc);
    float* mine = part + warp * kUnit * EP;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int col = j * 8 + 2 * q;
      mine[g * EP + col] = acc[j][0];
      mine[g * EP + col + 1] = acc[j][1];
      mine[(g + 8) * EP + col] = acc[j][2];
      mine[(g + 8) * EP + col + 1] = acc[j][3];
    }
    __syncthreads();
    // sum the 16 partials in a fixed order, add the bias
    for (int i = threadIdx.x; i < kUnit * EP; i += kRdThreads) {
      float v = part[i];
#pragma unroll
      for (int s = 1; s < kRdWarps; ++s) v += part[s * kUnit * EP + i];
      const int e = i % EP;
      if (r.bias != nullptr && e < E) v += __ldg(r.bias + e);
      part[i] = v;
    }
    __syncthreads();
    if (r.logits != nullptr) {
      for (int i = threadIdx.x; i < kUnit * E; i += kRdThreads) {
        const int rr = i / E, e = i % E, t = tok0 + rr;
        if (t < t_hi) r.logits[static_cast<int64_t>(t) * E + e] = part[rr * EP + e];
      }
    }
    {
      const int t = tok0 + warp;  // one token per warp
      if (t < t_hi) {
        int id;
        float wt;
        warp_gate<1>(part + warp * EP, E, k, r.raw_weights, id, wt);
        if (lane < k) {
          r.ids[static_cast<int64_t>(t) * k + lane] = id;
          r.w[static_cast<int64_t>(t) * k + lane] = wt;
          s_ids[(t - t_lo) * k + lane] = id;
        }
      }
    }
    __syncthreads();  // part is rewritten by the next group
  }

  // 2. ranks in the block, in flat (token, slot) order: 512 pairs per round,
  // match-any groups inside each warp, then an exclusive scan over the
  // warps per expert on top of the earlier rounds' counts; the block's counts
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (threadIdx.x < E) s_cnt[threadIdx.x] = 0;
  const int npairs = own * k;
  for (int base = 0; base < npairs; base += kRdThreads) {
    const int p = base + threadIdx.x;
    int e = p < npairs ? s_ids[p] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (lane < E) s_wcnt[warp][lane] = 0;
    __syncwarp();
    if (e >= 0 && (__ffs(m) - 1) == lane) s_wcnt[warp][e] = __popc(m);
    __syncthreads();
    if (threadIdx.x < E) {
      int run = s_cnt[threadIdx.x];
      for (int w = 0; w < kRdWarps; ++w) {
        const int c = s_wcnt[w][threadIdx.x];
        s_wcnt[w][threadIdx.x] = run;
        run += c;
      }
      s_cnt[threadIdx.x] = run;
    }
    __syncthreads();
    if (e >= 0) s_row[p] = s_wcnt[warp][e] + __popc(m & lt_mask);
    __syncthreads();  // s_wcnt is rewritten by the next round
  }
  if (threadIdx.x < E) a.chunk[static_cast<int64_t>(b) * E + threadIdx.x] = s_cnt[threadIdx.x];

  // 3. grid barrier (the block's count and rank stores are visible to all
  // blocks after it); one thread of the last warp counts the block's
  // departure while warps 0..E-1 start the column scans
  if (!grid_barrier_wait(a.bar, static_cast<unsigned>(G + a.test_stall), a.wait_limit_ns, a.err, &s_ok)) {
    if (threadIdx.x == 0) grid_barrier_depart(a.bar, static_cast<unsigned>(G));
    return;
  }
  if (threadIdx.x == kRdThreads - 32) grid_barrier_depart(a.bar, static_cast<unsigned>(G));

  // 4. column scans: warp e scans expert e's counts over the G rows, 32 rows
  // a round -> every block's base s_pref[b'][e] and the expert total
  if (warp < E) {
    const int e = warp;
    int cnt[kMaxGridRounds];  // all of the column's loads in flight before the scans
#pragma unroll
    for (int j = 0; j < kMaxGridRounds; ++j) {
      const int rr = j * 32 + lane;
      cnt[j] = rr < G ? __ldcg(a.chunk + static_cast<int64_t>(rr) * E + e) : 0;
    }
    int carry = 0;
#pragma unroll
    for (int j = 0; j < kMaxGridRounds; ++j) {
      const int r0 = j * 32;
      const int rr = r0 + lane;
      const int c = cnt[j];
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (rr < G) s_pref[rr * E + e] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_cnt[e] = carry;  // the expert's total
  }
  __syncthreads();
  if (warp == 0) {
    const int e = lane;
    const int total = e < E ? s_cnt[e] : 0;
    const int mt = (total + kTileM - 1) / kTileM;
    const int pt = (mt + 1) / 2;
    const int off = warp_exclusive_scan(e < E ? total : 0);
    const int moff = warp_exclusive_scan(e < E ? mt : 0);
    const int poff = warp_exclusive_scan(e < E ? pt : 0);
    if (e < E) {
      s_off[e] = off;
      s_moff[e] = moff;
      if (b == 0) {
        a.counts[e] = total;
        a.offsets[e] = off;
        a.mtile_off[e] = moff;
        if (e == E - 1) {
          a.offsets[E] = off + total;
          a.mtile_off[E] = moff + mt;
          if (moff + mt > a.max_mtiles) set_error(a.err, kErrDevice);
        }
        for (int i = moff; i < moff + mt && i < a.max_mtiles; ++i) a.mtile_expert[i] = e;
        if (a.ptile_off != nullptr) {
          a.ptile_off[e] = poff;
          if (e == E - 1) a.ptile_off[E] = poff + pt;
          for (int i = poff; i < poff + pt && i < a.max_mtiles; ++i) a.ptile_expert[i] = e;
        }
      }
    }
  }
  __syncthreads();

  // 5. global ranks of the block's pairs -> tok, inv; each pair's padded row;
  // then the row copy
  const int64_t rows = static_cast<int64_t>(a.max_mtiles) * kTileM;
  for (int i = threadIdx.x; i < own * k; i += kRdThreads) {
    const int t = t_lo + i / k;
    const int e = s_ids[i];
    int row = -1;
    if (e >= 0 && e < E) {
      const int rank = s_off[e] + s_pref[b * E + e] + s_row[i];
      if (rank >= 0 && rank < M) {
        a.inv[static_cast<int64_t>(t) * k + i % k] = rank;
        a.tok[rank] = t;
        const int64_t rw = static_cast<int64_t>(s_moff[e]) * kTileM + (rank - s_off[e]);
        if (rw >= 0 && rw < rows) row = static_cast<int>(rw);
      }
    }
    if (row < 0) set_error(a.err, kErrDevice);
    s_row[i] = row;
  }
  if (!a.copy_rows) return;
  __syncthreads();
  // items of 128 16-byte vectors of one token's row, dealt to the warps in
  // turn; each warp moves two items per round (eight loads in flight per lane)
  const int vec_per_row = d / 8;
  const int segs = (vec_per_row + kSegVec - 1) / kSegVec;
  const int n_items = own * segs;
  for (int it = warp; it < n_items; it += 2 * kRdWarps) {
    uint4 buf[2][kSegVec / 32];
    int tl[2] = {-1, -1};
    int v_base[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int item = it + h * kRdWarps;
      if (item >= n_items) continue;  // the same for the whole warp
      tl[h] = item / segs;
      v_base[h] = (item % segs) * kSegVec;
      const uint4* src = reinterpret_cast<const uint4*>(r.x + static_cast<int64_t>(t_lo + tl[h]) * d);
#pragma unroll
      for (int u = 0; u < kSegVec / 32; ++u) {
        const int v = v_base[h] + u * 32 + lane;
        if (v < vec_per_row) buf[h][u] = __ldg(src + v);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (tl[h] < 0) continue;
      for (int s = 0; s < k; ++s) {
        const int row = s_row[tl[h] * k + s];
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(a.xp + static_cast<int64_t>(row) * d);
#pragma unroll
        for (int u = 0; u < kSegVec / 32; ++u) {
          const int v = v_base[h] + u * 32 + lane;
          if (v < vec_per_row) dst[v] = buf[h][u];
        }
      }
    }
  }
}

template <int NT>
size_t smem_bytes(int own_max, int k, int G, int E) {
  return static_cast<size_t>(kRdWarps) * kUnit * NT * 8 * 4 + 8ull * own_max * k + 4ull * G * E;
}

}  // namespace

int route_dispatch_grid(int T, int num_sms) { return T > 0 ? std::min(num_sms, 32 * kMaxGridRounds) : 0; }

// tokens of the largest block share
int route_dispatch_own_max(int T, int grid) { return grid > 0 ? (T + grid - 1) / grid : 0; }

bool route_dispatch_supported(int T, int d, int E, int k, int num_sms) {
  if (E < 1 || E > kMaxExperts || k < 1 || k > E || d % 512 != 0 || T < 1) return false;
  const int grid = route_dispatch_grid(T, num_sms);
  const int own_max = route_dispatch_own_max(T, grid);
  const size_t smem = E <= 8 ? smem_bytes<1>(own_max, k, grid, E) : smem_bytes<2>(own_max, k, grid, E);
  if (smem > kSmemLimit) return false;
  int per_sm = 0;
  cudaError_t e = E <= 8 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_kernel<1>,
                                                                         kRdThreads, smem)
                         : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_kernel<2>,
                                                                         kRdThreads, smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return per_sm >= 1;
}

cudaError_t route_dispatch_prepare() {
  cudaError_t e = cudaFuncSetAttribute(route_dispatch_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_dispatch_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  return e;
}

cudaError_t launch_route_dispatch(const RouterArgs& r, const DispatchArgs& a, int grid, cudaStream_t s) {
  if (grid <= 0 || r.T <= 0) return cudaSuccess;
  if (r.E > kMaxExperts || r.d % 512 != 0 || a.bar == nullptr) return cudaErrorInvalidValue;
  const int own_max = route_dispatch_own_max(r.T, grid);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kRdThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (r.E <= 8) {
    cfg.dynamicSmemBytes = smem_bytes<1>(own_max, r.k, grid, r.E);
    return cudaLaunchKernelEx(&cfg, route_dispatch_kernel<1>, r, a, own_max);
  }
  cfg.dynamicSmemBytes = smem_bytes<2>(own_max, r.k, grid, r.E);
  return cudaLaunchKernelEx(&cfg, route_dispatch_kernel<2>, r, a, own_max);
}

}  // namespace cbmoe
