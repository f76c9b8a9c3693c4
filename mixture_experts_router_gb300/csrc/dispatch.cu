// Token dispatch: per-expert histogram, prefix sums and a stable permutation
// of the T*k (token, slot) pairs, then the row gather that builds the
// expert-grouped activations.  This is the dispatch kernel of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §2.3 (scatter each token to its k
// experts' input buffers), whose irregular scatter and warp divergence that
// page's §2.1 names as the cost.  Here the ranks come from warp match/ballot
// prefix counts in flat (token, slot) order, so the permutation is
// deterministic (expert ascending, then token ascending) and the row copies
// are plain coalesced 16-byte moves.
//
//   dispatch_count   : per chunk of 2048 pairs, counts per expert
//   dispatch_scan    : one block: per-expert totals, offsets, per-chunk row
//                      bases, the expert-aligned 128-row tile prefix and the
//                      tile -> expert map used by the grouped GEMMs
//   dispatch_scatter : per chunk: warp-aggregated ranks -> tok[], inv[]
//   dispatch_small   : the three above in one block, for small T*k
//   dispatch_scan_blocks : when the router already ranked each pair inside
//                      its block of tokens: one block scans the per-block
//                      counts (all of them staged in shared memory at once)
//                      into per-block row bases, totals, offsets and tiles
//   dispatch_copy    : each token's row of x into its k rows of Xp (and,
//                      after dispatch_scan_blocks, the global ranks: inv, tok)
//   dispatch_coop    : count, scan, ranks and row copy in one cooperative
//                      launch with one grid barrier (the default for the
//                      dispatch's own ranking)
#include "grid_barrier.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerWarp = kDispatchChunk / kWarps;  // 256 pairs, 8 rounds of 32

__global__ void __launch_bounds__(kThreads) dispatch_count(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int hist[256];
  for (int e = threadIdx.x; e < a.E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const int64_t M = static_cast<int64_t>(a.T) * a.k;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kDispatchChunk;
  for (int i = threadIdx.x; i < kDispatchChunk; i += kThreads) {
    const int64_t p = base + i;
    if (p < M) {
      const int e = a.ids[p];
      if (e >= 0 && e < a.E)
        atomicAdd(&hist[e], 1);
      else
        set_error(a.err, kErrDevice);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < a.E; e += kThreads)
    a.chunk[static_cast<int64_t>(blockIdx.x) * a.E + e] = hist[e];
}

// exclusive scan of one value per thread over a block of NW warps
template <int NW = kWarps>
__device__ int block_exclusive_scan(int v, int* tmp) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = (lane < NW) ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) tmp[lane] = s;
  }
  __syncthreads();
  const int r = x - v + (warp > 0 ? tmp[warp - 1] : 0);
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) dispatch_scan(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int tmp[kWarps];
  const int e = threadIdx.x;
  int total = 0;
  if (e < a.E) {
    for (int b = 0; b < a.n_chunks; ++b) {
      int* slot = a.chunk + static_cast<int64_t>(b) * a.E + e;
      const int c = *slot;
      *slot = total;  // exclusive within this expert
      total += c;
    }
  }
  const int mt = (total + kTileM - 1) / kTileM;
  const int pt = (mt + 1) / 2;
  const int off = block_exclusive_scan(e < a.E ? total : 0, tmp);
  const int moff = block_exclusive_scan(e < a.E ? mt : 0, tmp);
  const int poff = block_exclusive_scan(e < a.E ? pt : 0, tmp);
  if (e < a.E) {
    a.counts[e] = total;
    a.offsets[e] = off;
    a.mtile_off[e] = moff;
    if (e == a.E - 1) {
      a.offsets[a.E] = off + total;
      a.mtile_off[a.E] = moff + mt;
      if (moff + mt > a.max_mtiles) set_error(a.err, kErrDevice);
    }
    for (int b = 0; b < a.n_chunks; ++b) a.chunk[static_cast<int64_t>(b) * a.E + e] += off;
    for (int i = moff; i < moff + mt && i < a.max_mtiles; ++i) a.mtile_expert[i] = e;
    if (a.ptile_off != nullptr) {
      a.ptile_off[e] = poff;
      if (e == a.E - 1) a.ptile_off[a.E] = poff + pt;
      for (int i = poff; i < poff + pt && i < a.max_mtiles; ++i) a.ptile_expert[i] = e;
    }
  }
}

__global__ void __launch_bounds__(kThreads) dispatch_scatter(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int wh[kWarps][256];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < kWarps * 256; i += kThreads) (&wh[0][0])[i] = 0;
  __syncthreads();
  const int64_t M = static_cast<int64_t>(a.T) * a.k;
  const int64_t wbase = static_cast<int64_t>(blockIdx.x) * kDispatchChunk + warp * kPerWarp;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // pass 1: this warp's count per expert
  for (int r = 0; r < kPerWarp / 32; ++r) {
    const int64_t p = wbase + r * 32 + lane;
    int e = (p < M) ? a.ids[p] : -1;
    if (e < 0 || e >= a.E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (__ffs(m) - 1) == lane) wh[warp][e] += __popc(m);
  }
  __syncthreads();
  // per expert: exclusive over the warps, starting at this chunk's row base
  for (int e = threadIdx.x; e < a.E; e += kThreads) {
    int base = a.chunk[static_cast<int64_t>(blockIdx.x) * a.E + e];
    for (int w = 0; w < kWarps; ++w) {
      const int c = wh[w][e];
      wh[w][e] = base;
      base += c;
    }
  }
  __syncthreads();
  // pass 2: ranks in flat (token, slot) order
  for (int r = 0; r < kPerWarp / 32; ++r) {
    const int64_t p = wbase + r * 32 + lane;
    int e = (p < M) ? a.ids[p] : -1;
    if (e < 0 || e >= a.E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    int rank = 0;
    if (e >= 0) rank = wh[warp][e] + __popc(m & lt_mask);
    __syncwarp();
    if (e >= 0 && (__ffs(m) - 1) == lane) wh[warp][e] += __popc(m);
    __syncwarp();
    if (e >= 0) {
      if (rank < 0 || rank >= M) {
        set_error(a.err, kErrDevice);
      } else {
        a.tok[rank] = static_cast<int32_t>(p / a.k);
        a.inv[p] = rank;
      }
    }
  }
}

// Count, scan and ranks in one 1024-thread block, for T*k <= kDispatchSmallPairs: the
// 32 warps take consecutive runs of the flat (token, slot) pairs, so the
// warp-aggregated ranks come out in token order exactly as in the chunked
// kernels above.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / 32;

__global__ void __launch_bounds__(kSmallThreads) dispatch_small(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int wh[kSmallWarps][256];
  __shared__ int tmp[kSmallWarps];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < kSmallWarps * 256; i += kSmallThreads) (&wh[0][0])[i] = 0;
  __syncthreads();
  const int64_t M = static_cast<int64_t>(a.T) * a.k;
  const int64_t per_warp = ((M + kSmallWarps - 1) / kSmallWarps + 31) / 32 * 32;
  const int64_t wbase = warp * per_warp;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t r = 0; r < per_warp; r += 32) {
    const int64_t p = wbase + r + lane;
    int e = (p < M) ? a.ids[p] : -1;
    if (p < M && (e < 0 || e >= a.E)) set_error(a.err, kErrDevice);
    if (e < 0 || e >= a.E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (__ffs(m) - 1) == lane) wh[warp][e] += __popc(m);
  }
  __syncthreads();
  int total = 0;
  const int e = threadIdx.x;
  if (e < a.E) {
    for (int w = 0; w < kSmallWarps; ++w) {
      const int c = wh[w][e];
      wh[w][e] = total;
      total += c;
    }
  }
  const int mt = (total + kTileM - 1) / kTileM;
  const int pt = (mt + 1) / 2;
  const int off = block_exclusive_scan<kSmallWarps>(e < a.E ? total : 0, tmp);
  const int moff = block_exclusive_scan<kSmallWarps>(e < a.E ? mt : 0, tmp);
  const int poff = block_exclusive_scan<kSmallWarps>(e < a.E ? pt : 0, tmp);
  if (e < a.E) {
    a.counts[e] = total;
    a.offsets[e] = off;
    a.mtile_off[e] = moff;
    if (e == a.E - 1) {
      a.offsets[a.E] = off + total;
      a.mtile_off[a.E] = moff + mt;
      if (moff + mt > a.max_mtiles) set_error(a.err, kErrDevice);
    }
    for (int i = moff; i < moff + mt && i < a.max_mtiles; ++i) a.mtile_expert[i] = e;
    if (a.ptile_off != nullptr) {
      a.ptile_off[e] = poff;
      if (e == a.E - 1) a.ptile_off[a.E] = poff + pt;
      for (int i = poff; i < poff + pt && i < a.max_mtiles; ++i) a.ptile_expert[i] = e;
    }
    for (int w = 0; w < kSmallWarps; ++w) wh[w][e] += off;
  }
  __syncthreads();
  for (int64_t r = 0; r < per_warp; r += 32) {
    const int64_t p = wbase + r + lane;
    int e2 = (p < M) ? a.ids[p] : -1;
    if (e2 < 0 || e2 >= a.E) e2 = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e2);
    int rank = 0;
    if (e2 >= 0) rank = wh[warp][e2] + __popc(m & lt_mask);
    __syncwarp();
    if (e2 >= 0 && (__ffs(m) - 1) == lane) wh[warp][e2] += __popc(m);
    __syncwarp();
    if (e2 >= 0) {
      if (rank < 0 || rank >= M) {
        set_error(a.err, kErrDevice);
      } else {
        a.tok[rank] = static_cast<int32_t>(p / a.k);
        a.inv[p] = rank;
      }
    }
  }
}

constexpr int kScanThreads = 1024;
constexpr int kScanWarps = kScanThreads / 32;

// Per-expert totals -> counts, offsets, the 128-row tile prefix (and pairs)
// with their tile -> expert maps; thread e of the block handles expert e.
// Returns offsets[e] (0 for threads past E).  All threads must call it.
__device__ int publish_totals(const DispatchArgs& a, int total, int* tmp) {
  const int e = threadIdx.x;
  const int mt = (total + kTileM - 1) / kTileM;
  const int pt = (mt + 1) / 2;
  const int off = block_exclusive_scan<kScanWarps>(e < a.E ? total : 0, tmp);
  const int moff = block_exclusive_scan<kScanWarps>(e < a.E ? mt : 0, tmp);
  const int poff = block_exclusive_scan<kScanWarps>(e < a.E ? pt : 0, tmp);
  if (e < a.E) {
    a.counts[e] = total;
    a.offsets[e] = off;
    a.mtile_off[e] = moff;
    if (e == a.E - 1) {
      a.offsets[a.E] = off + total;
      a.mtile_off[a.E] = moff + mt;
      if (moff + mt > a.max_mtiles) set_error(a.err, kErrDevice);
    }
    for (int i = moff; i < moff + mt && i < a.max_mtiles; ++i) a.mtile_expert[i] = e;
    if (a.ptile_off != nullptr) {
      a.ptile_off[e] = poff;
      if (e == a.E - 1) a.ptile_off[a.E] = poff + pt;
      for (int i = poff; i < poff + pt && i < a.max_mtiles; ++i) a.ptile_expert[i] = e;
    }
  }
  return e < a.E ? off : 0;
}

// chunk[b][e] holds rank block b's count of expert e; it becomes the global
// rank of the block's first pair of e: offsets[e] + sum_{b' < b} chunk[b'][e].
// Shared memory: (n_rank_blocks + 1) rows of E + 1 counts (the odd row
// length keeps the per-expert column walk free of bank conflicts; the last
// row holds the totals).
__global__ void __launch_bounds__(kScanThreads) dispatch_scan_blocks(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  extern __shared__ int sc[];
  __shared__ int tmp[kScanWarps];
  __shared__ int s_off[256];
  const int nb = a.n_rank_blocks, E = a.E, ld = E + 1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < nb * E; i += kScanThreads) sc[(i / E) * ld + i % E] = a.chunk[i];
  __syncthreads();
  for (int e = warp; e < E; e += kScanWarps) {
    int carry = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      const int b = b0 + lane;
      const int v = b < nb ? sc[b * ld + e] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (b < nb) sc[b * ld + e] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) sc[nb * ld + e] = carry;
  }
  __syncthreads();
  const int total = threadIdx.x < E ? sc[nb * ld + threadIdx.x] : 0;
  const int off = publish_totals(a, total, tmp);
  if (threadIdx.x < E) s_off[threadIdx.x] = off;
  __syncthreads();
  for (int i = threadIdx.x; i < nb * E; i += kScanThreads) a.chunk[i] = sc[(i / E) * ld + i % E] + s_off[i % E];
}

// Row copy into the expert-grouped layout, token-major: one warp per token
// reads its row of x once (16-byte vectors, eight in flight per lane) and
// writes it to its k padded rows, row(t, s) = 128 tile_off[e] + inv - off[e].
// Padding rows of each expert's last tile are left as they are: no GEMM
// output row depends on another row.
__global__ void __launch_bounds__(kThreads) dispatch_copy(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int vec_per_row = a.d / 8;
  const int64_t rows = static_cast<int64_t>(a.max_mtiles) * kTileM;
  const int64_t M = static_cast<int64_t>(a.T) * a.k;
  for (int t = blockIdx.x * kWarps + warp; t < a.T; t += gridDim.x * kWarps) {
    int64_t dst_row = -1;
    if (lane < a.k) {
      const int64_t p = static_cast<int64_t>(t) * a.k + lane;
      const int e = a.ids[p];
      int r = a.inv[p];
      if (a.rank_block > 0 && e >= 0 && e < a.E) {
        r += a.chunk[static_cast<int64_t>(t / a.rank_block) * a.E + e];
        a.inv[p] = r;
        if (r >= 0 && r < M)
          a.tok[r] = t;
        else
          set_error(a.err, kErrDevice);
      }
      if (e >= 0 && e < a.E) dst_row = static_cast<int64_t>(a.mtile_off[e]) * kTileM + (r - a.offsets[e]);
      if (dst_row < 0 || dst_row >= rows) {
        set_error(a.err, kErrDevice);
        dst_row = -1;
      }
    }
    if (!a.copy_rows) continue;
    const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.d);
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * 32 + lane;
        if (v < vec_per_row) buf[u] = __ldg(src + v);
      }
      for (int s = 0; s < a.k; ++s) {
        const int64_t row = __shfl_sync(0xffffffffu, dst_row, s);
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(a.xp + row * a.d);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < vec_per_row) dst[v] = buf[u];
        }
      }
    }
  }
}

// The steps above in one cooperative launch of G co-resident blocks (the
// launch guarantees that all of them run at once, so each block's one wait
// at the grid barrier ends; the wait is bounded all the same).  Block b owns
// the tokens [b tpb, (b + 1) tpb) and with them the flat pairs
// [b tpb k, (b + 1) tpb k):
//   1. per-warp counts per expert of its pairs (warp w: a contiguous run,
//      as in dispatch_small), their sum to chunk[b][e]
//   2. the grid barrier
//   3. every block sums the G rows of counts itself: per-expert totals and
//      its own base sum_{b' < b} chunk[b'][e]; the expert prefix and the tile
//      maps follow (block 0 publishes them)
//   4. ranks of its pairs in flat (token, slot) order -> tok, inv
//   5. its tokens' rows of x into their k padded rows of Xp
constexpr int kCoopThreads = 1024;
constexpr int kCoopWarps = kCoopThreads / 32;

__global__ void __launch_bounds__(kCoopThreads) dispatch_coop(DispatchArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int wh[kCoopWarps][256];
  __shared__ int part_pre[kCoopThreads], part_tot[kCoopThreads];
  __shared__ int s_off[256], s_moff[256];
  __shared__ int tmp[kCoopWarps];
  __shared__ int s_ok;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x), E = a.E, k = a.k;
  const int64_t M = static_cast<int64_t>(a.T) * k;
  const int tpb = (a.T + G - 1) / G;
  const int t0 = static_cast<int>(min(static_cast<int64_t>(a.T), static_cast<int64_t>(b) * tpb));
  const int t1 = min(a.T, t0 + tpb);
  const int64_t p0 = static_cast<int64_t>(t0) * k, p1 = static_cast<int64_t>(t1) * k;
  const int64_t per_warp = ((p1 - p0 + kCoopWarps - 1) / kCoopWarps + 31) / 32 * 32;
  const int64_t wbase = p0 + warp * per_warp;
  const int64_t wend = min(p1, wbase + per_warp);
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int i = threadIdx.x; i < kCoopWarps * 256; i += kCoopThreads) (&wh[0][0])[i] = 0;
  __syncthreads();

  // 1. counts (the loop bound is the same for every lane of the warp)
  for (int64_t q = wbase; q < wend; q += 32) {
    const int64_t p = q + lane;
    int e = p < wend ? a.ids[p] : -1;
    if (p < wend && (e < 0 || e >= E)) set_error(a.err, kErrDevice);
    if (e < 0 || e >= E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (__ffs(m) - 1) == lane) wh[warp][e] += __popc(m);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kCoopThreads) {
    int c = 0;
    for (int w = 0; w < kCoopWarps; ++w) c += wh[w][e];
    a.chunk[static_cast<int64_t>(b) * E + e] = c;
  }

  // 2. grid barrier (the words reset themselves: no memset before the
  // launch); the block's last thread counts its departure while the others
  // start the column sums
  if (!grid_barrier_wait(a.bar, static_cast<unsigned>(G + a.test_stall), a.wait_limit_ns, a.err, &s_ok)) {
    if (threadIdx.x == 0) grid_barrier_depart(a.bar, static_cast<unsigned>(G));
    return;
  }
  if (threadIdx.x == kCoopThreads - 1) grid_barrier_depart(a.bar, static_cast<unsigned>(G));

  // 3. column sums: thread i < P E sums expert i % E over the rows
  // i / E, i / E + P, ... (consecutive threads read consecutive words of a
  // row; P = kCoopThreads / E >= 4 parts), up to kSumLoads loads in flight
  // at a time, then thread e adds the P parts
  constexpr int kSumLoads = 20;
  const int P = kCoopThreads / E;
  if (static_cast<int>(threadIdx.x) < P * E) {
    const int e = threadIdx.x % E, q = threadIdx.x / E;
    int pre = 0, tot = 0;
    for (int r0 = q; r0 < G; r0 += P * kSumLoads) {
      int c[kSumLoads];
#pragma unroll
      for (int i = 0; i < kSumLoads; ++i) {
        const int r = r0 + i * P;
        c[i] = r < G ? __ldcg(a.chunk + static_cast<int64_t>(r) * E + e) : 0;
      }
#pragma unroll
      for (int i = 0; i < kSumLoads; ++i) {
        tot += c[i];
        pre += r0 + i * P < b ? c[i] : 0;
      }
    }
    part_pre[threadIdx.x] = pre;
    part_tot[threadIdx.x] = tot;
  }
  __syncthreads();
  const int e = threadIdx.x;
  int total = 0, pre = 0;
  if (e < E)
    for (int q = 0; q < P; ++q) {
      total += part_tot[q * E + e];
      pre += part_pre[q * E + e];
    }
  const int mt = (total + kTileM - 1) / kTileM;
  const int pt = (mt + 1) / 2;
  const int off = block_exclusive_scan<kCoopWarps>(e < E ? total : 0, tmp);
  const int moff = block_exclusive_scan<kCoopWarps>(e < E ? mt : 0, tmp);
  const int poff = block_exclusive_scan<kCoopWarps>(e < E ? pt : 0, tmp);
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
    int base = off + pre;  // this block's first row of expert e, then each warp's
    for (int w = 0; w < kCoopWarps; ++w) {
      const int c = wh[w][e];
      wh[w][e] = base;
      base += c;
    }
  }
  __syncthreads();

  // 4. ranks
  for (int64_t q = wbase; q < wend; q += 32) {
    const int64_t p = q + lane;
    int e2 = p < wend ? a.ids[p] : -1;
    if (e2 < 0 || e2 >= E) e2 = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e2);
    int rank = 0;
    if (e2 >= 0) rank = wh[warp][e2] + __popc(m & lt_mask);
    __syncwarp();
    if (e2 >= 0 && (__ffs(m) - 1) == lane) wh[warp][e2] += __popc(m);
    __syncwarp();
    if (e2 >= 0) {
      if (rank < 0 || rank >= M) {
        set_error(a.err, kErrDevice);
      } else {
        a.tok[rank] = static_cast<int32_t>(p / k);
        a.inv[p] = rank;
      }
    }
  }
  if (!a.copy_rows) return;
  __syncthreads();  // this block's inv stores are visible to all its threads

  // 5. row copy: items of 128 16-byte vectors of one token's row, dealt to
  // the block's warps in turn (a whole row per warp would leave the block's
  // last warps idle: 54 tokens over 16 warps on the 128-expert layer); each
  // warp moves two items per round, eight 16-byte loads in flight per lane
  constexpr int kSegVec = 128;
  const int vec_per_row = a.d / 8;
  const int segs = (vec_per_row + kSegVec - 1) / kSegVec;
  const int n_items = (t1 - t0) * segs;
  const int64_t rows = static_cast<int64_t>(a.max_mtiles) * kTileM;
  for (int it = warp; it < n_items; it += 2 * kCoopWarps) {
    uint4 buf[2][kSegVec / 32];
    int64_t dst_row[2] = {-1, -1};
    int v_base[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int item = it + h * kCoopWarps;
      if (item >= n_items) continue;  // the same for the whole warp
      const int t = t0 + item / segs;
      v_base[h] = (item % segs) * kSegVec;
      if (lane < k) {
        const int64_t p = static_cast<int64_t>(t) * k + lane;
        const int ee = a.ids[p];
        if (ee >= 0 && ee < E) {
          dst_row[h] = static_cast<int64_t>(s_moff[ee]) * kTileM + (a.inv[p] - s_off[ee]);
          if (dst_row[h] < 0 || dst_row[h] >= rows) {
            set_error(a.err, kErrDevice);
            dst_row[h] = -1;
          }
        }
      }
      const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.d);
#pragma unroll
      for (int u = 0; u < kSegVec / 32; ++u) {
        const int v = v_base[h] + u * 32 + lane;
        if (v < vec_per_row) buf[h][u] = __ldg(src + v);
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (it + h * kCoopWarps >= n_items) continue;
      for (int s = 0; s < k; ++s) {
        const int64_t row = __shfl_sync(0xffffffffu, dst_row[h], s);
        if (row < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(a.xp + row * a.d);
#pragma unroll
        for (int u = 0; u < kSegVec / 32; ++u) {
          const int v = v_base[h] + u * 32 + lane;
          if (v < vec_per_row) dst[v] = buf[h][u];
        }
      }
    }
  }
}

}  // namespace

// The per-chunk counts of dispatch_count have the layout of the router's
// per-block counts ([chunk][E]), so the shared-memory block scan turns them
// into per-chunk row bases when they fit in max_words (kFusedScanWords after
// dispatch_prepare, else the 48 KB a launch gets without it); its columns are
// scanned by whole warps, where dispatch_scan walks each expert's chunks with
// one thread.
static cudaError_t launch_chunk_scan(const DispatchArgs& a, int max_words, cudaStream_t s) {
  if ((a.n_chunks + 1) * (a.E + 1) <= max_words && a.E <= 256) {
    DispatchArgs b = a;
    b.n_rank_blocks = a.n_chunks;
    return launch_kernel(dispatch_scan_blocks, 1, kScanThreads, (b.n_rank_blocks + 1) * (b.E + 1) * 4, s, b);
  }
  return launch_kernel(dispatch_scan, 1, kThreads, 0, s, a);
}

cudaError_t launch_dispatch_ranks(const DispatchArgs& a, int scan_words, cudaStream_t s) {
  if (a.n_chunks <= 0) return cudaSuccess;
  cudaError_t e = launch_kernel(dispatch_count, a.n_chunks, kThreads, 0, s, a);
  if (e == cudaSuccess) e = launch_chunk_scan(a, scan_words, s);
  if (e == cudaSuccess) e = launch_kernel(dispatch_scatter, a.n_chunks, kThreads, 0, s, a);
  return e;
}

cudaError_t dispatch_prepare() {
  return cudaFuncSetAttribute(dispatch_scan_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kFusedScanWords * 4);
}

int dispatch_coop_max_blocks(int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_coop, kCoopThreads, 0) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return per_sm > 0 ? num_sms : 0;
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s) {
  if (a.n_chunks <= 0) return cudaSuccess;
  if (a.rank_block <= 0 && a.coop_blocks > 0) {
    if (a.E > 256 || a.bar == nullptr) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.coop_blocks, 1, 1);
    cfg.blockDim = dim3(kCoopThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_coop, a);
  }
  if (a.rank_block > 0) {
    const int words = (a.n_rank_blocks + 1) * (a.E + 1);
    if (words > kFusedScanWords || a.E > 256) return cudaErrorInvalidValue;
    launch_kernel(dispatch_scan_blocks, 1, kScanThreads, words * 4, s, a);
    launch_kernel(dispatch_copy, a.gather_blocks, kThreads, 0, s, a);
    return cudaGetLastError();
  }
  if (static_cast<int64_t>(a.T) * a.k <= kDispatchSmallPairs) {
    launch_kernel(dispatch_small, 1, kSmallThreads, 0, s, a);
  } else {
    launch_kernel(dispatch_count, a.n_chunks, kThreads, 0, s, a);
    launch_chunk_scan(a, kFusedScanWords, s);
    launch_kernel(dispatch_scatter, a.n_chunks, kThreads, 0, s, a);
  }
  if (a.copy_rows) launch_kernel(dispatch_copy, a.gather_blocks, kThreads, 0, s, a);
  return cudaGetLastError();
}

}  // namespace cbmoe
