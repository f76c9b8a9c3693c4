// Router and dispatch in one cooperative launch for layers of 17 to 256
// experts (the 128-expert and 64-expert layers): the router of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2 (logits and top-k on the
// device) with the gate of "Colibri：面向MoE模型的高性能C语言推理引擎" §2.1,
// then the dispatch of the first page's §2.3 (per-expert histogram, prefix
// sum, stable permutation, row copy), without a kernel boundary between them.
//
// One block per SM.  Block b owns the tokens [b T / G, (b + 1) T / G):
//   1. the logits of its tokens on the tensor cores, up to 128 tokens per
//      pass: two producer threads stream, by TMA, the block's rows of x (a
//      box of just the rows it owns, so no SM loads a neighbour's rows) and
//      the router weights (E padded to NP rows, the padding read as zeros)
//      through two rings of shared-memory stages; one thread issues
//      M = 128, N = NP MMAs into TMEM, each K step of 16 into the next of
//      512 / NP accumulators (in turn), so that consecutive MMAs are
//      independent and no fp32 accumulation chain inside the tensor core
//      runs longer than d / (16 * 512 / NP) steps.  The epilogue sums the
//      accumulators in a fixed order, adds the bias and leaves the logits in
//      shared memory (over the then idle rings); one warp per 2 to 8 tokens
//      takes the gate;
//   2. ranks of its pairs within the block, in (token, slot) order
//      (match-any groups per warp, then a scan over the warps), and its
//      per-expert counts -> chunk[b][e];
//   3. one grid barrier (bounded by wall time; the barrier words reset
//      themselves, so the launch needs no memset before it);
//   4. every block sums the count rows itself: its base
//      sum_{b' < b} chunk[b'][e] and the expert totals (several threads per
//      expert, many loads in flight); the expert offsets and 128-row tile
//      maps follow by a scan, which block 0 publishes;
//   5. the global ranks of its pairs (offset + base + in-block rank) into tok
//      and inv, and the copy of its tokens' rows, Xp[row(t, s)] = x[t], whose
//      rows were read in step 1 a few microseconds earlier and come from L2
//      when x fits there (33.6 MB of the 128-expert layer does; the int8
//      layer's 134 MB is read from HBM again).
// Compared with the separate tcgen05 router (split-K partial logits, then a
// top-k kernel) and the cooperative dispatch, x crosses HBM once instead of
// twice and two kernel boundaries are gone.  The ranks are the canonical
// ones (expert ascending, then token ascending); the logits are sums of the
// same products in another order than the split-K router's.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "grid_barrier.cuh"
#include "router_common.cuh"

namespace cbmoe {
namespace {

using namespace router_detail;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int BM = 128;                    // token rows of one pass (one MMA M)
constexpr int BK = 64;                     // d per k-block (one 128-byte swizzled row)
constexpr int A_BYTES = BM * BK * 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxExperts = 256;
constexpr int kMaxGrid = 256;
constexpr int kMinTokensPerBlock = 16;     // fewer blocks at small T: each re-reads the router weights
constexpr int kSumLoads = 40;              // count-row loads in flight per thread
constexpr int kSegVec = 128;               // 16-byte vectors per copy item
constexpr int kSmemLimit = 200 * 1024;     // dynamic shared memory of a launch at most

// Two rings of stages, each with its own producer thread: x boxes (the
// block's rows, 128 bytes each per k-block, from HBM; as many stages as
// fit, up to kMaxXStages) and router-weight boxes (from L2; 8 stages, 4 at
// NP = 256).  The MMA reads a 128-row A tile from an x stage; rows past the
// box are whatever follows it in the ring (their accumulator rows are never
// read).  The MMA thread, not the loads, bounds the step: a tcgen05.mma of
// M = 128, K = 16 took about the same time for N = 64 and N = 128, so the
// rings only need to stay ahead of it.
constexpr int kMaxXStages = 16;
template <int NP>
struct RdtCfg {
  static constexpr int NACC = static_cast<int>(kTmemCols) / NP;
  static constexpr int W_BYTES = NP * BK * 2;
  static constexpr int WS = NP >= 256 ? 4 : 8;
  static constexpr int W_RING = WS * W_BYTES;
  static constexpr int X_RING = 176 * 1024 - W_RING;
  static constexpr int RING = X_RING + W_RING;   // x ring first: an A tile read past it stays inside
  static constexpr int LS = NP + 1;              // logits row stride in floats (conflict-free row writes)
  static constexpr int LOGIT_BYTES = BM * LS * 4;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int FIXED = 1024 + RING + BAR_BYTES;  // alignment slack, rings / logits, barriers
  static_assert(RING >= LOGIT_BYTES, "the logits fit over the rings");
  static_assert(X_RING >= 3 * A_BYTES, "x stages");
  static_assert((2 * kMaxXStages + 2 * 8 + 1) * 8 + 4 <= BAR_BYTES, "barrier space");
};

template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32)
    tmem_load32(taddr, r);
  else
    tmem_load16(taddr, r);
}

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

// NP: the expert count padded to a power of two (32..256), the MMA's N.
// Dynamic shared memory: the x and weight rings (later the logits of a
// pass, [128][NP + 1] fp32), the barriers, then the block's ids and their
// in-block ranks (then padded rows), [own_max][k] int32 each.
template <int NP>
__global__ void __launch_bounds__(kThreads, 1)
    route_dispatch_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                             const RouterArgs r, const DispatchArgs a, const int32_t own_max,
                             const int32_t box_rows) {
  using C = RdtCfg<NP>;
  constexpr int WS = C::WS, NACC = C::NACC, LS = C::LS;
  constexpr int PER = NP / 32;
  constexpr int CW = NP >= 128 ? 32 : 16;  // TMEM columns per load
  constexpr int GN = PER >= 8 ? 2 : PER >= 4 ? 4 : 8;  // tokens a warp gates at once
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, NP);
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  extern __shared__ uint8_t rdt_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rdt_raw) + 1023) & ~uintptr_t(1023));
  float* ls = reinterpret_cast<float*>(ring);                        // [BM][LS], after a pass's MMAs
  uint8_t* wring = ring + C::X_RING;
  uint64_t* xfull = reinterpret_cast<uint64_t*>(ring + C::RING);
  uint64_t* xempty = xfull + kMaxXStages;
  uint64_t* wfull = xempty + kMaxXStages;
  uint64_t* wempty = wfull + 8;
  uint64_t* tfull = wempty + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* s_ids = reinterpret_cast<int*>(ring + C::RING + C::BAR_BYTES);  // [own_max][k]
  int* s_row = s_ids + own_max * r.k;                                   // [own_max][k]
  __shared__ int s_cnt[kMaxExperts], s_base[kMaxExperts], s_off[kMaxExperts], s_moff[kMaxExperts];
  __shared__ int s_wcnt[kWarps][kMaxExperts];
  __shared__ int s_pb[kThreads], s_pt[kThreads];
  __shared__ int s_ok, s_fail;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const int T = r.T, E = r.E, k = r.k, d = r.d;
  const int64_t M = static_cast<int64_t>(T) * k;
  const int t_lo = static_cast<int>(static_cast<int64_t>(b) * T / G);
  const int t_hi = static_cast<int>(static_cast<int64_t>(b + 1) * T / G);
  const int own = t_hi - t_lo;
  const int kblocks = d / BK;
  const int x_bytes = box_rows * BK * 2;                               // a multiple of 1024
  const int XS = min(kMaxXStages, C::X_RING / x_bytes);

  for (int i = threadIdx.x; i < own * k; i += kThreads) s_ids[i] = -1;
  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < XS; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < WS; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 1);
    }
    mbar_init(tfull, 1);
    fence_barrier_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (own > 0 && warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = own > 0 ? *tmem_slot : 0u;
  grid_dep_launch();  // after the allocation: a dependent kernel's CTAs never hold this SM's TMEM first

  // 1. logits and gate, up to 128 tokens per pass; the ring positions run
  // on across passes (slot and phase kept incrementally)
  int xn = 0;                            // x producer: boxes loaded
  int wn = 0;                            // weight producer: boxes loaded
  int ms = 0, mw = 0;                    // MMA thread: x and weight slots
  uint32_t mxph = 0, mwph = 0;
  for (int p0 = t_lo, pass = 0; p0 < t_hi; p0 += BM, ++pass) {
    const int rows = min(BM, t_hi - p0);
    if (warp == 0 && lane == 0) {
      // x producer: slot n % XS is free once the MMA of k-block n - XS is done
      for (int kb = 0; kb < kblocks; ++kb, ++xn) {
        const int slot = xn % XS;
        if (xn >= XS && !mbar_wait(&xempty[slot], static_cast<uint32_t>(((xn / XS) - 1) & 1), a.wait_limit_ns)) {
          set_error(a.err, kErrTimeout);
          s_fail = 1;
          break;
        }
        mbar_arrive_expect_tx(&xfull[slot], static_cast<uint32_t>(x_bytes));
        tma_load_2d(ring + slot * x_bytes, &tm_x, &xfull[slot], kb * BK, p0);
      }
    } else if (warp == 2 && lane == 0) {
      // weight producer: slot n % WS is free once the MMA of k-block n - WS is done
      for (int kb = 0; kb < kblocks; ++kb, ++wn) {
        const int slot = wn % WS;
        if (wn >= WS && !mbar_wait(&wempty[slot], static_cast<uint32_t>(((wn / WS) - 1) & 1), a.wait_limit_ns)) {
          set_error(a.err, kErrTimeout);
          s_fail = 1;
          break;
        }
        mbar_arrive_expect_tx(&wfull[slot], static_cast<uint32_t>(C::W_BYTES));
        tma_load_2d(wring + slot * C::W_BYTES, &tm_w, &wfull[slot], kb * BK, 0);
      }
    } else if (warp == 1 && lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait(&xfull[ms], mxph, a.wait_limit_ns) || !mbar_wait(&wfull[mw], mwph, a.wait_limit_ns)) {
          set_error(a.err, kErrTimeout);
          s_fail = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sw128_desc(smem_u32(ring + ms * x_bytes));
        const uint64_t bdesc = sw128_desc(smem_u32(wring + mw * C::W_BYTES));
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // consecutive K steps go to different accumulators, so that no MMA
          // waits for the one before it
          const int g = kb * (BK / 16) + kk;
          tc_mma_f16(tmem_base + static_cast<uint32_t>((g % NACC) * NP), adesc + 2 * kk, bdesc + 2 * kk, IDESC,
                     g >= NACC ? 1u : 0u);
        }
        tc_commit(&xempty[ms]);
        tc_commit(&wempty[mw]);
        if (++ms == XS) {
          ms = 0;
          mxph ^= 1u;
        }
        if (++mw == WS) {
          mw = 0;
          mwph ^= 1u;
        }
      }
      if (ok) tc_commit(tfull);
    }
    if (threadIdx.x == 0) {
      s_ok = mbar_wait(tfull, static_cast<uint32_t>(pass & 1), a.wait_limit_ns) ? 1 : 0;
      if (!s_ok) {
        set_error(a.err, kErrTimeout);
        s_fail = 1;
      }
    }
    __syncthreads();
    if (!s_ok) break;  // the same for every thread
    tc_fence_after();
    {
      // warp w reads TMEM lanes 32 (w % 4).. (tokens) and the column chunks
      // w / 4, w / 4 + 4, ...; sums the accumulators in a fixed order
      const int q = warp & 3, cg = warp >> 2;
      const int row = q * 32 + lane;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int nacc = kblocks * (BK / 16) < NACC ? kblocks * (BK / 16) : NACC;
      for (int c0 = cg * CW; c0 < NP; c0 += 4 * CW) {
        float sum[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) sum[j] = 0.f;
        for (int acc = 0; acc < nacc; ++acc) {
          uint32_t v[CW];
          tmem_load_cols<CW>(tb + static_cast<uint32_t>(acc * NP + c0), v);
#pragma unroll
          for (int j = 0; j < CW; ++j) sum[j] += __uint_as_float(v[j]);
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) {
          const int e = c0 + j;
          float l = sum[j];
          if (r.bias != nullptr && e < E) l += __ldg(r.bias + e);
          ls[row * LS + e] = l;
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (r.logits != nullptr) {
      for (int i = threadIdx.x; i < rows * E; i += kThreads) {
        const int rr = i / E, e = i % E;
        r.logits[static_cast<int64_t>(p0 + rr) * E + e] = ls[rr * LS + e];
      }
    }
    for (int i0 = warp * GN; i0 < rows; i0 += kWarps * GN) {
      int id[GN];
      float wt[GN];
      warp_gate_rows<PER, GN>(ls + i0 * LS, LS, rows - i0, E, k, r.raw_weights, id, wt);
#pragma unroll
      for (int n = 0; n < GN; ++n) {
        if (i0 + n < rows && lane < k) {
          const int64_t t = p0 + i0 + n;
          r.ids[t * k + lane] = id[n];
          r.w[t * k + lane] = wt[n];
          s_ids[(p0 - t_lo + i0 + n) * k + lane] = id[n];
        }
      }
    }
    fence_proxy_async_smem();  // the logits' generic writes before the next pass's TMA writes
    __syncthreads();           // the ring is loaded again by the next pass
  }
  __syncthreads();
  if (s_fail && (warp == 0 || warp == 2) && lane == 0) {
    // after a timeout: every box loaded lands before the rings are left
    // (on the normal path the MMAs have consumed them all)
    const bool is_x = warp == 0;
    const int ns = is_x ? XS : WS;
    const int n = is_x ? xn : wn;
    for (int i = (n > ns ? n - ns : 0); i < n; ++i)
      if (!mbar_wait(is_x ? &xfull[i % ns] : &wfull[i % ns], static_cast<uint32_t>((i / ns) & 1), a.wait_limit_ns))
        set_error(a.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (own > 0 && warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }

  // 2. ranks in the block, in flat (token, slot) order: 512 pairs per round,
  // match-any groups inside each warp, then an exclusive scan over the
  // warps per expert on top of the earlier rounds' counts; the block's counts
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (threadIdx.x < E) s_cnt[threadIdx.x] = 0;
  const int npairs = own * k;
  for (int base = 0; base < npairs; base += kThreads) {
    const int p = base + threadIdx.x;
    int e = p < npairs ? s_ids[p] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t m = __match_any_sync(0xffffffffu, e);
    for (int x = lane; x < E; x += 32) s_wcnt[warp][x] = 0;
    __syncwarp();
    if (e >= 0 && (__ffs(m) - 1) == lane) s_wcnt[warp][e] = __popc(m);
    __syncthreads();
    if (threadIdx.x < E) {
      int run = s_cnt[threadIdx.x];
      for (int w = 0; w < kWarps; ++w) {
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

  // 3. grid barrier (every block's count and rank stores are visible after it)
  if (!grid_barrier_wait(a.bar, static_cast<unsigned>(G + a.test_stall), a.wait_limit_ns, a.err, &s_ok)) {
    if (threadIdx.x == 0) grid_barrier_depart(a.bar, static_cast<unsigned>(G));
    return;
  }
  if (threadIdx.x == kThreads - 32) grid_barrier_depart(a.bar, static_cast<unsigned>(G));

  // 4. per expert e: this block's base (the counts of blocks before it) and
  // the total, by P threads per expert over the rows h, h + P, ...
  {
    const int P = kThreads / E;
    if (threadIdx.x < P * E) {
      const int e = threadIdx.x % E, h = threadIdx.x / E;
      int below = 0, total = 0;
      for (int r0 = h; r0 < G; r0 += kSumLoads * P) {
        int v[kSumLoads];
#pragma unroll
        for (int u = 0; u < kSumLoads; ++u) {
          const int rr = r0 + u * P;
          v[u] = rr < G ? __ldcg(a.chunk + static_cast<int64_t>(rr) * E + e) : 0;
        }
#pragma unroll
        for (int u = 0; u < kSumLoads; ++u) {
          total += v[u];
          if (r0 + u * P < b) below += v[u];
        }
      }
      s_pb[threadIdx.x] = below;
      s_pt[threadIdx.x] = total;
    }
    __syncthreads();
    if (threadIdx.x < E) {
      int below = 0, total = 0;
      for (int h = 0; h < P; ++h) {
        below += s_pb[h * E + threadIdx.x];
        total += s_pt[h * E + threadIdx.x];
      }
      s_base[threadIdx.x] = below;
      s_cnt[threadIdx.x] = total;
    }
    __syncthreads();
  }
  // expert offsets and tile maps, 32 experts a round with carries; block 0
  // publishes them
  if (warp == 0) {
    int c_off = 0, c_m = 0, c_p = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int total = e < E ? s_cnt[e] : 0;
      const int mt = (total + kTileM - 1) / kTileM;
      const int pt = (mt + 1) / 2;
      const int off = c_off + warp_exclusive_scan(total);
      const int moff = c_m + warp_exclusive_scan(mt);
      const int poff = c_p + warp_exclusive_scan(pt);
      if (e < E) {
        s_off[e] = off;
        s_moff[e] = moff;
        if (b == 0) {
          a.counts[e] = total;
          a.offsets[e] = off;
          a.mtile_off[e] = moff;
          for (int i = moff; i < moff + mt && i < a.max_mtiles; ++i) a.mtile_expert[i] = e;
          if (a.ptile_off != nullptr) {
            a.ptile_off[e] = poff;
            for (int i = poff; i < poff + pt && i < a.max_mtiles; ++i) a.ptile_expert[i] = e;
          }
        }
      }
      c_off = __shfl_sync(0xffffffffu, off + total, 31);
      c_m = __shfl_sync(0xffffffffu, moff + mt, 31);
      c_p = __shfl_sync(0xffffffffu, poff + pt, 31);
    }
    if (b == 0 && lane == 0) {
      a.offsets[E] = c_off;
      a.mtile_off[E] = c_m;
      if (a.ptile_off != nullptr) a.ptile_off[E] = c_p;
      if (c_m > a.max_mtiles) set_error(a.err, kErrDevice);
    }
  }
  __syncthreads();

  // 5. global ranks of the block's pairs -> tok, inv; each pair's padded row;
  // then the row copy
  const int64_t rows_cap = static_cast<int64_t>(a.max_mtiles) * kTileM;
  for (int i = threadIdx.x; i < npairs; i += kThreads) {
    const int t = t_lo + i / k;
    const int e = s_ids[i];
    int row = -1;
    if (e >= 0 && e < E) {
      const int rank = s_off[e] + s_base[e] + s_row[i];
      if (rank >= 0 && rank < M) {
        a.inv[static_cast<int64_t>(t) * k + i % k] = rank;
        a.tok[rank] = t;
        const int64_t rw = static_cast<int64_t>(s_moff[e]) * kTileM + (rank - s_off[e]);
        if (rw >= 0 && rw < rows_cap) row = static_cast<int>(rw);
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
  for (int it = warp; it < n_items; it += 2 * kWarps) {
    uint4 buf[2][kSegVec / 32];
    int tl[2] = {-1, -1};
    int v_base[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int item = it + h * kWarps;
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

template <int NP>
size_t smem_bytes(int own_max, int k) {
  return static_cast<size_t>(RdtCfg<NP>::FIXED) + 8ull * own_max * k;
}

size_t smem_for(int np, int own_max, int k) {
  switch (np) {
    case 32: return smem_bytes<32>(own_max, k);
    case 64: return smem_bytes<64>(own_max, k);
    case 128: return smem_bytes<128>(own_max, k);
    default: return smem_bytes<256>(own_max, k);
  }
}

template <int NP>
cudaError_t launch_np(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& r, const DispatchArgs& a,
                      int grid, int own_max, int box_rows, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes<NP>(own_max, r.k);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_dispatch_tc_kernel<NP>, tm_x, tm_w, r, a, static_cast<int32_t>(own_max),
                            static_cast<int32_t>(box_rows));
}

int padded_experts(int E) {
  int np = 32;
  while (np < E) np *= 2;
  return np;
}

}  // namespace

int route_dispatch_tc_grid(int T, int num_sms) {
  if (T <= 0) return 0;
  const int by_tokens = (T + kMinTokensPerBlock - 1) / kMinTokensPerBlock;
  return std::min(std::min(num_sms, kMaxGrid), by_tokens);
}

int route_dispatch_tc_box_rows(int T, int grid) {
  const int own_max = route_dispatch_own_max(T, grid);
  const int rows = (own_max + 7) / 8 * 8;
  return rows < 8 ? 8 : rows > BM ? BM : rows;
}

bool route_dispatch_tc_supported(int T, int d, int E, int k, int num_sms) {
  if (E <= 16 || E > kMaxExperts || k < 1 || k > E || k > 32 || d % BK != 0 || d < BK || T < 1) return false;
  const int grid = route_dispatch_tc_grid(T, num_sms);
  if (static_cast<int64_t>(grid) * E > kFusedScanWords) return false;  // the count rows in chunk
  const int own_max = route_dispatch_own_max(T, grid);
  const int np = padded_experts(E);
  const size_t smem = smem_for(np, own_max, k);
  if (smem > kSmemLimit) return false;
  int per_sm = 0;
  cudaError_t e;
  switch (np) {
    case 32: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_tc_kernel<32>, kThreads, smem); break;
    case 64: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_tc_kernel<64>, kThreads, smem); break;
    case 128: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_tc_kernel<128>, kThreads, smem); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_dispatch_tc_kernel<256>, kThreads, smem);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return per_sm >= 1;
}

cudaError_t route_dispatch_tc_prepare() {
  cudaError_t e = cudaFuncSetAttribute(route_dispatch_tc_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_dispatch_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_dispatch_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_dispatch_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  return e;
}

cudaError_t launch_route_dispatch_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& r,
                                     const DispatchArgs& a, int grid, int box_rows, cudaStream_t s) {
  if (grid <= 0 || r.T <= 0) return cudaSuccess;
  if (r.E <= 16 || r.E > kMaxExperts || r.d % BK != 0 || a.bar == nullptr || box_rows < 1 || box_rows > BM)
    return cudaErrorInvalidValue;
  const int own_max = route_dispatch_own_max(r.T, grid);
  if (own_max > BM ? box_rows != BM : box_rows < own_max) return cudaErrorInvalidValue;
  switch (padded_experts(r.E)) {
    case 32: return launch_np<32>(tm_x, tm_w, r, a, grid, own_max, box_rows, s);
    case 64: return launch_np<64>(tm_x, tm_w, r, a, grid, own_max, box_rows, s);
    case 128: return launch_np<128>(tm_x, tm_w, r, a, grid, own_max, box_rows, s);
    default: return launch_np<256>(tm_x, tm_w, r, a, grid, own_max, box_rows, s);
  }
}

}  // namespace cbmoe
