// Grouped expert GEMMs (bf16) on CTA pairs with the 2-SM tensor-core MMA.
//
// Same math and epilogues as grouped_gemm.cu (gate/up with SwiGLU into bf16
// H, down into fp32 Y with bulk tensor stores), run by clusters of two CTAs
// on two SMs.  The down kernel can instead fuse the combine: each row's
// output, times its gate weight, is added into its token's fp32 row by
// vector reductions (the order of a token's k additions then varies from run
// to run, which changes no result for k <= 2: 0 + a + b = 0 + b + a).  The pair computes the two m-tiles (2p, 2p+1) of one expert
// against one 256-row weight tile with tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16), issued by one thread of the even CTA:
//
//   CTA r stages the A rows of m-tile 2p+r (128 x 64 per k-block) and
//   weight rows [128 r, 128 r + 128) of the tile (128 x 64); the two tensor
//   cores read each other's weight half, so each SM stages 32 KB per k-block
//   instead of 48 KB and the same shared memory holds a 6-deep ring;
//   each CTA's tensor memory receives its own 128 rows x 256 fp32 columns.
//
// Barriers: the TMA loads of both CTAs signal the even CTA's `full` barrier
// (whose producer expects both CTAs' bytes); the MMA thread's commits arrive
// on `empty` (stage free) and `tfull` (accumulator ready) in both CTAs; the
// epilogue warps of both CTAs arrive on the even CTA's `tempty`.
//
// A pair whose second m-tile does not exist (the last pair of an expert with
// an odd number of m-tiles) runs the M = 128 form of the 2-SM MMA instead:
// CTA r stages rows [64 r, 64 r + 64) of the single m-tile, and the MMA takes
// half the time.  Its accumulator (measured on GB300) holds, in each CTA,
// the CTA's 64 rows in TMEM lanes 0..63 against weight rows 0..127 and again
// in lanes 64..127 against weight rows 128..255, both in columns 0..127.  So
// in the down epilogue each warp stores its own 128-column half of Y, and in
// the gate/up epilogue (gate in lanes 0..63, up in lanes 64..127) the up
// warps hand their values to the gate warps through shared memory.
//
// Roles per CTA: warp 0 TMA producer, warp 1 TMEM allocation for the pair
// (and, in the even CTA, the MMA issuer), warps 2..5 epilogue.  All waits
// are bounded.  Cluster barriers after set-up (every barrier of the pair
// exists before any remote signal) and before the TMEM release (no remote
// arrive or tensor-memory read is still outstanding).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "swiglu.cuh"

namespace cbmoe {
namespace {

constexpr int BM = kTileM;  // rows per CTA
constexpr int BK = 64;
constexpr int BN = 256;
constexpr int HALF_ROWS = BN / 2;
constexpr int A_BYTES = BM * BK * 2;
constexpr int BH_BYTES = HALF_ROWS * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + BH_BYTES;  // per CTA
constexpr int THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN);
constexpr uint32_t IDESC_HALF = idesc_bf16_f32(BM, BN);  // M = 128: 64 rows per CTA
constexpr uint32_t EPI_BAR = 1;                          // named barrier of the epilogue warps
constexpr uint16_t PAIR_MASK = 0x3;
constexpr int STG_BYTES = EPI_WARPS * 2 * 32 * 128;

// Ring of A stages then weight-half stages; behind the ring the down
// kernel's store staging, or for gate/up an unused tile, so that an operand
// read of a full 256-row tile at the last stage would still fall inside the
// CTA's shared memory.
template <int KIND>
struct Cfg {
  static constexpr int STAGES = 6;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int STAGING = KIND == kDownF32 ? STG_BYTES : BH_BYTES;
  static constexpr int BYTES = RING + STAGING + 1024 + 256;
};
static_assert(Cfg<kGateUpSwiGLU>::BYTES <= 232448 && Cfg<kDownF32>::BYTES <= 232448, "shared memory per CTA");

struct PairTile {
  int m_tile;  // this CTA's m-tile (for a half pair, the pair's single m-tile)
  bool valid;
  bool half;   // the pair has one m-tile: M = 128, 64 of its rows per CTA
  int e;
  int n;
};

// Tile index -> (expert, N tile, pair); consecutive clusters take the pairs
// of one expert against the same weight tile.
__device__ __forceinline__ PairTile decode_pair_tile(int tile, const GemmArgs& p, int rank) {
  const int e = p.ptile_expert[tile / p.n_tiles];
  const int base = p.ptile_off[e];
  const int np = p.ptile_off[e + 1] - base;
  const int local = tile - base * p.n_tiles;
  const int pair = local % np;
  PairTile t;
  t.e = e;
  t.n = local / np;
  const int mt_e = p.mtile_off[e + 1] - p.mtile_off[e];
  const int idx = 2 * pair + rank;
  t.half = 2 * pair + 1 == mt_e;
  t.valid = t.half || idx < mt_e;
  t.m_tile = p.mtile_off[e] + (idx < mt_e ? idx : 2 * pair);
  return t;
}

template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_bh,
                             const __grid_constant__ CUtensorMap tm_out, const GemmArgs p) {
  using C = Cfg<KIND>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  uint8_t* staging = smem + C::RING;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING + C::STAGING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool even = rank == 0;
  const int cluster = blockIdx.x / 2, n_clusters = gridDim.x / 2;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);  // used in the even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * EPI_WARPS);  // used in the even CTA
    }
    fence_barrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_bh);
    if (KIND == kDownF32) prefetch_tensormap(&tm_out);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  const int total_tiles = p.ptile_off[p.E] * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t full_even = mapa_shared(smem_u32(full), 0);
      int64_t issued = 0;
      bool ok = true;
      for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters) {
        const PairTile t = decode_pair_tile(tile, p, rank);
        const int a_row = t.m_tile * BM + (t.half ? rank * (BM / 2) : 0);
        const int b_row = t.e * p.b_rows_per_expert + t.n * BN + rank * HALF_ROWS;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const int stage = static_cast<int>(issued % STAGES);
          const uint32_t phase = static_cast<uint32_t>((issued / STAGES) & 1);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          if (even) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          const uint32_t bar = full_even + static_cast<uint32_t>(stage * 8);
          tma_load_2d_pair(sa + stage * A_BYTES, &tm_a, bar, kb * BK, a_row);
          tma_load_2d_pair(sb + stage * BH_BYTES, &tm_bh, bar, kb * BK, b_row);
          ++issued;
        }
      }
      // The even CTA's full barriers count both CTAs' bytes, so waiting on
      // its last phases covers the odd CTA's loads in flight too.
      if (even)
        for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
          if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            break;
          }
    }
  } else if (warp == 1) {
    if (even && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster; ok && tile < total_tiles; tile += n_clusters) {
        const uint32_t idesc = decode_pair_tile(tile, p, 0).half ? IDESC_HALF : IDESC;
        if (!mbar_wait_cluster(&tempty[acc], p.test_stall ? acc_phase : acc_phase ^ 1u, p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_desc(smem_u32(sa + stage * A_BYTES));
          const uint64_t bdesc = sw128_desc(smem_u32(sb + stage * BH_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_f16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          tc_commit_pair_multicast(&empty[stage], PAIR_MASK);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(&tfull[acc], PAIR_MASK);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else {
    const int q = warp & 3;
    const uint32_t tempty_even = mapa_shared(smem_u32(tempty), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int n_stores = 0;
    for (int tile = cluster; tile < total_tiles; tile += n_clusters) {
      const PairTile t = decode_pair_tile(tile, p, rank);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_limit_ns)) {
        set_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (t.valid && KIND == kGateUpSwiGLU && t.half) {
        // half pair: gate in lanes 0..63, up of the same rows in lanes 64..127
        // (columns 0..127 both).  Warp q < 2 (gate) computes features 0..63
        // of rows 32q.., warp q + 2 (up) features 64..127 of the same rows;
        // per round j each hands the partner the 32-column chunk it needs
        // through a shared-memory slot (rows of 128 B, 16-byte chunks
        // swizzled by the row)
        const bool gate_warp = q < 2;
        uint8_t* mine = staging + ((q & 1) * 2 + (gate_warp ? 0 : 1)) * 4096;    // written by this warp
        uint8_t* theirs = staging + ((q & 1) * 2 + (gate_warp ? 1 : 0)) * 4096;  // written by the partner
        const int64_t row = static_cast<int64_t>(t.m_tile) * BM + rank * (BM / 2) + (q & 1) * 32 + lane;
        uint16_t* out_row = static_cast<uint16_t*>(p.out) + row * p.ld_out + t.n * (BN / 2);
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
          const int give = (gate_warp ? 2 + j : j) * 32;  // chunk the partner computes with
          const int keep = (gate_warp ? j : 2 + j) * 32;  // chunk this warp computes
          uint32_t v[32];
          tmem_load32(tbase + give, v);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(mine + lane * 128 + 16 * (c ^ (lane & 7))) =
                make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          tmem_load32(tbase + keep, v);
          named_bar_sync(EPI_BAR, EPI_WARPS * 32);
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(theirs + lane * 128 + 16 * (c ^ (lane & 7)));
            w[4 * c] = x.x;
            w[4 * c + 1] = x.y;
            w[4 * c + 2] = x.z;
            w[4 * c + 3] = x.w;
          }
          named_bar_sync(EPI_BAR, EPI_WARPS * 32);
          // gate warp: v = gate, w = up; up warp: v = up, w = gate
          uint32_t h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(gate_warp ? v[2 * i] : w[2 * i]);
            const float u0 = __uint_as_float(gate_warp ? w[2 * i] : v[2 * i]);
            const float g1 = __uint_as_float(gate_warp ? v[2 * i + 1] : w[2 * i + 1]);
            const float u1 = __uint_as_float(gate_warp ? w[2 * i + 1] : v[2 * i + 1]);
            h[i] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
          }
          uint4* dst = reinterpret_cast<uint4*>(out_row + keep);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        }
      } else if (t.valid) {
        // this lane's row within the m-tile, and the accumulator columns it
        // holds: all 256 for a full pair; for a half pair 128 of them, the
        // weight rows [128 (q / 2), +128) of the tile in columns 0..127
        const int row_in = t.half ? rank * (BM / 2) + (q & 1) * 32 : q * 32;
        const int ncols = t.half ? BN / 2 : BN;
        const int col0 = t.half ? (q >> 1) * (BN / 2) : 0;
        if constexpr (KIND == kGateUpSwiGLU) {
          const int64_t row = static_cast<int64_t>(t.m_tile) * BM + q * 32 + lane;
          uint16_t* out_row = static_cast<uint16_t*>(p.out) + row * p.ld_out + t.n * (BN / 2);
#pragma unroll 1
          for (int c0 = 0; c0 < BN / 2; c0 += 32) {
            uint32_t g[32], u[32];
            tmem_load32(tbase + c0, g);
            tmem_load32(tbase + BN / 2 + c0, u);
            uint32_t h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float h0 = silu(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
              const float h1 = silu(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
              h[j] = pack_bf16x2(h0, h1);
            }
            uint4* dst = reinterpret_cast<uint4*>(out_row + c0);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
          }
        } else if (p.comb_acc != nullptr) {
          // combine fused: the lane's row adds its gate-weighted output into
          // its token's accumulator row (fp32 reductions performed in L2);
          // padding rows past the expert's count add nothing
          const int local = (t.m_tile - p.mtile_off[t.e]) * BM + row_in + lane;
          const bool live = local < p.counts[t.e];
          float wt = 0.f;
          float* dst = p.comb_acc;
          if (live) {
            const int tk = p.tok[p.offsets[t.e] + local];
            const int64_t pr = static_cast<int64_t>(tk) * p.top_k;
            int sl = 0;
            while (sl + 1 < p.top_k && p.comb_ids[pr + sl] != t.e) ++sl;
            wt = p.comb_w[pr + sl];
            dst += static_cast<int64_t>(tk) * p.ld_out + t.n * BN + col0;
          }
#pragma unroll 1
          for (int c0 = 0; c0 < ncols; c0 += 32) {
            uint32_t r[32];
            tmem_load32(tbase + c0, r);
            if (live) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                red_add_f32x4(dst + c0 + 4 * j, wt * __uint_as_float(r[4 * j]), wt * __uint_as_float(r[4 * j + 1]),
                              wt * __uint_as_float(r[4 * j + 2]), wt * __uint_as_float(r[4 * j + 3]));
            }
          }
        } else {
          const int row0 = t.m_tile * BM + row_in;
#pragma unroll 1
          for (int c0 = 0; c0 < ncols; c0 += 32, ++n_stores) {
            uint32_t r[32];
            tmem_load32(tbase + c0, r);
            uint8_t* buf = staging + (q * 2 + (n_stores & 1)) * 4096;
            if (n_stores >= 2) {
              if (lane == 0) bulk_wait_group_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(buf + lane * 128 + 16 * (j ^ (lane & 7))) =
                  make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, buf, t.n * BN + col0 + c0, row0);
              bulk_commit_group();
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_even + static_cast<uint32_t>(acc * 8));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (KIND == kDownF32 && lane == 0) bulk_wait_group<0>();
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

template <int KIND>
cudaLaunchConfig_t pair_config(int grid, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<KIND>::BYTES;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap& tm_a, const CUtensorMap& tm_bh, const CUtensorMap& tm_out,
                        const GemmArgs& a, cudaStream_t s) {
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = pair_config<KIND>(a.grid, attr);
  cfg.stream = s;
  if (PdlScope::next()) {  // see launch_kernel
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<KIND>, tm_a, tm_bh, tm_out, a);
}

template <int KIND>
int max_pairs(int num_sms) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<KIND>(2 * (num_sms / 2), attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<KIND>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

cudaError_t grouped_gemm_pair_prepare(int num_sms, int* grid_gateup, int* grid_down) {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<kGateUpSwiGLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<kGateUpSwiGLU>::BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<kDownF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<kDownF32>::BYTES);
  if (e != cudaSuccess) return e;
  *grid_gateup = 2 * max_pairs<kGateUpSwiGLU>(num_sms);
  *grid_down = 2 * max_pairs<kDownF32>(num_sms);
  return cudaSuccess;
}

cudaError_t launch_grouped_gemm_pair(GemmKind kind, const CUtensorMap& tm_a, const CUtensorMap& tm_bh,
                                     const CUtensorMap& tm_out, const GemmArgs& a, cudaStream_t s) {
  if (a.grid < 2 || (a.grid & 1)) return cudaErrorInvalidConfiguration;
  if (kind == kGateUpSwiGLU) return launch_kind<kGateUpSwiGLU>(tm_a, tm_bh, tm_out, a, s);
  return launch_kind<kDownF32>(tm_a, tm_bh, tm_out, a, s);
}

}  // namespace cbmoe
