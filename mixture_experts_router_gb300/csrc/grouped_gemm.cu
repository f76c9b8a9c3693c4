// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// The expert matmuls of the MoE layer (the expert GEMM kernel of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §2.3, fused with the activation as in
// "discosf.com/news/4774337" §3.2, which hand-wrote its MMA in PTX for the same
// reason) run as one persistent kernel per projection over all experts:
//
//   gate/up : H[r, n*128 + j] = bf16( SiLU(acc[j]) * acc[128 + j] ),
//             acc = Xp[r] . Wgu[e][n]^T, where the repacked weight block n of
//             expert e holds gate rows n*128..n*128+127 followed by the same
//             up rows, so one 128x256 accumulator carries matching gate and
//             up columns (SwiGLU, w1 gate, w3 up:
//             "Colibri：面向MoE模型的高性能C语言推理引擎" §4.2)
//   down    : Y[r, n*256 + c] = acc[c], acc = H[r] . Wd[e][n]^T (fp32 out)
//
// Rows are the expert-grouped activations; every expert's block starts on a
// 128-row boundary, so an M-tile belongs to exactly one expert, and the tile
// list (expert-major, then N, then M) is derived on the device from the
// dispatch's tile prefix sums: the host never learns the expert counts.
//
// Per CTA (one per SM, persistent, static round-robin over tiles):
//   warp 0      : TMA producer (one thread): A 128x64 and B 256x64 bf16 boxes,
//                 128-byte swizzle, into a 4-stage ring guarded by mbarriers
//   warp 1      : owns the 512 TMEM columns; one thread issues
//                 tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16) x4
//                 per stage and commits stage release / accumulator ready
//   warps 2..5  : epilogue: tcgen05.ld 32 lanes x 32 columns, SwiGLU or fp32,
//                 16-byte global stores; two accumulators alternate so the
//                 epilogue of tile i overlaps the mainloop of tile i+1
// Every wait is bounded; a wait that runs out records CB_ERR_TIMEOUT in the
// status word and the CTA winds down (waiting for its own loads in flight
// and freeing its TMEM).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "swiglu.cuh"

namespace cbmoe {
namespace {

constexpr int BM = kTileM;               // 128 rows per tile
constexpr int BK = 64;                   // 64 bf16 = one 128-byte swizzled row
constexpr int BN = 256;                  // accumulator columns per tile
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int A32_ROWS = 32;              // rows of the short A box (tiles of few routed rows)
constexpr int A32_BYTES = A32_ROWS * BK * 2;
constexpr int B_BYTES = BN * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 2 * BN;   // two fp32 accumulators of 256 columns
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr int STG_BYTES = 4 * 2 * 32 * 128;  // down epilogue: 4 warps x 2 buffers x 32 rows x 128 B
template <int KIND>
struct Smem {
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int STAGING = KIND == kDownF32 ? STG_BYTES : 0;
  static constexpr int BYTES = RING + STAGING + 1024 + 256;
};

struct TileCoord {
  int m_tile;  // global 128-row tile index in the grouped rows
  int e;       // expert
  int n;       // N tile within the expert
};

__device__ __forceinline__ TileCoord decode_tile(int tile, const GemmArgs& p) {
  const int e = p.mtile_expert[tile / p.n_tiles];
  const int base = p.mtile_off[e];
  const int mt = p.mtile_off[e + 1] - base;
  const int local = tile - base * p.n_tiles;
  TileCoord c;
  c.e = e;
  c.n = local / mt;
  c.m_tile = base + local % mt;
  return c;
}

// The down kernel splits the last, partial wave of tiles along N: with G
// CTAs and R = tiles mod G leftover tiles, each leftover tile becomes S
// sub-tiles of BN / S columns (S = the largest of 1, 2, 4 with R S <= G), so
// the tail takes 1/S of a tile's time.  Work unit u < F = tiles - R is tile
// u; unit F + i is part i % S of tile F + i / S.
struct Work {
  TileCoord c;
  int nsub;  // columns (and weight rows) of this unit
  int col0;  // first output column within the expert
};

__device__ __forceinline__ void tail_split(int total_tiles, int grid, int& full, int& split) {
  const int r = total_tiles % grid;
  full = total_tiles - r;
  split = 1;
  if (r > 0) {
    if (4 * r <= grid)
      split = 4;
    else if (2 * r <= grid)
      split = 2;
  }
}

__device__ __forceinline__ Work decode_work(int u, const GemmArgs& p, int full, int split) {
  Work w;
  int tile = u, part = 0;
  w.nsub = BN;
  if (u >= full) {
    tile = full + (u - full) / split;
    part = (u - full) % split;
    w.nsub = BN / split;
  }
  w.c = decode_tile(tile, p);
  w.col0 = w.c.n * BN + part * w.nsub;
  return w;
}

template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_b64,
                        const __grid_constant__ CUtensorMap tm_a32, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  uint8_t* staging = smem + Smem<KIND>::RING;  // down: per-warp store buffers
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem<KIND>::RING + Smem<KIND>::STAGING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    fence_barrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
    if (p.counts != nullptr) prefetch_tensormap(&tm_a32);
    if (KIND == kDownF32) {
      prefetch_tensormap(&tm_out);
      prefetch_tensormap(&tm_b64);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  const int total_tiles = p.mtile_off[p.E] * p.n_tiles;
  int full_tiles = total_tiles, split = 1;
  if (KIND == kDownF32) tail_split(total_tiles, gridDim.x, full_tiles, split);
  const int total_units = full_tiles + (total_tiles - full_tiles) * split;

  if (KIND == kGateUpSwiGLU && warp == 0 && p.gather) {
    // ---------------------------- TMA producer, A rows gathered from x
    // Each lane owns 4 of the m-tile's 128 rows: their tokens, then one
    // tile::gather4 of those 4 rows per k-block (512 bytes at lane*512).
    // Padding rows of an expert's last tile repeat its first token; their
    // outputs land in padding rows of H that nothing reads.
    int64_t issued = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const Work w = decode_work(u, p, full_tiles, split);
      const int e = w.c.e;
      const int row0 = p.offsets[e] + (w.c.m_tile - p.mtile_off[e]) * BM;
      const int row_end = p.offsets[e] + p.counts[e];
      const int first = p.tok[row0];
      int tk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = row0 + 4 * lane + j;
        tk[j] = r < row_end ? p.tok[r] : first;
      }
      const int b_row = e * p.b_rows_per_expert + w.col0;
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        const int stage = static_cast<int>(issued % STAGES);
        const uint32_t phase = static_cast<uint32_t>((issued / STAGES) & 1);
        int got = 1;
        if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          if (lane == 0) set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tma_load_2d(sb + stage * B_BYTES, &tm_b, &full[stage], kb * BK, b_row);
        }
        __syncwarp();
        tma_gather4(sa + stage * A_BYTES + lane * 4 * 128, &tm_a, &full[stage], kb * BK, tk[0], tk[1], tk[2], tk[3]);
        ++issued;
      }
    }
    if (lane == 0)
      for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Work w = decode_work(u, p, full_tiles, split);
        const int a_row = w.c.m_tile * BM;
        const int b_row = w.c.e * p.b_rows_per_expert + w.col0;
        // A tile holding at most 32 routed rows (decode sizes) loads only its
        // first 32 rows: the accumulator's other rows are padding that no one
        // reads, and the SM's load traffic is then almost all weights
        const bool a32 = p.counts != nullptr &&
                         p.counts[w.c.e] - (w.c.m_tile - p.mtile_off[w.c.e]) * BM <= A32_ROWS;
        const uint32_t a_bytes = a32 ? A32_BYTES : A_BYTES;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], a_bytes + w.nsub * BK * 2);
          tma_load_2d(sa + stage * A_BYTES, a32 ? &tm_a32 : &tm_a, &full[stage], kb * BK, a_row);
          if (w.nsub == BN) {
            tma_load_2d(sb + stage * B_BYTES, &tm_b, &full[stage], kb * BK, b_row);
          } else {
            for (int i = 0; i < w.nsub / 64; ++i)
              tma_load_2d(sb + stage * B_BYTES + i * 64 * BK * 2, &tm_b64, &full[stage], kb * BK, b_row + 64 * i);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No load of ours may still be landing in shared memory when the CTA
      // exits: wait for the last load issued into each stage.
      for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i) {
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const int nsub = (u < full_tiles) ? BN : BN / split;
        const uint32_t idesc = (nsub == BN) ? IDESC : idesc_bf16_f32(BM, nsub);
        // (test_stall waits on the phase in progress, which no thread completes)
        if (!mbar_wait(&tempty[acc], p.test_stall ? acc_phase : acc_phase ^ 1u, p.wait_limit_ns)) {
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
          const uint64_t bdesc = sw128_desc(smem_u32(sb + stage * B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp's quarter of the 128 TMEM lanes
    int acc = 0;
    uint32_t acc_phase = 0;
    int n_stores = 0;  // bulk stores issued by this warp (down only)
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
      const Work w = decode_work(u, p, full_tiles, split);
      const TileCoord c = w.c;
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_limit_ns)) {
        set_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(c.m_tile) * BM + q * 32 + lane;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (KIND == kGateUpSwiGLU) {
        uint16_t* out_row = static_cast<uint16_t*>(p.out) + row * p.ld_out + c.n * (BN / 2);
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
      } else {
        // TMA-store epilogue: this warp's 32 rows x 32 fp32 columns go through
        // a 128-byte-swizzled staging buffer (two per warp, alternating), then
        // one bulk tensor store writes whole 128-byte row segments.
        const int row0 = c.m_tile * BM + q * 32;
#pragma unroll 1
        for (int c0 = 0; c0 < w.nsub; c0 += 32, ++n_stores) {
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
            tma_store_2d(&tm_out, buf, w.col0 + c0, row0);
            bulk_commit_group();
          }
        }
        (void)row;
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (KIND == kDownF32 && lane == 0) bulk_wait_group<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

int grouped_gemm_tile_n(GemmKind kind) { return kind == kGateUpSwiGLU ? BN / 2 : BN; }

cudaError_t grouped_gemm_prepare() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<kGateUpSwiGLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<kGateUpSwiGLU>::BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<kDownF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Smem<kDownF32>::BYTES);
}

cudaError_t launch_grouped_gemm(GemmKind kind, bool int8_weights, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const CUtensorMap& tm_out, const CUtensorMap& tm_b64, const CUtensorMap& tm_a32,
                                const GemmArgs& a, cudaStream_t s) {
  if (int8_weights) return cudaErrorNotSupported;
  if (kind == kGateUpSwiGLU)
    launch_kernel(grouped_gemm_kernel<kGateUpSwiGLU>, a.grid, THREADS, Smem<kGateUpSwiGLU>::BYTES, s, tm_a, tm_b,
                  tm_out, tm_b64, tm_a32, a);
  else
    launch_kernel(grouped_gemm_kernel<kDownF32>, a.grid, THREADS, Smem<kDownF32>::BYTES, s, tm_a, tm_b, tm_out,
                  tm_b64, tm_a32, a);
  return cudaGetLastError();
}

}  // namespace cbmoe
