// Grouped expert GEMMs with int8 weights (symmetric per-output-channel int8,
// "lshu.cn/news/53496" §4.3), dequantised to bf16 inside the kernel and run on
// the tcgen05 tensor cores.  Same math as the bf16 kernel, with the scales
// applied to the fp32 accumulator in the epilogue:
//
//   gate/up : H[r, n*64 + j] = bf16( SiLU(s_g[e][n*64+j] acc[j]) *
//                                    s_u[e][n*64+j] acc[64 + j] ),
//             weight block n of expert e = gate rows n*64.. then up rows n*64..
//   down    : Y[r, n*128 + c] = s_d[e][n*128 + c] acc[c]      (fp32 out)
//
// The int8 -> bf16 conversion is done by warps of this kernel and costs
// instruction issue slots, so every converted weight tile is used twice:
// a tile is a PAIR of 128-row m-tiles of the same expert against one N=128
// weight tile (two tcgen05.mma M=128 N=128 per K step, two accumulators).
// An expert with an odd number of m-tiles gives its last pair a second
// m-tile that is computed on a repeat of the first and not stored.
//
// Per CTA (one per SM, persistent, round-robin over pair tiles):
//   warp 0      : TMA producer of the two A boxes (2 x 128x64 bf16) of a stage
//   warp 1      : TMEM owner (512 columns = 2 buffers x 2 m-tiles x 128) and
//                 MMA issuer
//   warps 2..5  : epilogue (tcgen05.ld, scales, SwiGLU or fp32, 16-B stores)
//   warps 6..13 : int8 -> bf16 transform of each staged weight tile into the
//                 stage's 128-byte-swizzled B buffer, then fence to the async
//                 proxy and arrive on the stage barrier
//   warp 14     : TMA producer of the int8 weight tiles (128x64) into a
//                 6-slot ring, running up to 6 k-blocks ahead
// The down kernel's epilogue stages each warp's 32x32 fp32 blocks in
// 128-byte-swizzled shared memory and writes them with bulk tensor stores.
// Every wait is bounded (CB_ERR_TIMEOUT in the status word on expiry).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "int8_bf16.cuh"
#include "swiglu.cuh"

namespace cbmoe {
namespace {

constexpr int BM = kTileM;            // rows per m-tile
constexpr int BK = 64;                // K per stage (one 128-byte bf16 row)
constexpr int BN = 128;               // weight rows per tile
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB per m-tile
constexpr int B_BYTES = BN * BK * 2;  // 16 KB bf16
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int I8_SLOTS = 6;
constexpr int I8_BYTES = BN * BK;     // 8 KB int8
constexpr int N_XFORM_WARPS = 8;
constexpr int XFORM_WARP0 = 6;
constexpr int BPROD_WARP = XFORM_WARP0 + N_XFORM_WARPS;
constexpr int THREADS = 32 * (BPROD_WARP + 1);
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr int RING_BYTES = STAGES * STAGE_BYTES + I8_SLOTS * I8_BYTES;
constexpr int STG_BYTES = 4 * 2 * 32 * 128;  // down epilogue: 4 warps x 2 buffers x 32 rows x 128 B
template <int KIND>
struct Smem {
  static constexpr int STAGING = KIND == kDownF32 ? STG_BYTES : 0;
  static constexpr int BYTES = RING_BYTES + STAGING + 1024 + 256;
};

struct PairCoord {
  int m0;      // first m-tile (global index)
  bool two;    // second m-tile m0 + 1 is real
  int e;       // expert
  int n;       // N tile within the expert
};

__device__ __forceinline__ PairCoord decode_pair(int tile, const GemmArgs& p) {
  const int e = p.ptile_expert[tile / p.n_tiles];
  const int base = p.ptile_off[e];
  const int np = p.ptile_off[e + 1] - base;
  const int local = tile - base * p.n_tiles;
  const int pair = local % np;
  PairCoord c;
  c.e = e;
  c.n = local / np;
  const int mt_e = p.mtile_off[e + 1] - p.mtile_off[e];
  c.m0 = p.mtile_off[e] + 2 * pair;
  c.two = 2 * pair + 1 < mt_e;
  return c;
}

template <int KIND>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_int8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                             const __grid_constant__ CUtensorMap tm_out, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // stage s: A0 at s*STAGE_BYTES, A1 at +A_BYTES, B at +2*A_BYTES (all 1024-aligned)
  uint8_t* s8 = smem + STAGES * STAGE_BYTES;
  uint8_t* staging = smem + RING_BYTES;  // down: per-warp store buffers
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + RING_BYTES + Smem<KIND>::STAGING);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* i8_full = tempty + 2;
  uint64_t* i8_empty = i8_full + I8_SLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(i8_empty + I8_SLOTS);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + N_XFORM_WARPS);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    for (int i = 0; i < I8_SLOTS; ++i) {
      mbar_init(&i8_full[i], 1);
      mbar_init(&i8_empty[i], N_XFORM_WARPS);
    }
    fence_barrier_init();
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
    if (KIND == kDownF32) prefetch_tensormap(&tm_out);
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
  const int total_tiles = p.ptile_off[p.E] * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------- A producer
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const PairCoord c = decode_pair(tile, p);
        const int row0 = c.m0 * BM;
        const int row1 = (c.two ? c.m0 + 1 : c.m0) * BM;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const int stage = static_cast<int>(issued % STAGES);
          const uint32_t phase = static_cast<uint32_t>((issued / STAGES) & 1);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], 2 * A_BYTES);
          tma_load_2d(st, &tm_a, &full[stage], kb * BK, row0);
          tma_load_2d(st + A_BYTES, &tm_a, &full[stage], kb * BK, row1);
          ++issued;
        }
      }
      for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        // (test_stall waits on the phase in progress, which no thread completes)
        if (!mbar_wait(&tempty[acc], p.test_stall ? acc_phase : acc_phase ^ 1u, p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * 2 * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t a0 = sw128_desc(st), a1 = sw128_desc(st + A_BYTES), b = sw128_desc(st + 2 * A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
            tc_mma_f16(d0, a0 + 2 * k, b + 2 * k, IDESC, accum);
            tc_mma_f16(d0 + BN, a1 + 2 * k, b + 2 * k, IDESC, accum);
          }
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
  } else if (warp < 6) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    int n_stores = 0;  // bulk stores issued by this warp (down only)
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const PairCoord c = decode_pair(tile, p);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_limit_ns)) {
        set_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      for (int j = 0; j < (c.two ? 2 : 1); ++j) {
        const int64_t row = static_cast<int64_t>(c.m0 + j) * BM + q * 32 + lane;
        const uint32_t tbase =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * 2 * BN + j * BN);
        if constexpr (KIND == kGateUpSwiGLU) {
          constexpr int HALF = BN / 2;  // 64 gate + 64 up columns
          const int64_t col = static_cast<int64_t>(c.n) * HALF;
          uint16_t* out_row = static_cast<uint16_t*>(p.out) + row * p.ld_out + col;
          const float* sg = p.scale0 + static_cast<int64_t>(c.e) * p.ld_out + col;
          const float* su = p.scale1 + static_cast<int64_t>(c.e) * p.ld_out + col;
#pragma unroll 1
          for (int c0 = 0; c0 < HALF; c0 += 32) {
            uint32_t g[32], u[32];
            tmem_load32(tbase + c0, g);
            tmem_load32(tbase + HALF + c0, u);
            uint32_t h[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const float2 sgv = __ldg(reinterpret_cast<const float2*>(sg + c0 + 2 * jj));
              const float2 suv = __ldg(reinterpret_cast<const float2*>(su + c0 + 2 * jj));
              const float g0 = __uint_as_float(g[2 * jj]) * sgv.x, g1 = __uint_as_float(g[2 * jj + 1]) * sgv.y;
              const float u0 = __uint_as_float(u[2 * jj]) * suv.x, u1 = __uint_as_float(u[2 * jj + 1]) * suv.y;
              h[jj] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
            }
            uint4* dst = reinterpret_cast<uint4*>(out_row + c0);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
          }
        } else {
          const int64_t col = static_cast<int64_t>(c.n) * BN;
          const float* sd = p.scale0 + static_cast<int64_t>(c.e) * p.ld_out + col;
          const int row0 = (c.m0 + j) * BM + q * 32;
#pragma unroll 1
          for (int c0 = 0; c0 < BN; c0 += 32, ++n_stores) {
            uint32_t r[32];
            tmem_load32(tbase + c0, r);
            uint8_t* buf = staging + (q * 2 + (n_stores & 1)) * 4096;
            if (n_stores >= 2) {
              if (lane == 0) bulk_wait_group_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 s4 = __ldg(reinterpret_cast<const float4*>(sd + c0 + 4 * v));
              *reinterpret_cast<float4*>(buf + lane * 128 + 16 * (v ^ (lane & 7))) =
                  make_float4(__uint_as_float(r[4 * v]) * s4.x, __uint_as_float(r[4 * v + 1]) * s4.y,
                              __uint_as_float(r[4 * v + 2]) * s4.z, __uint_as_float(r[4 * v + 3]) * s4.w);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, buf, static_cast<int32_t>(col) + c0, row0);
              bulk_commit_group();
            }
          }
          (void)row;
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (KIND == kDownF32 && lane == 0) bulk_wait_group<0>();
  } else if (warp == BPROD_WARP) {
    if (lane == 0) {
      // --------------------------------------------- int8 weight producer
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const PairCoord c = decode_pair(tile, p);
        const int b_row = c.e * p.b_rows_per_expert + c.n * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const int slot = static_cast<int>(issued % I8_SLOTS);
          const uint32_t sphase = static_cast<uint32_t>((issued / I8_SLOTS) & 1);
          if (!mbar_wait(&i8_empty[slot], sphase ^ 1u, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&i8_full[slot], I8_BYTES);
          tma_load_2d(s8 + slot * I8_BYTES, &tm_b, &i8_full[slot], kb * BK, b_row);
          ++issued;
        }
      }
      for (int64_t i = (issued > I8_SLOTS ? issued - I8_SLOTS : 0); i < issued; ++i)
        if (!mbar_wait(&i8_full[i % I8_SLOTS], static_cast<uint32_t>((i / I8_SLOTS) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
    }
  } else {
    // ------------------------------------------------ int8 -> bf16 transform
    // Thread x converts 16 staged int8 codes (K elements 16c..16c+15 of row
    // r, chunk index ch = 4r + c) into two 16-byte bf16 chunks 2c and 2c+1 of
    // row r, stored at their 128-byte-swizzled positions r*128 +
    // 16*((2c + i) ^ (r & 7)).
    const int xt = threadIdx.x - 32 * XFORM_WARP0;
    int64_t it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int stage = static_cast<int>(it % STAGES);
        const uint32_t phase = static_cast<uint32_t>((it / STAGES) & 1);
        const int slot = static_cast<int>(it % I8_SLOTS);
        const uint32_t sphase = static_cast<uint32_t>((it / I8_SLOTS) & 1);
        if (!mbar_wait(&i8_full[slot], sphase, p.wait_limit_ns) ||
            !mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        const uint8_t* src = s8 + slot * I8_BYTES;
        uint8_t* dst = smem + stage * STAGE_BYTES + 2 * A_BYTES;
#pragma unroll
        for (int ch = xt; ch < BN * 4; ch += 32 * N_XFORM_WARPS) convert_chunk16(src + ch * 16, dst, ch >> 2, ch & 3);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&i8_empty[slot]);
          mbar_arrive(&full[stage]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

int grouped_gemm_int8_tile_n(GemmKind kind) { return kind == kGateUpSwiGLU ? BN / 2 : BN; }
int grouped_gemm_int8_gateup_block() { return BN / 2; }

cudaError_t grouped_gemm_int8_prepare() {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_int8_kernel<kGateUpSwiGLU>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<kGateUpSwiGLU>::BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_int8_kernel<kDownF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Smem<kDownF32>::BYTES);
}

cudaError_t launch_grouped_gemm_int8(GemmKind kind, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const CUtensorMap& tm_out, const GemmArgs& a, cudaStream_t s) {
  if (kind == kGateUpSwiGLU)
    launch_kernel(grouped_gemm_int8_kernel<kGateUpSwiGLU>, a.grid, THREADS, Smem<kGateUpSwiGLU>::BYTES, s, tm_a, tm_b, tm_out, a);
  else
    launch_kernel(grouped_gemm_int8_kernel<kDownF32>, a.grid, THREADS, Smem<kDownF32>::BYTES, s, tm_a, tm_b, tm_out, a);
  return cudaGetLastError();
}

}  // namespace cbmoe
