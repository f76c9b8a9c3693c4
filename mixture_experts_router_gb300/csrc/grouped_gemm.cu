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
// int8 experts (symmetric per-output-channel int8, "lshu.cn/news/53496" §4.3):
// the weight tile arrives as int8 and is turned into bf16 exactly inside the
// kernel; the channel scale multiplies the fp32 accumulator in the epilogue
// (acc_g * s_g[e][j], acc_u * s_u[e][j], acc * s_d[e][c]).
//
// Rows are the expert-grouped activations; every expert's block starts on a
// 128-row boundary, so an M-tile belongs to exactly one expert, and the tile
// list (expert-major, then N, then M) is derived on the device from the
// dispatch's tile prefix sums: the host never learns the expert counts.
//
// Per CTA (one per SM, persistent, static round-robin over tiles):
//   warp 0      : TMA producer (one thread): A 128x64 bf16 box and the B box
//                 (256x64 bf16, or 256x64 int8 into a 2-slot staging ring),
//                 128-byte swizzle, into a 4-stage ring guarded by mbarriers
//   warp 1      : owns the 512 TMEM columns; one thread issues
//                 tcgen05.mma.cta_group::1.kind::f16 (M=128, N=256, K=16) x4
//                 per stage and commits stage release / accumulator ready
//   warps 2..5  : epilogue: tcgen05.ld 32 lanes x 32 columns, SwiGLU or fp32,
//                 16-byte global stores; two accumulators alternate so the
//                 epilogue of tile i overlaps the mainloop of tile i+1
//   warps 6..9  : int8 only: convert each staged int8 tile to bf16 into the
//                 stage's B buffer in the swizzled layout the MMA reads, then
//                 fence to the async proxy and arrive on the stage barrier
// Every wait is bounded; a wait that runs out records CB_ERR_TIMEOUT in the
// status word and the CTA winds down (waiting for its own loads in flight
// and freeing its TMEM).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int BM = kTileM;               // 128 rows per tile
constexpr int BK = 64;                   // 64 bf16 = one 128-byte swizzled row
constexpr int BN = 256;                  // accumulator columns per tile
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int I8_BYTES = BN * BK;        // 16 KB of int8 per staged B tile
constexpr int N_XFORM_WARPS = 8;
constexpr uint32_t TMEM_COLS = 2 * BN;   // two fp32 accumulators of 256 columns
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

// bf16 weights: a 4-stage ring of (A, B) tiles filled by one TMA thread.
// int8 weights: a 3-stage (A, bf16 B) ring for the MMA plus a 5-slot ring of
// int8 B tiles with its own TMA thread, so weight loads run up to five
// k-blocks ahead of the MMA (about a DRAM latency) while the transform warps
// fill the bf16 B stages.
template <bool INT8>
struct Shape {
  static constexpr int STAGES = INT8 ? 3 : 4;
  static constexpr int I8_SLOTS = INT8 ? 5 : 1;
  static constexpr int XFORM_WARP0 = 6;
  static constexpr int BPROD_WARP = XFORM_WARP0 + N_XFORM_WARPS;
  static constexpr int THREADS = INT8 ? 32 * (BPROD_WARP + 1) : 192;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES + (INT8 ? I8_SLOTS * I8_BYTES : 0);
  static constexpr int SMEM_BYTES = RING_BYTES + 1024 + 256;
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

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// Four int8 codes (one 32-bit word) -> four bf16, exactly.  With m = q & 0x7F
// and s = q & 0x80, the bf16 words 0x4300|m and 0x4300|s are 128 + m and
// 128 (s = 0) or 256 (s = 0x80); their difference is m or m - 128, i.e. q,
// an integer below 2^8 in magnitude, so the bf16 subtraction is exact.
__device__ __forceinline__ void int8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t m = w & 0x7F7F7F7Fu, s = w & 0x80808080u;
  const uint32_t m01 = __byte_perm(m, 0x43434343u, 0x4140), m23 = __byte_perm(m, 0x43434343u, 0x4342);
  const uint32_t s01 = __byte_perm(s, 0x43434343u, 0x4140), s23 = __byte_perm(s, 0x43434343u, 0x4342);
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(m01), "r"(s01));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(m23), "r"(s23));
}

template <int KIND, bool INT8>
__global__ void __launch_bounds__(Shape<INT8>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const GemmArgs p) {
  constexpr int STAGES = Shape<INT8>::STAGES;
  constexpr int I8_SLOTS = Shape<INT8>::I8_SLOTS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  uint8_t* s8 = smem + STAGES * STAGE_BYTES;  // int8 staging ring (INT8 only)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Shape<INT8>::RING_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* i8_full = tempty + 2;
  uint64_t* i8_empty = i8_full + I8_SLOTS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(i8_empty + I8_SLOTS);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], INT8 ? 1 + N_XFORM_WARPS : 1);
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
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = p.mtile_off[p.E] * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------ TMA producer (A, and bf16 B)
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const TileCoord c = decode_tile(tile, p);
        const int a_row = c.m_tile * BM;
        const int b_row = c.e * p.b_rows_per_expert + c.n * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          const int stage = static_cast<int>(issued % STAGES);
          const uint32_t phase = static_cast<uint32_t>((issued / STAGES) & 1);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          if constexpr (INT8) {
            mbar_arrive_expect_tx(&full[stage], A_BYTES);
            tma_load_2d(sa + stage * A_BYTES, &tm_a, &full[stage], kb * BK, a_row);
          } else {
            mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
            tma_load_2d(sa + stage * A_BYTES, &tm_a, &full[stage], kb * BK, a_row);
            tma_load_2d(sb + stage * B_BYTES, &tm_b, &full[stage], kb * BK, b_row);
          }
          ++issued;
        }
      }
      // No load of ours may still be landing in shared memory when the CTA
      // exits: wait for the last load issued into each stage.
      for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.wait_limit_ns)) {
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
            tc_mma_f16(d_tmem, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb | k) != 0 ? 1u : 0u);
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
    const int q = warp & 3;  // this warp's quarter of the 128 TMEM lanes
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileCoord c = decode_tile(tile, p);
      if (!mbar_wait(&tfull[acc], acc_phase, p.wait_limit_ns)) {
        set_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(c.m_tile) * BM + q * 32 + lane;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (KIND == kGateUpSwiGLU) {
        uint16_t* out_row = static_cast<uint16_t*>(p.out) + row * p.ld_out + c.n * (BN / 2);
        const int64_t col0 = static_cast<int64_t>(c.e) * (p.ld_out) + c.n * (BN / 2);  // scale index base
#pragma unroll 1
        for (int c0 = 0; c0 < BN / 2; c0 += 32) {
          uint32_t g[32], u[32];
          tmem_load32(tbase + c0, g);
          tmem_load32(tbase + BN / 2 + c0, u);
          uint32_t h[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
            float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
            if constexpr (INT8) {
              g0 *= __ldg(p.scale0 + col0 + c0 + 2 * j);
              g1 *= __ldg(p.scale0 + col0 + c0 + 2 * j + 1);
              u0 *= __ldg(p.scale1 + col0 + c0 + 2 * j);
              u1 *= __ldg(p.scale1 + col0 + c0 + 2 * j + 1);
            }
            h[j] = pack_bf16x2(silu(g0) * u0, silu(g1) * u1);
          }
          uint4* dst = reinterpret_cast<uint4*>(out_row + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
        }
      } else {
        float* out_row = static_cast<float*>(p.out) + row * p.ld_out + c.n * BN;
        const int64_t col0 = static_cast<int64_t>(c.e) * p.ld_out + c.n * BN;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_load32(tbase + c0, r);
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            v[j] = __uint_as_float(r[j]);
            if constexpr (INT8) v[j] *= __ldg(p.scale0 + col0 + c0 + j);
          }
          float4* dst = reinterpret_cast<float4*>(out_row + c0);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if constexpr (INT8) {
    if (warp == Shape<INT8>::BPROD_WARP) {
      if (lane == 0) {
        // --------------------------------------------- TMA producer (int8 B)
        int64_t issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
          const TileCoord c = decode_tile(tile, p);
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
      // ----------------------------------------- int8 -> bf16 transform
      // N_XFORM_WARPS warps; thread x handles the 16-byte output chunks x,
      // x + 32 N_XFORM_WARPS, ... of the 256 rows x 8 chunks: chunk (r, c)
      // takes the 8 int8 codes at staged bytes r*64 + 8c and lands at
      // r*128 + 16*(c ^ (r & 7)), the 128-byte-swizzled position of K
      // elements 8c..8c+7 of row r.
      const int xt = threadIdx.x - 32 * Shape<INT8>::XFORM_WARP0;
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
          uint8_t* dst = sb + stage * B_BYTES;
#pragma unroll
          for (int ch = xt; ch < BN * 8; ch += 32 * N_XFORM_WARPS) {
            const int r = ch >> 3, cc = ch & 7;
            const uint2 w = *reinterpret_cast<const uint2*>(src + ch * 8);
            uint4 o;
            int8x4_to_bf16x4(w.x, o.x, o.y);
            int8x4_to_bf16x4(w.y, o.z, o.w);
            *reinterpret_cast<uint4*>(dst + r * 128 + 16 * (cc ^ (r & 7))) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&i8_empty[slot]);
            mbar_arrive(&full[stage]);
          }
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

template <int KIND, bool INT8>
cudaError_t set_smem() {
  return cudaFuncSetAttribute(grouped_gemm_kernel<KIND, INT8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Shape<INT8>::SMEM_BYTES);
}

}  // namespace

int grouped_gemm_tile_n(GemmKind kind) { return kind == kGateUpSwiGLU ? BN / 2 : BN; }

cudaError_t grouped_gemm_prepare() {
  cudaError_t e = set_smem<kGateUpSwiGLU, false>();
  if (e == cudaSuccess) e = set_smem<kDownF32, false>();
  if (e == cudaSuccess) e = set_smem<kGateUpSwiGLU, true>();
  if (e == cudaSuccess) e = set_smem<kDownF32, true>();
  return e;
}

cudaError_t launch_grouped_gemm(GemmKind kind, bool int8_weights, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                const GemmArgs& a, cudaStream_t s) {
  if (kind == kGateUpSwiGLU) {
    if (int8_weights)
      grouped_gemm_kernel<kGateUpSwiGLU, true>
          <<<a.grid, Shape<true>::THREADS, Shape<true>::SMEM_BYTES, s>>>(tm_a, tm_b, a);
    else
      grouped_gemm_kernel<kGateUpSwiGLU, false>
          <<<a.grid, Shape<false>::THREADS, Shape<false>::SMEM_BYTES, s>>>(tm_a, tm_b, a);
  } else {
    if (int8_weights)
      grouped_gemm_kernel<kDownF32, true><<<a.grid, Shape<true>::THREADS, Shape<true>::SMEM_BYTES, s>>>(tm_a, tm_b, a);
    else
      grouped_gemm_kernel<kDownF32, false>
          <<<a.grid, Shape<false>::THREADS, Shape<false>::SMEM_BYTES, s>>>(tm_a, tm_b, a);
  }
  return cudaGetLastError();
}

}  // namespace cbmoe
