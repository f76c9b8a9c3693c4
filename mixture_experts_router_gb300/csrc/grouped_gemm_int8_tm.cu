// Grouped expert GEMMs with int8 weights (symmetric per-output-channel int8,
// "lshu.cn/news/53496" §4.3), int4 weights (4-bit codes with a scale and a
// zero point per output channel, "m.nxbn.cn/news/47706" §3.2) or fp8 weights
// (e4m3 bytes with a scale per output channel, the FP8 of
// "discosf.com/news/4774337" §6.3), dequantised to bf16 inside the kernel,
// with the converted weights held in TENSOR MEMORY as the MMA's A operand.
// An int4 row of the tile holds q - z (its zero point taken off during the
// conversion, exact), an fp8 row the e4m3 values (exact in bf16); the scale
// is applied as for int8.
//
// The GEMM is computed transposed: D[weight row][token] = W[e] * Xp^T, with
// D in tensor memory (lane = weight row, column = token).  A tile is 128
// weight rows against the 256 tokens of a pair of 128-row m-tiles of one
// expert (both m-tiles' activation boxes sit back to back in shared memory),
// so each K step is ONE tcgen05.mma M=128 N=256 K=16 (N=128 when the pair
// has a single m-tile).  The tensor core accepts an MMA only as the previous
// one drains, so every barrier wait or commit of the issuing thread costs
// tensor time: one wait and one commit per 64-wide k-block keep that below
// the four MMAs' 512 cycles.
//
// The int8 codes go TMA -> shared memory -> registers -> exact bf16 ->
// tensor memory (tcgen05.st), so the converted weights never pass through
// shared memory and the tensor core reads only the activations from it.  The
// scales multiply the fp32 accumulator in the epilogue:
//
//   gate/up : H[r, n*64 + 16g + j] = bf16( SiLU(s_g D[32g + j][r]) * s_u D[32g + 16 + j][r] ),
//             weight rows of tile n: groups g = 0..3 of 16 gate rows then the
//             same 16 features' up rows, so a gate lane and its up lane are
//             16 lanes apart in one warp and pair up by a shuffle
//   down    : Y[r, n*128 + c] = s_d[e][n*128 + c] D[c][r]          (fp32 out)
//
// Tensor memory: the accumulator in columns 0..255 (single-buffered: the
// epilogue warps drain it into registers and release it before storing), and
// 4 converted weight slots of K = 64 (32 columns each) from column 256.
//
// Per CTA (one per SM, persistent, round-robin over pair tiles):
//   warp 0       : TMA producer of the activation boxes (128 x 64 bf16 each)
//   warp 1       : TMEM owner and MMA issuer
//   warp 2       : TMA producer of the int8 weight tiles (128 rows x 128 K)
//   warps 4..7   : int8 -> bf16 transform; warp 4+q writes lanes 32q..32q+31
//                  (one weight row per thread)
//   warps 8..15  : epilogue; warp 8+q drains lanes 32q..+31 of columns
//                  0..127 (first m-tile), warp 12+q the same lanes of 128..255
// Stage s of the 4-deep ring is an activation box pair in shared memory plus
// weight slot s in tensor memory: full[s] completes on the TMA bytes and the
// four transform warps' arrivals, empty[s] on the MMAs' commit.
// Every wait is bounded (CB_ERR_TIMEOUT in the status word on expiry).
//
// WIDE tiles (layers of at most 128 tokens, where every expert has at most
// one m-tile): a tile is the single m-tile against TWO 128-row weight blocks,
// two M=128 N=128 MMAs per K step into two accumulators (columns 0..127 and
// 128..255), so each k-block's handshake moves twice the weight bytes (at
// decode sizes the per-k-block waits, not the tensor core, bound the
// kernel).  A stage is then one activation box and a weight slot two 128-row
// boxes (the same 192 KB of shared memory); per stage the two converted
// blocks take 64 tensor-memory columns (256..511).  The conversion warps read
// each k-block's codes of both rows from shared memory and release the slot
// after its last k-block; the epilogue's two halves are the two weight blocks
// of the same tokens.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "int8_bf16.cuh"
#include "swiglu.cuh"

namespace cbmoe {
namespace {

constexpr int BM = kTileM;              // tokens per m-tile
constexpr int BK = 64;                  // K per stage (one 128-byte bf16 row)
constexpr int WROWS = 128;              // weight rows per tile (TMEM lanes)
constexpr int W_ROW_BYTES = 128;       // bytes per weight row of a slot (one TMA box row):
                                        // K = 128 int8 or 256 int4 codes
constexpr int STAGES = 4;
constexpr int A_BOX = BM * BK * 2;      // 16 KB: one m-tile's 64 K of activations
constexpr int STAGE_BYTES = 2 * A_BOX;
constexpr int A32_ROWS = 32;            // rows of the short activation box
constexpr int A32_BOX = A32_ROWS * BK * 2;
constexpr int W_SLOTS = 4;
constexpr int W_BYTES = WROWS * W_ROW_BYTES;  // 16 KB
constexpr int THREADS = 16 * 32;
constexpr int XFORM_WARP0 = 4;
constexpr int EPI_WARP0 = 8;
constexpr int GATEUP_GROUP = 16;        // gate/up rows interleaved in groups of this size
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL0 = 2 * BM;     // first weight slot column
constexpr uint32_t SLOT_COLS = BK / 2;  // 32 columns per weight slot
constexpr uint32_t IDESC2 = idesc_bf16_f32(WROWS, 2 * BM);
constexpr uint32_t IDESC1 = idesc_bf16_f32(WROWS, BM);
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + W_SLOTS * W_BYTES + 1024 + 512;

// Four one-byte weight codes -> four bf16 (int8 or e4m3), exactly.
template <int WF>
__device__ __forceinline__ void byte4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (WF == kWFp8)
    fp8x4_to_bf16x4(w, lo, hi);
  else
    int8x4_to_bf16x4(w, lo, hi);
}

struct PairCoord {
  int m0;      // first m-tile (global index)
  bool two;    // second m-tile m0 + 1 is real
  int e;       // expert
  int n;       // weight tile within the expert
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

template <int KIND, int WF, bool WIDE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_int8_tm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                                const __grid_constant__ CUtensorMap tm_x32, const GemmArgs p) {
  constexpr int KPS = WF == kWInt4 ? 4 : 2;  // k-blocks per weight slot
  constexpr int kStageBytes = WIDE ? A_BOX : STAGE_BYTES;     // activation boxes of a stage
  constexpr int kWBytes = WIDE ? 2 * W_BYTES : W_BYTES;        // weight boxes of a slot
  constexpr uint32_t kSlotCols = WIDE ? 2 * SLOT_COLS : SLOT_COLS;  // tensor-memory columns per stage
  static_assert(STAGES * kStageBytes + W_SLOTS * kWBytes == STAGES * STAGE_BYTES + W_SLOTS * W_BYTES,
                "both tilings use the same shared memory");
  static_assert(A_COL0 + STAGES * kSlotCols <= TMEM_COLS, "weight slots fit the tensor memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_w = smem + STAGES * kStageBytes;  // int8 weight slots (128-byte swizzled rows)
  uint64_t* full = reinterpret_cast<uint64_t*>(s_w + W_SLOTS * kWBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* w_full = empty + STAGES;
  uint64_t* w_empty = w_full + W_SLOTS;
  uint64_t* acc_full = w_empty + W_SLOTS;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* mma_done = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + 4);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < W_SLOTS; ++s) {
      mbar_init(&w_full[s], 1);
      mbar_init(&w_empty[s], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(mma_done, 1);
    fence_barrier_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
    if (p.counts != nullptr) prefetch_tensormap(&tm_x32);
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
      // ------------------------------------------- activation producer
      int64_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const PairCoord c = decode_pair(tile, p);
        // a single m-tile of at most 32 routed rows (decode sizes) loads only
        // its first 32 rows: the other token columns of the accumulator are
        // padding that no one reads, and the SM's loads are then mostly the
        // weights
        const bool a32 = p.counts != nullptr && !c.two &&
                         p.counts[c.e] - (c.m0 - p.mtile_off[c.e]) * BM <= A32_ROWS;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int stage = static_cast<int>(it % STAGES);
          if (!mbar_wait(&empty[stage], static_cast<uint32_t>(((it / STAGES) & 1) ^ 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * kStageBytes;
          mbar_arrive_expect_tx(&full[stage], c.two ? 2 * A_BOX : (a32 ? A32_BOX : A_BOX));
          tma_load_2d(st, a32 ? &tm_x32 : &tm_x, &full[stage], kb * BK, c.m0 * BM);
          if (c.two) tma_load_2d(st + A_BOX, &tm_x, &full[stage], kb * BK, (c.m0 + 1) * BM);
        }
      }
      // no copy may still be in flight into shared memory at exit
      for (int64_t i = (it > STAGES ? it - STAGES : 0); i < it; ++i)
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------------------------------------- int8 weight producer
      int64_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const PairCoord c = decode_pair(tile, p);
        const int w_row = c.e * p.b_rows_per_expert + c.n * (WIDE ? 2 * WROWS : WROWS);
        for (int j = 0; j < p.k_blocks / KPS; ++j, ++it) {
          const int slot = static_cast<int>(it % W_SLOTS);
          if (!mbar_wait(&w_empty[slot], static_cast<uint32_t>(((it / W_SLOTS) & 1) ^ 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&w_full[slot], kWBytes);
          tma_load_2d(s_w + slot * kWBytes, &tm_w, &w_full[slot], j * W_ROW_BYTES, w_row);
          if constexpr (WIDE) tma_load_2d(s_w + slot * kWBytes + W_BYTES, &tm_w, &w_full[slot], j * W_ROW_BYTES, w_row + WROWS);
        }
      }
      for (int64_t i = (it > W_SLOTS ? it - W_SLOTS : 0); i < it; ++i)
        if (!mbar_wait(&w_full[i % W_SLOTS], static_cast<uint32_t>((i / W_SLOTS) & 1), p.wait_limit_ns))
          set_error(p.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------- MMA issuer
      int64_t it = 0;
      uint32_t tphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
        const PairCoord c = decode_pair(tile, p);
        // (test_stall waits on the phase in progress, which no thread completes)
        if (!mbar_wait(acc_empty, p.test_stall ? tphase : tphase ^ 1u, p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        [[maybe_unused]] const uint32_t idesc = c.two ? IDESC2 : IDESC1;
        for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
          const int stage = static_cast<int>(it % STAGES);
          if (!mbar_wait(&full[stage], static_cast<uint32_t>((it / STAGES) & 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t b = sw128_desc(smem_u32(smem + stage * kStageBytes));
          const uint32_t a = tmem_base + A_COL0 + static_cast<uint32_t>(stage) * kSlotCols;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            if constexpr (WIDE) {
              const uint32_t acc = (kb | ks) != 0 ? 1u : 0u;
              tc_mma_f16_ts(tmem_base, a + 8 * ks, b + 2 * ks, IDESC1, acc);
              tc_mma_f16_ts(tmem_base + BM, a + SLOT_COLS + 8 * ks, b + 2 * ks, IDESC1, acc);
            } else {
              tc_mma_f16_ts(tmem_base, a + 8 * ks, b + 2 * ks, idesc, (kb | ks) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&empty[stage]);
        }
        if (!ok) break;
        tc_commit(acc_full);
        tphase ^= 1u;
      }
      // no MMA may still run when the tensor memory is freed
      tc_commit(mma_done);
      if (!mbar_wait(mma_done, 0, p.wait_limit_ns)) set_error(p.err, kErrTimeout);
    }
  } else if (WIDE && warp >= XFORM_WARP0 && warp < XFORM_WARP0 + 4) {
    // ---------------------------- int8 / int4 / fp8 -> bf16, wide tiles
    // Thread (q, lane) owns row r = 32q + lane of both weight blocks (TMEM
    // lane r of both regions).  Per k-block it reads that k-block's codes of
    // both rows from the slot (the TMA 128-byte swizzle as below), converts
    // them and stores them into the stage's two 32-column regions; the slot
    // is released after its last k-block.
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int64_t it = 0, wi = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      uint32_t zz[2] = {0u, 0u};  // int4: 0x4300 | zero point of block 0's and block 1's row r
      if constexpr (WF == kWInt4) {
        const PairCoord c = decode_pair(tile, p);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int nb = 2 * c.n + blk;
          int z;
          if constexpr (KIND == kGateUpSwiGLU) {
            const int feat = nb * (WROWS / 2) + (r / 32) * GATEUP_GROUP + (r % GATEUP_GROUP);
            z = __ldg((r % 32 < GATEUP_GROUP ? p.zero0 : p.zero1) + static_cast<int64_t>(c.e) * p.ld_out + feat);
          } else {
            z = __ldg(p.zero0 + static_cast<int64_t>(c.e) * p.ld_out + nb * WROWS + r);
          }
          zz[blk] = (0x4300u | static_cast<uint32_t>(z)) * 0x00010001u;
        }
      }
      int slot = 0;
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int stage = static_cast<int>(it % STAGES);
        if ((kb % KPS) == 0) {
          slot = static_cast<int>(wi % W_SLOTS);
          if (!mbar_wait(&w_full[slot], static_cast<uint32_t>((wi / W_SLOTS) & 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          ++wi;
        }
        if (!mbar_wait(&empty[stage], static_cast<uint32_t>(((it / STAGES) & 1) ^ 1), p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const uint8_t* row = s_w + slot * kWBytes + blk * W_BYTES + r * 128;
          uint32_t o[32];
          if constexpr (WF != kWInt4) {
            const int c0 = (kb & 1) * 4;  // 16-byte chunks c0..c0+3: this k-block's 64 codes
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const uint4 w = *reinterpret_cast<const uint4*>(row + (((c0 + cc) ^ (r & 7)) << 4));
              byte4_to_bf16x4<WF>(w.x, o[8 * cc + 0], o[8 * cc + 1]);
              byte4_to_bf16x4<WF>(w.y, o[8 * cc + 2], o[8 * cc + 3]);
              byte4_to_bf16x4<WF>(w.z, o[8 * cc + 4], o[8 * cc + 5]);
              byte4_to_bf16x4<WF>(w.w, o[8 * cc + 6], o[8 * cc + 7]);
            }
          } else {
            const int part = kb & 3;  // chunks 2 part, 2 part + 1: 64 codes
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const uint4 w = *reinterpret_cast<const uint4*>(row + (((2 * part + cc) ^ (r & 7)) << 4));
              uint32_t t[4];
              int4x8_minus_zero_to_bf16(w.x, zz[blk], t);
#pragma unroll
              for (int m = 0; m < 4; ++m) o[16 * cc + m] = t[m];
              int4x8_minus_zero_to_bf16(w.y, zz[blk], t);
#pragma unroll
              for (int m = 0; m < 4; ++m) o[16 * cc + 4 + m] = t[m];
              int4x8_minus_zero_to_bf16(w.z, zz[blk], t);
#pragma unroll
              for (int m = 0; m < 4; ++m) o[16 * cc + 8 + m] = t[m];
              int4x8_minus_zero_to_bf16(w.w, zz[blk], t);
#pragma unroll
              for (int m = 0; m < 4; ++m) o[16 * cc + 12 + m] = t[m];
            }
          }
          tmem_store32(lane_addr + A_COL0 + static_cast<uint32_t>(stage) * kSlotCols +
                           static_cast<uint32_t>(blk) * SLOT_COLS,
                       o);
        }
        if ((kb % KPS) == KPS - 1) {  // the slot's last k-block: its codes are all read
          __syncwarp();
          if (lane == 0) mbar_arrive(&w_empty[slot]);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
      }
    }
  } else if (!WIDE && warp >= XFORM_WARP0 && warp < XFORM_WARP0 + 4) {
    // ------------------------------------------- int8 / int4 -> bf16 transform
    // Thread (q, lane) owns weight row r = 32q + lane of the tile, i.e. TMEM
    // lane r.  Per weight slot (KPS k-blocks) it reads the row's 128 bytes
    // (16-byte chunk c at r*128 + 16*(c ^ (r & 7)), the TMA 128-byte swizzle);
    // per k-block it converts 64 codes exactly and stores them into the
    // stage's weight slot, column i holding K elements 2i, 2i + 1 of the
    // k-block (int8: 4 chunks of 16 codes; int4: 2 chunks of 32 codes, minus
    // the row's zero point).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int64_t it = 0, wi = 0;
    bool ok = true;
    uint4 v[8];
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      uint32_t zz = 0;  // int4: 0x4300 | zero point, in both bf16 halves
      if constexpr (WF == kWInt4) {
        const PairCoord c = decode_pair(tile, p);
        int z;
        if constexpr (KIND == kGateUpSwiGLU) {
          // rows of group g: 16 gate rows, then the same 16 features' up rows
          const int feat = c.n * (WROWS / 2) + (r / 32) * GATEUP_GROUP + (r % GATEUP_GROUP);
          z = __ldg((r % 32 < GATEUP_GROUP ? p.zero0 : p.zero1) + static_cast<int64_t>(c.e) * p.ld_out + feat);
        } else {
          z = __ldg(p.zero0 + static_cast<int64_t>(c.e) * p.ld_out + c.n * WROWS + r);
        }
        zz = (0x4300u | static_cast<uint32_t>(z)) * 0x00010001u;
      }
      for (int kb = 0; kb < p.k_blocks; ++kb, ++it) {
        const int stage = static_cast<int>(it % STAGES);
        if ((kb % KPS) == 0) {
          const int slot = static_cast<int>(wi % W_SLOTS);
          if (!mbar_wait(&w_full[slot], static_cast<uint32_t>((wi / W_SLOTS) & 1), p.wait_limit_ns)) {
            set_error(p.err, kErrTimeout);
            ok = false;
            break;
          }
          const uint8_t* row = s_w + slot * W_BYTES + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) v[c] = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) << 4));
          __syncwarp();
          if (lane == 0) mbar_arrive(&w_empty[slot]);
          ++wi;
        }
        if (!mbar_wait(&empty[stage], static_cast<uint32_t>(((it / STAGES) & 1) ^ 1), p.wait_limit_ns)) {
          set_error(p.err, kErrTimeout);
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t o[32];
        if constexpr (WF != kWInt4) {
          if ((kb & 1) == 0) {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              byte4_to_bf16x4<WF>(v[cc].x, o[8 * cc + 0], o[8 * cc + 1]);
              byte4_to_bf16x4<WF>(v[cc].y, o[8 * cc + 2], o[8 * cc + 3]);
              byte4_to_bf16x4<WF>(v[cc].z, o[8 * cc + 4], o[8 * cc + 5]);
              byte4_to_bf16x4<WF>(v[cc].w, o[8 * cc + 6], o[8 * cc + 7]);
            }
          } else {
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              byte4_to_bf16x4<WF>(v[4 + cc].x, o[8 * cc + 0], o[8 * cc + 1]);
              byte4_to_bf16x4<WF>(v[4 + cc].y, o[8 * cc + 2], o[8 * cc + 3]);
              byte4_to_bf16x4<WF>(v[4 + cc].z, o[8 * cc + 4], o[8 * cc + 5]);
              byte4_to_bf16x4<WF>(v[4 + cc].w, o[8 * cc + 6], o[8 * cc + 7]);
            }
          }
        } else {
          // chunks 2 (kb % 4) and 2 (kb % 4) + 1: 64 codes, 32 columns
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            if (part == (kb & 3)) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const uint4 w = v[2 * part + cc];
                uint32_t t[4];
                int4x8_minus_zero_to_bf16(w.x, zz, t);
#pragma unroll
                for (int m = 0; m < 4; ++m) o[16 * cc + m] = t[m];
                int4x8_minus_zero_to_bf16(w.y, zz, t);
#pragma unroll
                for (int m = 0; m < 4; ++m) o[16 * cc + 4 + m] = t[m];
                int4x8_minus_zero_to_bf16(w.z, zz, t);
#pragma unroll
                for (int m = 0; m < 4; ++m) o[16 * cc + 8 + m] = t[m];
                int4x8_minus_zero_to_bf16(w.w, zz, t);
#pragma unroll
                for (int m = 0; m < 4; ++m) o[16 * cc + 12 + m] = t[m];
              }
            }
          }
        }
        tmem_store32(lane_addr + A_COL0 + static_cast<uint32_t>(stage) * SLOT_COLS, o);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
      }
    }
  } else if (warp >= EPI_WARP0) {
    // ------------------------------------------------------------ epilogue
    // Warp 8+q (half 0) and 12+q (half 1) hold lanes 32q.. of the first and
    // second m-tile's 128 accumulator columns.  Each reads its columns, does
    // its arithmetic, releases the accumulator and only then stores.
    const int q = warp & 3;
    const int half = (warp - EPI_WARP0) / 4;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * BM);
    uint32_t tphase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const PairCoord c = decode_pair(tile, p);
      if (!mbar_wait(acc_full, tphase, p.wait_limit_ns)) {
        set_error(p.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      // WIDE: the halves are the two weight blocks of the same tokens
      const bool active = WIDE || half == 0 || c.two;
      const int64_t row0 = static_cast<int64_t>(c.m0 + (WIDE ? 0 : half)) * BM;
      const int nblk = WIDE ? 2 * c.n + half : c.n;  // weight block of this half
      if constexpr (KIND == kGateUpSwiGLU) {
        // lane j < 16 holds gate feature n*64 + 16q + j, lane j + 16 its up row:
        // per token pair (2m, 2m+1) a shuffle gives the gate lane u(2m) and
        // the up lane g(2m+1); each computes one h
        const bool gate = lane < GATEUP_GROUP;
        const int64_t feat = static_cast<int64_t>(nblk) * (WROWS / 2) + q * GATEUP_GROUP + (lane & (GATEUP_GROUP - 1));
        uint32_t hp[32];  // chunk ci, pair k: h of tokens ci*32 + 4k + (0|1) + {0, 2}
        if (active) {
          const float scale = __ldg((gate ? p.scale0 : p.scale1) + static_cast<int64_t>(c.e) * p.ld_out + feat);
#pragma unroll
          for (int ci = 0; ci < 4; ++ci) {
            uint32_t v[32];
            tmem_load32(lane_addr + ci * 32, v);
            float h[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const float a0 = __uint_as_float(v[2 * m]) * scale, a1 = __uint_as_float(v[2 * m + 1]) * scale;
              const float x = __shfl_xor_sync(0xffffffffu, gate ? a1 : a0, GATEUP_GROUP);
              h[m] = gate ? silu(a0) * x : silu(x) * a1;
            }
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) hp[ci * 8 + k2] = pack_bf16x2(h[2 * k2], h[2 * k2 + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        if (active) {
          uint16_t* hcol = static_cast<uint16_t*>(p.out) + (row0 + (gate ? 0 : 1)) * p.ld_out + feat;
#pragma unroll
          for (int ci = 0; ci < 4; ++ci)
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {
              const int t = ci * 32 + 4 * k2;  // token of h[2 k2] (gate lanes; up lanes one later)
              hcol[static_cast<int64_t>(t) * p.ld_out] = static_cast<uint16_t>(hp[ci * 8 + k2] & 0xFFFFu);
              hcol[static_cast<int64_t>(t + 2) * p.ld_out] = static_cast<uint16_t>(hp[ci * 8 + k2] >> 16);
            }
        }
      } else {
        if (active) {
          const int64_t col = static_cast<int64_t>(nblk) * WROWS + q * 32 + lane;
          const float scale = __ldg(p.scale0 + static_cast<int64_t>(c.e) * p.ld_out + col);
          float* ycol = static_cast<float*>(p.out) + row0 * p.ld_out + col;
#pragma unroll 1
          for (int ci = 0; ci < 4; ++ci) {
            uint32_t v[32];
            tmem_load32(lane_addr + ci * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              ycol[static_cast<int64_t>(ci * 32 + j) * p.ld_out] = __uint_as_float(v[j]) * scale;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      }
      tphase ^= 1u;
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

int grouped_gemm_int8_tm_tile_n(GemmKind kind) { return kind == kGateUpSwiGLU ? WROWS / 2 : WROWS; }
int grouped_gemm_int8_tm_gateup_block() { return GATEUP_GROUP; }

cudaError_t grouped_gemm_int8_tm_prepare() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto fn) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  };
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWInt8, false>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWInt8, false>);
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWInt4, false>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWInt4, false>);
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWFp8, false>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWFp8, false>);
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWInt8, true>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWInt8, true>);
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWInt4, true>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWInt4, true>);
  set(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, kWFp8, true>);
  set(grouped_gemm_int8_tm_kernel<kDownF32, kWFp8, true>);
  return e;
}

template <int WF, bool WIDE>
static void launch_wf(GemmKind kind, const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_x32,
                      const GemmArgs& a, cudaStream_t s) {
  if (kind == kGateUpSwiGLU)
    launch_kernel(grouped_gemm_int8_tm_kernel<kGateUpSwiGLU, WF, WIDE>, a.grid, THREADS, SMEM_BYTES, s, tm_x, tm_w,
                  tm_x32, a);
  else
    launch_kernel(grouped_gemm_int8_tm_kernel<kDownF32, WF, WIDE>, a.grid, THREADS, SMEM_BYTES, s, tm_x, tm_w,
                  tm_x32, a);
}

template <int WF>
static void launch_w(GemmKind kind, const CUtensorMap& tm_x, const CUtensorMap& tm_w, const CUtensorMap& tm_x32,
                     const GemmArgs& a, cudaStream_t s) {
  if (a.wide)
    launch_wf<WF, true>(kind, tm_x, tm_w, tm_x32, a, s);
  else
    launch_wf<WF, false>(kind, tm_x, tm_w, tm_x32, a, s);
}

cudaError_t launch_grouped_gemm_int8_tm(GemmKind kind, WeightFormat wf, const CUtensorMap& tm_x,
                                        const CUtensorMap& tm_w, const CUtensorMap& tm_x32, const GemmArgs& a,
                                        cudaStream_t s) {
  if (a.k_blocks % (wf == kWInt4 ? 4 : 2) != 0) return cudaErrorInvalidValue;
  switch (wf) {
    case kWInt8: launch_w<kWInt8>(kind, tm_x, tm_w, tm_x32, a, s); break;
    case kWInt4: launch_w<kWInt4>(kind, tm_x, tm_w, tm_x32, a, s); break;
    case kWFp8: launch_w<kWFp8>(kind, tm_x, tm_w, tm_x32, a, s); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace cbmoe
