// Router on the tcgen05 tensor cores: fp32 logits l = x Wr^T + b fused with
// the top-k gate (the router kernel of "Colibri：面向MoE架构的C语言级高效推理引擎"
// §3.2, routing decided on the device: "discosf.com/news/4774337" §5.1), with
// softmax renormalised over the k ("Colibri：面向MoE模型的高性能C语言推理引擎"
// §2.1): w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0); with raw_weights,
// w_s = l_s (no softmax, the first page's §3.2).
//
// A tile is 128 tokens; the whole expert dimension (E padded to NP, a power of
// two >= 16) is one UMMA N.  x is streamed by TMA (rows past T read as zeros),
// the router weights come by TMA too (rows past E read as zeros), and the
// K loop rotates over NACC = 512 / NP accumulators in TMEM (k-block kb adds
// into accumulator kb % NACC), so no fp32 accumulation chain in the tensor
// core is longer than ceil(d / (64 NACC)) k-blocks; the epilogue sums the
// NACC partials in a fixed order in fp32.  One epilogue thread owns one
// token: it adds the bias, keeps a sorted top-k in registers (order: number
// before NaN, larger first, lower index on ties) and writes ids and weights.
//
// Per CTA (persistent over 128-token tiles): warp 0 TMA producer, warp 1
// TMEM owner + MMA issuer, warps 2..5 epilogue.  Bounded waits as elsewhere.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

template <int NP>
struct RtCfg {
  static constexpr int NACC = 512 / NP > 32 ? 32 : 512 / NP;
  static constexpr int B_BYTES = NP * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  static constexpr int CW = NP < 32 ? NP : 32;  // epilogue column chunk
  static constexpr int STG_FLOATS = 128 * (CW + 1);  // per-row logit staging, padded
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STG_FLOATS * 4 + 1024 + 256;
};

// A candidate (logit v, expert e) as one 64-bit key whose unsigned order is
// the routing order: numbers by value (larger first; -0 folded into +0 so
// the two zeros tie), then NaN, then an empty slot (key 0); on equal values
// the lower expert index has the larger key.
__device__ __forceinline__ uint64_t rank_key(float v, int e) {
  uint32_t hi;
  if (isnan(v)) {
    hi = 1u;
  } else {
    const uint32_t b = __float_as_uint(v + 0.0f);
    hi = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    hi = hi < 2u ? 2u : hi;  // stay above NaN and empty (only -inf maps below)
  }
  return (static_cast<uint64_t>(hi) << 32) | static_cast<uint32_t>(~static_cast<uint32_t>(e));
}

template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32)
    tmem_load32(taddr, r);
  else
    tmem_load16(taddr, r);
}

template <int NP, int KMAX>
__global__ void __launch_bounds__(THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const RouterArgs a, const uint64_t wait_limit_ns) {
  using C = RtCfg<NP>;
  constexpr int STAGES = C::STAGES, NACC = C::NACC, CW = C::CW;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, NP);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);  // [128][CW + 1]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::STG_FLOATS * 4);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 128);
    fence_barrier_init();
    prefetch_tensormap(&tm_x);
    prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tiles = (a.T + BM - 1) / BM;
  const int kblocks = a.d / BK;
  const int nacc = kblocks < NACC ? kblocks : NACC;

  if (warp == 0) {
    if (lane == 0) {
      int64_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        for (int kb = 0; kb < kblocks; ++kb) {
          const int stage = static_cast<int>(issued % STAGES);
          const uint32_t phase = static_cast<uint32_t>((issued / STAGES) & 1);
          if (!mbar_wait(&empty[stage], phase ^ 1u, wait_limit_ns)) {
            set_error(a.err, kErrTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
          tma_load_2d(st, &tm_x, &full[stage], kb * BK, tile * BM);
          tma_load_2d(st + A_BYTES, &tm_w, &full[stage], kb * BK, 0);
          ++issued;
        }
      }
      for (int64_t i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        if (!mbar_wait(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), wait_limit_ns))
          set_error(a.err, kErrTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, tphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        if (!mbar_wait(tempty, tphase ^ 1u, wait_limit_ns)) {
          set_error(a.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, wait_limit_ns)) {
            set_error(a.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t adesc = sw128_desc(st), bdesc = sw128_desc(st + A_BYTES);
          const uint32_t d = tmem_base + static_cast<uint32_t>((kb % NACC) * NP);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_f16(d, adesc + 2 * k, bdesc + 2 * k, IDESC, (kb >= NACC || k > 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull);
        tphase ^= 1u;
      }
    }
  } else {
    const int q = warp & 3;
    uint32_t tphase = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      if (!mbar_wait(tfull, tphase, wait_limit_ns)) {
        set_error(a.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const int t = tile * BM + q * 32 + lane;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      uint64_t top[KMAX];   // sorted, best first
      float topv[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        top[j] = 0;
        topv[j] = 0.f;
      }
      uint64_t thr = 0;  // key of the k-th best so far
      float* my = stg + (q * 32 + lane) * (CW + 1);
      for (int c0 = 0; c0 < NP; c0 += CW) {
        if (c0 >= a.E) break;  // uniform across the warp
        float sum[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) sum[j] = 0.f;
        for (int acc = 0; acc < nacc; ++acc) {
          uint32_t r[CW];
          tmem_load_cols<CW>(tb + static_cast<uint32_t>(acc * NP + c0), r);
#pragma unroll
          for (int j = 0; j < CW; ++j) sum[j] += __uint_as_float(r[j]);
        }
        if (a.bias != nullptr) {
#pragma unroll
          for (int j = 0; j < CW; ++j)
            if (c0 + j < a.E) sum[j] += __ldg(a.bias + c0 + j);
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) my[j] = sum[j];
        __syncwarp();
        const int nj = a.E - c0 < CW ? a.E - c0 : CW;
#pragma unroll 4
        for (int j = 0; j < nj; ++j) {
          const int e = c0 + j;
          const float v = my[j];
          if (a.logits != nullptr && t < a.T) a.logits[static_cast<int64_t>(t) * a.E + e] = v;
          uint64_t key = rank_key(v, e);
          if (key > thr) {
            float kv = v;
#pragma unroll
            for (int s2 = 0; s2 < KMAX; ++s2) {
              const bool better = s2 < a.k && key > top[s2];
              const uint64_t tk = top[s2];
              const float tv = topv[s2];
              top[s2] = better ? key : tk;
              topv[s2] = better ? kv : tv;
              key = better ? tk : key;
              kv = better ? tv : kv;
            }
#pragma unroll
            for (int s2 = 0; s2 < KMAX; ++s2)
              if (s2 == a.k - 1) thr = top[s2];
          }
        }
        __syncwarp();
      }
      if (t < a.T) {
        const float l0 = topv[0];
        float ex[KMAX];
        float den = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < KMAX; ++s2) {
          ex[s2] = (s2 < a.k) ? expf(topv[s2] - l0) : 0.f;
          den += ex[s2];
        }
#pragma unroll
        for (int s2 = 0; s2 < KMAX; ++s2) {
          if (s2 < a.k) {
            a.ids[static_cast<int64_t>(t) * a.k + s2] = static_cast<int>(~static_cast<uint32_t>(top[s2]));
            a.w[static_cast<int64_t>(t) * a.k + s2] = a.raw_weights ? topv[s2] : ex[s2] / den;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
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

template <int NP, int KMAX>
cudaError_t launch_np(const CUtensorMap& tx, const CUtensorMap& tw, const RouterArgs& a, int grid,
                      cudaStream_t s) {
  router_tc_kernel<NP, KMAX><<<grid, THREADS, RtCfg<NP>::SMEM_BYTES, s>>>(tx, tw, a, kWaitLimitNs);
  return cudaGetLastError();
}

template <int NP>
cudaError_t launch_k(const CUtensorMap& tx, const CUtensorMap& tw, const RouterArgs& a, int grid, cudaStream_t s) {
  if (a.k <= 2) return launch_np<NP, 2>(tx, tw, a, grid, s);
  if (a.k <= 4) return launch_np<NP, 4>(tx, tw, a, grid, s);
  if (a.k <= 8) return launch_np<NP, 8>(tx, tw, a, grid, s);
  return launch_np<NP, 16>(tx, tw, a, grid, s);
}

template <int NP>
cudaError_t prepare_np() {
  cudaError_t e = cudaSuccess;
  auto set = [&](auto fn) {
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, RtCfg<NP>::SMEM_BYTES);
  };
  set(router_tc_kernel<NP, 2>);
  set(router_tc_kernel<NP, 4>);
  set(router_tc_kernel<NP, 8>);
  set(router_tc_kernel<NP, 16>);
  return e;
}

}  // namespace

int router_tc_rows(int E) {
  int np = 16;
  while (np < E) np *= 2;
  return np;
}

cudaError_t router_tc_prepare() {
  cudaError_t e = prepare_np<16>();
  if (e == cudaSuccess) e = prepare_np<32>();
  if (e == cudaSuccess) e = prepare_np<64>();
  if (e == cudaSuccess) e = prepare_np<128>();
  if (e == cudaSuccess) e = prepare_np<256>();
  return e;
}

cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a, int num_sms,
                             cudaStream_t s) {
  const int tiles = (a.T + BM - 1) / BM;
  if (tiles == 0) return cudaSuccess;
  const int grid = tiles < num_sms ? tiles : num_sms;
  switch (router_tc_rows(a.E)) {
    case 16: return launch_k<16>(tm_x, tm_w, a, grid, s);
    case 32: return launch_k<32>(tm_x, tm_w, a, grid, s);
    case 64: return launch_k<64>(tm_x, tm_w, a, grid, s);
    case 128: return launch_k<128>(tm_x, tm_w, a, grid, s);
    default: return launch_k<256>(tm_x, tm_w, a, grid, s);
  }
}

}  // namespace cbmoe
