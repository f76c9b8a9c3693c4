// Router on the tcgen05 tensor cores for wide expert counts: fp32 logits
// l = x Wr^T + b and the top-k gate (the router kernel of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2, routing decided on the device:
// "discosf.com/news/4774337" §5.1), with softmax renormalised over the k
// ("Colibri：面向MoE模型的高性能C语言推理引擎" §2.1):
// w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0); with raw_weights, w_s = l_s
// (no softmax, the first page's §3.2).
//
// Two kernels:
//
// router_tc_part_kernel: a unit is 128 tokens x one of KS slices of the
// model dimension, so a layer of few 128-token tiles still fills the GPU
// (KS units per tile).  The expert dimension (E padded to
// NP, a power of two >= 16) is one UMMA N.  x and the router weights are
// streamed by TMA (rows past T or E read as zeros); the K loop rotates over
// NACC = 256 / NP accumulators in TMEM, so no fp32 accumulation chain in
// the tensor core is longer than ceil(d / (64 KS NACC)) k-blocks.  The
// epilogue sums the NACC accumulators in a fixed order and writes the
// unit's partial logits part[ks][t][0..NP) with coalesced stores.
//
// router_topk_kernel: one warp per token sums the KS partials in slice order,
// adds the bias, optionally writes the logits, and takes the top k by k
// rounds of a warp-wide maximum (number before NaN, larger first, lower
// index on ties), then the weights.
//
// Bounded waits as elsewhere.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 256;

// Two CTAs share an SM (256 TMEM columns and at most 113 KB of shared memory
// each) for NP <= 64; from NP = 128 a stage is 32 KB or more and one CTA per
// SM with up to six stages in flight measured faster (skewed 128-expert
// layer: 25.6 vs 26.6 us for the router stage).
template <int NP>
struct RtCfg {
  static constexpr int NACC = 256 / NP;
  static constexpr int CTAS_PER_SM = NP >= 128 ? 1 : 2;
  static constexpr int B_BYTES = NP * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int CW = NP < 32 ? NP : 32;     // epilogue column chunk
  static constexpr int STG_FLOATS = 4 * 32 * 33;   // per-warp 32 x 32 transpose buffer, padded
  static constexpr int FIXED = STG_FLOATS * 4 + 1024 + 256;
  static constexpr int BUDGET = (CTAS_PER_SM == 2 ? 113 * 1024 : 200 * 1024) - FIXED;
  static constexpr int STAGES_RAW = BUDGET / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + FIXED;
  static_assert(STAGES >= 2, "router stages");
};

template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t (&r)[CW]) {
  if constexpr (CW == 32)
    tmem_load32(taddr, r);
  else
    tmem_load16(taddr, r);
}

struct PartArgs {
  int32_t T, d, E;
  int32_t ks;          // slices of the model dimension
  int32_t t_pad;       // rows of each slice's partial block (tiles * 128)
  float* part;         // [ks][t_pad][NP]
  int* err;
};

template <int NP>
__global__ void __launch_bounds__(THREADS, 2)
    router_tc_part_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                          const PartArgs a, const uint64_t wait_limit_ns) {
  using C = RtCfg<NP>;
  constexpr int STAGES = C::STAGES, NACC = C::NACC, CW = C::CW;
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, NP);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES);  // [4 warps][32][33]
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
    mbar_init(tempty, 4);
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
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  const int n_tiles = (a.T + BM - 1) / BM;
  const int n_units = n_tiles * a.ks;
  const int kblocks = a.d / BK;
  // unit u: tile u / ks, k-blocks [kb_lo, kb_hi) of slice u % ks
  auto k_range = [&](int u, int& lo, int& hi) {
    const int sl = u % a.ks;
    lo = sl * kblocks / a.ks;
    hi = (sl + 1) * kblocks / a.ks;
  };

  if (warp == 0) {
    if (lane == 0) {
      int64_t issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        int lo, hi;
        k_range(u, lo, hi);
        const int tile = u / a.ks;
        for (int kb = lo; kb < hi; ++kb) {
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
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        int lo, hi;
        k_range(u, lo, hi);
        if (!mbar_wait(tempty, tphase ^ 1u, wait_limit_ns)) {
          set_error(a.err, kErrTimeout);
          break;
        }
        tc_fence_after();
        for (int kb = lo; kb < hi; ++kb) {
          if (!mbar_wait(&full[stage], phase, wait_limit_ns)) {
            set_error(a.err, kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t adesc = sw128_desc(st), bdesc = sw128_desc(st + A_BYTES);
          const int j = kb - lo;
          const uint32_t d = tmem_base + static_cast<uint32_t>((j % NACC) * NP);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_f16(d, adesc + 2 * k, bdesc + 2 * k, IDESC, (j >= NACC || k > 0) ? 1u : 0u);
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
    // epilogue: warp q reads TMEM lanes 32q.. (tokens), sums the accumulators
    // of each 32-column chunk in a fixed order, transposes the 32 x 32 block
    // through shared memory and writes each token's 32 logits as one
    // 128-byte row segment
    const int q = warp & 3;
    float* tb32 = stg + q * 32 * 33;
    uint32_t tphase = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      int lo, hi;
      k_range(u, lo, hi);
      const int nacc = hi - lo < NACC ? hi - lo : NACC;
      if (!mbar_wait(tfull, tphase, wait_limit_ns)) {
        set_error(a.err, kErrTimeout);
        break;
      }
      tc_fence_after();
      const int tile = u / a.ks, sl = u % a.ks;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      float* dst = a.part + (static_cast<int64_t>(sl) * a.t_pad + tile * BM + q * 32) * NP;
      for (int c0 = 0; c0 < NP; c0 += CW) {
        float sum[CW];
#pragma unroll
        for (int j = 0; j < CW; ++j) sum[j] = 0.f;
        for (int acc = 0; acc < nacc; ++acc) {
          uint32_t r[CW];
          tmem_load_cols<CW>(tb + static_cast<uint32_t>(acc * NP + c0), r);
#pragma unroll
          for (int j = 0; j < CW; ++j) sum[j] += __uint_as_float(r[j]);
        }
#pragma unroll
        for (int j = 0; j < CW; ++j) tb32[lane * 33 + j] = sum[j];
        __syncwarp();
        if (lane < CW) {
#pragma unroll 4
          for (int i = 0; i < 32; ++i) dst[static_cast<int64_t>(i) * NP + c0 + lane] = tb32[i * 33 + lane];
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
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

// Order of a logit as an unsigned key: numbers by value (larger first; -0
// folded into +0 so the two zeros tie), then NaN; 0 marks an empty or taken
// candidate.  Ties between experts go to the lower index.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (isnan(v)) return 1u;
  const uint32_t b = __float_as_uint(v + 0.0f);
  const uint32_t h = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return h < 2u ? 2u : h;  // stay above NaN and empty (only -inf maps below)
}

// One warp per token: lane l owns experts l, l + 32, ... (NPL of them).  Each
// of the k rounds takes the warp's largest order key (a hardware warp
// reduction), then the lowest expert index among the lanes holding it.
template <int NPL, int KMAX>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ part, int ks, int t_pad, int np,
                                                          const RouterArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  const int lane = threadIdx.x % 32;
  const int t = blockIdx.x * 8 + threadIdx.x / 32;
  if (t >= a.T) return;
  float p[NPL][kRouterMaxSlices];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    const float* src = part + static_cast<int64_t>(t) * np + e;
#pragma unroll
    for (int sl = 0; sl < kRouterMaxSlices; ++sl)
      p[j][sl] = (e < a.E && sl < ks) ? __ldg(src + static_cast<int64_t>(sl) * t_pad * np) : 0.f;
  }
  float v[NPL];
  uint32_t key[NPL];
#pragma unroll
  for (int j = 0; j < NPL; ++j) {
    const int e = lane + 32 * j;
    float l = p[j][0];
#pragma unroll
    for (int sl = 1; sl < kRouterMaxSlices; ++sl)
      if (sl < ks) l += p[j][sl];
    if (e < a.E) {
      if (a.bias != nullptr) l += __ldg(a.bias + e);
      if (a.logits != nullptr) a.logits[static_cast<int64_t>(t) * a.E + e] = l;
    }
    v[j] = l;
    key[j] = e < a.E ? order_key(l) : 0u;
  }
  float topv[KMAX];
  int topi[KMAX];
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    topv[s] = 0.f;
    topi[s] = 0;
    if (s < a.k) {
      uint32_t bk = key[0];
      int bj = 0;
      float bv = v[0];
#pragma unroll
      for (int j = 1; j < NPL; ++j)
        if (key[j] > bk) {  // strictly larger: the lower index keeps a tie
          bk = key[j];
          bj = j;
          bv = v[j];
        }
      const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t we = __reduce_min_sync(0xffffffffu, bk == wk ? static_cast<uint32_t>(lane + 32 * bj) : ~0u);
      const int owner = static_cast<int>(we & 31u);
      topv[s] = __shfl_sync(0xffffffffu, bv, owner);
      topi[s] = static_cast<int>(we);
      if (lane == owner) {
#pragma unroll
        for (int j = 0; j < NPL; ++j)
          if (j == bj) key[j] = 0u;
      }
    }
  }
  const float l0 = topv[0];
  float ex[KMAX];
  float den = 0.f;
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    ex[s] = (s < a.k) ? expf(topv[s] - l0) : 0.f;
    den += ex[s];
  }
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    if (s < a.k && lane == s) {
      a.ids[static_cast<int64_t>(t) * a.k + s] = topi[s];
      a.w[static_cast<int64_t>(t) * a.k + s] = a.raw_weights ? topv[s] : ex[s] / den;
    }
  }
}

template <int NP>
cudaError_t launch_np(const CUtensorMap& tx, const CUtensorMap& tw, const RouterArgs& a, int ks, int t_pad,
                      float* part, int num_sms, cudaStream_t s) {
  PartArgs pa{a.T, a.d, a.E, ks, t_pad, part, a.err};
  const int units = (a.T + BM - 1) / BM * ks;
  const int slots = RtCfg<NP>::CTAS_PER_SM * num_sms;
  const int grid = units < slots ? units : slots;
  launch_kernel(router_tc_part_kernel<NP>, grid, THREADS, RtCfg<NP>::SMEM_BYTES, s, tx, tw, pa, kWaitLimitNs);
  constexpr int NPL = NP < 32 ? 1 : NP / 32;
  const int blocks = (a.T + 7) / 8;
  if (a.k <= 2)
    launch_kernel(router_topk_kernel<NPL, 2>, blocks, 256, 0, s, part, ks, t_pad, NP, a);
  else if (a.k <= 4)
    launch_kernel(router_topk_kernel<NPL, 4>, blocks, 256, 0, s, part, ks, t_pad, NP, a);
  else if (a.k <= 8)
    launch_kernel(router_topk_kernel<NPL, 8>, blocks, 256, 0, s, part, ks, t_pad, NP, a);
  else
    launch_kernel(router_topk_kernel<NPL, 16>, blocks, 256, 0, s, part, ks, t_pad, NP, a);
  return cudaGetLastError();
}

template <int NP>
cudaError_t prepare_np() {
  return cudaFuncSetAttribute(router_tc_part_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              RtCfg<NP>::SMEM_BYTES);
}

}  // namespace

int router_tc_rows(int E) {
  int np = 16;
  while (np < E) np *= 2;
  return np;
}

int router_tc_slices(int T, int d, int E, int num_sms) {
  const int tiles = (T + BM - 1) / BM;
  if (tiles == 0) return 1;
  const int slots = (router_tc_rows(E) >= 128 ? 1 : 2) * num_sms;
  int ks = (slots + tiles / 2) / tiles;
  const int kblocks = d / BK;
  if (ks > kRouterMaxSlices) ks = kRouterMaxSlices;
  if (ks > kblocks) ks = kblocks;
  return ks < 1 ? 1 : ks;
}

cudaError_t router_tc_prepare() {
  cudaError_t e = prepare_np<16>();
  if (e == cudaSuccess) e = prepare_np<32>();
  if (e == cudaSuccess) e = prepare_np<64>();
  if (e == cudaSuccess) e = prepare_np<128>();
  if (e == cudaSuccess) e = prepare_np<256>();
  return e;
}

cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a, float* part,
                             int num_sms, cudaStream_t s) {
  const int tiles = (a.T + BM - 1) / BM;
  if (tiles == 0) return cudaSuccess;
  const int ks = router_tc_slices(a.T, a.d, a.E, num_sms);
  const int t_pad = tiles * BM;
  switch (router_tc_rows(a.E)) {
    case 16: return launch_np<16>(tm_x, tm_w, a, ks, t_pad, part, num_sms, s);
    case 32: return launch_np<32>(tm_x, tm_w, a, ks, t_pad, part, num_sms, s);
    case 64: return launch_np<64>(tm_x, tm_w, a, ks, t_pad, part, num_sms, s);
    case 128: return launch_np<128>(tm_x, tm_w, a, ks, t_pad, part, num_sms, s);
    default: return launch_np<256>(tm_x, tm_w, a, ks, t_pad, part, num_sms, s);
  }
}

}  // namespace cbmoe
