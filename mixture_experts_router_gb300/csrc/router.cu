// Router: fp32 logits l = x Wr^T + b fused with the top-k gate (the router
// kernel of "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2: linear projection
// then top-k; routing decided on the device with no host round trip,
// "discosf.com/news/4774337" §5.1).  Softmax is applied and renormalised
// over the k ("Colibri：面向MoE模型的高性能C语言推理引擎" §2.1); since its full
// denominator cancels, w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0).
//
// One block owns a tile of TT tokens and all E experts.  The logit GEMM runs
// on CUDA cores in fp32 (bf16 products are exact in fp32) with a per-32
// partial sum, keeping the logit error near 1e-6.  The logits stay in shared
// memory; one warp per token then takes k rounds of a warp arg-max in the
// order (number before NaN, larger first, lower index on ties).
#include <cuda_bf16.h>

#include "internal.h"

namespace cbmoe {
namespace {

constexpr int kThreads = 256;
constexpr int kDK = 32;  // d elements per shared-memory step


struct Cand {
  float v;
  int idx;
  int cls;  // 0 number, 1 NaN, 2 not available (padding or already taken)
};

__device__ __forceinline__ bool ranks_before(const Cand& a, const Cand& b) {
  if (a.cls != b.cls) return a.cls < b.cls;
  if (a.cls == 0 && a.v != b.v) return a.v > b.v;
  return a.idx < b.idx;
}

template <int EX, int TN, int TM>
struct RouterCfg {
  static constexpr int ROWS = kThreads / EX;  // thread rows over tokens
  static constexpr int TT = ROWS * TM;        // tokens per block
  static constexpr int EP = EX * TN;          // padded expert count
  static constexpr int GEMM_FLOATS = kDK * (TT + EP);
  static constexpr int LOGIT_FLOATS = TT * (EP + 1);
  static constexpr int SMEM_BYTES = 4 * (GEMM_FLOATS > LOGIT_FLOATS ? GEMM_FLOATS : LOGIT_FLOATS);
};

template <int EX, int TN, int TM>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(RouterArgs a) {
  using C = RouterCfg<EX, TN, TM>;
  constexpr int ROWS = C::ROWS, TT = C::TT, EP = C::EP;
  extern __shared__ float sm[];
  float* xs = sm;             // [kDK][TT]
  float* ws = sm + kDK * TT;  // [kDK][EP]
  const int tid = threadIdx.x;
  const int tx = tid % EX, ty = tid / EX;
  const int t0 = blockIdx.x * TT;

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < a.d; k0 += kDK) {
    for (int v = tid; v < TT * (kDK / 8); v += kThreads) {
      const int r = v / (kDK / 8), c8 = v % (kDK / 8);
      const int t = t0 + r;
      uint4 q = make_uint4(0, 0, 0, 0);
      if (t < a.T) q = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(t) * a.d + k0 + c8 * 8));
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[(c8 * 8 + 2 * j) * TT + r] = __uint_as_float(u[j] << 16);
        xs[(c8 * 8 + 2 * j + 1) * TT + r] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    }
    for (int v = tid; v < EP * (kDK / 8); v += kThreads) {
      const int e = v / (kDK / 8), c8 = v % (kDK / 8);
      uint4 q = make_uint4(0, 0, 0, 0);
      if (e < a.E) q = __ldg(reinterpret_cast<const uint4*>(a.wr + static_cast<size_t>(e) * a.d + k0 + c8 * 8));
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ws[(c8 * 8 + 2 * j) * EP + e] = __uint_as_float(u[j] << 16);
        ws[(c8 * 8 + 2 * j + 1) * EP + e] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    }
    __syncthreads();
    float part[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) part[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < kDK; ++kk) {
      float xv[TM], wv[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) xv[i] = xs[kk * TT + ty + i * ROWS];
#pragma unroll
      for (int j = 0; j < TN; ++j) wv[j] = ws[kk * EP + tx + j * EX];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) part[i][j] = fmaf(xv[i], wv[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] += part[i][j];
    __syncthreads();
  }

  float* ls = sm;  // [TT][EP + 1]
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int r = ty + i * ROWS, e = tx + j * EX;
      float v = acc[i][j];
      if (a.bias != nullptr && e < a.E) v += __ldg(a.bias + e);
      ls[r * (EP + 1) + e] = v;
    }
  __syncthreads();

  if (a.logits != nullptr) {
    for (int v = tid; v < TT * a.E; v += kThreads) {
      const int r = v / a.E, e = v % a.E, t = t0 + r;
      if (t < a.T) a.logits[static_cast<size_t>(t) * a.E + e] = ls[r * (EP + 1) + e];
    }
  }

  constexpr int PER = (EP + 31) / 32;
  const int warp = tid / 32, lane = tid % 32;
  for (int r = warp; r < TT; r += kThreads / 32) {
    const int t = t0 + r;
    if (t >= a.T) break;
    Cand c[PER];
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = lane + 32 * p;
      if (e < a.E) {
        const float v = ls[r * (EP + 1) + e];
        c[p] = Cand{v, e, isnan(v) ? 1 : 0};
      } else {
        c[p] = Cand{0.f, e, 2};
      }
    }
    float my_v = 0.f, l0 = 0.f;
    int my_i = 0;
    for (int s = 0; s < a.k; ++s) {
      Cand b = c[0];
#pragma unroll
      for (int p = 1; p < PER; ++p)
        if (ranks_before(c[p], b)) b = c[p];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        Cand o;
        o.v = __shfl_xor_sync(0xffffffffu, b.v, off);
        o.idx = __shfl_xor_sync(0xffffffffu, b.idx, off);
        o.cls = __shfl_xor_sync(0xffffffffu, b.cls, off);
        if (ranks_before(o, b)) b = o;
      }
      if ((b.idx & 31) == lane) {
#pragma unroll
        for (int p = 0; p < PER; ++p)
          if (p == (b.idx >> 5)) c[p].cls = 2;
      }
      if (s == 0) l0 = b.v;
      if (lane == s) {
        my_v = b.v;
        my_i = b.idx;
      }
    }
    const float ex = (lane < a.k) ? expf(my_v - l0) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane < a.k) {
      a.ids[static_cast<size_t>(t) * a.k + lane] = my_i;
      a.w[static_cast<size_t>(t) * a.k + lane] = ex / sum;
    }
  }
}

template <int EX, int TN, int TM>
cudaError_t launch_cfg(const RouterArgs& a, cudaStream_t s) {
  using C = RouterCfg<EX, TN, TM>;
  const int blocks = (a.T + C::TT - 1) / C::TT;
  if (blocks == 0) return cudaSuccess;
  router_topk_kernel<EX, TN, TM><<<blocks, kThreads, C::SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t router_prepare() { return cudaSuccess; }

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  if (a.E <= 8) return launch_cfg<8, 1, 1>(a, s);
  if (a.E <= 16) return launch_cfg<16, 1, 2>(a, s);
  if (a.E <= 32) return launch_cfg<16, 2, 2>(a, s);
  if (a.E <= 64) return launch_cfg<16, 4, 4>(a, s);
  if (a.E <= 128) return launch_cfg<16, 8, 4>(a, s);
  return launch_cfg<16, 16, 2>(a, s);
}

}  // namespace cbmoe
