// Combine: out[t] = sum_s w[t][s] * Y[row(t, s)], the weighted sum of the k
// expert outputs by gating score (the combine kernel of
// "Colibri：面向MoE架构的C语言级高效推理引擎" §2.3).  Y is fp32; the sum is fp32
// FMA in slot order, rounded once to bf16 (or stored as fp32).
//
// One block per token: the k padded row indices are resolved once into
// shared memory (row = tile_base(e) + (inv - offset(e))), then each thread
// streams 8 columns at a time with 16-byte loads from the k rows.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxK = 16;

template <bool F32OUT>
__global__ void __launch_bounds__(kThreads) combine_kernel(CombineArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ int64_t rows[kMaxK];
  __shared__ float ws[kMaxK];
  const int t = blockIdx.x;
  if (threadIdx.x < a.k) {
    const int s = threadIdx.x;
    const int e = a.ids[static_cast<int64_t>(t) * a.k + s];
    const int r = a.inv[static_cast<int64_t>(t) * a.k + s];
    rows[s] = static_cast<int64_t>(a.mtile_off[e]) * kTileM + (r - a.offsets[e]);
    ws[s] = a.w[static_cast<int64_t>(t) * a.k + s];
  }
  __syncthreads();
  const int nvec = a.d / 8;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int s = 0; s < a.k; ++s) {
      const float4* src = reinterpret_cast<const float4*>(a.y + rows[s] * a.d) + 2 * v;
      const float4 p = __ldg(src), q = __ldg(src + 1);
      const float wv = ws[s];
      acc[0] = fmaf(wv, p.x, acc[0]);
      acc[1] = fmaf(wv, p.y, acc[1]);
      acc[2] = fmaf(wv, p.z, acc[2]);
      acc[3] = fmaf(wv, p.w, acc[3]);
      acc[4] = fmaf(wv, q.x, acc[4]);
      acc[5] = fmaf(wv, q.y, acc[5]);
      acc[6] = fmaf(wv, q.z, acc[6]);
      acc[7] = fmaf(wv, q.w, acc[7]);
    }
    if constexpr (F32OUT) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + static_cast<int64_t>(t) * a.d) + 2 * v;
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint4 o;
      __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6], acc[7]);
      o.x = *reinterpret_cast<uint32_t*>(&b0);
      o.y = *reinterpret_cast<uint32_t*>(&b1);
      o.z = *reinterpret_cast<uint32_t*>(&b2);
      o.w = *reinterpret_cast<uint32_t*>(&b3);
      reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + static_cast<int64_t>(t) * a.d)[v] = o;
    }
  }
}

// The combine fused into the down GEMM leaves each token's fp32 sum in acc;
// this pass rounds it once to bf16 (or copies it out as fp32).
template <bool F32OUT>
__global__ void __launch_bounds__(kThreads) combine_acc_kernel(const float* __restrict__ acc, int64_t n8, void* out) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t v = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; v < n8; v += stride) {
    const float4 p = __ldg(reinterpret_cast<const float4*>(acc) + 2 * v);
    const float4 q = __ldg(reinterpret_cast<const float4*>(acc) + 2 * v + 1);
    if constexpr (F32OUT) {
      reinterpret_cast<float4*>(out)[2 * v] = p;
      reinterpret_cast<float4*>(out)[2 * v + 1] = q;
    } else {
      __nv_bfloat162 b0 = __floats2bfloat162_rn(p.x, p.y);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(p.z, p.w);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(q.x, q.y);
      __nv_bfloat162 b3 = __floats2bfloat162_rn(q.z, q.w);
      uint4 o;
      o.x = *reinterpret_cast<uint32_t*>(&b0);
      o.y = *reinterpret_cast<uint32_t*>(&b1);
      o.z = *reinterpret_cast<uint32_t*>(&b2);
      o.w = *reinterpret_cast<uint32_t*>(&b3);
      reinterpret_cast<uint4*>(out)[v] = o;
    }
  }
}

}  // namespace

cudaError_t launch_combine_acc(const float* acc, int64_t n_elems, void* out, int out_f32, int grid, cudaStream_t s) {
  const int64_t n8 = n_elems / 8;
  if (n8 <= 0) return cudaSuccess;
  const int64_t need = (n8 + kThreads - 1) / kThreads;
  const int g = static_cast<int>(need < grid ? need : grid);
  if (out_f32)
    launch_kernel(combine_acc_kernel<true>, g, kThreads, 0, s, acc, n8, out);
  else
    launch_kernel(combine_acc_kernel<false>, g, kThreads, 0, s, acc, n8, out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.out_f32)
    launch_kernel(combine_kernel<true>, a.T, kThreads, 0, s, a);
  else
    launch_kernel(combine_kernel<false>, a.T, kThreads, 0, s, a);
  return cudaGetLastError();
}

}  // namespace cbmoe
