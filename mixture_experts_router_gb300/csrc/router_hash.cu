// Hash router ("lshu.cn/news/53496" §2): a light projection r = x W_h of
// each token to hash_dims (<= 8) values, each mapped to a 20-bit integer
// h_i = (int32)(r_i * 1e6) & 0xFFFFF, and the token's single expert
// (h_0 ^ h_1 ^ ...) mod E with weight 1.  The routing is a pure function of
// the token, so it is reproduced bit for bit: the page's expression is C on a
// float routing vector, so r_i is a float sum taken left to right over d of
// the bf16 products (exact in float), r_i * 1e6 is a double product (exact),
// and the conversion truncates toward zero, saturating at the int32 range
// (NaN -> 0), which is what cvt.rzi.s32.f64 does.
//
// The left-to-right order makes each r_i one chain of d dependent float adds.
// A block takes 16 tokens; a thread keeps the sums of two dimensions of one
// token (two independent chains sharing each x value).  W_h is kept in fp32
// (widened exactly at set-up).  The block's rows of x and the hash_dims rows
// of W_h arrive 128 elements at a time by cp.async into a ring of 5 buffers
// (rows past T zero-filled), 4 chunks in flight while one is summed.  Every
// thread adds its products in increasing element order, loading each 32
// elements before their adds; a product of two bf16 values is exact in
// float, so a fused multiply-add rounds once, like the add alone.  The 4
// threads of a token are 4 consecutive lanes; their hashes are XOR-ed with
// shuffles.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace cbmoe {
namespace {

constexpr int kHashTokens = 16;
constexpr int kHashDimsMax = 8;
constexpr int kDimsPerThread = 2;                       // independent sums per thread
constexpr int kLanesPerToken = kHashDimsMax / kDimsPerThread;
constexpr int kHashThreads = kHashTokens * kLanesPerToken;
constexpr int kChunk = 128;            // elements of d per staging round
constexpr int kStages = 5;             // staging buffers: 4 chunks in flight
constexpr int kXStride = kChunk + 8;   // bf16 per staged row (16-byte rows, spread banks)
constexpr int kXBuf = kHashTokens * kXStride;   // bf16
constexpr int kWStride = kChunk + 4;             // fp32 per staged W_h row (spread banks)
constexpr int kWBuf = kHashDimsMax * kWStride;   // fp32
static_assert(kStages * (kWBuf * 4 + kXBuf * 2) <= 48 * 1024, "static shared memory");

__device__ __forceinline__ float bf16_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// 16-byte global -> shared copy; src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void stage_chunk(const HashRouterArgs& a, int t0, int c0, uint16_t* xs, float* ws) {
  for (int v = threadIdx.x; v < kHashTokens * kChunk / 8; v += kHashThreads) {
    const int row = v / (kChunk / 8), col = (v % (kChunk / 8)) * 8;
    const int t = t0 + row;
    const uint16_t* src = a.x + static_cast<int64_t>(t < a.T ? t : 0) * a.d + c0 + col;
    cp_async16(xs + row * kXStride + col, src, t < a.T ? 16 : 0);
  }
  for (int v = threadIdx.x; v < a.hash_dims * kChunk / 4; v += kHashThreads) {
    const int row = v / (kChunk / 4), col = (v % (kChunk / 4)) * 4;
    cp_async16(ws + row * kWStride + col, a.wh + static_cast<int64_t>(row) * a.d + c0 + col, 16);
  }
}

__global__ void __launch_bounds__(kHashThreads) router_hash_kernel(HashRouterArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  __shared__ __align__(16) float ws[kStages][kWBuf];
  __shared__ __align__(16) uint16_t xs[kStages][kXBuf];
  const int tl = threadIdx.x / kLanesPerToken;
  const int dim0 = (threadIdx.x % kLanesPerToken) * kDimsPerThread;  // this thread's dims: dim0, dim0 + 1
  const int t0 = blockIdx.x * kHashTokens;
  const int n_chunks = a.d / kChunk;
  float r0 = 0.0f, r1 = 0.0f;
  // one cp.async group per chunk (empty past the last chunk), so that after
  // committing chunk c + kStages - 1, waiting until kStages - 1 groups are
  // pending means chunk c has landed
  for (int c = 0; c < kStages - 1; ++c) {
    if (c < n_chunks) stage_chunk(a, t0, c * kChunk, xs[c], ws[c]);
    cp_async_commit();
  }
  for (int c = 0; c < n_chunks; ++c) {
    const int ahead = c + kStages - 1;
    if (ahead < n_chunks) stage_chunk(a, t0, ahead * kChunk, xs[ahead % kStages], ws[ahead % kStages]);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const uint16_t* xr = xs[c % kStages] + tl * kXStride;
    const float* w0 = ws[c % kStages] + dim0 * kWStride;
    const float* w1 = w0 + kWStride;
    // 32 elements at a time: all loads first (16-byte vectors of x and of this
    // thread's W_h row), then the 32 dependent adds.  A product of two bf16
    // values is exact in float, so the fused multiply-add rounds once, like
    // the add alone: the same result as the separate multiply and add.
#pragma unroll 1
    for (int j0 = 0; j0 < kChunk; j0 += 32) {
      float xv[32], wv0[32], wv1[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(xr + j0 + 8 * q);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          xv[8 * q + 2 * p] = __uint_as_float(u[p] << 16);
          xv[8 * q + 2 * p + 1] = __uint_as_float(u[p] & 0xFFFF0000u);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 a0 = *reinterpret_cast<const float4*>(w0 + j0 + 4 * q);
        const float4 a1 = *reinterpret_cast<const float4*>(w1 + j0 + 4 * q);
        wv0[4 * q] = a0.x;
        wv0[4 * q + 1] = a0.y;
        wv0[4 * q + 2] = a0.z;
        wv0[4 * q + 3] = a0.w;
        wv1[4 * q] = a1.x;
        wv1[4 * q + 1] = a1.y;
        wv1[4 * q + 2] = a1.z;
        wv1[4 * q + 3] = a1.w;
      }
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        r0 = __fmaf_rn(xv[q], wv0[q], r0);
        r1 = __fmaf_rn(xv[q], wv1[q], r1);
      }
    }
    __syncthreads();
  }
  uint32_t h = 0;
  if (dim0 < a.hash_dims) h = static_cast<uint32_t>(__double2int_rz(__dmul_rn(static_cast<double>(r0), 1e6))) & 0xFFFFFu;
  if (dim0 + 1 < a.hash_dims)
    h ^= static_cast<uint32_t>(__double2int_rz(__dmul_rn(static_cast<double>(r1), 1e6))) & 0xFFFFFu;
  h ^= __shfl_xor_sync(0xffffffffu, h, 2);
  h ^= __shfl_xor_sync(0xffffffffu, h, 1);
  const int t = t0 + tl;
  if (dim0 == 0 && t < a.T) {
    a.ids[t] = static_cast<int32_t>(h % static_cast<uint32_t>(a.E));
    a.w[t] = 1.0f;
  }
}

// bf16 -> fp32, exactly
__global__ void widen_bf16(const uint16_t* src, int64_t n, float* dst) {
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[e] = bf16_to_float(src[e]);
}

}  // namespace

cudaError_t prepare_hash_weights(const uint16_t* wh, int hash_dims, int d, float* wh_f32, cudaStream_t s) {
  if (hash_dims < 1 || hash_dims > kHashDimsMax) return cudaErrorInvalidValue;
  launch_kernel(widen_bf16, 64, 256, 0, s, wh, static_cast<int64_t>(hash_dims) * d, wh_f32);
  return cudaGetLastError();
}

cudaError_t launch_router_hash(const HashRouterArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.hash_dims < 1 || a.hash_dims > kHashDimsMax || a.d % kChunk != 0) return cudaErrorInvalidValue;
  launch_kernel(router_hash_kernel, (a.T + kHashTokens - 1) / kHashTokens, kHashThreads, 0, s, a);
  return cudaGetLastError();
}

}  // namespace cbmoe
