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
// A block takes 32 tokens; thread (token tl, dimension i) keeps one float
// sum.  The tokens' rows of x and W_h are staged through shared memory 256
// elements at a time (W_h transposed, so the 8 dimensions of one element are
// 16 contiguous bytes), and every thread adds its products in increasing
// element order with separate multiply and add, so the order and the
// roundings are exactly those of the definition.  The 8 threads of a token
// are 8 consecutive lanes; their hashes are XOR-ed with lane shuffles.
#include <cuda_bf16.h>

#include "internal.h"

namespace cbmoe {
namespace {

constexpr int kHashTokens = 32;
constexpr int kHashDimsMax = 8;
constexpr int kHashThreads = kHashTokens * kHashDimsMax;
constexpr int kChunk = 256;               // elements of d per staging round
constexpr int kXStride = kChunk + 8;      // bf16 per staged row (16-byte rows, spread banks)

__device__ __forceinline__ float bf16_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__global__ void __launch_bounds__(kHashThreads) router_hash_kernel(HashRouterArgs a) {
  __shared__ __align__(16) uint16_t xs[kHashTokens * kXStride];
  __shared__ __align__(16) uint16_t whs[kChunk * kHashDimsMax];
  const int tid = threadIdx.x;
  const int tl = tid / kHashDimsMax, dim = tid % kHashDimsMax;
  const int t0 = blockIdx.x * kHashTokens;
  float r = 0.0f;
  for (int c0 = 0; c0 < a.d; c0 += kChunk) {
    // x rows of the block's tokens (rows past T are zeros), 16-byte vectors
    for (int v = tid; v < kHashTokens * kChunk / 8; v += kHashThreads) {
      const int row = v / (kChunk / 8), col = (v % (kChunk / 8)) * 8;
      const int t = t0 + row;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (t < a.T) val = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<int64_t>(t) * a.d + c0 + col));
      *reinterpret_cast<uint4*>(xs + row * kXStride + col) = val;
    }
    // W_h transposed: whs[j][i] = W_h[i][c0 + j] (zero for i >= hash_dims)
    for (int e = tid; e < kChunk * kHashDimsMax; e += kHashThreads) {
      const int j = e / kHashDimsMax, i = e % kHashDimsMax;
      whs[e] = i < a.hash_dims ? a.wh[static_cast<int64_t>(i) * a.d + c0 + j] : static_cast<uint16_t>(0);
    }
    __syncthreads();
    const uint16_t* xr = xs + tl * kXStride;
#pragma unroll 8
    for (int j = 0; j < kChunk; ++j) r = __fadd_rn(r, __fmul_rn(bf16_to_float(xr[j]), bf16_to_float(whs[j * kHashDimsMax + dim])));
    __syncthreads();
  }
  uint32_t h = 0;
  if (dim < a.hash_dims) h = static_cast<uint32_t>(__double2int_rz(__dmul_rn(static_cast<double>(r), 1e6))) & 0xFFFFFu;
  h ^= __shfl_xor_sync(0xffffffffu, h, 4);
  h ^= __shfl_xor_sync(0xffffffffu, h, 2);
  h ^= __shfl_xor_sync(0xffffffffu, h, 1);
  const int t = t0 + tl;
  if (dim == 0 && t < a.T) {
    a.ids[t] = static_cast<int32_t>(h % static_cast<uint32_t>(a.E));
    a.w[t] = 1.0f;
  }
}

}  // namespace

cudaError_t launch_router_hash(const HashRouterArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  if (a.hash_dims < 1 || a.hash_dims > kHashDimsMax || a.d % kChunk != 0) return cudaErrorInvalidValue;
  router_hash_kernel<<<(a.T + kHashTokens - 1) / kHashTokens, kHashThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace cbmoe
