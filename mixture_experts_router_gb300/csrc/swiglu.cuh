// SwiGLU epilogue helpers shared by the gate/up GEMM kernels:
// h = SiLU(g) * u with SiLU(z) = z / (1 + e^-z), rounded to bf16.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace cbmoe {

// SiLU from the hardware exponential and the fast divide (a few fp32 ulp,
// far below the bf16 rounding of h).  The limits stay exact: for z -> -inf
// the denominator grows past 2^126 and the quotient is 0; for z -> +inf it
// is 1 and the result z.
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

}  // namespace cbmoe
