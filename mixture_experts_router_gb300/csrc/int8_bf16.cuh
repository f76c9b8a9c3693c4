// Exact int8 -> bf16 conversion of staged weight codes, shared by the int8
// grouped GEMM kernels.
#pragma once
#include <cstdint>

namespace cbmoe {

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

// 16 staged int8 codes (K elements 16c..16c+15 of a weight row) -> the two
// 16-byte bf16 chunks 2c and 2c+1 of that row in a 128-byte-swizzled K-major
// tile (row r at r * 128, chunk i at 16 * (i ^ (r & 7))).
__device__ __forceinline__ void convert_chunk16(const uint8_t* src, uint8_t* tile, int r, int c) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  uint4 o0, o1;
  int8x4_to_bf16x4(w.x, o0.x, o0.y);
  int8x4_to_bf16x4(w.y, o0.z, o0.w);
  int8x4_to_bf16x4(w.z, o1.x, o1.y);
  int8x4_to_bf16x4(w.w, o1.z, o1.w);
  uint8_t* row = tile + r * 128;
  *reinterpret_cast<uint4*>(row + 16 * ((2 * c) ^ (r & 7))) = o0;
  *reinterpret_cast<uint4*>(row + 16 * ((2 * c + 1) ^ (r & 7))) = o1;
}

// Eight packed 4-bit codes (one 32-bit word; byte m holds element 2m in its
// low nibble and 2m + 1 in its high nibble) minus a zero point z -> four
// bf16x2 words o[m] = {q_2m - z, q_2m+1 - z}, exactly.  Each nibble n sits in
// the low byte of the bf16 word 0x4300|n = 128 + n; subtracting the word
// 0x4300|z = 128 + z (zz holds it in both halves) leaves n - z, an integer
// of magnitude <= 15.
__device__ __forceinline__ void int4x8_minus_zero_to_bf16(uint32_t w, uint32_t zz, uint32_t (&o)[4]) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    // bytes {lo_m, -, hi_m, -}, then 0x43 into the high byte of each half
    const uint32_t t = __byte_perm(lo, hi, static_cast<uint32_t>(m | ((4 + m) << 8)));
    uint32_t v;
    asm("lop3.b32 %0, %1, 0x00FF00FF, 0x43004300, 0xEA;" : "=r"(v) : "r"(t));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(o[m]) : "r"(v), "r"(zz));
  }
}

// Four e4m3 bytes (one 32-bit word; sign, 4 exponent bits with bias 7, 3
// mantissa bits) -> four bf16, exactly: lo = {b0, b1}, hi = {b2, b3}.  Each
// byte's sign goes to bit 15 and its exponent and mantissa to bits 10..4 of a
// bf16 word, which is then the byte's value times 2^-120 (exponent bias 127
// instead of 7; an e4m3 subnormal lands on a bf16 subnormal with the same
// mantissa bits).  The bf16 product with 2^120 restores the value; it is
// exact, being a power-of-two scaling into bf16's normal range.  The NaN
// bytes (exponent 15, mantissa 7) are not valid weights and map to 480.
__device__ __forceinline__ void fp8x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t01 = __byte_perm(w, 0u, 0x4140), t23 = __byte_perm(w, 0u, 0x4342);  // {b, 0} per half
  uint32_t v01, v23;
  asm("lop3.b32 %0, %1, 0x80008000, %2, 0xEA;" : "=r"(v01) : "r"(t01 << 8), "r"((t01 & 0x007F007Fu) << 4));
  asm("lop3.b32 %0, %1, 0x80008000, %2, 0xEA;" : "=r"(v23) : "r"(t23 << 8), "r"((t23 & 0x007F007Fu) << 4));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(v01), "r"(0x7B807B80u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(v23), "r"(0x7B807B80u));
}

}  // namespace cbmoe
