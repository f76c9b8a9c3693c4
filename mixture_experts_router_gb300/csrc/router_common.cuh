// Pieces of the mma.sync router shared by the router kernel (router.cu) and
// the fused router + dispatch launch (route_dispatch.cu): the logit GEMM of
// one 16-token m-tile over a slice of d, and the warp gate (top-k in the
// order number before NaN, larger first, lower index on ties; softmax
// renormalised over the k, or the raw logits).
//
// The gate is the one of "Colibri：面向MoE模型的高性能C语言推理引擎" §2.1
// (softmax, top-k, weights renormalised over the k; since the full softmax
// denominator cancels, w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0)), and
// of "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2 with raw_weights (top-k
// straight on the raw logits, which are then the weights).
#pragma once
#include <cstdint>

namespace cbmoe {
namespace router_detail {

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Logits of one 16-token m-tile against NTW n-tiles of 8 experts over the
// slice [dbeg, dbeg + dslice) of d (dslice a multiple of 32), accumulated in
// acc (the m16n8 fragment: rows g and g + 8, columns 2q and 2q + 1, g = lane
// / 4, q = lane % 4).  A dot product does not depend on the order of its
// terms, so the MMA's 16 k-slots are mapped onto d such that each thread's
// four k-slots of one MMA are four consecutive elements: a thread loads 8
// consecutive bf16 (16 bytes) of a row of x and of W_r per 32-element step
// and feeds two MMAs from them.  UNR steps are loaded before any MMA runs, so
// each thread keeps several 16-byte loads in flight.  Rows past T and experts
// past E read as zero.
template <int NTW, int UNR>
__device__ __forceinline__ void tile_logits(const uint16_t* x, const uint16_t* wr, int T, int d, int E, int tok0,
                                            int e0, int dbeg, int dslice, float (&acc)[NTW][4]) {
  const int lane = threadIdx.x % 32;
  const int g = lane >> 2, q = lane & 3;
  const int r0 = tok0 + g, r1 = tok0 + g + 8;
  const uint4* xa_ptr =
      reinterpret_cast<const uint4*>(x + static_cast<int64_t>(min(r0, T - 1)) * d + dbeg + 8 * q);
  const uint4* xb_ptr =
      reinterpret_cast<const uint4*>(x + static_cast<int64_t>(min(r1, T - 1)) * d + dbeg + 8 * q);
  const bool va = r0 < T, vb = r1 < T;
  const uint4* w_ptr[NTW];
  bool wv[NTW];
#pragma unroll
  for (int j = 0; j < NTW; ++j) {
    const int e = e0 + j * 8 + g;
    wv[j] = e < E;
    w_ptr[j] = reinterpret_cast<const uint4*>(wr + static_cast<int64_t>(min(e, E - 1)) * d + dbeg + 8 * q);
  }
#pragma unroll
  for (int j = 0; j < NTW; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int c = 0; c < dslice; c += 32 * UNR) {
    uint4 xa[UNR], xb[UNR], w[UNR][NTW];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const bool in = c + 32 * u < dslice;
      const int off = (c + 32 * u) / 8;  // in uint4 units
      xa[u] = (in && va) ? __ldg(xa_ptr + off) : zero;
      xb[u] = (in && vb) ? __ldg(xb_ptr + off) : zero;
#pragma unroll
      for (int j = 0; j < NTW; ++j) w[u][j] = (in && wv[j]) ? __ldg(w_ptr[j] + off) : zero;
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u)
#pragma unroll
      for (int j = 0; j < NTW; ++j) {
        mma_bf16(acc[j], xa[u].x, xb[u].x, xa[u].y, xb[u].y, w[u][j].x, w[u][j].y);
        mma_bf16(acc[j], xa[u].z, xb[u].z, xa[u].w, xb[u].w, w[u][j].z, w[u][j].w);
      }
  }
}

// Order of a logit as an unsigned key, larger first: numbers by value (-0
// folded into +0, so the two zeros tie), then NaN (1); 0 is left for a
// candidate that is padding or already taken.
__device__ __forceinline__ uint32_t gate_key(float v) {
  if (isnan(v)) return 1u;
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  const uint32_t h = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return h < 2u ? 2u : h;  // numbers stay above NaN (only NaN bit patterns could map lower)
}

// The gate of one token from its logits row ls[0..E) (shared memory), by one
// warp: k rounds of a warp arg-max.  Lane l holds experts l, l + 32, ...
// (PER of them); a round takes the largest key in the lane (the lower
// expert on equal keys), then the warp's largest key and, among the lanes
// holding it, the lowest expert index (two warp reductions).  Lane s < k
// returns the s-th expert in (id) and its weight (w); other lanes return
// id = -1.  Registers only: the candidates are never indexed by a value.
template <int PER>
__device__ __forceinline__ void warp_gate(const float* ls, int E, int k, int raw_weights, int& id, float& w) {
  const int lane = threadIdx.x % 32;
  float v[PER];
  uint32_t key[PER];
#pragma unroll
  for (int p = 0; p < PER; ++p) {
    const int e = lane + 32 * p;
    v[p] = e < E ? ls[e] : 0.f;
    key[p] = e < E ? gate_key(v[p]) : 0u;
  }
  float my_v = 0.f, l0 = 0.f;
  int my_i = -1;
  for (int s = 0; s < k; ++s) {
    uint32_t bk = key[0];
    int bj = 0;
    float bv = v[0];
#pragma unroll
    for (int p = 1; p < PER; ++p)
      if (key[p] > bk) {  // strictly larger: the lower expert keeps a tie
        bk = key[p];
        bj = p;
        bv = v[p];
      }
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t we = __reduce_min_sync(0xffffffffu, bk == wk ? static_cast<uint32_t>(lane + 32 * bj) : ~0u);
    const int owner = static_cast<int>(we & 31u);
    const float sv = __shfl_sync(0xffffffffu, bv, owner);
    if (lane == owner) {
#pragma unroll
      for (int p = 0; p < PER; ++p)
        if (p == bj) key[p] = 0u;
    }
    if (s == 0) l0 = sv;
    if (lane == s) {
      my_v = sv;
      my_i = static_cast<int>(we);
    }
  }
  const float ex = (lane < k) ? expf(my_v - l0) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  id = lane < k ? my_i : -1;
  w = raw_weights ? my_v : ex / sum;
}

// warp_gate for up to N rows at once (rows ls, ls + stride, ...; the first
// nrows of them are tokens): the same steps for each row, interleaved so
// that the rows' reductions overlap.  Lane s < k of row n returns its s-th
// expert in id[n] and its weight in w[n]; rows past nrows return nothing
// meaningful.
template <int PER, int N>
__device__ __forceinline__ void warp_gate_rows(const float* ls, int stride, int nrows, int E, int k,
                                               int raw_weights, int (&id)[N], float (&w)[N]) {
  const int lane = threadIdx.x % 32;
  float v[N][PER];
  uint32_t key[N][PER];
#pragma unroll
  for (int n = 0; n < N; ++n)
#pragma unroll
    for (int p = 0; p < PER; ++p) {
      const int e = lane + 32 * p;
      const bool in = n < nrows && e < E;
      v[n][p] = in ? ls[n * stride + e] : 0.f;
      key[n][p] = in ? gate_key(v[n][p]) : 0u;
    }
  float my_v[N], l0[N];
  int my_i[N];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    my_v[n] = 0.f;
    l0[n] = 0.f;
    my_i[n] = -1;
  }
  for (int s = 0; s < k; ++s) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
      uint32_t bk = key[n][0];
      int bj = 0;
      float bv = v[n][0];
#pragma unroll
      for (int p = 1; p < PER; ++p)
        if (key[n][p] > bk) {  // strictly larger: the lower expert keeps a tie
          bk = key[n][p];
          bj = p;
          bv = v[n][p];
        }
      const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
      const uint32_t we =
          __reduce_min_sync(0xffffffffu, bk == wk ? static_cast<uint32_t>(lane + 32 * bj) : ~0u);
      const int owner = static_cast<int>(we & 31u);
      const float sv = __shfl_sync(0xffffffffu, bv, owner);
      if (lane == owner) {
#pragma unroll
        for (int p = 0; p < PER; ++p)
          if (p == bj) key[n][p] = 0u;
      }
      if (s == 0) l0[n] = sv;
      if (lane == s) {
        my_v[n] = sv;
        my_i[n] = static_cast<int>(we);
      }
    }
  }
#pragma unroll
  for (int n = 0; n < N; ++n) {
    const float ex = (lane < k) ? expf(my_v[n] - l0[n]) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    id[n] = lane < k ? my_i[n] : -1;
    w[n] = raw_weights ? my_v[n] : ex / sum;
  }
}

}  // namespace router_detail
}  // namespace cbmoe
