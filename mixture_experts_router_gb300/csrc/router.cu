// Router: fp32 logits l = x Wr^T + b fused with the top-k gate (the router
// kernel of "Colibri：面向MoE架构的C语言级高效推理引擎" §3.2: linear projection
// then top-k; routing decided on the device with no host round trip,
// "discosf.com/news/4774337" §5.1).  Softmax is applied and renormalised
// over the k ("Colibri：面向MoE模型的高性能C语言推理引擎" §2.1); since its full
// denominator cancels, w_s = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0).
// With raw_weights the weights are the selected logits themselves (top-k
// straight on the raw logits, no softmax: the first page's §3.2).
//
// The logit GEMM [T x d] x [d x E] runs on the tensor cores with
// mma.sync m16n8k16 (bf16 products are exact, fp32 accumulation).  It is a
// thin GEMM (E <= 256 columns): the operands go straight from global memory
// into registers, no shared-memory staging.  Because a dot product does not
// depend on the order of its terms, the MMA's 16 k-slots are mapped onto d
// so that each thread's four k-slots of one MMA are four consecutive
// elements: a thread loads 8 consecutive bf16 (16 bytes) of a row of x and of
// Wr per 32-element step and feeds two MMAs from them.
//
// Each warp computes a 16-token m-tile against NTW n-tiles of 8 experts over
// a slice of d.  A block of up to 16 warps splits d KS ways (memory parallelism for
// small E, where the kernel is bound by reading x) and the experts NS ways
// (register budget for E > 128).  Partial logits are summed in a fixed order
// in shared memory, the bias is added, and one warp per token takes k rounds
// of a warp arg-max in the order (number before NaN, larger first, lower
// index on ties).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "route_ranks.cuh"
#include "router_common.cuh"

namespace cbmoe {
namespace {

using namespace router_detail;

constexpr int kMaxWarps = 16;

// NT: n-tiles of 8 experts in total (E padded to 8 NT); KS: d split; NS:
// expert split; MTB: 16-token m-tiles per block; the block has KS NS MTB
// warps.
template <int NT, int KS, int NS, int MTB>
struct RCfg {
  static constexpr int WARPS = KS * NS * MTB;
  static constexpr int THREADS = 32 * WARPS;
  static_assert(WARPS <= kMaxWarps, "at most 16 warps per block");
  static constexpr int NTW = NT / NS;      // n-tiles per warp
  static constexpr int EP = NT * 8;        // padded experts
  static constexpr int TB = 16 * MTB;      // tokens per block
  static constexpr int SMEM = KS * TB * EP * 4;
};

template <int NT, int KS, int NS, int MTB>
__global__ void __launch_bounds__(RCfg<NT, KS, NS, MTB>::THREADS) router_mma_kernel(RouterArgs a) {
  grid_dep_wait();    // what earlier kernels in the stream wrote is visible from here
  grid_dep_launch();
  using C = RCfg<NT, KS, NS, MTB>;
  constexpr int NTW = C::NTW, EP = C::EP, TB = C::TB;
  constexpr int kThreads = C::THREADS, kWarps = C::WARPS;
  extern __shared__ float part[];  // [KS][TB][EP], then part[0] holds the logits
  __shared__ int s_ids[TB * 16];   // the block's routing ids, for the fused dispatch ranks
  __shared__ int s_cnt[256];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane >> 2, q = lane & 3;
  const int ks = warp % KS;
  const int ns = (warp / KS) % NS;
  const int mt = warp / (KS * NS);
  const int tok0 = blockIdx.x * TB + mt * 16;
  const int dslice = a.d / KS;
  const int dbeg = ks * dslice;

  // UNR 32-element steps per iteration: more loads in flight for fewer n-tiles
  constexpr int UNR = NTW <= 2 ? 8 : (NTW <= 4 ? 2 : 1);
  float acc[NTW][4];
  tile_logits<NTW, UNR>(a.x, a.wr, a.T, a.d, a.E, tok0, ns * NTW * 8, dbeg, dslice, acc);

  // partial logits -> shared memory
  float* mine = part + (static_cast<int64_t>(ks) * TB + mt * 16) * EP;
#pragma unroll
  for (int j = 0; j < NTW; ++j) {
    const int col = (ns * NTW + j) * 8 + 2 * q;
    mine[g * EP + col] = acc[j][0];
    mine[g * EP + col + 1] = acc[j][1];
    mine[(g + 8) * EP + col] = acc[j][2];
    mine[(g + 8) * EP + col + 1] = acc[j][3];
  }
  __syncthreads();
  // sum the KS partials in a fixed order, add the bias
  for (int i = threadIdx.x; i < TB * EP; i += kThreads) {
    float v = part[i];
#pragma unroll
    for (int s = 1; s < KS; ++s) v += part[static_cast<int64_t>(s) * TB * EP + i];
    const int e = i % EP;
    if (a.bias != nullptr && e < a.E) v += __ldg(a.bias + e);
    part[i] = v;
  }
  __syncthreads();
  const float* ls = part;  // [TB][EP]
  const int t_base = blockIdx.x * TB;

  if (a.logits != nullptr) {
    for (int i = threadIdx.x; i < TB * a.E; i += kThreads) {
      const int r = i / a.E, e = i % a.E, t = t_base + r;
      if (t < a.T) a.logits[static_cast<int64_t>(t) * a.E + e] = ls[r * EP + e];
    }
  }

  constexpr int PER = (EP + 31) / 32;
  for (int r = warp; r < TB; r += kWarps) {
    const int t = t_base + r;
    if (t >= a.T) break;
    int my_i;
    float my_w;
    warp_gate<PER>(ls + r * EP, a.E, a.k, a.raw_weights, my_i, my_w);
    if (lane < a.k) {
      a.ids[static_cast<int64_t>(t) * a.k + lane] = my_i;
      a.w[static_cast<int64_t>(t) * a.k + lane] = my_w;
      s_ids[r * 16 + lane] = my_i;
    }
  }

  // Fused dispatch ranks: this block is one rank block of TB tokens.  Warp 0
  // takes its tokens 32 at a time in token order.
  if (a.blk_counts != nullptr) {
    __syncthreads();
    if (warp == 0) {
      for (int e = lane; e < a.E; e += 32) s_cnt[e] = 0;
      __syncwarp();
      for (int r0 = 0; r0 < TB; r0 += 32) {
        const int r = r0 + lane, t = t_base + r;
        const bool valid = r < TB && t < a.T;
        int ids_l[16], rank[16];
#pragma unroll
        for (int s2 = 0; s2 < 16; ++s2) ids_l[s2] = (valid && s2 < a.k) ? s_ids[r * 16 + s2] : -1;
        warp_expert_ranks<16>(ids_l, a.k, valid, a.E, s_cnt, rank);
        if (valid) {
#pragma unroll
          for (int s2 = 0; s2 < 16; ++s2)
            if (s2 < a.k) a.local_rank[static_cast<int64_t>(t) * a.k + s2] = rank[s2];
        }
      }
      __syncwarp();
      for (int e = lane; e < a.E; e += 32) a.blk_counts[static_cast<int64_t>(blockIdx.x) * a.E + e] = s_cnt[e];
    }
  }
}

template <int NT, int KS, int NS, int MTB>
cudaError_t launch_cfg(const RouterArgs& a, cudaStream_t s) {
  using C = RCfg<NT, KS, NS, MTB>;
  const int blocks = (a.T + C::TB - 1) / C::TB;
  if (blocks == 0) return cudaSuccess;
  launch_kernel(router_mma_kernel<NT, KS, NS, MTB>, blocks, C::THREADS, C::SMEM, s, a);
  return cudaGetLastError();
}

template <int NT, int KS, int NS, int MTB>
cudaError_t prepare_cfg() {
  using C = RCfg<NT, KS, NS, MTB>;
  return cudaFuncSetAttribute(router_mma_kernel<NT, KS, NS, MTB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              C::SMEM);
}

}  // namespace

// Configurations by expert count: small E splits d 8 ways over 16 tokens
// per block; large E keeps up to 16 n-tiles (128 experts) per warp.
#define CBMOE_ROUTER_CONFIGS(X) \
  X(1, 16, 1, 1)                \
  X(2, 16, 1, 1)                \
  X(1, 8, 1, 1)                 \
  X(2, 8, 1, 1)                 \
  X(4, 4, 1, 2)                 \
  X(8, 2, 1, 4)                 \
  X(16, 2, 1, 4)                \
  X(32, 1, 2, 4)

cudaError_t router_prepare() {
  cudaError_t e = cudaSuccess;
#define X(nt, ks, ns, mtb) \
  if (e == cudaSuccess) e = prepare_cfg<nt, ks, ns, mtb>();
  CBMOE_ROUTER_CONFIGS(X)
#undef X
  return e;
}

// tokens per block (16 MTB) of the configuration launch_router picks
int router_rank_block(int E) {
  const int nt = (E + 7) / 8;
  if (nt <= 2) return 16;
  if (nt <= 4) return 32;
  return 64;
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t s) {
  const int nt = (a.E + 7) / 8;
  // small E is bound by reading x: 16 warps split d 16 ways when d allows
  if (nt <= 1) return a.d % 512 == 0 ? launch_cfg<1, 16, 1, 1>(a, s) : launch_cfg<1, 8, 1, 1>(a, s);
  if (nt <= 2) return a.d % 512 == 0 ? launch_cfg<2, 16, 1, 1>(a, s) : launch_cfg<2, 8, 1, 1>(a, s);
  if (nt <= 4) return launch_cfg<4, 4, 1, 2>(a, s);
  if (nt <= 8) return launch_cfg<8, 2, 1, 4>(a, s);
  if (nt <= 16) return launch_cfg<16, 2, 1, 4>(a, s);
  return launch_cfg<32, 1, 2, 4>(a, s);
}

}  // namespace cbmoe
