// Declarations shared by the library's own translation units: the launchers
// of each kernel and the argument blocks they take.  Not part of the ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace cbmoe {

// Rows of one GEMM M-tile; every expert's block of rows in the permuted
// activations is padded to a multiple of it, so no tile spans two experts.
constexpr int kTileM = 128;
// Device status codes written by kernels (same values as cb_status_t).
constexpr int kErrTimeout = 6;
constexpr int kErrDevice = 7;
// Default bound on any device-side wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Kernel launches of this library go through launch_kernel.  Inside a
// PdlScope that is on, every launch after the first `plain_first` ones
// carries programmatic stream serialization: the kernel may start (and run
// its prologue) while the previous one in the stream finishes.  Every kernel
// of the library calls grid_dep_wait before it reads what an earlier kernel
// wrote, so the results do not depend on it.
struct PdlScope {
  static bool& flag() {
    static thread_local bool on = false;
    return on;
  }
  static int& plain() {
    static thread_local int n = 0;
    return n;
  }
  bool prev_on;
  int prev_plain;
  PdlScope(bool on, int plain_first) : prev_on(flag()), prev_plain(plain()) {
    flag() = on;
    plain() = plain_first;
  }
  ~PdlScope() {
    flag() = prev_on;
    plain() = prev_plain;
  }
  // whether the launch being made carries the attribute
  static bool next() {
    if (!flag()) return false;
    if (plain() > 0) {
      --plain();
      return false;
    }
    return true;
  }
};

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PdlScope::next() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Record a device-side error: the first one wins.
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ------------------------------------------------------------------ router
struct RouterArgs {
  const uint16_t* x;     // bf16 [T][d]
  const uint16_t* wr;    // bf16 [E][d]
  const float* bias;     // [E] or nullptr
  int32_t T, d, E, k;
  int32_t* ids;          // [T][k]
  float* w;              // [T][k]
  float* logits;         // [T][E] or nullptr
  int* err;
  // fused dispatch ranks (mma router; or nullptr): per block b of
  // router_rank_block(E) tokens and
  // expert e, blk_counts[b E + e] = the block's pairs routed to e, and per
  // pair local_rank[t k + s] = its rank among the block's pairs of its expert
  // in (token, slot) order
  int32_t* blk_counts;
  int32_t* local_rank;
  int32_t raw_weights;   // 1: w = the selected raw logits (no softmax)
};
// hash router: x [T][d] (bf16) and W_h [hash_dims][d] widened to fp32 ->
// ids [T], w [T] = 1
struct HashRouterArgs {
  const uint16_t* x;
  const float* wh;
  int32_t T, d, E, hash_dims;
  int32_t* ids;
  float* w;
};
cudaError_t launch_router_hash(const HashRouterArgs& a, cudaStream_t s);
// W_h bf16 [hash_dims][d] -> fp32 (exact) for HashRouterArgs::wh
cudaError_t prepare_hash_weights(const uint16_t* wh, int hash_dims, int d, float* wh_f32, cudaStream_t s);
// tokens per block of the mma router, each one rank block of the fused
// dispatch ranks (the tcgen05 router leaves the ranking to the dispatch)
int router_rank_block(int E);
cudaError_t launch_router(const RouterArgs& a, cudaStream_t s);
cudaError_t router_prepare();  // one-time function attributes
// tcgen05 router: x and Wr through TMA (tm_x: [T][d] box 64x128; tm_w: [E][d]
// box 64 x router_tc_rows(E)); units of 128 tokens x one of
// router_tc_slices(..) slices of d write partial logits to `part`
// ([slices][128 ceil(T/128)][router_tc_rows(E)] fp32, at most
// kRouterMaxSlices slices), then one warp per token takes the top k
constexpr int kRouterMaxSlices = 4;
cudaError_t launch_router_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& a, float* part,
                             int num_sms, cudaStream_t s);
cudaError_t router_tc_prepare();
int router_tc_rows(int E);
int router_tc_slices(int T, int d, int E, int num_sms);

// ---------------------------------------------------------------- dispatch
struct DispatchArgs {
  const int32_t* ids;    // [T*k]
  const uint16_t* x;     // bf16 [T][d]
  int32_t T, k, E, d;
  int32_t n_chunks;      // ceil(T*k / kDispatchChunk)
  int32_t* chunk;        // [n_chunks][E] per-chunk counts, then per-chunk row bases
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* mtile_off;    // [E+1] prefix sum of ceil(counts/kTileM)
  int32_t* mtile_expert; // [max_mtiles] expert owning each m-tile
  int32_t max_mtiles;
  int32_t* ptile_off;    // [E+1] prefix sum of ceil(mtiles/2): pairs of m-tiles (or nullptr)
  int32_t* ptile_expert; // [max_mtiles] expert owning each pair (or nullptr)
  int32_t* tok;          // [T*k]
  int32_t* inv;          // [T*k]
  uint16_t* xp;          // bf16 [max_mtiles*kTileM][d]
  int32_t gather_blocks;  // blocks of the row copy
  int32_t copy_rows;      // 0: the GEMM gathers its rows from x itself, skip the copy
  int* err;
  // > 0: the router already wrote per-block counts into chunk ([n_rank_blocks][E])
  // and in-block ranks into inv; the dispatch scans the block counts and the
  // row-copy kernel turns the ranks into global ones
  int32_t rank_block;     // tokens per rank block
  int32_t n_rank_blocks;
  // > 0: the dispatch's own ranking and the row copy run as one cooperative
  // launch of this many blocks (chunk then holds [coop_blocks][E] counts),
  // meeting once at a grid barrier on bar[0..1] (zero between launches: the
  // kernel sets the words back itself, grid_barrier.cuh)
  int32_t coop_blocks;
  unsigned int* bar;
  uint64_t wait_limit_ns;
  int32_t test_stall;     // test only: the barrier waits for one block more than exist
};
constexpr int kDispatchChunk = 2048;
constexpr int64_t kDispatchSmallPairs = 16384;  // T*k ranked by the one-block kernel
// the fused-rank scan holds (n_rank_blocks + 1) x (E + 1) counts in shared memory
constexpr int kFusedScanWords = 49152;
cudaError_t dispatch_prepare();  // one-time function attributes
// routed pairs up to which the cooperative dispatch is the default
constexpr int64_t kCoopMaxPairs = 65536;
// blocks of the cooperative dispatch that can be resident at once on
// num_sms SMs (at most one per SM; 0 if none)
int dispatch_coop_max_blocks(int num_sms);
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t s);
// histogram, prefix sums and ranks only (no row gather; x and xp unused);
// the block scan is used up to scan_words words of shared memory
// (kFusedScanWords once dispatch_prepare has run on the device); returns the
// first launch's error, launching nothing after it
cudaError_t launch_dispatch_ranks(const DispatchArgs& a, int scan_words, cudaStream_t s);

// ---------------------------------------------- router + dispatch, fused
// The mma router and the dispatch (ranks, tok/inv, tile maps, row copy) in
// one cooperative launch of `grid` blocks, one per SM, for E <= 16 and d a
// multiple of 512 (route_dispatch_supported checks the shared memory and the
// residency).  Uses a.chunk ([grid][E]), a.bar (the grid barrier's two words),
// a.test_stall and a.wait_limit_ns; the router's blk_counts/local_rank are
// unused.
bool route_dispatch_supported(int T, int d, int E, int k, int num_sms);
int route_dispatch_grid(int T, int num_sms);
cudaError_t route_dispatch_prepare();  // one-time function attributes
cudaError_t launch_route_dispatch(const RouterArgs& r, const DispatchArgs& a, int grid, cudaStream_t s);
// tokens of the largest block share of a launch of `grid` blocks
int route_dispatch_own_max(int T, int grid);
// The tcgen05 router and the dispatch in one cooperative launch, for
// 16 < E <= 256 and d a multiple of 64 (route_dispatch_tc_supported checks
// the shared memory, the count rows and the residency).  tm_x: x, bf16
// [T][d], box 64 x route_dispatch_tc_box_rows(T, grid) (the rows a block
// owns); tm_w: the router weights, box 64 x router_tc_rows(E).  Uses
// a.chunk ([grid][E]), a.bar, a.test_stall and a.wait_limit_ns.
bool route_dispatch_tc_supported(int T, int d, int E, int k, int num_sms);
int route_dispatch_tc_grid(int T, int num_sms);
int route_dispatch_tc_box_rows(int T, int grid);
cudaError_t route_dispatch_tc_prepare();  // one-time function attributes
cudaError_t launch_route_dispatch_tc(const CUtensorMap& tm_x, const CUtensorMap& tm_w, const RouterArgs& r,
                                     const DispatchArgs& a, int grid, int box_rows, cudaStream_t s);

// ----------------------------------------------------------------- combine
struct CombineArgs {
  const float* y;        // fp32 [max_mtiles*kTileM][d]
  const float* w;        // [T][k]
  const int32_t* ids;    // [T][k]
  const int32_t* inv;    // [T][k]
  const int32_t* offsets;   // [E+1]
  const int32_t* mtile_off; // [E+1]
  int32_t T, k, d;
  void* out;             // bf16 or fp32 [T][d]
  int out_f32;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t s);
// out[t] = round(acc[t]) for the down GEMM's fused combine: acc fp32 [T][d]
// -> out bf16 (or fp32 when out_f32) [T][d]
cudaError_t launch_combine_acc(const float* acc, int64_t n_elems, void* out, int out_f32, int grid, cudaStream_t s);

// ------------------------------------------------------------ grouped GEMM
struct GemmArgs {
  const int32_t* mtile_off;     // [E+1]
  const int32_t* mtile_expert;  // [max_mtiles]
  const int32_t* ptile_off;     // [E+1] m-tile pairs (int8 and pair kernels)
  const int32_t* ptile_expert;  // [max_mtiles]
  int32_t E;
  int32_t n_tiles;              // N tiles per expert
  int32_t k_blocks;             // K / 64
  int32_t b_rows_per_expert;    // rows of the B operand per expert
  void* out;                    // H bf16 or Y fp32
  int64_t ld_out;               // elements per output row
  const float* scale0;          // int8 / int4: gate (or down) per-channel scales
  const float* scale1;          // int8 / int4: up scales
  const uint8_t* zero0;         // int4: gate (or down) per-channel zero points
  const uint8_t* zero1;         // int4: up zero points
  int* err;
  uint64_t wait_limit_ns;
  int32_t grid;                 // persistent CTAs
  int32_t test_stall;           // test only: MMA warp waits on a phase nothing completes
  // gate/up with gathered A: tm_a is x [T][d] with a 64 x 1 box; rows of
  // m-tile mt of expert e are tokens tok[offsets[e] + 128 (mt - mtile_off[e]) + i]
  int32_t gather;
  const int32_t* tok;
  const int32_t* offsets;
  const int32_t* counts;
  // down on CTA pairs with the combine fused into its epilogue (comb_acc
  // non-null; tok, offsets and counts set): row `local` of expert e, for
  // local < counts[e], is token t = tok[offsets[e] + local] at the slot s with
  // comb_ids[t k + s] = e; the epilogue adds comb_w[t k + s] * Y-row into
  // comb_acc[t] (fp32 [T][ld_out], zero beforehand) instead of storing Y
  float* comb_acc;
  const int32_t* comb_ids;
  const float* comb_w;
  int32_t top_k;
  // quantised tensor-memory GEMMs: tiles of one m-tile against two weight
  // blocks (every expert must have at most one m-tile; n_tiles counts pairs
  // of weight blocks)
  int32_t wide;
};
enum GemmKind { kGateUpSwiGLU = 0, kDownF32 = 1 };
// tm_out: the fp32 output Y [rows][d] with a 32 x 32 box and the 128-byte
// swizzle, used by the down kernels' TMA-store epilogue; tm_b64: the down
// weights with a 64-row box, for the narrower tail tiles (both ignored by
// gate/up); tm_a32: the A operand with a 32-row box, for m-tiles of at most
// 32 routed rows (used when a.counts is set; not with gathered rows)
cudaError_t launch_grouped_gemm(GemmKind kind, bool int8_weights, const CUtensorMap& tm_a,
                                const CUtensorMap& tm_b, const CUtensorMap& tm_out, const CUtensorMap& tm_b64,
                                const CUtensorMap& tm_a32, const GemmArgs& a, cudaStream_t s);
cudaError_t grouped_gemm_prepare();  // one-time function attributes
int grouped_gemm_tile_n(GemmKind kind);  // output columns per tile
// bf16 on CTA pairs with the 2-SM MMA (M = 256 over m-tiles 2p, 2p+1 of one
// expert): tm_bh is the weight tensor with a 128-row box (each CTA's half of
// a 256-row tile); prepare returns the persistent grids (2 x co-resident
// clusters, 0 if none)
cudaError_t launch_grouped_gemm_pair(GemmKind kind, const CUtensorMap& tm_a, const CUtensorMap& tm_bh,
                                     const CUtensorMap& tm_out, const GemmArgs& a, cudaStream_t s);
cudaError_t grouped_gemm_pair_prepare(int num_sms, int* grid_gateup, int* grid_down);
// int8 weights: tiles are pairs of m-tiles against 128 weight rows
cudaError_t launch_grouped_gemm_int8(GemmKind kind, const CUtensorMap& tm_a, const CUtensorMap& tm_b,
                                     const CUtensorMap& tm_out, const GemmArgs& a, cudaStream_t s);
cudaError_t grouped_gemm_int8_prepare();
int grouped_gemm_int8_tile_n(GemmKind kind);
int grouped_gemm_int8_gateup_block();  // gate/up rows interleaved in blocks of this size
// int8, int4 or fp8 weights converted into tensor memory (the MMA's A
// operand): tiles are 128 weight rows against a pair of m-tiles; tm_x: the
// activations (128 x 64 boxes), tm_w: the weight bytes with a 128 x 128 box
// and the 128-byte swizzle (kWInt8: int8 codes; kWFp8: e4m3 codes; kWInt4:
// packed int4 codes with zero points, slots of K = 256)
enum WeightFormat { kWInt8 = 0, kWInt4 = 1, kWFp8 = 2 };
// (tm_x32: the activations with a 32-row box, for a single m-tile of at most
// 32 routed rows; used when a.counts is set)
cudaError_t launch_grouped_gemm_int8_tm(GemmKind kind, WeightFormat wf, const CUtensorMap& tm_x,
                                        const CUtensorMap& tm_w, const CUtensorMap& tm_x32, const GemmArgs& a,
                                        cudaStream_t s);
cudaError_t grouped_gemm_int8_tm_prepare();
int grouped_gemm_int8_tm_tile_n(GemmKind kind);
int grouped_gemm_int8_tm_gateup_block();  // gate/up rows interleaved in blocks of this size

}  // namespace cbmoe
