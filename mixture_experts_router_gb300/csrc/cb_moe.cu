// Host side of the C ABI in cb_moe.h: argument validation, the one-time
// allocation of every device buffer, the weight re-layout, the TMA tensor
// maps, and the launch sequence of one forward pass.
//
// Mirrors the init / infer / free triple and the "C decides, CUDA executes"
// split of "Colibri：面向MoE架构的C语言级高效推理引擎" §2.2-§2.3: the host fixes
// launch shapes from (T, d, f, E, k) once, and every forward only enqueues
// kernels on the caller's stream.  All memory is taken at init
// ("discosf.com/news/4774337" §3.1) from one allocation carved into
// 256-byte-aligned regions (the memory-pool offsets of "lshu.cn/news/53496"
// §3), and dimensions must be multiples of 256 (same page, §3).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "cb_moe.h"
#include "internal.h"

using namespace cbmoe;

struct cb_moe {
  cb_moe_config_t cfg;
  int num_sms;
  char* block;
  uint64_t block_bytes;
  // weights (handle-owned copies)
  uint16_t* wr;
  float* wh;  // hash router projection [hash_dims][d] widened to fp32, or nullptr
  float* bias;
  void* wgu;  // [E][f/B][2][B][d]: gate rows then up rows per B-row block (B = 128 bf16; int8: 16 or 64)
  void* wd;   // [E][d][f]
  float *sg, *su, *sd;
  uint8_t *zg, *zu, *zd;  // int4 zero points
  // workspace
  uint16_t* xp;  // [mpad][d]
  uint16_t* hb;  // [mpad][f]
  float* y;      // [mpad][d]
  int32_t* ids;
  float* w;
  float* logits;
  float* rpart;  // tcgen05 router's partial logits
  int32_t *chunk, *counts, *offsets, *mtile_off, *mtile_expert, *ptile_off, *ptile_expert, *tok, *inv;
  int* err;
  unsigned int* coop_bar;  // grid barrier of the cooperative dispatch
  int32_t coop_blocks;     // > 0: the dispatch's own ranking runs as one cooperative launch
  uint64_t guard_off[48];  // CB_FLAG_GUARDS: offsets of the guard bands in the block
  int32_t n_guards;
  uint16_t *x_stage[2], *out_stage[2];  // host-buffer forwards: double-buffered device copies of x and out
  // Host-buffer forwards run on the handle's own streams: the copy of x in,
  // the layer, the copy of out back.  Successive calls alternate between the
  // two staging slots, so one call's copies overlap another call's layer.
  cudaStream_t hs_in, hs_comp, hs_out;
  cudaEvent_t hin_done[2], hfwd_done[2], hout_done[2];
  int host_slot;
  cudaEvent_t ev_last;     // completion of the last forward enqueued on this handle
  bool last_valid;
  int32_t max_mtiles, n_chunks;
  cudaEvent_t ev[CB_N_STAGES + 1];
  bool timing;             // record the stage events in forwards now
  bool timing_events;      // the events exist (CB_FLAG_STAGE_TIMING at init)
  bool router_tc;          // tcgen05 router (else the mma.sync router)
  bool use_graphs;         // replay each forward variant from a captured CUDA graph
  bool pair_gu, pair_dn;   // bf16 gate/up, down GEMMs on CTA pairs (2-SM MMA)
  int32_t rd_grid;         // > 0: router and dispatch run as one cooperative launch of this many blocks
  int32_t rd_box;          // the tcgen05 form's x box rows (a block's token share)
  bool short_a;            // 1-CTA bf16 GEMMs load 32-row A boxes for m-tiles of at most 32 routed rows
  bool quant_wide;         // quantised GEMMs take one m-tile against two weight blocks per tile
  int32_t rank_block;      // > 0: the router ranks pairs in blocks of this many tokens
  int32_t n_rank_blocks;
  int pair_grid_gu, pair_grid_dn;
  struct GraphSlot {
    const void* a;
    const void* b;
    bool timing;           // captured with the stage events
    cudaGraphExec_t exec;
  } graphs[4];             // bf16 forward, fp32-out forward, host-buffer forward (two staging slots)
  bool gather_a;           // gate/up GEMM gathers its rows from x (no Xp copy)
  bool int8_tm;            // int8 GEMMs convert their weights into tensor memory
  bool use_pdl;            // programmatic dependent launch between the forward's kernels
  bool fused_combine;      // the CTA-pair down GEMM adds its rows into the token sums
  const void* tm_x_src;    // x pointer tm_x was encoded for
  const void* tm_xg_src;   // x pointer tm_xg was encoded for
  CUtensorMap tm_a_gu, tm_b_gu, tm_a_dn, tm_b_dn, tm_b_dn64, tm_b_gu128, tm_b_dn128, tm_y, tm_x, tm_xg, tm_wr,
      tm_a_gu32, tm_a_dn32,
      tm_w_gu8, tm_w_dn8;
};

namespace {

// CB_FLAG_GUARDS: a band of this many bytes of kGuardByte after every
// non-empty workspace region
constexpr uint64_t kGuardBytes = 4096;
constexpr int kGuardByte = 0xA5;
constexpr int kMaxGuards = 48;

struct Layout {
  uint64_t guard_off[kMaxGuards];
  int32_t n_guards;
  uint64_t off_wr, off_bias, off_wgu, off_wd, off_sg, off_su, off_sd, off_wh, off_zg, off_zu, off_zd;
  uint64_t off_xp, off_hb, off_y, off_ids, off_w, off_logits, off_rpart, off_chunk, off_counts, off_offsets, off_mtile_off,
      off_mtile_expert, off_ptile_off, off_ptile_expert, off_tok, off_inv, off_err, off_bar, off_xs, off_os;
  uint64_t total;
  int32_t max_mtiles, n_chunks;
};

uint64_t align256(uint64_t v) { return (v + 255) & ~uint64_t(255); }

Layout plan(const cb_moe_config_t& c) {
  Layout L{};
  const uint64_t T = c.n_tokens, d = c.d_model, f = c.d_ff, E = c.n_experts, k = c.top_k;
  const uint64_t wbits = c.wdtype == CB_W_INT4 ? 4 : c.wdtype == CB_W_BF16 ? 16 : 8;  // bits per weight
  const bool quant = c.wdtype != CB_W_BF16;
  const uint64_t M = T * k;
  L.max_mtiles = static_cast<int32_t>((M + E * (kTileM - 1)) / kTileM + 1);
  L.n_chunks = static_cast<int32_t>((M + kDispatchChunk - 1) / kDispatchChunk);
  const uint64_t mpad = static_cast<uint64_t>(L.max_mtiles) * kTileM;
  uint64_t o = 0;
  const uint64_t guard = (c.flags & CB_FLAG_GUARDS) ? kGuardBytes : 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t at = o;
    o = align256(o + bytes);
    if (guard != 0 && bytes != 0 && L.n_guards < kMaxGuards) {
      L.guard_off[L.n_guards++] = o;
      o += guard;
    }
    return at;
  };
  L.off_wr = take(E * d * 2);
  L.off_bias = take(E * 4);
  L.off_wgu = take(E * 2 * f * d * wbits / 8);
  L.off_wd = take(E * d * f * wbits / 8);
  L.off_sg = take(quant ? E * f * 4 : 0);
  L.off_su = take(quant ? E * f * 4 : 0);
  L.off_sd = take(quant ? E * d * 4 : 0);
  L.off_zg = take(c.wdtype == CB_W_INT4 ? E * f : 0);
  L.off_zu = take(c.wdtype == CB_W_INT4 ? E * f : 0);
  L.off_zd = take(c.wdtype == CB_W_INT4 ? E * d : 0);
  L.off_wh = take(c.router_mode == CB_ROUTER_HASH ? static_cast<uint64_t>(c.hash_dims) * d * 4 : 0);  // fp32
  L.off_xp = take(mpad * d * 2);
  L.off_hb = take(mpad * f * 2);
  L.off_y = take(mpad * d * 4);
  L.off_ids = take(M * 4);
  L.off_w = take(M * 4);
  L.off_logits = take((c.flags & CB_FLAG_KEEP_LOGITS) ? T * E * 4 : 0);
  // partial logits of the tcgen05 router: slices x 128-token tiles x E padded
  L.off_rpart = take(static_cast<uint64_t>(kRouterMaxSlices) * ((T + 127) / 128) * 128 *
                     static_cast<uint64_t>(router_tc_rows(static_cast<int>(E))) * 4);
  // per-chunk counts of the dispatch's own ranking, or the router's per-block
  // counts of the fused ranking (at most kFusedScanWords)
  L.off_chunk = take(std::max<uint64_t>(static_cast<uint64_t>(L.n_chunks) * E, kFusedScanWords) * 4);
  L.off_counts = take(E * 4);
  L.off_offsets = take((E + 1) * 4);
  L.off_mtile_off = take((E + 1) * 4);
  L.off_mtile_expert = take(static_cast<uint64_t>(L.max_mtiles) * 4);
  L.off_ptile_off = take((E + 1) * 4);
  L.off_ptile_expert = take(static_cast<uint64_t>(L.max_mtiles) * 4);
  L.off_tok = take(M * 4);
  L.off_inv = take(M * 4);
  L.off_err = take(64);
  L.off_bar = take(64);
  L.off_xs = take(2 * T * d * 2);
  L.off_os = take(2 * T * d * 2);
  L.total = o;
  return L;
}

cb_status_t validate_config(const cb_moe_config_t* c) {
  if (c == nullptr) return CB_ERR_INVALID_ARG;
  if (c->n_tokens < 0 || c->d_model <= 0 || c->d_ff <= 0 || c->n_experts <= 0 || c->top_k <= 0)
    return CB_ERR_INVALID_ARG;
  if (c->top_k > c->n_experts) return CB_ERR_INVALID_ARG;
  if (c->wdtype != CB_W_BF16 && c->wdtype != CB_W_INT8 && c->wdtype != CB_W_INT4 && c->wdtype != CB_W_FP8)
    return CB_ERR_INVALID_ARG;
  if (c->d_model % 256 != 0 || c->d_ff % 256 != 0) return CB_ERR_UNSUPPORTED;
  if (c->n_experts > 256 || c->top_k > 16) return CB_ERR_UNSUPPORTED;
  if (c->router_mode < CB_ROUTER_SOFTMAX_TOPK || c->router_mode > CB_ROUTER_HASH) return CB_ERR_INVALID_ARG;
  if (c->router_mode == CB_ROUTER_HASH &&
      (c->top_k != 1 || c->hash_dims < 1 || c->hash_dims > CB_MAX_HASH_DIMS))
    return CB_ERR_INVALID_ARG;
  if ((c->flags & ~(CB_FLAG_KEEP_LOGITS | CB_FLAG_STAGE_TIMING | CB_FLAG_TEST_STALL |
                   CB_FLAG_TEST_STALL_DISPATCH | CB_FLAG_GUARDS)) != 0)
    return CB_ERR_INVALID_ARG;
  // 32-bit row and tile indices everywhere
  const uint64_t M = static_cast<uint64_t>(c->n_tokens) * c->top_k;
  const uint64_t rows = M + static_cast<uint64_t>(c->n_experts) * kTileM;
  if (rows >= (1ull << 31) || static_cast<uint64_t>(c->n_experts) * 2 * c->d_ff >= (1ull << 31) ||
      static_cast<uint64_t>(c->n_experts) * c->d_model >= (1ull << 31))
    return CB_ERR_UNSUPPORTED;
  return CB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool fault_injected(const char* what) {
  const char* v = std::getenv("CB_MOE_INJECT_FAULT");
  return v != nullptr && std::strcmp(v, what) == 0;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D row-major tensor [outer][inner] with a box of box_outer x box_inner
// elements, 128-byte swizzled (bf16 operands) or unswizzled (int8 staging).
bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t elem_bytes, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

cb_status_t enqueue_forward(cb_moe_t* h, const void* x, void* out, bool f32out, cudaStream_t s) {
  const cb_moe_config_t& c = h->cfg;
  if (fault_injected("launch")) return CB_ERR_CUDA;
  // the forward's first kernel follows arbitrary work of the caller and is
  // launched plainly; the others may start while their predecessor finishes
  // (not on the legacy default stream)
  PdlScope pdl(h->use_pdl && s != nullptr, 1);
  // external event nodes when captured, so stage timing works through a
  // graph; plain records otherwise
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (h->timing && cudaStreamIsCapturing(s, &cap) != cudaSuccess) return CB_ERR_CUDA;
  const unsigned int ev_flags = cap == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
  auto mark = [&](int i) {
    return !h->timing || cudaEventRecordWithFlags(h->ev[i], s, ev_flags) == cudaSuccess;
  };
  if (!mark(0)) return CB_ERR_CUDA;
  const bool fuse = h->fused_combine && h->pair_dn && c.wdtype == CB_W_BF16;
  const uint64_t td = static_cast<uint64_t>(c.n_tokens) * c.d_model;
  // the fused combine's token sums (in the Y buffer, which it does not use)
  // start from zero
  if (fuse && cudaMemsetAsync(h->y, 0, td * 4, s) != cudaSuccess) return CB_ERR_CUDA;

  RouterArgs ra{};
  ra.x = static_cast<const uint16_t*>(x);
  ra.wr = h->wr;
  ra.bias = h->bias;
  ra.T = c.n_tokens;
  ra.d = c.d_model;
  ra.E = c.n_experts;
  ra.k = c.top_k;
  ra.ids = h->ids;
  ra.w = h->w;
  ra.logits = h->logits;
  ra.err = h->err;
  if (h->rank_block > 0) {
    ra.blk_counts = h->chunk;
    ra.local_rank = h->inv;
  }
  ra.raw_weights = c.router_mode == CB_ROUTER_RAW_LOGITS ? 1 : 0;
  if (c.router_mode == CB_ROUTER_HASH) {
    HashRouterArgs ha{};
    ha.x = static_cast<const uint16_t*>(x);
    ha.wh = h->wh;
    ha.T = c.n_tokens;
    ha.d = c.d_model;
    ha.E = c.n_experts;
    ha.hash_dims = c.hash_dims;
    ha.ids = h->ids;
    ha.w = h->w;
    if (launch_router_hash(ha, s) != cudaSuccess || !mark(1)) return CB_ERR_CUDA;
  } else if (h->router_tc) {
    if (h->tm_x_src != x) {
      const uint32_t box = h->rd_grid > 0 ? static_cast<uint32_t>(h->rd_box) : 128u;
      if (!make_tmap(&h->tm_x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.d_model, c.n_tokens, 64, box))
        return CB_ERR_CUDA;
      h->tm_x_src = x;
    }
    if (h->rd_grid <= 0 &&
        (launch_router_tc(h->tm_x, h->tm_wr, ra, h->rpart, h->num_sms, s) != cudaSuccess || !mark(1)))
      return CB_ERR_CUDA;
  } else if (h->rd_grid <= 0) {
    if (launch_router(ra, s) != cudaSuccess || !mark(1)) return CB_ERR_CUDA;
  }

  DispatchArgs da{};
  da.ids = h->ids;
  da.x = static_cast<const uint16_t*>(x);
  da.T = c.n_tokens;
  da.k = c.top_k;
  da.E = c.n_experts;
  da.d = c.d_model;
  da.n_chunks = h->n_chunks;
  da.chunk = h->chunk;
  da.counts = h->counts;
  da.offsets = h->offsets;
  da.mtile_off = h->mtile_off;
  da.mtile_expert = h->mtile_expert;
  da.max_mtiles = h->max_mtiles;
  da.ptile_off = h->ptile_off;
  da.ptile_expert = h->ptile_expert;
  da.tok = h->tok;
  da.inv = h->inv;
  da.xp = h->xp;
  da.gather_blocks = static_cast<int32_t>(std::min<int64_t>(h->num_sms * 8, (c.n_tokens + 7) / 8));
  da.copy_rows = h->gather_a ? 0 : 1;
  da.err = h->err;
  da.rank_block = h->rank_block;
  da.n_rank_blocks = h->n_rank_blocks;
  da.coop_blocks = h->coop_blocks;
  da.bar = h->coop_bar;
  da.wait_limit_ns = kWaitLimitNs;
  if (c.flags & CB_FLAG_TEST_STALL_DISPATCH) {
    da.test_stall = 1;
    da.wait_limit_ns = 1000000ull;  // 1 ms
  }
  if (h->rd_grid > 0 && c.router_mode != CB_ROUTER_HASH) {
    // router and dispatch in one launch: the router stage ends with it and
    // the dispatch stage is empty
    ra.blk_counts = nullptr;
    ra.local_rank = nullptr;
    const cudaError_t e = h->router_tc ? launch_route_dispatch_tc(h->tm_x, h->tm_wr, ra, da, h->rd_grid, h->rd_box, s)
                                       : launch_route_dispatch(ra, da, h->rd_grid, s);
    if (e != cudaSuccess || !mark(1) || !mark(2)) return CB_ERR_CUDA;
  } else if (launch_dispatch(da, s) != cudaSuccess || !mark(2)) {
    return CB_ERR_CUDA;
  }

  const bool int4w = c.wdtype == CB_W_INT4;
  const bool int8w = c.wdtype != CB_W_BF16;  // quantized weights (int8, int4 or fp8)
  const WeightFormat wf = int4w ? kWInt4 : c.wdtype == CB_W_FP8 ? kWFp8 : kWInt8;
  GemmArgs ga{};
  ga.mtile_off = h->mtile_off;
  ga.mtile_expert = h->mtile_expert;
  ga.ptile_off = h->ptile_off;
  ga.ptile_expert = h->ptile_expert;
  ga.E = c.n_experts;
  ga.n_tiles = c.d_ff / (int8w ? (h->int8_tm ? grouped_gemm_int8_tm_tile_n(kGateUpSwiGLU)
                                              : grouped_gemm_int8_tile_n(kGateUpSwiGLU))
                                : grouped_gemm_tile_n(kGateUpSwiGLU));
  ga.k_blocks = c.d_model / 64;
  ga.b_rows_per_expert = 2 * c.d_ff;
  ga.out = h->hb;
  ga.ld_out = c.d_ff;
  ga.scale0 = h->sg;
  ga.scale1 = h->su;
  ga.zero0 = h->zg;
  ga.zero1 = h->zu;
  ga.err = h->err;
  ga.wait_limit_ns = kWaitLimitNs;
  ga.grid = h->num_sms;
  const CUtensorMap* tm_a_gu = &h->tm_a_gu;
  if (h->gather_a) {
    if (h->tm_xg_src != x) {
      if (!make_tmap(&h->tm_xg, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.d_model, c.n_tokens, 64, 1))
        return CB_ERR_CUDA;
      h->tm_xg_src = x;
    }
    tm_a_gu = &h->tm_xg;
    ga.gather = 1;
    ga.tok = h->tok;
    ga.offsets = h->offsets;
    ga.counts = h->counts;
  }
  if (c.flags & CB_FLAG_TEST_STALL) {
    ga.test_stall = 1;
    ga.wait_limit_ns = 1000000ull;  // 1 ms
  }
  const bool pair_gu = !int8w && h->pair_gu && !h->gather_a;
  const bool pair_dn = !int8w && h->pair_dn;
  cudaError_t e1;
  if (int8w && h->int8_tm) {
    GemmArgs g1 = ga;
    g1.counts = h->short_a ? h->counts : nullptr;  // 32-row activation boxes for single m-tiles of few rows
    if (h->quant_wide) {  // one m-tile against two weight blocks per tile
      g1.wide = 1;
      g1.n_tiles = ga.n_tiles / 2;
    }
    e1 = launch_grouped_gemm_int8_tm(kGateUpSwiGLU, wf, h->tm_a_gu, h->tm_w_gu8, h->tm_a_gu32, g1, s);
  } else if (int8w) {
    e1 = launch_grouped_gemm_int8(kGateUpSwiGLU, h->tm_a_gu, h->tm_b_gu, h->tm_y, ga, s);
  } else if (pair_gu) {
    GemmArgs gp = ga;
    gp.grid = h->pair_grid_gu;
    e1 = launch_grouped_gemm_pair(kGateUpSwiGLU, h->tm_a_gu, h->tm_b_gu128, h->tm_y, gp, s);
  } else {
    GemmArgs g1 = ga;
    if (!h->gather_a && h->short_a) g1.counts = h->counts;  // 32-row A boxes for tiles of few rows
    e1 = launch_grouped_gemm(kGateUpSwiGLU, false, *tm_a_gu, h->tm_b_gu, h->tm_y, h->tm_b_dn64, h->tm_a_gu32, g1, s);
  }
  if (e1 != cudaSuccess || !mark(3)) return CB_ERR_CUDA;

  GemmArgs gd = ga;
  gd.gather = 0;
  gd.test_stall = 0;
  gd.wait_limit_ns = kWaitLimitNs;
  gd.n_tiles = c.d_model / (int8w ? (h->int8_tm ? grouped_gemm_int8_tm_tile_n(kDownF32) : grouped_gemm_int8_tile_n(kDownF32))
                                   : grouped_gemm_tile_n(kDownF32));
  gd.k_blocks = c.d_ff / 64;
  gd.b_rows_per_expert = c.d_model;
  gd.out = h->y;
  gd.ld_out = c.d_model;
  gd.scale0 = h->sd;
  gd.scale1 = nullptr;
  gd.zero0 = h->zd;
  gd.zero1 = nullptr;
  cudaError_t e2;
  if (int8w && h->int8_tm) {
    GemmArgs g2 = gd;
    g2.counts = h->short_a ? h->counts : nullptr;
    if (h->quant_wide) {
      g2.wide = 1;
      g2.n_tiles = gd.n_tiles / 2;
    }
    e2 = launch_grouped_gemm_int8_tm(kDownF32, wf, h->tm_a_dn, h->tm_w_dn8, h->tm_a_dn32, g2, s);
  } else if (int8w) {
    e2 = launch_grouped_gemm_int8(kDownF32, h->tm_a_dn, h->tm_b_dn, h->tm_y, gd, s);
  } else if (pair_dn) {
    GemmArgs gp = gd;
    gp.grid = h->pair_grid_dn;
    if (fuse) {
      gp.comb_acc = h->y;
      gp.comb_ids = h->ids;
      gp.comb_w = h->w;
      gp.top_k = c.top_k;
      gp.tok = h->tok;
      gp.offsets = h->offsets;
      gp.counts = h->counts;
    }
    e2 = launch_grouped_gemm_pair(kDownF32, h->tm_a_dn, h->tm_b_dn128, h->tm_y, gp, s);
  } else {
    GemmArgs g2 = gd;
    g2.counts = h->short_a ? h->counts : nullptr;
    e2 = launch_grouped_gemm(kDownF32, false, h->tm_a_dn, h->tm_b_dn, h->tm_y, h->tm_b_dn64, h->tm_a_dn32, g2, s);
  }
  if (e2 != cudaSuccess || !mark(4)) return CB_ERR_CUDA;

  if (fuse) {
    if (launch_combine_acc(h->y, static_cast<int64_t>(td), out, f32out ? 1 : 0, h->num_sms * 8, s) != cudaSuccess ||
        !mark(5))
      return CB_ERR_CUDA;
    return CB_OK;
  }
  CombineArgs ca{};
  ca.y = h->y;
  ca.w = h->w;
  ca.ids = h->ids;
  ca.inv = h->inv;
  ca.offsets = h->offsets;
  ca.mtile_off = h->mtile_off;
  ca.T = c.n_tokens;
  ca.k = c.top_k;
  ca.d = c.d_model;
  ca.out = out;
  ca.out_f32 = f32out ? 1 : 0;
  if (launch_combine(ca, s) != cudaSuccess || !mark(5)) return CB_ERR_CUDA;
  return CB_OK;
}

// Enqueue body(s) through a CUDA graph cached per forward variant and keyed
// by its buffer pointers (a, b): the first call for a key captures the
// kernel launches into a graph and instantiates it, later calls replay it,
// which removes the launch gaps between the layer's kernels.  Without graphs
// (the legacy default stream, a stream the caller is already capturing, or
// a capture that fails) the launches are enqueued directly.
template <class Body>
cb_status_t run_graphed(cb_moe_t* h, int slot, const void* a, const void* b, cudaStream_t s, Body body) {
  if (!h->use_graphs || s == nullptr) return body(s);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return body(s);
  }
  if (cs != cudaStreamCaptureStatusNone) return body(s);
  cb_moe::GraphSlot& g = h->graphs[slot];
  if (g.exec == nullptr || g.a != a || g.b != b || g.timing != h->timing) {
    if (g.exec != nullptr) {
      cudaGraphExecDestroy(g.exec);
      g.exec = nullptr;
    }
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      cudaGetLastError();
      return body(s);
    }
    const cb_status_t st = body(s);
    cudaGraph_t graph = nullptr;
    const cudaError_t ec = cudaStreamEndCapture(s, &graph);
    cudaGraphExec_t exec = nullptr;
    const bool ok = st == CB_OK && ec == cudaSuccess && graph != nullptr &&
                    cudaGraphInstantiate(&exec, graph, 0) == cudaSuccess;
    if (graph != nullptr) cudaGraphDestroy(graph);
    if (!ok) {
      cudaGetLastError();
      return body(s);
    }
    g.exec = exec;
    g.a = a;
    g.b = b;
    g.timing = h->timing;
  }
  return cudaGraphLaunch(g.exec, s) == cudaSuccess ? CB_OK : CB_ERR_CUDA;
}

cb_status_t check_forward_args(const cb_moe_t* h, const void* x, const void* out, uint64_t out_elem_bytes) {
  if (h == nullptr || x == nullptr || out == nullptr) return CB_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out)) return CB_ERR_ALIGNMENT;
  const uint64_t xb = static_cast<uint64_t>(h->cfg.n_tokens) * h->cfg.d_model * 2;
  const uint64_t ob = static_cast<uint64_t>(h->cfg.n_tokens) * h->cfg.d_model * out_elem_bytes;
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), oa = reinterpret_cast<uintptr_t>(out);
  if (xb > 0 && xa < oa + ob && oa < xa + xb) return CB_ERR_INVALID_ARG;  // overlap
  return CB_OK;
}

bool create_sync_objects(cb_moe_t* h) {
  bool ok = true;
  for (cudaStream_t* s : {&h->hs_in, &h->hs_comp, &h->hs_out})
    ok = ok && cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; i < 2; ++i)
    for (cudaEvent_t* e : {&h->hin_done[i], &h->hfwd_done[i], &h->hout_done[i]})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  ok = ok && cudaEventCreateWithFlags(&h->ev_last, cudaEventDisableTiming) == cudaSuccess;
  // the events start out complete, so the first calls wait on nothing
  for (int i = 0; ok && i < 2; ++i)
    for (cudaEvent_t e : {h->hin_done[i], h->hfwd_done[i], h->hout_done[i]})
      ok = ok && cudaEventRecord(e, h->hs_comp) == cudaSuccess;
  return ok;
}

void destroy_sync_objects(cb_moe_t* h) {
  for (cudaStream_t s : {h->hs_in, h->hs_comp, h->hs_out})
    if (s != nullptr) cudaStreamDestroy(s);
  for (int i = 0; i < 2; ++i)
    for (cudaEvent_t e : {h->hin_done[i], h->hfwd_done[i], h->hout_done[i]})
      if (e != nullptr) cudaEventDestroy(e);
  if (h->ev_last != nullptr) cudaEventDestroy(h->ev_last);
}

// Forwards of one handle share its workspace, so each waits for the last one
// enqueued, whichever stream ran it, and then becomes the last one.  A stream
// that the caller is capturing into a graph is left to the caller's ordering.
bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs != cudaStreamCaptureStatusNone;
}

bool wait_last_forward(cb_moe_t* h, cudaStream_t s) {
  return !h->last_valid || cudaStreamWaitEvent(s, h->ev_last, 0) == cudaSuccess;
}

bool mark_last_forward(cb_moe_t* h, cudaStream_t s) {
  if (cudaEventRecord(h->ev_last, s) != cudaSuccess) return false;
  h->last_valid = true;
  return true;
}

// A device forward (bf16 or fp32 output) on the caller's stream.
template <class Body>
cb_status_t device_forward(cb_moe_t* h, int slot, const void* x, void* out, cudaStream_t s, Body body) {
  const bool cap = capturing(s);
  if (!cap && !wait_last_forward(h, s)) return CB_ERR_CUDA;
  const cb_status_t st = run_graphed(h, slot, x, out, s, body);
  if (st == CB_OK && !cap && !mark_last_forward(h, s)) return CB_ERR_CUDA;
  return st;
}

}  // namespace

extern "C" {

const char* cb_status_string(cb_status_t s) {
  switch (s) {
    case CB_OK: return "ok";
    case CB_ERR_INVALID_ARG: return "invalid argument";
    case CB_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case CB_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case CB_ERR_OOM: return "device allocation failed";
    case CB_ERR_CUDA: return "CUDA call or kernel launch failed";
    case CB_ERR_TIMEOUT: return "device-side wait timed out";
    case CB_ERR_DEVICE: return "device-side range check failed";
  }
  return "unknown status";
}

cb_status_t cb_moe_kernels_per_forward(const cb_moe_t* h, int32_t* n) {
  if (h == nullptr || n == nullptr) return CB_ERR_INVALID_ARG;
  const cb_moe_config_t& c = h->cfg;
  if (c.n_tokens == 0) {  // a forward of no tokens launches nothing
    *n = 0;
    return CB_OK;
  }
  int32_t dispatch;
  const bool fused = h->rd_grid > 0 && c.router_mode != CB_ROUTER_HASH;
  if (fused)
    dispatch = 0;  // in the router's launch
  else if (h->rank_block > 0)
    dispatch = 2;  // block-count scan + row copy (which also finalises the ranks)
  else if (h->coop_blocks > 0)
    dispatch = 1;  // count, scan, ranks and row copy in one cooperative launch
  else
    dispatch = (static_cast<int64_t>(c.n_tokens) * c.top_k <= kDispatchSmallPairs ? 1 : 3) + (h->gather_a ? 0 : 1);
  // the separate tcgen05 router: partials + top-k
  const int32_t router = (h->router_tc && c.router_mode != CB_ROUTER_HASH && !fused) ? 2 : 1;
  *n = router + dispatch + 2 + 1;
  return CB_OK;
}

cb_status_t cb_moe_device_bytes(const cb_moe_config_t* cfg, uint64_t* bytes) {
  if (bytes == nullptr) return CB_ERR_INVALID_ARG;
  const cb_status_t st = validate_config(cfg);
  if (st != CB_OK) return st;
  *bytes = plan(*cfg).total;
  return CB_OK;
}

cb_status_t cb_moe_init(const cb_moe_config_t* cfg, const cb_moe_weights_t* wts, cb_moe_t** out) {
  if (out == nullptr) return CB_ERR_INVALID_ARG;
  *out = nullptr;
  cb_status_t st = validate_config(cfg);
  if (st != CB_OK) return st;
  const bool hashr = cfg->router_mode == CB_ROUTER_HASH;
  if (wts == nullptr || (wts->w_router == nullptr && !hashr) || wts->w_gate == nullptr || wts->w_up == nullptr ||
      wts->w_down == nullptr || (hashr && wts->w_hash == nullptr))
    return CB_ERR_INVALID_ARG;
  const bool int4w = cfg->wdtype == CB_W_INT4;
  const bool fp8w = cfg->wdtype == CB_W_FP8;
  const bool int8w = cfg->wdtype != CB_W_BF16;  // quantized weights (int8, int4 or fp8)
  if (int4w && (wts->z_gate == nullptr || wts->z_up == nullptr || wts->z_down == nullptr))
    return CB_ERR_UNSUPPORTED;
  if (int8w && (wts->s_gate == nullptr || wts->s_up == nullptr || wts->s_down == nullptr))
    return CB_ERR_UNSUPPORTED;
  const void* ptrs[] = {wts->w_router, wts->router_bias, wts->w_gate, wts->w_up, wts->w_down,
                        wts->s_gate,   wts->s_up,        wts->s_down, wts->w_hash};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return CB_ERR_ALIGNMENT;

  DeviceGuard guard(cfg->device);
  if (!guard.ok) return CB_ERR_UNSUPPORTED;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return CB_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return CB_ERR_UNSUPPORTED;

  const Layout L = plan(*cfg);
  cb_moe_t* h = new (std::nothrow) cb_moe_t();
  if (h == nullptr) return CB_ERR_OOM;
  static_assert(sizeof(h->guard_off) / sizeof(h->guard_off[0]) == kMaxGuards, "guard table");
  for (int i = 0; i < L.n_guards; ++i) h->guard_off[i] = L.guard_off[i];
  h->n_guards = L.n_guards;
  h->cfg = *cfg;
  h->num_sms = prop.multiProcessorCount;
  h->max_mtiles = L.max_mtiles;
  h->n_chunks = L.n_chunks;
  h->block_bytes = L.total;
  if (fault_injected("oom") || cudaMalloc(&h->block, L.total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return CB_ERR_OOM;
  }
  char* b = h->block;
  h->wr = reinterpret_cast<uint16_t*>(b + L.off_wr);
  h->wh = hashr ? reinterpret_cast<float*>(b + L.off_wh) : nullptr;
  h->bias = wts->router_bias ? reinterpret_cast<float*>(b + L.off_bias) : nullptr;
  h->wgu = b + L.off_wgu;
  h->wd = b + L.off_wd;
  h->sg = int8w ? reinterpret_cast<float*>(b + L.off_sg) : nullptr;
  h->su = int8w ? reinterpret_cast<float*>(b + L.off_su) : nullptr;
  h->sd = int8w ? reinterpret_cast<float*>(b + L.off_sd) : nullptr;
  h->zg = int4w ? reinterpret_cast<uint8_t*>(b + L.off_zg) : nullptr;
  h->zu = int4w ? reinterpret_cast<uint8_t*>(b + L.off_zu) : nullptr;
  h->zd = int4w ? reinterpret_cast<uint8_t*>(b + L.off_zd) : nullptr;
  h->xp = reinterpret_cast<uint16_t*>(b + L.off_xp);
  h->hb = reinterpret_cast<uint16_t*>(b + L.off_hb);
  h->y = reinterpret_cast<float*>(b + L.off_y);
  h->ids = reinterpret_cast<int32_t*>(b + L.off_ids);
  h->w = reinterpret_cast<float*>(b + L.off_w);
  h->logits = (cfg->flags & CB_FLAG_KEEP_LOGITS) ? reinterpret_cast<float*>(b + L.off_logits) : nullptr;
  h->rpart = reinterpret_cast<float*>(b + L.off_rpart);
  h->chunk = reinterpret_cast<int32_t*>(b + L.off_chunk);
  h->counts = reinterpret_cast<int32_t*>(b + L.off_counts);
  h->offsets = reinterpret_cast<int32_t*>(b + L.off_offsets);
  h->mtile_off = reinterpret_cast<int32_t*>(b + L.off_mtile_off);
  h->mtile_expert = reinterpret_cast<int32_t*>(b + L.off_mtile_expert);
  h->ptile_off = reinterpret_cast<int32_t*>(b + L.off_ptile_off);
  h->ptile_expert = reinterpret_cast<int32_t*>(b + L.off_ptile_expert);
  h->tok = reinterpret_cast<int32_t*>(b + L.off_tok);
  h->inv = reinterpret_cast<int32_t*>(b + L.off_inv);
  h->err = reinterpret_cast<int*>(b + L.off_err);
  h->coop_bar = reinterpret_cast<unsigned int*>(b + L.off_bar);
  for (int i = 0; i < 2; ++i) {
    h->x_stage[i] = reinterpret_cast<uint16_t*>(b + L.off_xs) + static_cast<uint64_t>(i) * cfg->n_tokens * cfg->d_model;
    h->out_stage[i] = reinterpret_cast<uint16_t*>(b + L.off_os) + static_cast<uint64_t>(i) * cfg->n_tokens * cfg->d_model;
  }

  const uint64_t E = cfg->n_experts, d = cfg->d_model, f = cfg->d_ff;
  const uint64_t eb = int8w ? 1 : 2;                      // element bytes of the bf16 / int8 maps
  const uint64_t wbits = int4w ? 4 : int8w ? 8 : 16;      // bits per expert weight
  bool ok = cudaMemset(h->block + L.off_xp, 0, L.off_ids - L.off_xp) == cudaSuccess &&
            cudaMemset(h->block + L.off_ids, 0, L.total - L.off_ids) == cudaSuccess;
  if (wts->w_router != nullptr)
    ok = ok && cudaMemcpy(h->wr, wts->w_router, E * d * 2, cudaMemcpyDeviceToDevice) == cudaSuccess;
  else
    ok = ok && cudaMemset(h->wr, 0, E * d * 2) == cudaSuccess;
  if (hashr)
    ok = ok && prepare_hash_weights(static_cast<const uint16_t*>(wts->w_hash), cfg->hash_dims, static_cast<int>(d),
                                    h->wh, nullptr) == cudaSuccess;
  if (ok && h->bias) ok = cudaMemcpy(h->bias, wts->router_bias, E * 4, cudaMemcpyDeviceToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(h->wd, wts->w_down, E * d * f * wbits / 8, cudaMemcpyDeviceToDevice) == cudaSuccess;
  if (ok && int8w) {
    ok = cudaMemcpy(h->sg, wts->s_gate, E * f * 4, cudaMemcpyDeviceToDevice) == cudaSuccess &&
         cudaMemcpy(h->su, wts->s_up, E * f * 4, cudaMemcpyDeviceToDevice) == cudaSuccess &&
         cudaMemcpy(h->sd, wts->s_down, E * d * 4, cudaMemcpyDeviceToDevice) == cudaSuccess;
  }
  if (ok && int4w) {
    ok = cudaMemcpy(h->zg, wts->z_gate, E * f, cudaMemcpyDeviceToDevice) == cudaSuccess &&
         cudaMemcpy(h->zu, wts->z_up, E * f, cudaMemcpyDeviceToDevice) == cudaSuccess &&
         cudaMemcpy(h->zd, wts->z_down, E * d, cudaMemcpyDeviceToDevice) == cudaSuccess;
  }
  // gate/up interleave: block n of expert e = gate rows [Bn, Bn+B) then the same up rows
  // int8 expert GEMMs: weights converted into tensor memory as the MMA's A
  // operand (default), or CB_MOE_INT8=smem for the kernel that converts them
  // into shared memory as the B operand; the two interleave gate and up rows
  // in blocks of different sizes.  int4 weights have the first kernel only.
  {
    const char* iv = std::getenv("CB_MOE_INT8");
    h->int8_tm = int4w || fp8w || !(iv != nullptr && std::strcmp(iv, "smem") == 0);
  }
  const uint64_t brows =
      int8w ? (h->int8_tm ? grouped_gemm_int8_tm_gateup_block() : grouped_gemm_int8_gateup_block()) : 128;
  const uint64_t blk = brows * d * wbits / 8;  // bytes of one block of weight rows
  const uint64_t nblk = E * (f / brows);
  ok = ok && cudaMemcpy2D(h->wgu, 2 * blk, wts->w_gate, blk, blk, nblk, cudaMemcpyDeviceToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy2D(static_cast<char*>(h->wgu) + blk, 2 * blk, wts->w_up, blk, blk, nblk,
                          cudaMemcpyDeviceToDevice) == cudaSuccess;
  const uint64_t mpad = static_cast<uint64_t>(h->max_mtiles) * kTileM;
  const CUtensorMapDataType wdt = int8w ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  ok = ok && make_tmap(&h->tm_a_gu, h->xp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, mpad, 64, 128);
  const CUtensorMapSwizzle wsw = int8w ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  const uint32_t brows_box = int8w ? 128 : 256;
  ok = ok && make_tmap(&h->tm_a_dn, h->hb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, f, mpad, 64, 128);
  // 32-row boxes of the same activations, for the 1-CTA GEMMs' m-tiles of at
  // most 32 routed rows
  ok = ok && make_tmap(&h->tm_a_gu32, h->xp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, mpad, 64, 32);
  ok = ok && make_tmap(&h->tm_a_dn32, h->hb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, f, mpad, 64, 32);
  ok = ok && make_tmap(&h->tm_y, h->y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, mpad, 32, 32);
  if (!int4w) {  // the bf16 and shared-memory int8 GEMMs' weight maps
    ok = ok && make_tmap(&h->tm_b_gu, h->wgu, wdt, eb, d, E * 2 * f, 64, brows_box, wsw);
    ok = ok && make_tmap(&h->tm_b_dn, h->wd, wdt, eb, f, E * d, 64, brows_box, wsw);
    ok = ok && make_tmap(&h->tm_b_dn64, h->wd, wdt, eb, f, E * d, 64, 64, wsw);
  }
  if (int8w) {  // the tensor-memory int8 / int4 GEMMs: rows of bytes (K or K/2 of them)
    ok = ok && make_tmap(&h->tm_w_gu8, h->wgu, wdt, 1, d * wbits / 8, E * 2 * f, 128, 128);
    ok = ok && make_tmap(&h->tm_w_dn8, h->wd, wdt, 1, f * wbits / 8, E * d, 128, 128);
  }
  if (!int8w) {
    ok = ok && make_tmap(&h->tm_b_gu128, h->wgu, wdt, eb, d, E * 2 * f, 64, 128, wsw);
    ok = ok && make_tmap(&h->tm_b_dn128, h->wd, wdt, eb, f, E * d, 64, 128, wsw);
  }
  ok = ok && grouped_gemm_prepare() == cudaSuccess && grouped_gemm_int8_prepare() == cudaSuccess &&
       grouped_gemm_int8_tm_prepare() == cudaSuccess &&
       router_prepare() == cudaSuccess && router_tc_prepare() == cudaSuccess && dispatch_prepare() == cudaSuccess &&
       route_dispatch_prepare() == cudaSuccess && route_dispatch_tc_prepare() == cudaSuccess;
  // router: tcgen05 for wide expert counts, the mma.sync split-K router for
  // E <= 16 (bound by reading x, where more CTAs help); CB_MOE_ROUTER=tc|mma
  // overrides the choice
  {
    const char* rv = std::getenv("CB_MOE_ROUTER");
    h->router_tc = cfg->n_experts > 16;
    if (rv != nullptr && std::strcmp(rv, "tc") == 0) h->router_tc = true;
    if (rv != nullptr && std::strcmp(rv, "mma") == 0) h->router_tc = false;
    // The gate/up rows are copied into the grouped activations by the
    // dispatch and loaded as 128-row TMA tiles.  CB_MOE_GATHER=1 (bf16
    // layers) instead gathers them straight from x with TMA tile::gather4,
    // which skips the copy but measured 3.3x slower in the GEMM on GB300
    // (32 four-row gathers per k-block); it is kept for callers short of
    // memory.
    const char* gv = std::getenv("CB_MOE_GATHER");
    h->gather_a = !int8w && gv != nullptr && std::strcmp(gv, "1") == 0;
    // bf16 GEMMs on CTA pairs (2-SM MMA).  Measured on GB300 once experts
    // average two or more m-tiles (T k >= 256 E): gate/up 4-8 % and down
    // 4-9 % faster than on single CTAs; a decode-size layer, whose experts
    // have one m-tile each, is faster on single CTAs.
    // CB_MOE_PAIR=1|0|gateup|down overrides.
    const char* pv = std::getenv("CB_MOE_PAIR");
    const int64_t routed = static_cast<int64_t>(cfg->n_tokens) * cfg->top_k;
    h->pair_gu = routed >= 256ll * cfg->n_experts;
    h->pair_dn = h->pair_gu;
    if (pv != nullptr) {
      h->pair_gu = std::strcmp(pv, "1") == 0 || std::strcmp(pv, "gateup") == 0;
      h->pair_dn = std::strcmp(pv, "1") == 0 || std::strcmp(pv, "down") == 0;
    }
    if (int8w) h->pair_gu = h->pair_dn = false;
    if (h->pair_gu || h->pair_dn) {
      ok = ok && grouped_gemm_pair_prepare(h->num_sms, &h->pair_grid_gu, &h->pair_grid_dn) == cudaSuccess;
      if (h->pair_grid_gu < 2 || h->pair_grid_dn < 2) h->pair_gu = h->pair_dn = false;
    }
    // The 1-CTA bf16 GEMMs and the quantised GEMMs load only the first 32
    // rows of an m-tile that has at most 32 routed rows (decode sizes: 8 rows
    // per expert at T = 64, k = 2, E = 8), so their load traffic is almost
    // all weights.  CB_MOE_SHORT_A=0 loads whole 128-row tiles.
    const char* sav = std::getenv("CB_MOE_SHORT_A");
    h->short_a = !(sav != nullptr && std::strcmp(sav, "0") == 0);
    // With at most 128 tokens every expert has at most one m-tile (a token's
    // k experts are distinct), and the quantised GEMMs are bound by their
    // per-k-block handshake, not the tensor core: each of their tiles then
    // pairs the m-tile with two weight blocks, twice the weight bytes per
    // handshake.  CB_MOE_WIDE_QUANT=0 keeps one weight block per tile.
    const char* wqv = std::getenv("CB_MOE_WIDE_QUANT");
    h->quant_wide = int8w && h->int8_tm && cfg->n_tokens <= kTileM &&
                    !(wqv != nullptr && std::strcmp(wqv, "0") == 0);
    // the combine fused into the CTA-pair down GEMM with CB_MOE_FUSED_COMBINE=1
    // (bf16 weights, layers that run the pair down kernel): each routed row
    // adds w * Y-row into its token's fp32 sum by vector reductions, and one
    // pass rounds the sums to the output; Y is neither stored nor re-read.
    // Measured on GB300 it does not pay: the reductions slow the down GEMM
    // more than the combine pass costs (128-expert layer 0.377 vs 0.348 ms,
    // Mixtral prefill 1.900 vs 1.875 ms); off by default.
    const char* fcv = std::getenv("CB_MOE_FUSED_COMBINE");
    h->fused_combine = h->pair_dn && fcv != nullptr && std::strcmp(fcv, "1") == 0;
    // programmatic dependent launch between the forward's kernels with
    // CB_MOE_PDL=1.  Measured on GB300 it does not pay: decode layer -0.4 %,
    // 128-expert layer +1.7 % (the next kernel's early CTAs wait beside the
    // running one), Mixtral prefill unchanged per SM clock; off by default.
    const char* pdv = std::getenv("CB_MOE_PDL");
    h->use_pdl = pdv != nullptr && std::strcmp(pdv, "1") == 0;
    // forwards replay captured CUDA graphs unless CB_MOE_GRAPHS=0
    const char* grv = std::getenv("CB_MOE_GRAPHS");
    h->use_graphs = !(grv != nullptr && std::strcmp(grv, "0") == 0);
    // With the mma router, each router block ranks its routed pairs while the
    // ids are at hand, and one small scan of the per-block counts replaces the
    // dispatch's own counting passes, when those counts fit the scan's shared
    // memory.  (Measured on GB300: router + dispatch 44.6 vs 47.9 us at the
    // Mixtral prefill layer.  In the tcgen05 router the per-expert ballots
    // cost more than they save: +10 us on the 128-expert layer, so it is not
    // built there.)  CB_MOE_FUSED_RANKS=0 keeps the dispatch's ranking.
    const char* fv = std::getenv("CB_MOE_FUSED_RANKS");
    const int rb = router_rank_block(cfg->n_experts);
    const int64_t nb = (static_cast<int64_t>(cfg->n_tokens) + rb - 1) / rb;
    h->rank_block = 0;
    h->n_rank_blocks = 0;
    const bool fused_ranks = !(fv != nullptr && std::strcmp(fv, "0") == 0);
    if (!h->router_tc && !hashr && (nb + 1) * (cfg->n_experts + 1) <= kFusedScanWords && fused_ranks) {
      h->rank_block = rb;
      h->n_rank_blocks = static_cast<int32_t>(nb);
    }
    // The router, the ranking and the row copy run as one cooperative launch
    // that reads x from HBM once (the copy finds its rows in L2) and needs no
    // scan kernel in between: with the mma router for up to 16 experts (d a
    // multiple of 512), with the tcgen05 router for 17 to 256 (d a multiple
    // of 64).  CB_MOE_ROUTE_DISPATCH=0 keeps the separate router and dispatch
    // kernels; CB_MOE_FUSED_RANKS=0 implies it.
    const char* rdv = std::getenv("CB_MOE_ROUTE_DISPATCH");
    h->rd_grid = 0;
    h->rd_box = 0;
    const bool rd_ok = !hashr && fused_ranks && !(rdv != nullptr && std::strcmp(rdv, "0") == 0) &&
                       static_cast<int64_t>(cfg->n_tokens) * cfg->top_k + 128ll * cfg->n_experts < (1ll << 31);
    if (rd_ok && !h->router_tc &&
        route_dispatch_supported(cfg->n_tokens, cfg->d_model, cfg->n_experts, cfg->top_k, h->num_sms)) {
      h->rd_grid = route_dispatch_grid(cfg->n_tokens, h->num_sms);
      h->rank_block = 0;
      h->n_rank_blocks = 0;
    } else if (rd_ok && h->router_tc &&
               route_dispatch_tc_supported(cfg->n_tokens, cfg->d_model, cfg->n_experts, cfg->top_k, h->num_sms)) {
      h->rd_grid = route_dispatch_tc_grid(cfg->n_tokens, h->num_sms);
      h->rd_box = route_dispatch_tc_box_rows(cfg->n_tokens, h->rd_grid);
    }
    // Otherwise (tcgen05 and hash routers, or CB_MOE_FUSED_RANKS=0) the
    // dispatch ranks the pairs itself.  Up to 65536 routed pairs its
    // counting, scan, ranking and row copy run as one cooperative launch of
    // one block per SM: measured on GB300, the 128-expert layer's dispatch
    // takes 38.3 us instead of 43.2 us with the separate count / scan /
    // scatter / copy kernels, while the int8 layer's (98304 pairs, an 805 MB
    // row copy) takes 172.2 us instead of 170.3 us.  CB_MOE_DISPATCH=split |
    // coop overrides.
    const char* dv = std::getenv("CB_MOE_DISPATCH");
    const bool coop_pref = dv != nullptr ? std::strcmp(dv, "coop") == 0 : routed <= kCoopMaxPairs;
    h->coop_blocks = 0;
    if (h->rank_block == 0 && h->rd_grid == 0 && cfg->n_experts <= 256 && coop_pref) {
      int g = dispatch_coop_max_blocks(h->num_sms);
      g = std::min(g, kFusedScanWords / cfg->n_experts);  // rows of counts the chunk buffer holds
      g = std::min(g, cfg->n_tokens);
      h->coop_blocks = std::max(g, 0);
    }
  }
  ok = ok && make_tmap(&h->tm_wr, h->wr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, E, 64,
                       static_cast<uint32_t>(router_tc_rows(cfg->n_experts)));
  h->timing = (cfg->flags & CB_FLAG_STAGE_TIMING) != 0;
  h->timing_events = h->timing;
  for (int i = 0; ok && h->timing && i <= CB_N_STAGES; ++i) ok = cudaEventCreate(&h->ev[i]) == cudaSuccess;
  // the guard bands last: the workspace memsets above span them
  for (int i = 0; ok && i < h->n_guards; ++i)
    ok = cudaMemset(h->block + h->guard_off[i], kGuardByte, kGuardBytes) == cudaSuccess;
  ok = ok && create_sync_objects(h);
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    destroy_sync_objects(h);
    cudaFree(h->block);
    delete h;
    return CB_ERR_CUDA;
  }
  // CB_MOE_LOG=1: one line on stderr with the paths this handle runs
  const char* lv = std::getenv("CB_MOE_LOG");
  if (lv != nullptr && std::strcmp(lv, "1") == 0) {
    static const char* const kW[] = {"bf16", "int8", "int4", "fp8"};
    static const char* const kR[] = {"softmax", "raw", "hash"};
    const char* router = cfg->router_mode == CB_ROUTER_HASH ? "hash" : h->router_tc ? "tcgen05" : "mma";
    const char* dispatch = h->rd_grid > 0 ? "fused-with-router" : h->rank_block > 0 ? "router-ranked"
                           : h->coop_blocks > 0 ? "cooperative" : "split";
    const char* gemm = int8w ? (h->int8_tm ? "tensor-memory quantised" : "shared-memory int8")
                             : (h->pair_gu || h->pair_dn) ? "cta-pair" : "single-cta";
    std::fprintf(stderr,
                 "cbmoe: T=%d d=%d f=%d E=%d k=%d weights=%s gate=%s router=%s dispatch=%s gemm=%s "
                 "pair=%d/%d graphs=%d pdl=%d fused_combine=%d guards=%d workspace=%.1f MB sms=%d\n",
                 cfg->n_tokens, cfg->d_model, cfg->d_ff, cfg->n_experts, cfg->top_k, kW[cfg->wdtype],
                 kR[cfg->router_mode], router, dispatch, gemm, h->pair_gu ? 1 : 0, h->pair_dn ? 1 : 0,
                 h->use_graphs ? 1 : 0, h->use_pdl ? 1 : 0, h->fused_combine ? 1 : 0, h->n_guards,
                 static_cast<double>(L.total) / 1e6, h->num_sms);
  }
  *out = h;
  return CB_OK;
}

cb_status_t cb_moe_forward(cb_moe_t* h, const void* x, void* out, void* stream) {
  const cb_status_t st = check_forward_args(h, x, out, 2);
  if (st != CB_OK) return st;
  if (h->cfg.n_tokens == 0) return CB_OK;
  if (fault_injected("launch")) return CB_ERR_CUDA;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return CB_ERR_CUDA;
  return device_forward(h, 0, x, out, static_cast<cudaStream_t>(stream),
                        [&](cudaStream_t s) { return enqueue_forward(h, x, out, false, s); });
}

cb_status_t cb_moe_forward_f32out(cb_moe_t* h, const void* x, float* out, void* stream) {
  const cb_status_t st = check_forward_args(h, x, out, 4);
  if (st != CB_OK) return st;
  if (h->cfg.n_tokens == 0) return CB_OK;
  if (fault_injected("launch")) return CB_ERR_CUDA;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return CB_ERR_CUDA;
  return device_forward(h, 1, x, out, static_cast<cudaStream_t>(stream),
                        [&](cudaStream_t s) { return enqueue_forward(h, x, out, true, s); });
}

cb_status_t cb_moe_forward_host(cb_moe_t* h, const void* x_host, void* out_host, void* stream) {
  if (h == nullptr || x_host == nullptr || out_host == nullptr) return CB_ERR_INVALID_ARG;
  if (h->cfg.n_tokens == 0) return CB_OK;
  if (fault_injected("launch")) return CB_ERR_CUDA;
  const cudaStream_t user = static_cast<cudaStream_t>(stream);
  if (capturing(user)) return CB_ERR_UNSUPPORTED;  // the copies run on the handle's own streams
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok) return CB_ERR_CUDA;
  const uint64_t bytes = static_cast<uint64_t>(h->cfg.n_tokens) * h->cfg.d_model * 2;
  const int b = h->host_slot;
  h->host_slot ^= 1;
  // 1. x into staging slot b, once the layer that last read the slot is done
  if (cudaStreamWaitEvent(h->hs_in, h->hfwd_done[b], 0) != cudaSuccess ||
      cudaMemcpyAsync(h->x_stage[b], x_host, bytes, cudaMemcpyHostToDevice, h->hs_in) != cudaSuccess ||
      cudaEventRecord(h->hin_done[b], h->hs_in) != cudaSuccess)
    return CB_ERR_CUDA;
  // 2. the layer, after its input copy, after the copy out of the slot's
  // previous result, and after the handle's last forward
  if (cudaStreamWaitEvent(h->hs_comp, h->hin_done[b], 0) != cudaSuccess ||
      cudaStreamWaitEvent(h->hs_comp, h->hout_done[b], 0) != cudaSuccess || !wait_last_forward(h, h->hs_comp))
    return CB_ERR_CUDA;
  const cb_status_t st = run_graphed(h, 2 + b, h->x_stage[b], h->out_stage[b], h->hs_comp, [&](cudaStream_t s) {
    return enqueue_forward(h, h->x_stage[b], h->out_stage[b], false, s);
  });
  if (st != CB_OK) return st;
  if (cudaEventRecord(h->hfwd_done[b], h->hs_comp) != cudaSuccess || !mark_last_forward(h, h->hs_comp))
    return CB_ERR_CUDA;
  // 3. out back to the host, then the caller's stream waits for it
  if (cudaStreamWaitEvent(h->hs_out, h->hfwd_done[b], 0) != cudaSuccess ||
      cudaMemcpyAsync(out_host, h->out_stage[b], bytes, cudaMemcpyDeviceToHost, h->hs_out) != cudaSuccess ||
      cudaEventRecord(h->hout_done[b], h->hs_out) != cudaSuccess ||
      cudaStreamWaitEvent(user, h->hout_done[b], 0) != cudaSuccess)
    return CB_ERR_CUDA;
  return CB_OK;
}

cb_status_t cb_moe_routing(const cb_moe_t* h, cb_routing_view_t* v) {
  if (h == nullptr || v == nullptr) return CB_ERR_INVALID_ARG;
  v->ids = h->ids;
  v->w = h->w;
  v->counts = h->counts;
  v->offsets = h->offsets;
  v->tok = h->tok;
  v->inv = h->inv;
  v->logits = h->logits;
  v->tile_offsets = h->mtile_off;
  return CB_OK;
}

cb_status_t cb_moe_stage_times(cb_moe_t* h, float* ms, int32_t n) {
  if (h == nullptr || ms == nullptr || n < CB_N_STAGES) return CB_ERR_INVALID_ARG;
  if (!h->timing) return CB_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok || cudaEventSynchronize(h->ev[CB_N_STAGES]) != cudaSuccess) return CB_ERR_CUDA;
  for (int i = 0; i < CB_N_STAGES; ++i)
    if (cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) return CB_ERR_CUDA;
  return CB_OK;
}

cb_status_t cb_moe_set_stage_timing(cb_moe_t* h, int32_t on) {
  if (h == nullptr || !h->timing_events) return CB_ERR_INVALID_ARG;
  h->timing = on != 0;
  return CB_OK;
}

cb_status_t cb_moe_check_guards(cb_moe_t* h) {
  if (h == nullptr || h->n_guards == 0) return CB_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) return CB_ERR_CUDA;
  std::vector<uint8_t> band(kGuardBytes);
  for (int i = 0; i < h->n_guards; ++i) {
    if (cudaMemcpy(band.data(), h->block + h->guard_off[i], kGuardBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
      return CB_ERR_CUDA;
    for (uint8_t v : band)
      if (v != kGuardByte) return CB_ERR_DEVICE;
  }
  return CB_OK;
}

cb_status_t cb_moe_last_error(cb_moe_t* h) {
  if (h == nullptr) return CB_ERR_INVALID_ARG;
  DeviceGuard guard(h->cfg.device);
  if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) return CB_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CB_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(h->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CB_ERR_CUDA;
  return static_cast<cb_status_t>(v);
}

cb_status_t cb_moe_free(cb_moe_t* h) {
  if (h == nullptr) return CB_OK;
  cb_status_t st = CB_OK;
  {
    DeviceGuard guard(h->cfg.device);
    if (!guard.ok || cudaDeviceSynchronize() != cudaSuccess) st = CB_ERR_CUDA;
    for (int i = 0; h->timing_events && i <= CB_N_STAGES; ++i)
      if (h->ev[i] != nullptr) cudaEventDestroy(h->ev[i]);
    for (auto& g : h->graphs)
      if (g.exec != nullptr) cudaGraphExecDestroy(g.exec);
    destroy_sync_objects(h);
    if (cudaFree(h->block) != cudaSuccess) st = CB_ERR_CUDA;
  }
  delete h;
  return st;
}

}  // extern "C"
