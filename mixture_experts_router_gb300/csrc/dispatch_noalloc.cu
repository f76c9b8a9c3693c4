// cb_moe_dispatch_noalloc: the token dispatch (per-expert counts, prefix-sum
// offsets, stable permutation) for callers that must not allocate device
// memory.
//
// Some callers of this library cannot call cudaMalloc.  Typical cases are an
// inference server or framework whose own caching allocator has already
// reserved the GPU's memory and does not let plug-ins allocate behind its
// back, and latency-critical loops that cannot afford the implicit device
// synchronisation a cudaMalloc/cudaFree may cause.  The handle-based API
// allocates its whole workspace in cb_moe_init, which such a caller cannot
// do.  This entry point needs no handle and allocates nothing: the caller
// passes the routing ids (input) and the dispatch arrays (outputs), and the
// kernels' scratch (per-chunk counts and row bases, tile offsets, tile ->
// expert map, and a status word when the caller gives none) lives in one
// file-scope device array of fixed size, CB_NOALLOC_SCRATCH_BYTES (1 MiB).
// Every GPU that loads the library holds that array until the process exits.
//
// In host code the array's name is only a host-side stand-in, so the device
// address is looked up with cudaGetSymbolAddress once per device, with that
// device current.  The same set-up raises the shared-memory limit of the
// block-scan kernel (cudaFuncSetAttribute, which allocates nothing), so the
// call does not depend on a handle having been made on the device.  The
// first call on each device does this set-up (which may also load the
// library's kernels onto the device), so make that first call before any
// stream capture.  The set-up is keyed on the device's current CUDA context
// as well: after cudaDeviceReset the next call looks the address up again
// in the new context.
//
// All calls share the one array and it keeps the last call's contents.
// Every scratch word a call reads is written earlier in the same call, and
// the status word is cleared at the start of each call.  Calls whose work
// overlaps on the GPU (different streams, different host threads) race on
// the array: serialise them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "cb_moe.h"
#include "internal.h"

using namespace cbmoe;

namespace {

constexpr int64_t kScratchWords = CB_NOALLOC_SCRATCH_BYTES / 4;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_dispatch_scratch[kScratchWords];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry points (the library
// links no driver library), or nullptr if it cannot be had.
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return static_cast<CtxGetCurrentFn>(nullptr);
    }
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

CUcontext current_context() {
  CUcontext c = nullptr;
  CtxGetCurrentFn fn = ctx_get_current();
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_dispatch_scratch on `device` (the current device), or
// nullptr when the set-up fails.  Set up once per device and context: the
// address lookup, and the block scan's shared-memory limit.  Without a way to
// name the context the set-up runs on every call.
int32_t* scratch_on(int device) {
  struct Entry {
    CUcontext ctx;
    int32_t* addr;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  Entry& en = cache[device];
  const CUcontext before = current_context();
  if (before != nullptr && en.ctx == before && en.addr != nullptr) return en.addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || dispatch_prepare() != cudaSuccess) {
    cudaGetLastError();
    en = Entry{nullptr, nullptr};
    return nullptr;
  }
  en = Entry{current_context(), static_cast<int32_t*>(p)};
  return en.addr;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" cb_status_t cb_moe_dispatch_noalloc(const int32_t* ids, int32_t n_tokens, int32_t top_k,
                                               int32_t n_experts, int32_t* counts, int32_t* offsets,
                                               int32_t* tok, int32_t* inv, int32_t* status, void* stream) {
  if (n_tokens < 0 || top_k < 1 || n_experts < 1 || top_k > n_experts) return CB_ERR_INVALID_ARG;
  if (n_experts > 256 || top_k > 16) return CB_ERR_UNSUPPORTED;
  if (counts == nullptr || offsets == nullptr) return CB_ERR_INVALID_ARG;
  if (n_tokens > 0 && (ids == nullptr || tok == nullptr || inv == nullptr)) return CB_ERR_INVALID_ARG;
  const void* ptrs[] = {ids, counts, offsets, tok, inv, status};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned4(p)) return CB_ERR_ALIGNMENT;

  // scratch words: per-chunk counts, tile offsets, tile -> expert map, status
  const int64_t M = static_cast<int64_t>(n_tokens) * top_k;
  const int64_t n_chunks = (M + kDispatchChunk - 1) / kDispatchChunk;
  const int64_t max_mtiles = (M + static_cast<int64_t>(n_experts) * (kTileM - 1)) / kTileM + 1;
  const int64_t need = n_chunks * n_experts + (n_experts + 1) + max_mtiles + 1;
  if (need > kScratchWords) return CB_ERR_UNSUPPORTED;  // beyond the static scratch: T*k too large

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return CB_ERR_CUDA;
  int32_t* scratch = scratch_on(device);
  if (scratch == nullptr) return CB_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  int32_t* chunk = scratch;
  int32_t* mtile_off = chunk + n_chunks * n_experts;
  int32_t* mtile_expert = mtile_off + (n_experts + 1);
  int32_t* err = status != nullptr ? status : mtile_expert + max_mtiles;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return CB_ERR_CUDA;
  if (M == 0) {
    if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * n_experts, s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (n_experts + 1), s) != cudaSuccess)
      return CB_ERR_CUDA;
    return CB_OK;
  }

  DispatchArgs a{};
  a.ids = ids;
  a.T = n_tokens;
  a.k = top_k;
  a.E = n_experts;
  a.n_chunks = static_cast<int32_t>(n_chunks);
  a.chunk = chunk;
  a.counts = counts;
  a.offsets = offsets;
  a.mtile_off = mtile_off;
  a.mtile_expert = mtile_expert;
  a.max_mtiles = static_cast<int32_t>(max_mtiles);
  a.tok = tok;
  a.inv = inv;
  a.err = err;
  return launch_dispatch_ranks(a, kFusedScanWords, s) == cudaSuccess ? CB_OK : CB_ERR_CUDA;
}
