/*
 * cb_moe.h -- C ABI of a GB300 (sm_103a) Mixture-of-Experts FFN layer forward.
 *
 * The layer (the MoE pipeline of "Colibri：面向MoE架构的C语言级高效推理引擎" §2.1,
 * with the init / infer / free host interface of its §2.3):
 *
 *   l[t][e]   = sum_i x[t][i] Wr[e][i] + b[e]                (fp32 logits)
 *   ids[t][:] = the k experts with the largest logits, ties to the lower
 *               index, in (logit descending, index ascending) order
 *   w[t][s]   = exp(l[t][ids[t][s]] - l[t][ids[t][0]]) / sum_{j<k} (same)
 *               (softmax, top-k, renormalised over the k: the gate of
 *               "Colibri：面向MoE模型的高性能C语言推理引擎" §1 and §2.1)
 *   dispatch  : per-expert counts, prefix-sum offsets, and a stable
 *               permutation (expert ascending, then token ascending)
 *   H[r]      = bf16( SiLU(Xp[r] Wg[e]^T) * (Xp[r] Wu[e]^T) )  (SwiGLU,
 *               w1 = gate, w3 = up, w2 = down: same page §4.2)
 *   Y[r]      = H[r] Wd[e]^T                                  (fp32)
 *   out[t]    = bf16( sum_s w[t][s] Y[row(t,s)] )             (combine)
 *
 * int8 experts: W[e][j][i] = s[e][j] * Q[e][j][i] with one fp32 scale per
 * output channel (symmetric per-channel int8, "lshu.cn/news/53496" §4.3);
 * int4 experts: W[e][j][i] = s[e][j] * (q[e][j][i] - z[e][j]) with a scale
 * and an integer zero point per output channel ("m.nxbn.cn/news/47706"
 * §3.2); fp8 experts: W[e][j][i] = s[e][j] * v(c[e][j][i]) for e4m3 bytes c
 * ("discosf.com/news/4774337" §6.3).  The codes (minus the zero point)
 * become bf16 exactly inside the GEMM and the scale multiplies the fp32
 * accumulator.
 *
 * Conventions for every call below:
 *  - bf16 means IEEE bfloat16 stored as 16-bit words; all matrices are
 *    row-major, weights channel-last [out_features][in_features] (first
 *    page §3.1).
 *  - "device" pointers are CUDA device (or managed) memory on the handle's
 *    device, 16-byte aligned; "host" pointers are ordinary host memory
 *    (pinned for asynchronous copies).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued on it (the host-buffer forward uses the
 *    handle's own streams and makes `stream` wait for its result); no call
 *    below synchronises the device except cb_moe_init, cb_moe_free,
 *    cb_moe_last_error and cb_moe_check_guards.
 *  - Errors in arguments are reported before anything is enqueued.  A
 *    non-zero status never leaves a partial forward behind.
 *  - A handle is not thread safe; one forward may be in flight per handle
 *    (each forward reuses the handle's workspace).
 */
#ifndef CB_MOE_H
#define CB_MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CB_API __attribute__((visibility("default")))
#else
#define CB_API
#endif

typedef enum {
  CB_OK = 0,
  CB_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, k > E, x aliasing out, unknown
                              router_mode, hash router with top_k != 1, hash_dims
                              outside 1..CB_MAX_HASH_DIMS or no w_hash          */
  CB_ERR_UNSUPPORTED = 2,  /* d_model or d_ff not a multiple of 256, E > 256, k > 16,
                              wrong GPU (not compute capability 10.3), missing scales     */
  CB_ERR_ALIGNMENT = 3,    /* a pointer not 16-byte aligned                               */
  CB_ERR_OOM = 4,          /* a device allocation in cb_moe_init failed                   */
  CB_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed                 */
  CB_ERR_TIMEOUT = 6,      /* a device-side wait ran past its bound (cb_moe_last_error)   */
  CB_ERR_DEVICE = 7        /* a device-side range check failed, e.g. an expert id out of
                              range or a row past the workspace (cb_moe_last_error)      */
} cb_status_t;

/* Expert weight formats.  CB_W_INT8: symmetric int8 codes q with an fp32
 * scale s per output channel, W = s q ("lshu.cn/news/53496" §4.3).
 * CB_W_INT4: 4-bit codes q in 0..15 with an fp32 scale s and an integer zero
 * point z (uint8, 0..15) per output channel, W = s (q - z)
 * ("m.nxbn.cn/news/47706" §3.2, a channel read as an output row); the codes
 * are packed two to a byte along the input dimension, element 2m in the low
 * nibble of byte m and element 2m + 1 in its high nibble.
 * CB_W_FP8: one e4m3 byte per weight (sign, 4 exponent bits with bias 7, 3
 * mantissa bits: (1 + M/8) 2^(E-7), or (M/8) 2^-6 for E = 0; the NaN bytes
 * 0x7F and 0xFF are not valid weights) with an fp32 scale s per output
 * channel, W = s v(byte): the FP8 of "discosf.com/news/4774337" §6.3, read
 * as the e4m3 format Transformer Engine uses for forward-pass weights.  The
 * layout and scales are those of CB_W_INT8. */
typedef enum { CB_W_BF16 = 0, CB_W_INT8 = 1, CB_W_INT4 = 2, CB_W_FP8 = 3 } cb_wdtype_t;

/*
 * config.router_mode: how each token picks its experts and their weights.
 *  CB_ROUTER_SOFTMAX_TOPK: logits l = x Wr^T + b; the k largest (ties to the
 *    lower index); softmax renormalised over the k,
 *    w_s = exp(l_s - l_0) / sum_j exp(l_j - l_0) ("Colibri：面向MoE模型的高性能C语言
 *    推理引擎" §1, §2.1).  The default.
 *  CB_ROUTER_RAW_LOGITS: the same k experts, and each weight is the raw logit
 *    itself, w_s = l_s: top-k on the raw logits without a softmax
 *    ("Colibri：面向MoE架构的C语言级高效推理引擎" §3.2).
 *  CB_ROUTER_HASH: one expert per token (top_k must be 1, weight 1) from a
 *    d x hash_dims projection r = x W_h ("lshu.cn/news/53496" §2): each r_i a
 *    float sum, left to right over d, of the exact bf16 products; h_i =
 *    (int32)((double)r_i * 1e6) & 0xFFFFF with the int32 conversion
 *    truncating toward zero and saturating (NaN -> 0); expert =
 *    (h_0 ^ h_1 ^ ...) mod E.  No logits are computed (w_router and
 *    router_bias are ignored).
 */
typedef enum { CB_ROUTER_SOFTMAX_TOPK = 0, CB_ROUTER_RAW_LOGITS = 1, CB_ROUTER_HASH = 2 } cb_router_mode_t;
#define CB_MAX_HASH_DIMS 8

/* config.flags */
#define CB_FLAG_KEEP_LOGITS 0x1u   /* also store the fp32 router logits [T][E] */
#define CB_FLAG_STAGE_TIMING 0x2u  /* record CUDA events between the stages of each
                                      forward (see cb_moe_stage_times)          */
#define CB_FLAG_TEST_STALL 0x4u    /* test only: in every forward the gate/up GEMM
                                      waits on a barrier phase that nothing
                                      completes, with all its waits bounded to
                                      1 ms, so the device timeout path runs: the
                                      forward finishes (its output is garbage)
                                      and cb_moe_last_error returns
                                      CB_ERR_TIMEOUT                            */
#define CB_FLAG_GUARDS 0x10u       /* testing and debugging: a 4096-byte band of
                                      0xA5 follows every workspace region;
                                      cb_moe_check_guards reports whether a
                                      kernel wrote into one                     */
#define CB_FLAG_TEST_STALL_DISPATCH 0x8u /* test only: the cooperative dispatch's
                                      grid barrier waits for one block more
                                      than the launch has, bounded to 1 ms:
                                      every block gives up and returns, the
                                      routing tables keep their previous
                                      values (zeros after init), the output is
                                      garbage and cb_moe_last_error returns
                                      CB_ERR_TIMEOUT                            */

typedef struct {
  int32_t n_tokens;   /* T: tokens in every forward on this handle (>= 0)         */
  int32_t d_model;    /* d: multiple of 256                                      */
  int32_t d_ff;       /* f: multiple of 256                                      */
  int32_t n_experts;  /* E: 1..256                                               */
  int32_t top_k;      /* k: 1..min(E, 16)                                        */
  int32_t wdtype;     /* cb_wdtype_t of the expert weights                       */
  int32_t device;     /* CUDA device ordinal                                     */
  uint32_t flags;     /* CB_FLAG_*                                               */
  int32_t router_mode; /* cb_router_mode_t (0 = softmax top-k)                    */
  int32_t hash_dims;  /* CB_ROUTER_HASH: 1..CB_MAX_HASH_DIMS columns of W_h; else 0 */
} cb_moe_config_t;

/* Expert and router weights: device pointers, read only during cb_moe_init. */
typedef struct {
  const void *w_router;     /* bf16 [E][d]                                        */
  const float *router_bias; /* fp32 [E], or NULL for no bias                      */
  const void *w_gate;       /* bf16, int8 or e4m3 [E][f][d]; int4 [E][f][d/2] (w1) */
  const void *w_up;         /* bf16, int8 or e4m3 [E][f][d]; int4 [E][f][d/2] (w3) */
  const void *w_down;       /* bf16, int8 or e4m3 [E][d][f]; int4 [E][d][f/2] (w2) */
  const float *s_gate;      /* fp32 [E][f]  int8, int4 and fp8, else NULL         */
  const float *s_up;        /* fp32 [E][f]  int8, int4 and fp8, else NULL         */
  const float *s_down;      /* fp32 [E][d]  int8, int4 and fp8, else NULL         */
  const void *w_hash;       /* bf16 [hash_dims][d], CB_ROUTER_HASH only, else NULL */
  const uint8_t *z_gate;    /* uint8 [E][f] zero points 0..15, int4 only, else NULL */
  const uint8_t *z_up;      /* uint8 [E][f] zero points, int4 only, else NULL     */
  const uint8_t *z_down;    /* uint8 [E][d] zero points, int4 only, else NULL     */
} cb_moe_weights_t;

typedef struct cb_moe cb_moe_t;   /* opaque handle */

/*
 * Create a layer.  Validates the config (sizes, alignment, GPU), allocates
 * every device buffer the layer will ever use (weights, workspace sized for
 * n_tokens), and copies the weights into handle-owned memory, re-laid out
 * for the GEMMs (gate and up rows interleaved in blocks of 128).  The caller
 * may free its own weight buffers when this returns.  Synchronous.
 * Returns CB_OK and *out, or an error with *out = NULL and nothing leaked.
 */
CB_API cb_status_t cb_moe_init(const cb_moe_config_t *cfg, const cb_moe_weights_t *weights, cb_moe_t **out);

/*
 * One forward pass: x bf16 [T][d] (device) -> out bf16 [T][d] (device).
 * x and out are caller-owned, must not overlap, and must stay valid until
 * the stream has run the work.  Asynchronous on `stream`; no allocation,
 * no host synchronisation.  Device-side failures (bounds, timeouts) are
 * reported later by cb_moe_last_error.
 */
CB_API cb_status_t cb_moe_forward(cb_moe_t *h, const void *x, void *out, void *stream);
/* The forwards of one handle share its workspace.  Each waits for the
 * handle's previous forward, on whatever stream that one ran, unless `stream`
 * is being captured into a graph (then the caller's graph orders them). */

/* Same pass with the combine storing fp32 instead of bf16: out fp32 [T][d]. */
CB_API cb_status_t cb_moe_forward_f32out(cb_moe_t *h, const void *x, float *out, void *stream);

/*
 * Same pass from host memory: x_host (bf16 [T][d]) in, out_host (bf16 [T][d])
 * back.  The input copy, the layer and the output copy run on three streams
 * of the handle, through two handle-owned device staging slots that
 * successive calls alternate between, so one call's copies run beside the
 * next or previous call's layer.  The call does not wait for earlier work on
 * `stream`; later work on `stream` waits for out_host to be written.  With
 * page-locked host buffers the call returns before the copies finish: both
 * buffers must stay untouched until `stream` has been synchronised.
 * CB_ERR_UNSUPPORTED while `stream` is being captured into a graph.
 */
CB_API cb_status_t cb_moe_forward_host(cb_moe_t *h, const void *x_host, void *out_host, void *stream);

/* Device pointers of the routing of the last forward (valid until the next
 * forward or cb_moe_free; read after synchronising its stream). */
typedef struct {
  const int32_t *ids;       /* [T][k] expert ids, slot order                       */
  const float *w;           /* [T][k] gate weights (renormalised softmax, raw
                               logits, or 1 under the hash router)              */
  const int32_t *counts;    /* [E]   rows per expert                               */
  const int32_t *offsets;   /* [E+1] exclusive prefix sum of counts                */
  const int32_t *tok;       /* [T*k] token of each row (expert-major, stable)      */
  const int32_t *inv;       /* [T][k] row of each (token, slot)                    */
  const float *logits;      /* [T][E] fp32 logits with bias, or NULL unless
                               CB_FLAG_KEEP_LOGITS (not written by the hash
                               router)                                          */
  const int32_t *tile_offsets; /* [E+1] prefix sum of ceil(counts/128): the
                               expert-aligned 128-row tiles of the GEMM layout   */
} cb_routing_view_t;

CB_API cb_status_t cb_moe_routing(const cb_moe_t *h, cb_routing_view_t *view);

/*
 * Durations in milliseconds of the stages of the last forward on a handle
 * created with CB_FLAG_STAGE_TIMING, measured by CUDA events recorded on the
 * forward's stream: ms[0] router, ms[1] dispatch (count, scan, scatter,
 * gather), ms[2] gate/up GEMM + SwiGLU, ms[3] down GEMM, ms[4] combine.
 * Waits for the last event.  n must be >= CB_N_STAGES.
 */
#define CB_N_STAGES 5
CB_API cb_status_t cb_moe_stage_times(cb_moe_t *h, float *ms, int32_t n);

/*
 * Turns the stage events on (on != 0) or off for the forwards enqueued after
 * this call, on a handle created with CB_FLAG_STAGE_TIMING (its events exist);
 * CB_ERR_INVALID_ARG for any other handle.  The events are nodes between the
 * stages' kernels, so forwards without them run a little faster: a caller can
 * time its steps with the events off and take stage times from other steps.
 * cb_moe_stage_times reports the last forward that recorded them.  Host-side
 * only; the handle's captured graphs are keyed on the setting.
 */
CB_API cb_status_t cb_moe_set_stage_timing(cb_moe_t *h, int32_t on);

/* Synchronise the device, return the handle's device status word (CB_OK,
 * CB_ERR_TIMEOUT or CB_ERR_DEVICE) and clear it. */
CB_API cb_status_t cb_moe_last_error(cb_moe_t *h);

/* On a handle created with CB_FLAG_GUARDS: synchronises the device and checks
 * every guard band.  CB_OK when all are intact, CB_ERR_DEVICE when a byte of
 * one changed (a kernel wrote past the end of a workspace region),
 * CB_ERR_INVALID_ARG on a handle without guards. */
CB_API cb_status_t cb_moe_check_guards(cb_moe_t *h);

/*
 * Dispatch without any device allocation (the pages have no counterpart of
 * this call; it exists for callers that cannot allocate device memory, such
 * as a host program whose own allocator has reserved the GPU's memory, or a
 * loop that cannot afford cudaMalloc's implicit synchronisation).
 *
 * From routing ids[T][k] (device, each row k distinct experts in [0, E)) it
 * writes counts[E], offsets[E+1], tok[T*k] and inv[T][k] exactly as the
 * dispatch of cb_moe_forward does (rows of expert e in ascending token
 * order).  `status` (device int32, or NULL) receives 0 or CB_ERR_DEVICE
 * (an id out of range) once the stream has run the call.  With status ==
 * NULL that error is not reported anywhere: the call still returns CB_OK,
 * and the pairs with bad ids are missing from tok and inv.  Pass a status
 * word unless the ids are known to be in range.  All pointers are
 * caller-owned device memory, 4-byte aligned; the call is asynchronous on
 * `stream` and runs on the current device.
 *
 * Scratch lives in one static device array of CB_NOALLOC_SCRATCH_BYTES per
 * GPU, held until the process exits; the call returns CB_ERR_UNSUPPORTED
 * without launching anything when
 *   ceil(T*k/2048)*E + (E+1) + ((T*k + 127*E)/128 + 1) + 1
 * 32-bit words exceed it (about T*k <= 2 million pairs at E = 256).  The
 * first call on each device (and the first after that device's context has
 * changed, e.g. after cudaDeviceReset) looks the array's address up and sets
 * a kernel attribute (no allocation; it may load the library's kernels onto
 * the device): make it before any stream capture.  All calls
 * share the array, so calls that overlap on the GPU race: keep them on one
 * stream.  Returns CB_ERR_INVALID_ARG / CB_ERR_UNSUPPORTED / CB_ERR_ALIGNMENT
 * on bad arguments, CB_ERR_CUDA if a launch fails.
 */
#define CB_NOALLOC_SCRATCH_BYTES (1u << 20)
CB_API cb_status_t cb_moe_dispatch_noalloc(const int32_t *ids, int32_t n_tokens, int32_t top_k, int32_t n_experts,
                                           int32_t *counts, int32_t *offsets, int32_t *tok, int32_t *inv,
                                           int32_t *status, void *stream);

/* Number of kernels one forward of this handle launches (router, dispatch
 * kernels, the two grouped GEMMs, combine), fixed at init by the shapes and
 * the kernel choices made there.  Returns CB_ERR_INVALID_ARG on NULL. */
CB_API cb_status_t cb_moe_kernels_per_forward(const cb_moe_t *h, int32_t *n);

/* Bytes of device memory a handle with this config holds (weights + workspace). */
CB_API cb_status_t cb_moe_device_bytes(const cb_moe_config_t *cfg, uint64_t *bytes);

/* Free every buffer of the handle (synchronises the device first).  NULL is OK. */
CB_API cb_status_t cb_moe_free(cb_moe_t *h);

/* Static description of a status code. */
CB_API const char *cb_status_string(cb_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* CB_MOE_H */
