/*
 * moe.h -- C ABI of libmoe: forward pass of one sparse Mixture-of-Experts
 * FFN layer on an NVIDIA B300 (sm_103a).
 *
 * What the layer computes (the pages describe a gating network that picks a
 * few experts per token -- kongchang.com, section "Architecture: The 40B
 * Total vs. 2.5B Active Trade-off" -- with 256 routed experts, 6 selected per
 * token and one always-active shared expert -- evermx.com review, section
 * "Sparse architecture"; futurpulse.com, section "How does Flint use 39.8B
 * parameters efficiently?"):
 *
 *   l[t][e]  = sum_i x[t][i] * Wr[e][i] + b[e]                 (fp32 router)
 *   idx[t]   = the k experts with the largest l[t][.], larger logit first,
 *              lower expert index first on equal logits
 *   gate[t]  = softmax of l[t][idx[t][0..k)]   (renormalised top-k gates)
 *   E_e(v)   = Wd_e ( silu(Wg_e v) * (Wu_e v) ),  silu(z) = z / (1 + e^-z)
 *   y[t]     = sum_j gate[t][j] * E_{idx[t][j]}(x[t])  +  S(x[t])  [+ x[t]]
 *
 * where S is the shared expert (same SwiGLU form, weight 1).  The pages give
 * counts, not the router function, gate normalisation or activation; the
 * readings above are the ones this library implements.
 *
 * Conventions for every function below:
 *  - Pointers named *_host are host memory; every other data pointer is
 *    device memory of the current CUDA device.
 *  - Nothing throws, exits or traps.  Argument errors are found on the host
 *    before any launch and leave no side effect.
 *  - Work is enqueued on the caller's stream; moe_route and moe_forward do
 *    not synchronise and do not allocate.  One handle serves one stream at
 *    a time (the handle's workspace is reused by every call).
 *  - T == 0 is a no-op returning MOE_OK.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_H__
typedef struct CUstream_st* cudaStream_t;
#endif

typedef struct moe_layer* moe_handle;          /* opaque, owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL where a pointer is required, bad size, T > max_tokens, misaligned */
  MOE_ERR_UNSUPPORTED = 2,   /* shape or dtype combination this build does not implement */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch error, no device, ...) */
  MOE_ERR_OOM = 4,           /* workspace allocation failed in moe_create */
  MOE_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out (reported by moe_check) */
  MOE_ERR_RANGE = 6          /* a value out of its range, reported by the check calls: NVFP4 weights on the
                                tensor-core path, an intermediate h / xs^2 saturated f16 (moe_check); a
                                negative decode position (moe_attn_check) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_NVFP4 = 2 } moe_dtype;

/* Which expert-FFN kernels moe_forward uses. */
typedef enum {
  MOE_PATH_AUTO = 0,   /* T <= 8 with bf16 weights and activations, E <= 256 and d, F, F_s multiples of
                          256: one persistent cooperative launch (routing, gate/up, down with grid-wide
                          barriers between them); otherwise the tcgen05 grouped GEMM when the weights
                          allow it, else the GEMV kernels */
  MOE_PATH_GEMV = 1,   /* always the weight-streaming GEMV kernels */
  MOE_PATH_TC = 2      /* always the tcgen05 grouped GEMM: bf16 activations with bf16 weights (d, F, F_s
                          multiples of 128) or NVFP4 weights (multiples of 256; the codes are decoded into
                          tensor memory and x and h are carried in f16 with exact power-of-two scales) */
} moe_path;

typedef struct {
  int32_t d;             /* hidden width; multiple of 64, at most 6400 */
  int32_t ffn;           /* routed expert FFN width F; multiple of 64 */
  int32_t shared_ffn;    /* shared expert FFN width F_s (multiple of 64), 0 = no shared expert */
  int32_t num_experts;   /* E, 1..512 */
  int32_t top_k;         /* k, 1..8, k <= E */
  int32_t max_tokens;    /* largest T any call will pass; sizes the workspace */
  int32_t act_dtype;     /* MOE_F32 or MOE_BF16: type of x and y */
  int32_t weight_dtype;  /* MOE_F32 (with F32 activations), MOE_BF16 or MOE_NVFP4 (with BF16 activations) */
  int32_t add_residual;  /* nonzero: y = x + moe(x) */
  int32_t path;          /* moe_path */
  int32_t gemv_max_tokens; /* MOE_PATH_AUTO: T <= this uses the GEMV kernels even when tcgen05 could; 0 = never */
  int32_t wait_timeout_ms; /* limit of every device-side spin wait; 0 = default (2000 ms) */
  int32_t deterministic;   /* 1: the tcgen05 paths combine each token's expert outputs in a fixed order
                              (gate-weighted per-slot rows, summed in selection order, then the shared
                              expert and x), so repeated calls agree bit for bit; 0 (default): they add
                              into an fp32 accumulator with atomics, in arrival order (equal up to fp32
                              rounding order).  The persistent and GEMV paths are fixed-order either way.
                              Costs a [max_tokens (k + 1)][d] fp32 buffer and its traffic. */
} moe_config;

/*
 * Weights, borrowed: device pointers that must stay valid and unchanged for
 * the handle's lifetime (no copy is made).  All are 16-byte aligned.
 *
 * F32 / BF16 weights (row-major, the reduction dimension contiguous):
 *   router_w [E][d] fp32, router_b [E] fp32 or NULL (= zeros)
 *   w_gate, w_up [E][F][d];  w_down [E][d][F]
 *   ws_gate, ws_up [F_s][d]; ws_down [d][F_s]     (ignored when shared_ffn == 0)
 * NVFP4 weights: the same pointers hold packed e2m1 codes, two per byte,
 *   element 2i in the low nibble, rows of K/2 bytes (K = reduction width);
 *   s_* hold one e4m3 scale per 16 consecutive elements of a row
 *   ([rows][K/16] bytes); t_* hold one fp32 scale per matrix ([E] for
 *   routed experts, [1] for the shared expert).  Weight = e2m1 * e4m3 * fp32.
 */
typedef struct {
  const float* router_w;
  const float* router_b;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const void* ws_gate;
  const void* ws_up;
  const void* ws_down;
  const uint8_t* s_gate;
  const uint8_t* s_up;
  const uint8_t* s_down;
  const uint8_t* ss_gate;
  const uint8_t* ss_up;
  const uint8_t* ss_down;
  const float* t_gate;
  const float* t_up;
  const float* t_down;
  const float* ts_gate;
  const float* ts_up;
  const float* ts_down;
} moe_weights;

/* Human-readable name of a status; never NULL. */
const char* moe_status_string(moe_status s);

/*
 * Validate cfg and w, allocate the workspace for cfg->max_tokens tokens and
 * build the tensor maps over the weights.  On success *out owns that
 * memory until moe_destroy.  On failure *out is NULL and nothing is held.
 * `stream` is used for the workspace's initial clearing (synchronised
 * before return).
 */
moe_status moe_create(const moe_config* cfg, const moe_weights* w, cudaStream_t stream,
                      moe_handle* out);

/* Free the handle and its workspace (synchronises the device first). NULL is a no-op. */
moe_status moe_destroy(moe_handle h);

/*
 * Routing only: the gating network that scores each token against the routed
 * experts and keeps a few of them (kongchang.com, section "Architecture: The
 * 40B Total vs. 2.5B Active Trade-off"), 6 of 256 per token in Flint
 * (evermx.com review, Feature Overview, "Sparse architecture").  The router
 * function, tie rule and renormalisation are this library's readings (top of
 * this file).
 *
 * x [T][d] (act_dtype), 16-byte aligned.  Writes idx [T][k] int32 (larger
 * gate first) and gate [T][k] fp32 (required), and counts [E] int32 = tokens
 * routed to each expert (optional, NULL to skip).  All buffers are
 * caller-owned device memory.  Errors: MOE_ERR_INVALID_ARG for a NULL handle,
 * x, idx or gate, T < 0 or T > max_tokens, or misaligned pointers (checked
 * before any launch); MOE_ERR_CUDA if a launch fails.
 */
moe_status moe_route(moe_handle h, const void* x, int32_t T, int32_t* idx, float* gate,
                     int32_t* counts, cudaStream_t stream);

/*
 * Full layer: routing as in moe_route, each selected expert and the
 * always-active shared expert on the token (evermx.com review, Feature
 * Overview, "Sparse architecture"; futurpulse.com, section "How does Flint use
 * 39.8B parameters efficiently?"), gate-weighted sum, and the residual add
 * that joins the 47 MoE layers when add_residual is set (swarmz.net, section
 * "The architecture, in plain terms").
 *
 * x [T][d] and y [T][d] in act_dtype, caller-owned device memory, 16-byte
 * aligned, not overlapping.  idx_out [T][k] and gate_out [T][k] receive the
 * routing when non-NULL.  T <= max_tokens.  Errors: MOE_ERR_INVALID_ARG for a
 * NULL handle or buffer, T out of range, misalignment or overlapping x and y
 * (checked before any launch); MOE_ERR_CUDA if a launch fails.  Device-side
 * timeouts and f16 saturation show up in moe_check.
 */
moe_status moe_forward(moe_handle h, const void* x, int32_t T, void* y, int32_t* idx_out,
                       float* gate_out, cudaStream_t stream);

/*
 * Full layer on host buffers: copies x_host [T][d] to the device, runs
 * moe_forward and copies y back to y_host [T][d]; returns after y_host is
 * written (synchronises `stream`).  Page-locked host memory makes the copies
 * asynchronous DMA; pageable memory works but is slower.
 */
moe_status moe_forward_host(moe_handle h, const void* x_host, int32_t T, void* y_host,
                            cudaStream_t stream);

/*
 * The token-slot grouping of the last moe_route / moe_forward call on this
 * handle (with the same T).  Grouping token-slots by expert is the scheduling
 * step the pages single out for MoE throughput (kongchang.com, section
 * "Architecture: The 40B Total vs. 2.5B Active Trade-off"; uneven expert use:
 * futurpulse.com, section "How does Flint use 39.8B parameters efficiently?"): offsets [E+1] (exclusive scan of counts),
 * tok_of_slot [T*k] (token of each grouped slot; slots of one expert are
 * contiguous and in (token, j) order) and slot_of [T][k] (grouped position
 * of slot (t, j)).  Any output may be NULL.  Enqueued on `stream`.
 */
moe_status moe_get_grouping(moe_handle h, int32_t T, int32_t* offsets, int32_t* tok_of_slot,
                            int32_t* slot_of, cudaStream_t stream);

/*
 * Synchronise `stream`, then report and clear the device error word:
 * MOE_ERR_TIMEOUT if a bounded wait ran out since the last check,
 * MOE_ERR_RANGE if an f16 intermediate saturated since then (NVFP4 on the tensor cores),
 * MOE_ERR_CUDA if the stream reported an error, else MOE_OK.
 */
moe_status moe_check(moe_handle h, cudaStream_t stream);

/*
 * Failure-detection self-test (no counterpart on the pages): launch one
 * kernel whose thread waits on an mbarrier that nothing completes, with the
 * wait limited to timeout_us microseconds (1..5,000,000).  The wait runs out,
 * the kernel records MOE_ERR_TIMEOUT in the device error word and returns;
 * moe_check then reports it.  The GPU is not hung and the context stays usable.
 */
moe_status moe_debug_expire_wait(moe_handle h, int32_t timeout_us, cudaStream_t stream);

/*
 * Failure injection (no counterpart on the pages; test support): from now on
 * the nth device allocation the library makes (counting from 1) fails as if
 * the device were out of memory; nth == 0 switches injection off.  The count
 * is process-wide.  Lets a test check that moe_create reports MOE_ERR_OOM
 * and holds nothing afterwards, without exhausting a GPU.  nth < 0 returns
 * MOE_ERR_INVALID_ARG.
 */
moe_status moe_debug_fail_alloc(int32_t nth);

/* Kernels of the layer, as counted by the profiling calls below. */
typedef enum {
  MOE_K_ROUTE = 0,         /* router + top-k + grouping */
  MOE_K_GEMV_GATEUP = 1,   /* weight-streaming gate/up + SwiGLU */
  MOE_K_GEMV_DOWN = 2,     /* weight-streaming down + gated combine */
  MOE_K_TC_GATHER = 3,     /* tcgen05 unit lists, slot-ordered copy of the activations (f16 with scales
                              for NVFP4 weights); after a large-batch router also the slots' grouped
                              positions */
  MOE_K_TC_GATEUP = 4,     /* tcgen05 gate/up + SwiGLU */
  MOE_K_TC_DOWN = 5,       /* tcgen05 down + gated accumulate */
  MOE_K_TC_FINALIZE = 6,   /* fp32 accumulator -> output */
  MOE_K_FUSED = 7,         /* the persistent kernel: routing, gate/up and down in one launch (T <= 8) */
  MOE_K_COUNT = 8
} moe_kernel_id;

/*
 * Per-kernel timing (no counterpart on the pages; measurement support).
 * enable != 0: every later moe_route / moe_forward on this handle records a
 * CUDA event pair around each kernel it launches (pairs come from a pool of
 * max_launches created here; launches beyond it are not timed).  Recording
 * events between kernels serialises them, so timed calls lose the overlap
 * that programmatic dependent launch gives untimed ones.  enable == 0 stops
 * recording and frees the pool.
 */
moe_status moe_profile_enable(moe_handle h, int32_t enable, int32_t max_launches);

/*
 * Synchronise the device, then write per kernel id the summed duration in
 * milliseconds (ms[MOE_K_COUNT]) and the number of timed launches
 * (launches[MOE_K_COUNT]) since the last read, and reset the counts.
 */
moe_status moe_profile_read(moe_handle h, float* ms, int32_t* launches);

/* ------------------------------------------------------------------ stacks */

typedef struct moe_stack* moe_stack_handle;    /* opaque, owned by the library */

/*
 * A stack of MoE layers joined by residual adds, x_{l+1} = bf16(x_l +
 * moe_l(x_l)): the 47 MoE layers of the Flint decoder (swarmz.net, section
 * "The architecture, in plain terms"; the rounding of the residual stream to
 * the activation type between layers is this library's reading).
 *
 * cfg: the shape shared by every layer; add_residual must be nonzero.
 * layers: n_layers (1..4096) weight sets as in moe_create, borrowed for the
 * handle's lifetime.  Creates one moe_create handle per layer (the per-layer
 * path) and, when the shapes allow it, sets up a persistent decode kernel:
 * bf16 activations with bf16 weights (T <= 8) or NVFP4 weights (T <= 32), at
 * most 256 routed experts, d, F and F_s multiples of 256, a device of compute
 * capability 10.x that launches cooperative grids.  That kernel runs every
 * layer of the stack in one launch -- the counterpart of the decode
 * megakernel the pages describe (evermx.com review, Feature Overview,
 * "Kernels and inference").
 * Errors: those of moe_create; MOE_ERR_INVALID_ARG for a NULL argument,
 * n_layers out of range or add_residual == 0; MOE_ERR_OOM if the stack's own
 * workspace cannot be allocated.  On failure *out is NULL and nothing is held.
 */
moe_status moe_stack_create(const moe_config* cfg, const moe_weights* layers, int32_t n_layers,
                            cudaStream_t stream, moe_stack_handle* out);

/* Free the stack, its layer handles and workspace (synchronises the device). NULL is a no-op. */
moe_status moe_stack_destroy(moe_stack_handle h);

/* 1 if moe_stack_forward with T tokens runs the persistent kernel, else 0 (per-layer path).  An
 * NVFP4 stack asked for x_trace runs the per-layer path (same kernels, one launch per layer). */
int32_t moe_stack_uses_persistent(moe_stack_handle h, int32_t T);

/*
 * Run the whole stack: y = layer_{L-1}( ... layer_0(x)), each layer with its
 * residual add.  x [T][d] and y [T][d] in act_dtype, device memory, 16-byte
 * aligned, not overlapping; T <= max_tokens.  Optional traces (NULL to skip):
 * x_trace [L + 1][T][d] receives x and every layer's output (16-byte aligned);
 * idx_trace [L][T][k] int32 and gate_trace [L][T][k] fp32 (both or neither)
 * receive every layer's routing.  Enqueued on `stream`, no host
 * synchronisation.  Errors: MOE_ERR_INVALID_ARG for bad arguments (checked
 * before any launch), MOE_ERR_CUDA if a launch fails (the persistent kernel
 * needs all of its CTAs resident at once: one per SM).  Device-side timeouts
 * show up in moe_stack_check.
 */
moe_status moe_stack_forward(moe_stack_handle h, const void* x, int32_t T, void* y, void* x_trace,
                             int32_t* idx_trace, float* gate_trace, cudaStream_t stream);

/*
 * Synchronise `stream`, then report and clear the error words of the
 * persistent kernel and of every layer handle (as moe_check).
 */
moe_status moe_stack_check(moe_stack_handle h, cudaStream_t stream);

/* ------------------------------------------------------------------ sliding-window attention */

typedef struct moe_attn* moe_attn_handle;      /* opaque, owned by the library */

typedef struct {
  int32_t d;              /* hidden width, a multiple of 256 */
  int32_t n_q;            /* query heads */
  int32_t n_kv;           /* key/value heads; n_q / n_kv <= 8 query heads share one */
  int32_t head_dim;       /* 128 */
  int32_t window;         /* positions attended: the current one and window - 1 before it; at most 4096 */
  int32_t max_batch;      /* largest B (sequences per call), 1..8 */
  int32_t use_rope;       /* nonzero: rotate queries and keys (the sliding-window layers) */
  int32_t add_residual;   /* nonzero: y = x + attn(x) */
  int32_t wait_timeout_ms;/* limit of every device-side wait; 0 = 2000 ms */
  float rope_base;        /* RoPE base (10,000 in this library's reading) */
  float eps;              /* RMSNorm epsilon */
} moe_attn_config;

/* Borrowed device pointers: wq [n_q 128][d], wk and wv [n_kv 128][d], wo
   [d][n_q 128] bf16 (16-byte aligned); q_norm and k_norm [128] fp32 (the
   per-head RMSNorm scales); sinks [n_q] fp32 (one learned logit per head). */
typedef struct {
  const void* wq;
  const void* wk;
  const void* wv;
  const void* wo;
  const float* q_norm;
  const float* k_norm;
  const float* sinks;
} moe_attn_weights;

/*
 * Sliding-window grouped-query attention for decode: 35 of Flint's 49 layers
 * attend over the current token and the 512 before it, with 32 query heads
 * over 4 key/value heads of dimension 128, a per-head QK RMSNorm, learned
 * per-head sinks and RoPE (swarmz.net, section "The architecture, in plain
 * terms"; futurpulse.com, section "How does Flint use 39.8B parameters
 * efficiently?").  Per sequence b at position p: q = Wq x, k = Wk x, v = Wv
 * x; q and k RMS-normalised per head (times q_norm / k_norm) and rotated by
 * RoPE (pairs i, i + 64, angle p base^(-i / 64)); the new k, v written to the
 * cache slot p % window as bf16; o_h = softmax over the window's keys of
 * q_h . k / sqrt(128), with sink_h as one more logit in the denominator, times
 * the values; y = Wo o (+ x).  The readings the pages leave open are listed
 * at the top of this library's design notes.
 *
 * Errors: MOE_ERR_INVALID_ARG (NULL, non-positive sizes, misalignment),
 * MOE_ERR_UNSUPPORTED (head_dim != 128, n_q / n_kv > 8, n_q > 64, d not a
 * multiple of 256, window > 4096, max_batch > 8, no cooperative launch),
 * MOE_ERR_OOM, MOE_ERR_CUDA.
 */
moe_status moe_attn_create(const moe_attn_config* cfg, const moe_attn_weights* w, moe_attn_handle* out);

/*
 * One decode step of B sequences (B <= max_batch), one cooperative launch:
 * x [B][d] bf16, pos [B] int32 (device memory, so a captured graph can be
 * replayed at new positions), k_cache and v_cache [B][window][n_kv][128] bf16
 * (caller-owned ring buffers; slot p % window holds position p; this call
 * writes slot pos[b] % window), y [B][d] bf16.  All device pointers, 16-byte
 * aligned (pos 4-byte), x and y not overlapping.  Enqueued on `stream`.
 * Errors: MOE_ERR_INVALID_ARG (checked before any launch), MOE_ERR_CUDA;
 * timeouts show up in moe_attn_check, and so does a negative position
 * (MOE_ERR_RANGE; that sequence is computed as if at position 0).
 */
moe_status moe_attn_decode(moe_attn_handle h, const void* x, int32_t B, const int32_t* pos, void* k_cache,
                           void* v_cache, void* y, cudaStream_t stream);

/* Synchronise `stream`, then report and clear the error word (MOE_ERR_TIMEOUT, MOE_ERR_RANGE or MOE_OK). */
moe_status moe_attn_check(moe_attn_handle h, cudaStream_t stream);

/* Free the handle (synchronises the device). NULL is a no-op. */
moe_status moe_attn_destroy(moe_attn_handle h);

/* ------------------------------------------------------------------ 4-bit output layer */

typedef struct moe_head* moe_head_handle;      /* opaque, owned by the library */

/*
 * The output layer (lm_head) quantised to 4 bits: the pages say it was, since
 * it is a large share of the weights read per token, and that the shipped
 * low-bit model is NVFP4 (evermx.com review, Feature Overview,
 * "Quantization").  logits[t][v] = sum_i x[t][i] W[v][i], W = e2m1 code x
 * e4m3 block scale (one per 16 values along d) x fp32 matrix scale.
 *
 * codes [vocab][d / 2] bytes (element 2i in the low nibble), scales
 * [vocab][d / 16] e4m3 codes, tscale [1] fp32: device memory, borrowed for
 * the handle's lifetime, codes and scales 16-byte aligned.  d a multiple of
 * 256, vocab a multiple of 64.  wait_timeout_ms limits every device-side wait
 * (0 = 2000 ms).  Errors: MOE_ERR_INVALID_ARG (NULL, non-positive sizes,
 * misalignment), MOE_ERR_UNSUPPORTED (shape), MOE_ERR_OOM, MOE_ERR_CUDA.
 */
moe_status moe_head_create(int32_t d, int32_t vocab, int32_t max_tokens, const uint8_t* codes,
                           const uint8_t* scales, const float* tscale, int32_t wait_timeout_ms,
                           moe_head_handle* out);

/*
 * logits [T][vocab] fp32 (device, 16-byte aligned) from x [T][d] bf16 (device,
 * 16-byte aligned), T <= max_tokens; one launch per 8 tokens, enqueued on
 * `stream`.  The weights are decoded exactly to f16 in registers and x is
 * carried in f16 with an exact power-of-two scale per token; products are
 * accumulated in fp32.  Errors: MOE_ERR_INVALID_ARG (checked before any
 * launch), MOE_ERR_CUDA (launch); timeouts show up in moe_head_check.
 */
moe_status moe_head_forward(moe_head_handle h, const void* x, int32_t T, float* logits, cudaStream_t stream);

/* Synchronise `stream`, then report and clear the head's error word (MOE_ERR_TIMEOUT or MOE_OK). */
moe_status moe_head_check(moe_head_handle h, cudaStream_t stream);

/* Free the handle (synchronises the device). NULL is a no-op. */
moe_status moe_head_destroy(moe_head_handle h);

/*
 * Routing without any device allocation (no counterpart on the pages).
 *
 * For callers that cannot call cudaMalloc -- plugins whose host process owns
 * all device memory, runtimes that forbid allocation after start-up, or
 * latency-critical paths that must not enter an allocator, which may
 * synchronise the device -- and so cannot create a handle.  Computes what
 * moe_route computes (same kernel and arithmetic): idx [T][k] int32, gate
 * [T][k] fp32, and optionally counts [E] int32, from x [T][d] (act_dtype
 * MOE_F32 or MOE_BF16, 16-byte aligned), router_w [E][d] fp32 (16-byte
 * aligned) and router_b [E] fp32 or NULL.
 *
 * Limits: 1 <= T <= 64, E <= 512, k <= 8 (k <= E), d a multiple of 64 and at
 * most 6400; larger sizes return MOE_ERR_INVALID_ARG.  Scratch lives in one fixed array of about
 * 144 KiB inside the library's device image; every device that loads the
 * library holds it until the process exits.  The first call on a device looks
 * up that array's device address (cudaGetSymbolAddress) once, so make the
 * first call on each device before any stream capture.  All calls share the
 * array and it keeps the last call's contents: calls that overlap on the GPU
 * (other streams, other host threads) race and must be serialised.  Calls no
 * cudaMalloc, cudaFree or allocating library routine.  The address is cached
 * for the life of the process: after a cudaDeviceReset of a device, do not
 * call this function on that device again.
 */
moe_status moe_route_noalloc(const void* x, int32_t T, int32_t d, int32_t num_experts, int32_t top_k,
                             int32_t act_dtype, const float* router_w, const float* router_b,
                             int32_t* idx, float* gate, int32_t* counts, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
