// Internal types shared by the host API (moe_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "moe.h"

namespace moe {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 8;
constexpr int kSmallT = 64;          // largest T the single-kernel small-batch router handles
constexpr int kGemvChunkT = 64;      // GEMV path: tokens per pass (longer batches run in passes)
constexpr int kFinRows = 32;         // GEMV down: rows finalised together by the last contributor
constexpr int kTcBN = 128;           // tcgen05 path: largest token tile (MMA N)
constexpr int kTcBM = 128;           // tcgen05 path: weight rows per tile (MMA M)
constexpr int kTcBK = 64;            // tcgen05 path: reduction step per stage (128 bytes of bf16)
constexpr int kTokMajorT = 512;      // tcgen05 path: T at which the down pass turns token-major
constexpr int kMaxKSplit = 8;        // tcgen05 path: most parts a small batch's gate/up tiles split into along K
constexpr int kTc4BN = 64;           // NVFP4 tcgen05 path: largest token tile
constexpr int kTc4KS = 256;          // NVFP4 tcgen05 path: reduction step per stage (16 scale bytes per row)
constexpr unsigned kErrTimeout = 1u << 5;
constexpr unsigned kErrRange = 1u << 6;     // an f16 intermediate saturated (NVFP4 tcgen05 path)

// One unit of tcgen05 work: expert (E = the shared expert), weight-row tile,
// first slot (for the shared expert: first token) and token count (<= kTcBN).
struct __align__(16) TcUnit {   // one 16-byte load or store
  int32_t expert, m_tile, slot0, n;
};

// Device workspace owned by a handle.
struct Workspace {
  int32_t* idx;           // [max_T][k]   routing when the caller passes no buffer
  float* gate;            // [max_T][k]
  float* logits;          // [kSmallT][E] small-batch router scratch
  uint32_t* sel;          // [ceil(max_T/32)][E] token-selection bitmap words (large-batch routers)
  int32_t* bcnt;          // [ceil(max_T/32)][E] per-block expert counts (large-batch routers)
  int32_t* bpref;         // [ceil(max_T/32)][E] exclusive prefix of bcnt over blocks
  int32_t* counts;        // [E + 1]
  int32_t* offsets;       // [E + 2]
  int32_t* tok_of_slot;   // [max_T * k]  token of each grouped slot
  int32_t* src_of_slot;   // [max_T * k]  original slot t * k + j of each grouped slot
  int32_t* slot_of;       // [max_T * k]
  int32_t* active;        // [E + 1] routed experts with tokens, ascending; active[E] = how many
  TcUnit* units_gu;       // tcgen05 gate/up units
  TcUnit* units_dn;       // tcgen05 down units
  int32_t* n_units;       // [2] unit counts (gate/up, down)
  int32_t* uprefix;       // [2][E + 1] first unit-list entry of each routed expert after the shared ones
  float* h32;             // [min(max_T, kGemvChunkT) * (k + 1)][F_max] GEMV intermediate
  __nv_bfloat16* h16;     // [max(max_T, ...) * (k + 1)][F_max] bf16 intermediate (tcgen05 and bf16 GEMV)
  __nv_bfloat16* xp;      // tcgen05 slot-ordered copy of the activations: bf16 [max_T * k][d], or for
                          // NVFP4 weights f16 [max_T * (k + 1)][d] (routed slots, then the tokens)
  float* xs;              // [max_T * (k + 1)] power-of-two scale of each f16 row of xp
  float* ypart;           // [min(max_T, kGemvChunkT) * (k + 1)][d] GEMV down partials
  __half* xh16;           // [min(max_T, kGemvChunkT)][d] NVFP4 GEMV: f16 activations, scaled per token
  float* xsc;             // [min(max_T, kGemvChunkT)] their power-of-two scales
  float* yacc;            // [max_T][d] tcgen05 fp32 accumulator
  float* oslot;           // [max_T (k + 1)][d] gate-weighted down outputs per slot (deterministic mode), or null
  uint32_t* counters;     // router tickets: [0] grid, [1 + b] per token chunk / block
  __nv_bfloat16* wr_split;  // [3][E][d] router weights as bf16 hi, mid, lo (tensor-core router)
  uint64_t* cand;         // [max_T][E / 64][kMaxTopK] tensor-core router: per-slice selection keys
  uint32_t* fin;          // [kGemvChunkT][d / 32] GEMV down completion counts (kept at zero between calls)
  float* gu_part;         // [kMaxKSplit][min(max_T, 64) * (k + 1)][2][F_max] partial gate/up sums (split tiles)
  uint32_t* gu_cnt;       // [4 per gate/up tile] arrivals of a split tile's parts (kept at zero between calls)
  uint32_t* ready;        // [E + 4] tcgen05 gate/up progress (kept at zero between calls): [e] finished
                          // tile quarters of expert e ([E] = the shared expert), [E + 1] CTA quarters
                          // done clearing y_acc, [E + 2] CTA quarters done with all their tiles;
                          // [E + 3] the down pass's next unit to claim
  unsigned int* err;      // device error word
  void* x_stage;          // [max_T][d] moe_forward_host staging
  void* y_stage;
  size_t bytes;           // total allocated
};

// Optional per-launch timing: event pairs recorded around each kernel.
struct Prof {
  std::vector<cudaEvent_t> ev;     // pool, 2 per launch
  std::vector<int> kid;            // kernel id of each recorded pair
  int pending = -1;
  bool on() const { return !ev.empty(); }
  void begin(int id, cudaStream_t s) {
    pending = -1;
    if (!on() || 2 * (kid.size() + 1) > ev.size()) return;
    pending = id;
    cudaEventRecord(ev[2 * kid.size()], s);
  }
  void end(cudaStream_t s) {
    if (pending < 0) return;
    cudaEventRecord(ev[2 * kid.size() + 1], s);
    kid.push_back(pending);
    pending = -1;
  }
};

// Parameters shared by the routing kernels.
struct RouteArgs {
  const void* x;          // [T][d] f32 or bf16
  int T, d, E, k;
  int act_bf16;
  const float* Wr;        // [E][d]
  const float* b;         // [E] or nullptr
  int32_t* idx;           // [T][k]
  float* gate;            // [T][k]
  int32_t* counts_out;    // [E] or nullptr
  Workspace ws;
  int build_tc_units;     // also build tcgen05 unit lists
  int dn_rows;            // Wd rows per down tile (128 weight-major, 256 token-major)
  int tile_n;             // token tile of the unit lists (kTcBN, or kTc4BN for NVFP4 weights)
  int gu_split;           // parts along K of every gate/up tile (1 = none)
  int F, Fs;              // widths (for unit lists)
  int has_shared;
};

// Parameters of the GEMV expert kernels.
struct GemvArgs {
  const void* x;          // [T][d]
  void* y;                // [T][d]
  const int32_t* idx;     // [T][k] (unused by the kernels; the grouping carries it)
  const float* gate;      // [T][k]
  int T, d, F, Fs, E, k;
  int act_bf16, add_residual;
  const void* wg; const void* wu; const void* wd;       // routed stacks
  const void* sg; const void* su; const void* sd;       // shared
  const uint8_t* sc_g; const uint8_t* sc_u; const uint8_t* sc_d;   // nvfp4 block scales
  const uint8_t* ssc_g; const uint8_t* ssc_u; const uint8_t* ssc_d;
  const float* ts_g; const float* ts_u; const float* ts_d;         // nvfp4 tensor scales
  const float* tss_g; const float* tss_u; const float* tss_d;
  Workspace ws;
};

// Raise `func`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device, so it is set once per
// (device, kernel) pair; the bookkeeping is guarded by a mutex, so several
// host threads may make first calls at once.  Make the first call on each
// device before any stream capture.
cudaError_t ensure_smem_limit(const void* func, int bytes);
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel* func, int bytes) {
  return ensure_smem_limit(reinterpret_cast<const void*>(func), bytes);
}

// cuTensorMapEncodeTiled (through the runtime's driver entry point): a rank-D
// tensor with dims[0] contiguous, strides_bytes[i] = byte stride of dimension
// i + 1, box extents box[], no interleave, L2 256-byte promotion, zero fill.
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Every device allocation of the library goes through here, so that
// moe_debug_fail_alloc can make the nth one fail.
cudaError_t dev_malloc(void** p, size_t bytes);

// Largest hidden width d: the small-batch router stages 8 tokens x d fp32
// activations in shared memory under a 200 KiB limit.
constexpr int kRouteSmallSmem = 200 * 1024;
constexpr int kMaxHidden = kRouteSmallSmem / (8 * 4);

// Launchers (return the launch status).
cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s, Prof* prof);
// Tensor-core router for T > 64 with bf16 activations (E a multiple of 64).
cudaError_t launch_route_tc(const RouteArgs& a, const CUtensorMap* tm_x, const CUtensorMap* tm_wr, uint64_t* cand,
                            uint64_t wait_ns, cudaStream_t s, Prof* prof);
// Grouped slot positions after a large-batch router (wpb bitmap words per block).
cudaError_t launch_place(const int32_t* idx, const Workspace& ws, int T, int E, int k, int wpb, cudaStream_t s);

// Grouped position of slot (t, expert e) after a large-batch router: the
// expert's offset, the counts of earlier token blocks, and the earlier tokens
// of this block (from the selection bitmap; blocks of 32 * wpb tokens).
__device__ __forceinline__ int slot_position(const Workspace& ws, int E, int t, int e, int wpb) {
  const int w = t >> 5, b = w / wpb;
  int pos = __ldcg(ws.offsets + e) + __ldcg(ws.bpref + (size_t)b * E + e);
  for (int ww = b * wpb; ww < w; ++ww) pos += __popc(__ldcg(ws.sel + (size_t)ww * E + e));
  return pos + __popc(__ldcg(ws.sel + (size_t)w * E + e) & ((1u << (t & 31)) - 1u));
}

// Splits fp32 router weights w[n] into bf16 hi, mid, lo (out[3][n]).
cudaError_t launch_router_split(const float* w, __nv_bfloat16* out, size_t n, cudaStream_t s);
cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int num_sms, cudaStream_t s, Prof* prof, uint64_t wait_ns);
// Shapes the GEMV kernels are built for: rows of d values span 1, 2, 4 or 8
// x 512 bytes; rows of F values span 16, 32, 64 or 128 chunks of 16 bytes;
// the shared expert, if any, has the routed width.
bool gemv_supported(int wfmt, int d, int F, int Fs);
cudaError_t launch_debug_wait(unsigned int* err, uint64_t limit_ns, cudaStream_t s);

struct TcArgs {
  const CUtensorMap* tm_x;      // x [T][d] (box 64 x kTcBN)
  const CUtensorMap* tm_xp;     // slot-ordered x copy [max_T*k][d] (box 64 x kTcBN)
  const CUtensorMap* tm_wg;     // [E*F][d]
  const CUtensorMap* tm_wu;
  const CUtensorMap* tm_sg;     // [Fs][d]
  const CUtensorMap* tm_su;
  const CUtensorMap* tm_wd;     // [E*d][F]
  const CUtensorMap* tm_sd;     // [d][Fs]
  const CUtensorMap* tm_wd256;  // [E*d][F], box 64 x 256 (token-major down pass)
  const CUtensorMap* tm_sd256;  // [d][Fs], box 64 x 256
  int dn_rows;                  // Wd rows per down tile: 128 (weight-major) or 256 (token-major)
  const CUtensorMap* tm_h;      // [slots][F_max] (box 64 x kTcBN)
  const void* x;
  void* y;
  const float* gate;            // [T][k]
  const int32_t* idx;           // [T][k]
  int wpb;                      // > 0: the gather kernel places slots (bitmap words per router block)
  int T, d, F, Fs, E, k, add_residual;
  int gu_split;                 // parts along K of every gate/up tile (as given to the router)
  Workspace ws;
  uint64_t wait_ns;
  int max_units_gu, max_units_dn;
};
cudaError_t launch_tc(const TcArgs& a, int num_sms, cudaStream_t s, Prof* prof);
// Most unit-list entries a call can produce (token tiles of tile_n).
int tc_max_units_gu(int T, int d, int F, int Fs, int E, int k, int tile_n);
int tc_max_units_dn(int T, int d, int F, int Fs, int E, int k, int tile_n);
// y = bf16(y_acc (+ x)) over T x d values, or with ws.oslot set the fixed-order
// sum of each token's per-slot rows (selection order, then the shared expert's
// row) (+ x); clears ready[0 .. n_ready).
cudaError_t launch_tc_finalize(const Workspace& ws, const void* x, void* y, int T, int d, int k, bool has_shared,
                               bool residual, unsigned int* ready, int n_ready, int num_sms, cudaStream_t s,
                               Prof* prof);

// NVFP4 weights on the tensor cores.  Tensor maps over the packed codes
// (bytes [rows][K / 2], box 128 B x 128 rows, 128-byte swizzle) and the block
// scales (bytes [rows][K / 16], box 16 B x 128 rows); xp / h rows are f16
// (box 64 x 16, 128-byte swizzle).
struct Tc4Args {
  const CUtensorMap* q[3];      // routed codes: gate, up, down
  const CUtensorMap* sc[3];     // routed block scales
  const CUtensorMap* sq[3];     // shared-expert codes
  const CUtensorMap* ssc[3];    // shared-expert block scales
  const CUtensorMap* tm_xp;     // f16 activation rows [max_T * (k + 1)][d]
  const CUtensorMap* tm_h;      // f16 intermediate rows [max_T * (k + 1)][F_max]
  const float* ts[3];           // routed per-matrix scales [E]
  const float* tss[3];          // shared per-matrix scales [1]
  const void* x;
  void* y;
  const float* gate;
  const int32_t* idx;
  int wpb;                      // > 0: the gather kernel places slots (bitmap words per router block)
  int T, d, F, Fs, E, k, add_residual;
  Workspace ws;
  uint64_t wait_ns;
  int max_units_gu, max_units_dn;
};
cudaError_t launch_tc4(const Tc4Args& a, int num_sms, cudaStream_t s, Prof* prof);

// ---------------------------------------------------------------- persistent stack decode
constexpr int kSdMaxT = 8;          // tokens per call of the persistent stack kernel
constexpr int kSdConsumers = 8;     // consumer warps per CTA

// Weights of one layer of a stack (device pointers, bf16 experts, fp32 router).
struct StackLayerPtrs {
  const float* wr;
  const float* br;                  // nullptr = zeros
  const __nv_bfloat16* wg;          // [E][F][d]
  const __nv_bfloat16* wu;
  const __nv_bfloat16* wd;          // [E][d][F]
  const __nv_bfloat16* sg;          // [Fs][d]
  const __nv_bfloat16* su;
  const __nv_bfloat16* sd;          // [d][Fs]
};

// Tensor maps of one layer for the persistent kernel (device memory, [L][kSdMaps]):
// 3-D views {64 values, rows, K / 64 chunks} of the bf16 weight stacks, box
// {64, 8, 4} for gate / up and {64, 16, 4} for down, 128-byte swizzle.
constexpr int kMapWg = 0, kMapWu = 1, kMapWd = 2, kMapSg = 3, kMapSu = 4, kMapSd = 5, kSdMaps = 6;

struct StackArgs {
  const StackLayerPtrs* layers;     // [L], device memory
  const CUtensorMap* maps;          // [L][kSdMaps], device memory
  int L;
  const __nv_bfloat16* x_in;        // [T][d]
  __nv_bfloat16* y_out;             // [T][d]
  __nv_bfloat16* xbuf;              // [2][kSdMaxT][d] residual stream between layers
  float* logits;                    // [4][kSdMaxT][E] partial router logits (quarter rows)
  __nv_bfloat16* h;                 // [kSdMaxT * (k + 1)][Fmax]
  __nv_bfloat16* x_trace;           // [L + 1][T][d] or nullptr
  int32_t* idx_trace;               // [L][T][k] or nullptr
  float* gate_trace;                // [L][T][k] (with idx_trace)
  unsigned* bar;                    // grid barrier counter, zero at launch
  unsigned* err;                    // device error word
  int T, d, F, Fs, E, k;
  int add_residual;                 // y = x + moe(x) (always set for a stack)
  int32_t* g_offsets;               // [E + 1] grouping of layer 0 (exclusive scan of the counts), or nullptr
  int32_t* g_tok_of_slot;           // [T k] with g_offsets
  int32_t* g_slot_of;               // [T k] with g_offsets
  uint64_t wait_ns;
};
size_t stack_decode_smem_bytes(int d, int F, int Fs, int k);
// Whether the persistent kernel can serve a layer of this configuration on
// the current device: bf16 weights and activations, at most 256 experts (one
// warp's top-k), at most 8 per token, widths in whole 256-value segments, a
// device of compute capability 10.x that launches cooperative grids, and its
// shared-memory plan within the device's opt-in limit.  *query_ok = false
// when a device query failed.
bool stack_decode_supported(const moe_config& c, bool* query_ok);
// The kSdMaps 3-D tile views of one layer's weights ({64 values, rows, K / 64},
// 128-byte swizzle; 8-row boxes for gate/up, 16-row boxes for down).
bool stack_layer_views(const moe_config& c, const moe_weights& w, CUtensorMap* maps);

// ---------------------------------------------------------------- persistent decode kernel, NVFP4 weights
constexpr int kS4MaxT = 32;          // tokens per launch of the NVFP4 persistent kernel
constexpr int kS4Consumers = 8;      // consumer warps per CTA
// Tensor maps of one layer, [L][kS4Maps]: index 2 m (codes) and 2 m + 1
// (block scales) for m = routed gate, up, down, shared gate, up, down.
constexpr int kS4Maps = 12;
struct Stack4LayerPtrs {
  const float* wr;                  // [E][d] router (fp32)
  const float* br;                  // [E] or nullptr
  const float* tg; const float* tu; const float* td;      // [E] tensor scales of the routed matrices
  const float* tsg; const float* tsu; const float* tsd;   // [1] tensor scales of the shared matrices
};
struct Stack4Args {
  const Stack4LayerPtrs* layers;    // [L], device memory
  const CUtensorMap* maps;          // [L][kS4Maps], device memory
  int L;
  const __nv_bfloat16* x_in;        // [T][d]
  __nv_bfloat16* y_out;             // [T][d]
  __nv_bfloat16* xbuf;              // [2][kS4MaxT][d] residual stream between layers (L > 1)
  float* logits;                    // [ceil(d / 512)][kS4MaxT][E] partial router logits (512-value parts)
  __half* xh;                       // [kS4MaxT][d] x / xs as f16
  float* xsc;                       // [kS4MaxT] xs: a power of two per token
  __half* h;                        // [kS4MaxT (k + 1)][Fmax] h / xs^2 as f16 (routed slots, then the shared rows)
  float* o;                         // [kS4MaxT (k + 1)][d] gate-weighted down outputs per slot
  int32_t* topk_e;                  // [kS4MaxT k] selections published across the grid (T > 8)
  float* topk_g;                    // [kS4MaxT k] their gates
  int32_t* idx_trace;               // [L][T][k] or nullptr
  float* gate_trace;                // [L][T][k] or nullptr
  int32_t* g_offsets;               // [E + 1] grouping of layer 0, or nullptr
  int32_t* g_tok_of_slot;           // [T k] with g_offsets
  int32_t* g_slot_of;               // [T k] with g_offsets
  unsigned* bar;                    // grid barrier counter, zero at launch
  unsigned* err;                    // device error word
  int T, d, F, Fs, E, k, add_residual;
  uint64_t wait_ns;
};
size_t stack_decode_fp4_smem_bytes();
// Whether the NVFP4 persistent kernel can serve this configuration on the
// current device (NVFP4 weights with bf16 activations, E <= 256, k <= 8,
// d, F, F_s multiples of 256, compute capability 10.x, cooperative launch,
// shared memory within the opt-in limit).  *query_ok = false when a device
// query failed.
bool stack_decode_fp4_supported(const moe_config& c, bool* query_ok);
// The kS4Maps tile maps of one layer (codes: 128-byte boxes with the 128-byte
// swizzle; block scales: 16-byte boxes; 32-row boxes for gate/up, 64 for down).
bool stack_layer_views_fp4(const moe_config& c, const moe_weights& w, CUtensorMap* maps);
cudaError_t launch_stack_decode_fp4(const Stack4Args& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- sliding-window attention (decode)
constexpr int kAtMaxT = 8;          // sequences per attention launch

struct AttnArgs {
  CUtensorMap tm[4];                // Wq, Wk, Wv, Wo as 3-D views {64, rows, K / 64}, box {64, 16, 4}
  const __nv_bfloat16* x;           // [B][d]
  __nv_bfloat16* y;                 // [B][d]
  const int32_t* pos;               // [B] position of each sequence's new token
  __nv_bfloat16* k_cache;           // [B][window][n_kv][128]
  __nv_bfloat16* v_cache;
  const float* q_norm;              // [128]
  const float* k_norm;              // [128]
  const float* sinks;               // [n_q]
  float* qkv;                       // [8][n_q 128 + 2 n_kv 128] projections
  __nv_bfloat16* ob;                // [8][n_q 128] attention output per head
  float* part;                      // [B n_kv splits][8][130] per-split (o, max, sum)
  unsigned* split_cnt;              // [B n_kv] splits finished (kept at zero between calls)
  unsigned* bar;                    // grid barrier counter, zero at launch
  unsigned* err;
  const unsigned long long* rope_turns;   // [64] base^(-2 i / 128) / (2 pi) as 64-bit fractions of a turn
  int B, d, n_q, n_kv, window, use_rope, add_residual, splits;
  float eps;
  uint64_t wait_ns;
};
size_t attn_decode_smem_bytes(int d, int n_q);
cudaError_t launch_attn_decode(const AttnArgs& a, int num_sms, cudaStream_t s);

// ---------------------------------------------------------------- 4-bit output layer
constexpr int kHdMaxT = 8;          // tokens per launch of the output-layer kernel
constexpr int kHdConsumers = 8;

struct HeadArgs {
  CUtensorMap tm_codes;             // codes, box 128 bytes x 64 rows, 128-byte swizzle
  CUtensorMap tm_scales;            // scales, box 16 bytes x 64 rows
  const uint8_t* codes;             // [V][d / 2] e2m1 pairs, element 2i in the low nibble
  const uint8_t* scales;            // [V][d / 16] e4m3 block scales
  const float* tscale;              // [1] matrix scale
  const __nv_bfloat16* x;           // [T][d]
  float* logits;                    // [T][V]
  int T, d, V;
  unsigned* err;
  uint64_t wait_ns;
};
size_t lm_head_smem_bytes(int d);
cudaError_t launch_lm_head(const HeadArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_stack_decode(const StackArgs& a, int num_sms, cudaStream_t s);

}  // namespace moe
