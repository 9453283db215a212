// Host side of the C ABI declared in include/moe.h: argument validation,
// workspace ownership, tensor maps, kernel sequencing on the caller's stream.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "moe_internal.cuh"

using namespace moe;

struct moe_layer {
  moe_config cfg;
  moe_weights w;
  Workspace ws;
  int device = 0;
  int num_sms = 0;
  bool tc_capable = false;
  bool gemv_capable = false;
  bool rtc_capable = false;    // tensor-core router for T > 64
  int n_counters = 64;
  uint64_t wait_ns = 0;
  int max_units_gu = 0, max_units_dn = 0;
  int max_tiles_small = 0;     // gate/up tiles of a batch of at most 64 tokens (split bookkeeping)
  CUtensorMap tm_wg, tm_wu, tm_wd, tm_sg, tm_su, tm_sd, tm_h, tm_xp, tm_wr, tm_wd256, tm_sd256;
  bool tok_major_ok = false;   // 256-row down maps exist
  bool fp4 = false;            // NVFP4 weights (tcgen05 path decodes them into tensor memory)
  CUtensorMap q4[3], sc4[3], sq4[3], ssc4[3];   // NVFP4 codes / block scales: gate, up, down (routed, shared)
  void* block = nullptr;
  // The persistent decode kernels run as a stack of one layer (bf16 weights:
  // T <= kSdMaxT; NVFP4 weights: T <= kS4MaxT)
  bool sd_capable = false;
  bool s4_capable = false;
  CUtensorMap* s4_maps = nullptr;
  Stack4LayerPtrs* s4_layer = nullptr;
  __half* s4_xh = nullptr;
  float* s4_xsc = nullptr;
  __half* s4_h = nullptr;
  float* s4_o = nullptr;
  int32_t* s4_topk_e = nullptr;
  float* s4_topk_g = nullptr;
  void* sd_block = nullptr;          // layer pointers, tensor maps, partial logits, h, barrier counter
  StackLayerPtrs* sd_layer = nullptr;
  CUtensorMap* sd_maps = nullptr;
  float* sd_logits = nullptr;
  __nv_bfloat16* sd_h = nullptr;
  unsigned* sd_bar = nullptr;
  Prof prof;
};

namespace moe {

cudaError_t ensure_smem_limit(const void* func, int bytes) {
  struct Done { int dev; const void* func; int bytes; };
  static std::mutex mu;
  static std::vector<Done> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Done& d : done)
    if (d.dev == dev && d.func == func && d.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (Done& d : done)
    if (d.dev == dev && d.func == func) {
      d.bytes = bytes;
      return cudaSuccess;
    }
  done.push_back({dev, func, bytes});
  return cudaSuccess;
}

std::atomic<int> g_fail_alloc{0};   // > 0: allocations left until the injected failure

cudaError_t dev_malloc(void** p, size_t bytes) {
  int v = g_fail_alloc.load();
  while (v > 0 && !g_fail_alloc.compare_exchange_weak(v, v - 1)) {
  }
  if (v == 1) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

}  // namespace moe

namespace {

inline size_t act_bytes(const moe_config& c) { return c.act_dtype == MOE_F32 ? 4 : 2; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

bool gemv_shape_ok(const moe_config& c) { return gemv_supported(c.weight_dtype, c.d, c.ffn, c.shared_ffn); }

bool tc_shape_ok(const moe_config& c) {
  if (c.act_dtype != MOE_BF16) return false;
  if (c.weight_dtype == MOE_BF16)
    return c.d % kTcBM == 0 && c.ffn % kTcBM == 0 && c.shared_ffn % kTcBM == 0;
  // NVFP4: stages of 256 K values (16 block-scale bytes per row)
  return c.weight_dtype == MOE_NVFP4 && c.d % kTc4KS == 0 && c.ffn % kTc4KS == 0 && c.shared_ffn % kTc4KS == 0;
}
inline int tile_n_of(const moe_config& c) { return c.weight_dtype == MOE_NVFP4 ? kTc4BN : kTcBN; }

// Parts along K for the bf16 gate/up tiles of a small batch.  A batch of a
// few tokens touches few experts, so one unit per (expert, row tile) leaves
// most SMs idle; splitting along K spreads the weight stream over more SMs at
// the cost of a partial-sum round trip per tile.  Measured on B300 (whole
// layer, 16-layer rotation, graph replay): T = 1: 46.8 us unsplit, 39.1 us in
// 4 parts; T = 8: 87.4 / 83.4 us in 2 parts; from T = 32 on every split was
// slower (T = 64: 240 us unsplit, 260 us in 2 parts).
int gu_split_for(const moe_config& c, int T, int num_sms) {
  (void)num_sms;
  if (c.weight_dtype != MOE_BF16 || c.d / kTcBK < 4) return 1;
  if (T <= 2) return 4;
  if (T <= 12) return 2;
  return 1;
}

moe_status validate_config(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->d <= 0 || c->ffn <= 0 || c->shared_ffn < 0 || c->max_tokens <= 0) return MOE_ERR_INVALID_ARG;
  if (c->num_experts < 1 || c->top_k < 1 || c->top_k > c->num_experts) return MOE_ERR_INVALID_ARG;
  if (c->path < MOE_PATH_AUTO || c->path > MOE_PATH_TC || c->gemv_max_tokens < 0 || c->wait_timeout_ms < 0 ||
      c->deterministic < 0 || c->deterministic > 1)
    return MOE_ERR_INVALID_ARG;
  if (c->d % 64 || c->ffn % 64 || c->shared_ffn % 64) return MOE_ERR_UNSUPPORTED;
  if (c->d > kMaxHidden) return MOE_ERR_UNSUPPORTED;
  if (c->num_experts > kMaxExperts || c->top_k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  const bool combo = (c->act_dtype == MOE_F32 && c->weight_dtype == MOE_F32) ||
                     (c->act_dtype == MOE_BF16 && (c->weight_dtype == MOE_BF16 || c->weight_dtype == MOE_NVFP4));
  if (!combo) return MOE_ERR_UNSUPPORTED;
  const bool gemv = gemv_shape_ok(*c), tc = tc_shape_ok(*c);
  if (!gemv && !tc) return MOE_ERR_UNSUPPORTED;
  if (c->path == MOE_PATH_TC && !tc) return MOE_ERR_UNSUPPORTED;
  if (c->path == MOE_PATH_GEMV && !gemv) return MOE_ERR_UNSUPPORTED;
  if ((long long)c->max_tokens * c->top_k > (1LL << 30)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status validate_weights(const moe_config& c, const moe_weights* w) {
  if (!w || !w->router_w || !w->w_gate || !w->w_up || !w->w_down) return MOE_ERR_INVALID_ARG;
  const void* need[] = {w->router_w, w->w_gate, w->w_up, w->w_down};
  for (const void* p : need)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (w->router_b && (reinterpret_cast<uintptr_t>(w->router_b) & 3u)) return MOE_ERR_INVALID_ARG;
  if (c.shared_ffn > 0) {
    if (!w->ws_gate || !w->ws_up || !w->ws_down) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down)) return MOE_ERR_INVALID_ARG;
  }
  if (c.weight_dtype == MOE_NVFP4) {
    const void* s[] = {w->s_gate, w->s_up, w->s_down, w->t_gate, w->t_up, w->t_down};
    for (const void* p : s)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (c.shared_ffn > 0) {
      const void* ss[] = {w->ss_gate, w->ss_up, w->ss_down, w->ts_gate, w->ts_up, w->ts_down};
      for (const void* p : ss)
        if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    }
  }
  return MOE_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 tensor [rows][cols] (cols contiguous), box {box_cols, box_rows}, 128-byte swizzle.
bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D f16 tensor [rows][cols], box {box_cols, box_rows}, 128-byte swizzle.
bool make_map_f16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D byte tensor [rows][cols], box {box_cols, box_rows}; 128-byte swizzle or none.
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace moe {

bool encode_tiled(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return fn(m, type, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe

namespace {

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

RouteArgs route_args(const moe_layer* h, const void* x, int T, int32_t* idx, float* gate, int32_t* counts,
                     bool tc_units) {
  RouteArgs a;
  a.x = x;
  a.T = T;
  a.d = h->cfg.d;
  a.E = h->cfg.num_experts;
  a.k = h->cfg.top_k;
  a.act_bf16 = h->cfg.act_dtype == MOE_BF16;
  a.Wr = h->w.router_w;
  a.b = h->w.router_b;
  a.idx = idx;
  a.gate = gate;
  a.counts_out = counts;
  a.ws = h->ws;
  a.build_tc_units = tc_units ? 1 : 0;
  a.dn_rows = (tc_units && !h->fp4 && T >= kTokMajorT && h->tok_major_ok) ? 2 * kTcBN : kTcBM;
  a.tile_n = tile_n_of(h->cfg);
  a.gu_split = tc_units ? gu_split_for(h->cfg, T, h->num_sms) : 1;
  a.F = h->cfg.ffn;
  a.Fs = h->cfg.shared_ffn;
  a.has_shared = h->cfg.shared_ffn > 0;
  return a;
}

GemvArgs gemv_args(const moe_layer* h, const void* x, void* y, const float* gate, int T) {
  GemvArgs a;
  const moe_weights& w = h->w;
  a.x = x;
  a.y = y;
  a.idx = nullptr;
  a.gate = gate;
  a.T = T;
  a.d = h->cfg.d;
  a.F = h->cfg.ffn;
  a.Fs = h->cfg.shared_ffn;
  a.E = h->cfg.num_experts;
  a.k = h->cfg.top_k;
  a.act_bf16 = h->cfg.act_dtype == MOE_BF16;
  a.add_residual = h->cfg.add_residual != 0;
  a.wg = w.w_gate; a.wu = w.w_up; a.wd = w.w_down;
  a.sg = w.ws_gate; a.su = w.ws_up; a.sd = w.ws_down;
  a.sc_g = w.s_gate; a.sc_u = w.s_up; a.sc_d = w.s_down;
  a.ssc_g = w.ss_gate; a.ssc_u = w.ss_up; a.ssc_d = w.ss_down;
  a.ts_g = w.t_gate; a.ts_u = w.t_up; a.ts_d = w.t_down;
  a.tss_g = w.ts_gate; a.tss_u = w.ts_up; a.tss_d = w.ts_down;
  a.ws = h->ws;
  return a;
}

moe_status check_call(const moe_layer* h, const void* x, int32_t T) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !aligned16(x))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// Routing: the tensor-core router for large bf16 batches, else the fp32 SIMT
// kernels.  tm_x (box 64 x 128 over x) is built here when needed and returned.
moe_status do_route(moe_layer* h, const void* x, int32_t T, int32_t* idx, float* gate, int32_t* counts,
                    bool tc_units, CUtensorMap* tm_x, bool* have_tm_x, cudaStream_t s) {
  const RouteArgs ra = route_args(h, x, T, idx, gate, counts, tc_units);
  if (T > kSmallT && h->rtc_capable) {
    if (!*have_tm_x) {
      if (!make_map_bf16(tm_x, x, (uint64_t)T, (uint64_t)h->cfg.d, kTcBN, kTcBK)) return MOE_ERR_CUDA;
      *have_tm_x = true;
    }
    return cuda_status(launch_route_tc(ra, tm_x, &h->tm_wr, h->ws.cand, h->wait_ns, s, &h->prof));
  }
  return cuda_status(launch_route(ra, h->num_sms, s, &h->prof));
}

// The persistent decode kernel as a stack of one layer: its layer pointers and
// tensor maps in device memory, its scratch (partial logits, h, the grid
// barrier counter).  Leaves sd_capable false when the shapes or the device do
// not allow it (the other paths serve every T then).
moe_status setup_fused4(moe_layer* h, cudaStream_t stream);

moe_status setup_fused(moe_layer* h, cudaStream_t stream) {
  const moe_config& c = h->cfg;
  if (c.weight_dtype == MOE_NVFP4) return setup_fused4(h, stream);
  bool query_ok = true;
  if (!stack_decode_supported(c, &query_ok)) return query_ok ? MOE_OK : MOE_ERR_CUDA;
  CUtensorMap maps[kSdMaps];
  std::memset(maps, 0, sizeof(maps));
  if (!stack_layer_views(c, h->w, maps)) return MOE_OK;
  const moe_weights& w = h->w;
  const StackLayerPtrs lp{w.router_w, w.router_b,
                          static_cast<const __nv_bfloat16*>(w.w_gate), static_cast<const __nv_bfloat16*>(w.w_up),
                          static_cast<const __nv_bfloat16*>(w.w_down), static_cast<const __nv_bfloat16*>(w.ws_gate),
                          static_cast<const __nv_bfloat16*>(w.ws_up), static_cast<const __nv_bfloat16*>(w.ws_down)};
  const size_t Fmax = c.ffn > c.shared_ffn ? c.ffn : c.shared_ffn;
  const size_t nmaps = up256(sizeof(maps)), nlp = up256(sizeof(lp));
  const size_t nlog = up256((size_t)4 * kSdMaxT * c.num_experts * 4);
  const size_t nh = up256((size_t)kSdMaxT * (c.top_k + 1) * Fmax * 2);
  if (dev_malloc(&h->sd_block, nmaps + nlp + nlog + nh + 256) != cudaSuccess) {
    cudaGetLastError();
    h->sd_block = nullptr;
    return MOE_ERR_OOM;
  }
  uint8_t* p = static_cast<uint8_t*>(h->sd_block);
  h->sd_maps = reinterpret_cast<CUtensorMap*>(p); p += nmaps;
  h->sd_layer = reinterpret_cast<StackLayerPtrs*>(p); p += nlp;
  h->sd_logits = reinterpret_cast<float*>(p); p += nlog;
  h->sd_h = reinterpret_cast<__nv_bfloat16*>(p); p += nh;
  h->sd_bar = reinterpret_cast<unsigned*>(p);
  if (cudaMemcpyAsync(h->sd_maps, maps, sizeof(maps), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(h->sd_layer, &lp, sizeof(lp), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->sd_block);
    h->sd_block = nullptr;
    return MOE_ERR_CUDA;
  }
  h->sd_capable = true;
  return MOE_OK;
}

// The NVFP4 persistent kernel as a stack of one layer: tensor maps, layer
// pointers and scratch (partial logits, the f16 copy of x and its scales, h,
// the per-slot down outputs, the barrier counter).
moe_status setup_fused4(moe_layer* h, cudaStream_t stream) {
  const moe_config& c = h->cfg;
  bool query_ok = true;
  if (!stack_decode_fp4_supported(c, &query_ok)) return query_ok ? MOE_OK : MOE_ERR_CUDA;
  CUtensorMap maps[kS4Maps];
  std::memset(maps, 0, sizeof(maps));
  if (!stack_layer_views_fp4(c, h->w, maps)) return MOE_OK;
  const moe_weights& w = h->w;
  const Stack4LayerPtrs lp{w.router_w, w.router_b, w.t_gate, w.t_up, w.t_down, w.ts_gate, w.ts_up, w.ts_down};
  const size_t Fmax = c.ffn > c.shared_ffn ? c.ffn : c.shared_ffn, E = c.num_experts, d = c.d;
  const size_t slots = (size_t)kS4MaxT * (c.top_k + 1);
  const size_t nmaps = up256(sizeof(maps)), nlp = up256(sizeof(lp));
  const size_t nlog = up256((d + 511) / 512 * kS4MaxT * E * 4), nxh = up256((size_t)kS4MaxT * d * 2);
  const size_t nxs = up256((size_t)kS4MaxT * 4), nh = up256(slots * Fmax * 2), no = up256(slots * d * 4);
  const size_t ntk = up256((size_t)kS4MaxT * kMaxTopK * 4);
  if (dev_malloc(&h->sd_block, nmaps + nlp + nlog + nxh + nxs + nh + no + 2 * ntk + 256) != cudaSuccess) {
    cudaGetLastError();
    h->sd_block = nullptr;
    return MOE_ERR_OOM;
  }
  uint8_t* p = static_cast<uint8_t*>(h->sd_block);
  h->s4_maps = reinterpret_cast<CUtensorMap*>(p); p += nmaps;
  h->s4_layer = reinterpret_cast<Stack4LayerPtrs*>(p); p += nlp;
  h->sd_logits = reinterpret_cast<float*>(p); p += nlog;
  h->s4_xh = reinterpret_cast<__half*>(p); p += nxh;
  h->s4_xsc = reinterpret_cast<float*>(p); p += nxs;
  h->s4_h = reinterpret_cast<__half*>(p); p += nh;
  h->s4_o = reinterpret_cast<float*>(p); p += no;
  h->s4_topk_e = reinterpret_cast<int32_t*>(p); p += ntk;
  h->s4_topk_g = reinterpret_cast<float*>(p); p += ntk;
  h->sd_bar = reinterpret_cast<unsigned*>(p);
  if (cudaMemcpyAsync(h->s4_maps, maps, sizeof(maps), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(h->s4_layer, &lp, sizeof(lp), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->sd_block);
    h->sd_block = nullptr;
    return MOE_ERR_CUDA;
  }
  h->s4_capable = true;
  return MOE_OK;
}

moe_status run_fused4(moe_layer* h, const void* x, int32_t T, void* y, int32_t* idx_out, float* gate_out,
                      cudaStream_t s) {
  const moe_config& c = h->cfg;
  if (cudaMemsetAsync(h->sd_bar, 0, 4, s) != cudaSuccess) return cuda_status(cudaGetLastError());
  Stack4Args a;
  a.layers = h->s4_layer;
  a.maps = h->s4_maps;
  a.L = 1;
  a.x_in = static_cast<const __nv_bfloat16*>(x);
  a.y_out = static_cast<__nv_bfloat16*>(y);
  a.xbuf = nullptr;                  // one layer: x_in -> y_out
  a.logits = h->sd_logits;
  a.xh = h->s4_xh;
  a.xsc = h->s4_xsc;
  a.h = h->s4_h;
  a.o = h->s4_o;
  a.topk_e = h->s4_topk_e;
  a.topk_g = h->s4_topk_g;
  a.idx_trace = idx_out;
  a.gate_trace = gate_out;
  a.g_offsets = h->ws.offsets;       // kept for moe_get_grouping
  a.g_tok_of_slot = h->ws.tok_of_slot;
  a.g_slot_of = h->ws.slot_of;
  a.bar = h->sd_bar;
  a.err = h->ws.err;
  a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
  a.add_residual = c.add_residual != 0;
  a.wait_ns = h->wait_ns;
  h->prof.begin(MOE_K_FUSED, s);
  const cudaError_t e = launch_stack_decode_fp4(a, h->num_sms, s);
  h->prof.end(s);
  return cuda_status(e);
}

moe_status run_fused(moe_layer* h, const void* x, int32_t T, void* y, int32_t* idx_out, float* gate_out,
                     cudaStream_t s) {
  const moe_config& c = h->cfg;
  if (cudaMemsetAsync(h->sd_bar, 0, 4, s) != cudaSuccess) return cuda_status(cudaGetLastError());
  StackArgs a;
  a.layers = h->sd_layer;
  a.maps = h->sd_maps;
  a.L = 1;
  a.x_in = static_cast<const __nv_bfloat16*>(x);
  a.y_out = static_cast<__nv_bfloat16*>(y);
  a.xbuf = nullptr;                  // one layer: x_in -> y_out
  a.logits = h->sd_logits;
  a.h = h->sd_h;
  a.x_trace = nullptr;
  a.idx_trace = idx_out;             // routing of the layer, each written when given
  a.gate_trace = gate_out;
  a.bar = h->sd_bar;
  a.err = h->ws.err;
  a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
  a.add_residual = c.add_residual != 0;
  a.g_offsets = h->ws.offsets;       // kept for moe_get_grouping
  a.g_tok_of_slot = h->ws.tok_of_slot;
  a.g_slot_of = h->ws.slot_of;
  a.wait_ns = h->wait_ns;
  h->prof.begin(MOE_K_FUSED, s);
  const cudaError_t e = launch_stack_decode(a, h->num_sms, s);
  h->prof.end(s);
  return cuda_status(e);
}

moe_status run_forward(moe_layer* h, const void* x, int32_t T, void* y, int32_t* idx_out, float* gate_out,
                       cudaStream_t s) {
  const moe_config& c = h->cfg;
  // AUTO, small batches: the persistent kernel (routing, gate/up and down in
  // one launch with grid-wide barriers between the phases)
  if (c.path == MOE_PATH_AUTO && h->sd_capable && T <= kSdMaxT && T > c.gemv_max_tokens)
    return run_fused(h, x, T, y, idx_out, gate_out, s);
  if (c.path == MOE_PATH_AUTO && h->s4_capable && T <= kS4MaxT && T > c.gemv_max_tokens)
    return run_fused4(h, x, T, y, idx_out, gate_out, s);
  int32_t* idx = idx_out ? idx_out : h->ws.idx;
  float* gate = gate_out ? gate_out : h->ws.gate;
  // AUTO: the tensor-core path whenever the weights allow it (it streams the
  // weights faster than the GEMV kernels at every batch size measured), unless
  // the caller asked for GEMV up to gemv_max_tokens.
  const bool tc = c.path == MOE_PATH_TC ||
                  (c.path == MOE_PATH_AUTO && h->tc_capable && (T > c.gemv_max_tokens || !h->gemv_capable));
  if (tc && h->fp4) {
    CUtensorMap tm_x;
    bool have_tm_x = false;
    moe_status st = do_route(h, x, T, idx, gate, nullptr, true, &tm_x, &have_tm_x, s);
    if (st != MOE_OK) return st;
    const moe_weights& w = h->w;
    Tc4Args a;
    for (int m = 0; m < 3; ++m) {
      a.q[m] = &h->q4[m]; a.sc[m] = &h->sc4[m]; a.sq[m] = &h->sq4[m]; a.ssc[m] = &h->ssc4[m];
    }
    a.ts[0] = w.t_gate; a.ts[1] = w.t_up; a.ts[2] = w.t_down;
    a.tss[0] = w.ts_gate; a.tss[1] = w.ts_up; a.tss[2] = w.ts_down;
    a.tm_xp = &h->tm_xp;
    a.tm_h = &h->tm_h;
    a.x = x;
    a.y = y;
    a.gate = gate;
    a.idx = idx;
    a.wpb = T > kSmallT ? (h->rtc_capable ? 4 : 1) : 0;
    a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
    a.add_residual = c.add_residual != 0;
    a.ws = h->ws;
    a.wait_ns = h->wait_ns;
    a.max_units_gu = tc_max_units_gu(T, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, kTc4BN);
    a.max_units_dn = tc_max_units_dn(T, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, kTc4BN);
    return cuda_status(launch_tc4(a, h->num_sms, s, &h->prof));
  }
  if (tc) {
    CUtensorMap tm_x;
    bool have_tm_x = false;
    moe_status st = do_route(h, x, T, idx, gate, nullptr, true, &tm_x, &have_tm_x, s);
    if (st != MOE_OK) return st;
    if (!have_tm_x && !make_map_bf16(&tm_x, x, (uint64_t)T, (uint64_t)c.d, kTcBN, kTcBK)) return MOE_ERR_CUDA;
    TcArgs a;
    a.tm_x = &tm_x;
    a.tm_xp = &h->tm_xp;
    a.tm_wg = &h->tm_wg; a.tm_wu = &h->tm_wu; a.tm_sg = &h->tm_sg; a.tm_su = &h->tm_su;
    a.tm_wd = &h->tm_wd; a.tm_sd = &h->tm_sd; a.tm_h = &h->tm_h;
    a.tm_wd256 = &h->tm_wd256; a.tm_sd256 = &h->tm_sd256;
    a.dn_rows = (T >= kTokMajorT && h->tok_major_ok) ? 2 * kTcBN : kTcBM;
    a.x = x;
    a.y = y;
    a.gate = gate;
    a.idx = idx;
    a.wpb = T > kSmallT ? (h->rtc_capable ? 4 : 1) : 0;
    a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
    a.add_residual = c.add_residual != 0;
    a.ws = h->ws;
    a.wait_ns = h->wait_ns;
    a.gu_split = gu_split_for(c, T, h->num_sms);
    a.max_units_gu = a.gu_split * tc_max_units_gu(T, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, kTcBN);
    a.max_units_dn = tc_max_units_dn(T, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, kTcBN);
    return cuda_status(launch_tc(a, h->num_sms, s, &h->prof));
  }
  const size_t es = act_bytes(c);
  for (int t0 = 0; t0 < T; t0 += kGemvChunkT) {
    const int tc_ = T - t0 < kGemvChunkT ? T - t0 : kGemvChunkT;
    const uint8_t* xc = static_cast<const uint8_t*>(x) + (size_t)t0 * c.d * es;
    uint8_t* yc = static_cast<uint8_t*>(y) + (size_t)t0 * c.d * es;
    int32_t* ic = idx + (size_t)t0 * c.top_k;
    float* gc = gate + (size_t)t0 * c.top_k;
    CUtensorMap tm_x;
    bool have_tm_x = false;
    moe_status st = do_route(h, xc, tc_, ic, gc, nullptr, false, &tm_x, &have_tm_x, s);
    if (st != MOE_OK) return st;
    st = cuda_status(launch_gemv(gemv_args(h, xc, yc, gc, tc_), c.weight_dtype, h->num_sms, s, &h->prof, h->wait_ns));
    if (st != MOE_OK) return st;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or dtype not supported";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime error";
    case MOE_ERR_OOM: return "MOE_ERR_OOM: device allocation failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: device-side wait ran out";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE: an intermediate value saturated its format";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_create(const moe_config* cfg, const moe_weights* w, cudaStream_t stream, moe_handle* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status st = validate_config(cfg);
  if (st != MOE_OK) return st;
  st = validate_weights(*cfg, w);
  if (st != MOE_OK) return st;

  moe_layer* h = new (std::nothrow) moe_layer();
  if (!h) return MOE_ERR_OOM;
  h->cfg = *cfg;
  h->w = *w;
  const moe_config& c = h->cfg;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_CUDA;
  }
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, h->device);
  h->tc_capable = tc_shape_ok(c) && cc_major == 10;
  h->fp4 = c.weight_dtype == MOE_NVFP4;
  h->gemv_capable = gemv_shape_ok(c);
  h->rtc_capable = cc_major == 10 && c.act_dtype == MOE_BF16 && c.num_experts % 64 == 0 && c.d % 64 == 0;
  if ((c.path == MOE_PATH_TC && !h->tc_capable) || (!h->tc_capable && !h->gemv_capable)) {
    delete h;
    return MOE_ERR_UNSUPPORTED;
  }
  h->wait_ns = (uint64_t)(c.wait_timeout_ms > 0 ? c.wait_timeout_ms : 2000) * 1000000ull;

  const size_t Tm = (size_t)c.max_tokens, E = c.num_experts, k = c.top_k, d = c.d;
  const size_t Fmax = c.ffn > c.shared_ffn ? c.ffn : c.shared_ffn;
  const size_t Tg = Tm < (size_t)kGemvChunkT ? Tm : (size_t)kGemvChunkT;
  const size_t nblk = (Tm + 31) / 32;
  if (h->tc_capable) {
    h->max_units_gu = tc_max_units_gu(c.max_tokens, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, tile_n_of(c));
    if (!h->fp4) {   // split gate/up tiles of batches up to 64 tokens
      const int ts = c.max_tokens < kSmallT ? c.max_tokens : kSmallT;
      h->max_tiles_small = tc_max_units_gu(ts, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, kTcBN);
      const int m = kMaxKSplit * h->max_tiles_small;
      if (m > h->max_units_gu) h->max_units_gu = m;
    }
    h->max_units_dn = tc_max_units_dn(c.max_tokens, c.d, c.ffn, c.shared_ffn, c.num_experts, c.top_k, tile_n_of(c));
  }
  struct Part { void** dst; size_t bytes; };
  Workspace& ws = h->ws;
  Part parts[] = {
      {(void**)&ws.idx, Tm * k * 4},
      {(void**)&ws.gate, Tm * k * 4},
      {(void**)&ws.logits, (size_t)kSmallT * E * 4},
      {(void**)&ws.sel, nblk * E * 4},
      {(void**)&ws.bcnt, nblk * E * 4},
      {(void**)&ws.bpref, nblk * E * 4},
      {(void**)&ws.counts, (E + 1) * 4},
      {(void**)&ws.offsets, (E + 2) * 4},
      {(void**)&ws.tok_of_slot, Tm * k * 4},
      {(void**)&ws.src_of_slot, Tm * k * 4},
      {(void**)&ws.slot_of, Tm * k * 4},
      {(void**)&ws.active, (E + 1) * 4},
      {(void**)&ws.units_gu, (size_t)(h->max_units_gu > 0 ? h->max_units_gu : 1) * sizeof(TcUnit)},
      {(void**)&ws.units_dn, (size_t)(h->max_units_dn > 0 ? h->max_units_dn : 1) * sizeof(TcUnit)},
      {(void**)&ws.n_units, 2 * 4},
      {(void**)&ws.uprefix, (size_t)2 * (E + 1) * 4},
      {(void**)&ws.h32, Tg * (k + 1) * Fmax * 4},
      {(void**)&ws.h16, (h->tc_capable ? Tm : Tg) * (k + 1) * Fmax * 2},
      {(void**)&ws.xp, h->tc_capable ? Tm * (h->fp4 ? k + 1 : k) * d * 2 : 16},
      {(void**)&ws.xs, h->tc_capable && h->fp4 ? Tm * (k + 1) * 4 : 16},
      {(void**)&ws.ypart, Tg * (k + 1) * d * 4},
      {(void**)&ws.xh16, c.weight_dtype == MOE_NVFP4 ? Tg * d * 2 : 16},
      {(void**)&ws.xsc, c.weight_dtype == MOE_NVFP4 ? Tg * 4 : 16},
      {(void**)&ws.yacc, h->tc_capable ? Tm * d * 4 : 16},
      {(void**)&ws.oslot, h->tc_capable && c.deterministic ? Tm * (k + 1) * d * 4 : 16},
      {(void**)&ws.counters, (size_t)(64 + (Tm + 127) / 128) * 4},
      {(void**)&ws.wr_split, h->rtc_capable ? 3 * E * d * 2 : 16},
      {(void**)&ws.cand, h->rtc_capable ? Tm * (E / 64) * kMaxTopK * 8 : 16},
      {(void**)&ws.fin, Tg * (d / kFinRows) * 4},
      {(void**)&ws.ready, (E + 4) * 4},
      {(void**)&ws.gu_part, h->max_tiles_small > 0 ? (size_t)kMaxKSplit * (Tm < (size_t)kSmallT ? Tm : (size_t)kSmallT) * (k + 1) * 2 * Fmax * 4 : 16},
      {(void**)&ws.gu_cnt, (size_t)(h->max_tiles_small > 0 ? h->max_tiles_small : 1) * 4 * 4},
      {(void**)&ws.err, 16},
      {&ws.x_stage, Tm * d * act_bytes(c)},
      {&ws.y_stage, Tm * d * act_bytes(c)},
  };
  size_t total = 0;
  for (const Part& p : parts) total += up256(p.bytes);
  ws.bytes = total;
  if (dev_malloc(&h->block, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  size_t off = 0;
  for (const Part& p : parts) {
    *p.dst = static_cast<uint8_t*>(h->block) + off;
    off += up256(p.bytes);
  }
  if (!(h->tc_capable && c.deterministic)) ws.oslot = nullptr;   // accumulate mode
  // Counters and the error word start at zero; the rest is written before it is read.
  h->n_counters = (int)(64 + (Tm + 127) / 128);
  cudaError_t e = cudaMemsetAsync(ws.counters, 0, (size_t)h->n_counters * 4, stream);
  if (e == cudaSuccess && h->rtc_capable) e = launch_router_split(w->router_w, ws.wr_split, E * d, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws.fin, 0, Tg * (d / kFinRows) * 4, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws.ready, 0, (E + 4) * 4, stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(ws.gu_cnt, 0, (size_t)(h->max_tiles_small > 0 ? h->max_tiles_small : 1) * 4 * 4, stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws.err, 0, 16, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->block);
    delete h;
    return MOE_ERR_CUDA;
  }
  if (h->rtc_capable && !make_map_bf16(&h->tm_wr, ws.wr_split, 3 * E, d, 64, kTcBK)) h->rtc_capable = false;
  if (h->tc_capable && h->fp4) {
    const uint64_t F = c.ffn, Fs = c.shared_ffn;
    const void* qs[3] = {w->w_gate, w->w_up, w->w_down};
    const void* ss[3] = {w->s_gate, w->s_up, w->s_down};
    const void* sq[3] = {w->ws_gate, w->ws_up, w->ws_down};
    const void* sss[3] = {w->ss_gate, w->ss_up, w->ss_down};
    const uint64_t rows[3] = {E * F, E * F, E * d}, srows[3] = {Fs, Fs, d}, kk[3] = {d, d, F}, skk[3] = {d, d, Fs};
    bool ok = make_map_f16(&h->tm_xp, ws.xp, Tm * (k + 1), d, 16, 64) &&
              make_map_f16(&h->tm_h, ws.h16, Tm * (k + 1), Fmax, 16, 64);
    for (int m = 0; m < 3 && ok; ++m) {
      ok = make_map_u8(&h->q4[m], qs[m], rows[m], kk[m] / 2, 128, 128, true) &&
           make_map_u8(&h->sc4[m], ss[m], rows[m], kk[m] / 16, 128, 16, false);
      if (ok && Fs > 0)
        ok = make_map_u8(&h->sq4[m], sq[m], srows[m], skk[m] / 2, 128, 128, true) &&
             make_map_u8(&h->ssc4[m], sss[m], srows[m], skk[m] / 16, 128, 16, false);
    }
    if (!ok) {
      if (c.path == MOE_PATH_TC) {
        cudaFree(h->block);
        delete h;
        return MOE_ERR_CUDA;
      }
      h->tc_capable = false;
    }
  } else if (h->tc_capable) {
    const uint64_t F = c.ffn, Fs = c.shared_ffn;
    bool ok = make_map_bf16(&h->tm_wg, w->w_gate, E * F, d, kTcBM, kTcBK) &&
              make_map_bf16(&h->tm_wu, w->w_up, E * F, d, kTcBM, kTcBK) &&
              make_map_bf16(&h->tm_wd, w->w_down, E * d, F, kTcBM, kTcBK) &&
              make_map_bf16(&h->tm_h, ws.h16, Tm * (k + 1), Fmax, kTcBN, kTcBK) &&
              make_map_bf16(&h->tm_xp, ws.xp, Tm * k, d, kTcBN, kTcBK);
    if (ok && Fs > 0)
      ok = make_map_bf16(&h->tm_sg, w->ws_gate, Fs, d, kTcBM, kTcBK) &&
           make_map_bf16(&h->tm_su, w->ws_up, Fs, d, kTcBM, kTcBK) &&
           make_map_bf16(&h->tm_sd, w->ws_down, d, Fs, kTcBM, kTcBK);
    if (ok && d % (2 * kTcBN) == 0) {
      h->tok_major_ok = make_map_bf16(&h->tm_wd256, w->w_down, E * d, F, 2 * kTcBN, kTcBK) &&
                        (Fs == 0 || make_map_bf16(&h->tm_sd256, w->ws_down, d, Fs, 2 * kTcBN, kTcBK));
      if (Fs == 0) h->tm_sd256 = h->tm_wd256;
    }
    if (!ok) {
      if (c.path == MOE_PATH_TC) {
        cudaFree(h->block);
        delete h;
        return MOE_ERR_CUDA;
      }
      h->tc_capable = false;
    }
  }
  if (c.path == MOE_PATH_AUTO) {
    moe_status sst = setup_fused(h, stream);
    if (sst != MOE_OK) {
      cudaFree(h->block);
      delete h;
      return sst;
    }
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle h) {
  if (!h) return MOE_OK;
  cudaError_t e = cudaDeviceSynchronize();
  for (cudaEvent_t ev : h->prof.ev) cudaEventDestroy(ev);
  cudaError_t f = cudaFree(h->block);
  if (h->sd_block && cudaFree(h->sd_block) != cudaSuccess) f = cudaErrorInvalidValue;
  delete h;
  return (e == cudaSuccess && f == cudaSuccess) ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_route(moe_handle h, const void* x, int32_t T, int32_t* idx, float* gate, int32_t* counts,
                     cudaStream_t stream) {
  moe_status st = check_call(h, x, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!idx || !gate) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(gate) & 3u) ||
      (reinterpret_cast<uintptr_t>(counts) & 3u))
    return MOE_ERR_INVALID_ARG;
  CUtensorMap tm_x;
  bool have_tm_x = false;
  moe_status st2 = do_route(h, x, T, idx, gate, counts, false, &tm_x, &have_tm_x, stream);
  if (st2 != MOE_OK || T <= kSmallT) return st2;
  // large-batch routers leave the per-slot placement to a separate pass
  return cuda_status(launch_place(idx, h->ws, T, h->cfg.num_experts, h->cfg.top_k, h->rtc_capable ? 4 : 1, stream));
}

moe_status moe_forward(moe_handle h, const void* x, int32_t T, void* y, int32_t* idx_out, float* gate_out,
                       cudaStream_t stream) {
  moe_status st = check_call(h, x, T);
  if (st != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  if (!y || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const size_t nb = (size_t)T * h->cfg.d * act_bytes(h->cfg);
  if (ranges_overlap(x, nb, y, nb)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx_out) & 3u) || (reinterpret_cast<uintptr_t>(gate_out) & 3u))
    return MOE_ERR_INVALID_ARG;
  return run_forward(h, x, T, y, idx_out, gate_out, stream);
}

moe_status moe_forward_host(moe_handle h, const void* x_host, int32_t T, void* y_host, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return MOE_ERR_INVALID_ARG;
  const size_t nb = (size_t)T * h->cfg.d * act_bytes(h->cfg);
  cudaError_t e = cudaMemcpyAsync(h->ws.x_stage, x_host, nb, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  moe_status st = run_forward(h, h->ws.x_stage, T, h->ws.y_stage, nullptr, nullptr, stream);
  if (st != MOE_OK) return st;
  e = cudaMemcpyAsync(y_host, h->ws.y_stage, nb, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return cuda_status(e);
}

moe_status moe_get_grouping(moe_handle h, int32_t T, int32_t* offsets, int32_t* tok_of_slot, int32_t* slot_of,
                            cudaStream_t stream) {
  if (!h || T < 0 || T > h->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  const size_t n = (size_t)T * h->cfg.top_k * 4;
  cudaError_t e = cudaSuccess;
  if (offsets)
    e = cudaMemcpyAsync(offsets, h->ws.offsets, (h->cfg.num_experts + 1) * 4, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess && tok_of_slot && n)
    e = cudaMemcpyAsync(tok_of_slot, h->ws.tok_of_slot, n, cudaMemcpyDeviceToDevice, stream);
  if (e == cudaSuccess && slot_of && n)
    e = cudaMemcpyAsync(slot_of, h->ws.slot_of, n, cudaMemcpyDeviceToDevice, stream);
  return cuda_status(e);
}

moe_status moe_check(moe_handle h, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  unsigned int word = 0;
  e = cudaMemcpy(&word, h->ws.err, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (word) {
    e = cudaMemset(h->ws.err, 0, sizeof(word));
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (word & kErrRange) return MOE_ERR_RANGE;
  return MOE_OK;
}

moe_status moe_debug_fail_alloc(int32_t nth) {
  if (nth < 0) return MOE_ERR_INVALID_ARG;
  g_fail_alloc.store(nth);
  return MOE_OK;
}

moe_status moe_debug_expire_wait(moe_handle h, int32_t timeout_us, cudaStream_t stream) {
  if (!h || timeout_us < 1 || timeout_us > 5000000) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_debug_wait(h->ws.err, (uint64_t)timeout_us * 1000ull, stream));
}

moe_status moe_profile_enable(moe_handle h, int32_t enable, int32_t max_launches) {
  if (!h || (enable && (max_launches < 1 || max_launches > (1 << 20)))) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  for (cudaEvent_t ev : h->prof.ev) cudaEventDestroy(ev);
  h->prof.ev.clear();
  h->prof.kid.clear();
  if (!enable) return MOE_OK;
  h->prof.ev.resize(2 * (size_t)max_launches);
  for (auto& ev : h->prof.ev) {
    if (cudaEventCreate(&ev) != cudaSuccess) {
      cudaGetLastError();
      ev = nullptr;
      for (cudaEvent_t e : h->prof.ev)
        if (e) cudaEventDestroy(e);
      h->prof.ev.clear();
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

moe_status moe_profile_read(moe_handle h, float* ms, int32_t* launches) {
  if (!h || !ms || !launches) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < MOE_K_COUNT; ++i) {
    ms[i] = 0.f;
    launches[i] = 0;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  for (size_t i = 0; i < h->prof.kid.size(); ++i) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, h->prof.ev[2 * i], h->prof.ev[2 * i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
    ms[h->prof.kid[i]] += t;
    launches[h->prof.kid[i]] += 1;
  }
  h->prof.kid.clear();
  return MOE_OK;
}

}  // extern "C"
