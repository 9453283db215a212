// Host side of the stack entry points (moe_stack_* in include/moe.h): a stack
// of MoE layers joined by residual adds, run either by the persistent decode
// kernel (one launch for all layers, small batches) or layer by layer through
// moe_forward.
#include <new>
#include <vector>

#include "moe_internal.cuh"

namespace moe {

bool stack_decode_supported(const moe_config& c, bool* query_ok) {
  *query_ok = true;
  int dev = 0, coop = 0, cc_major = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    *query_ok = false;
    return false;
  }
  return c.act_dtype == MOE_BF16 && c.weight_dtype == MOE_BF16 && c.num_experts <= 256 && c.top_k <= 8 &&
         c.d % 256 == 0 && c.ffn % 256 == 0 && c.shared_ffn % 256 == 0 && cc_major == 10 && coop &&
         stack_decode_smem_bytes(c.d, c.ffn, c.shared_ffn, c.top_k) <= (size_t)smem_optin;
}

bool stack_layer_views(const moe_config& c, const moe_weights& w, CUtensorMap* m) {
  auto view = [](CUtensorMap* t, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    const uint64_t dims[3] = {64, rows, K / 64}, strides[2] = {K * 2, 128};
    const uint32_t box[3] = {64, box_rows, 4};
    return encode_tiled(t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  const uint64_t E = c.num_experts, d = c.d, F = c.ffn, Fs = c.shared_ffn;
  bool ok = view(m + kMapWg, w.w_gate, E * F, d, 8) && view(m + kMapWu, w.w_up, E * F, d, 8) &&
            view(m + kMapWd, w.w_down, E * d, F, 16);
  if (ok && Fs > 0)
    ok = view(m + kMapSg, w.ws_gate, Fs, d, 8) && view(m + kMapSu, w.ws_up, Fs, d, 8) &&
         view(m + kMapSd, w.ws_down, d, Fs, 16);
  return ok;
}

}  // namespace moe

using namespace moe;

struct moe_stack {
  moe_config cfg;
  int L = 0;
  int device = 0;
  int num_sms = 0;
  std::vector<moe_handle> layers;    // one handle per layer (per-layer path)
  bool persistent = false;           // the persistent bf16 kernel serves T <= kSdMaxT
  bool persistent4 = false;          // the persistent NVFP4 kernel serves T <= kS4MaxT
  StackLayerPtrs* d_layers = nullptr;
  CUtensorMap* d_maps = nullptr;
  Stack4LayerPtrs* d_layers4 = nullptr;
  void* block4 = nullptr;            // NVFP4 kernel: maps, layer pointers, x f16 copy and scales, h, o, top-k
  CUtensorMap* d_maps4 = nullptr;
  __half* xh = nullptr;
  float* xsc = nullptr;
  __half* h4 = nullptr;
  float* o4 = nullptr;
  int32_t* topk_e = nullptr;
  float* topk_g = nullptr;
  void* block = nullptr;             // xbuf, logits, h, barrier counter, error word, chain buffers
  __nv_bfloat16* xbuf = nullptr;
  float* logits = nullptr;
  __nv_bfloat16* h = nullptr;
  unsigned* bar = nullptr;
  unsigned* err = nullptr;
  void* chain[2] = {nullptr, nullptr};
  uint64_t wait_ns = 0;
};

namespace {

inline size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

void free_stack(moe_stack* s) {
  for (moe_handle h : s->layers) moe_destroy(h);
  if (s->block) cudaFree(s->block);
  if (s->block4) cudaFree(s->block4);
  if (s->d_layers) cudaFree(s->d_layers);
  if (s->d_maps) cudaFree(s->d_maps);
  delete s;
}

}  // namespace

extern "C" {

moe_status moe_stack_create(const moe_config* cfg, const moe_weights* layers, int32_t n_layers, cudaStream_t stream,
                            moe_stack_handle* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !layers || n_layers < 1 || n_layers > 4096) return MOE_ERR_INVALID_ARG;
  if (!cfg->add_residual) return MOE_ERR_INVALID_ARG;
  moe_stack* s = new (std::nothrow) moe_stack();
  if (!s) return MOE_ERR_OOM;
  s->cfg = *cfg;
  s->L = n_layers;
  const moe_config& c = s->cfg;
  for (int l = 0; l < n_layers; ++l) {
    moe_handle h = nullptr;
    const moe_status st = moe_create(cfg, &layers[l], stream, &h);
    if (st != MOE_OK) {
      free_stack(s);
      return st;
    }
    s->layers.push_back(h);
  }
  bool query_ok = true;
  s->persistent = stack_decode_supported(c, &query_ok);
  if (!query_ok || cudaGetDevice(&s->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&s->num_sms, cudaDevAttrMultiProcessorCount, s->device) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return MOE_ERR_CUDA;
  }
  s->wait_ns = (uint64_t)(c.wait_timeout_ms > 0 ? c.wait_timeout_ms : 2000) * 1000000ull;
  const int Fmax = c.ffn > c.shared_ffn ? c.ffn : c.shared_ffn;
  const size_t es = c.act_dtype == MOE_F32 ? 4 : 2;
  // residual stream between layers and partial logits, sized for both persistent kernels
  const size_t nx = (size_t)kS4MaxT * c.d * 2;
  const size_t nlog = (size_t)((c.d + 511) / 512 > 4 ? (c.d + 511) / 512 : 4) * kS4MaxT * c.num_experts * 4;
  const size_t nh = (size_t)kSdMaxT * (c.top_k + 1) * Fmax * 2, nchain = (size_t)c.max_tokens * c.d * es;
  const size_t total = up256(2 * nx) + up256(nlog) + up256(nh) + 256 + 256 + 2 * up256(nchain);
  if (dev_malloc(&s->block, total) != cudaSuccess) {
    cudaGetLastError();
    s->block = nullptr;
    free_stack(s);
    return MOE_ERR_OOM;
  }
  uint8_t* p = static_cast<uint8_t*>(s->block);
  s->xbuf = reinterpret_cast<__nv_bfloat16*>(p); p += up256(2 * nx);
  s->logits = reinterpret_cast<float*>(p); p += up256(nlog);
  s->h = reinterpret_cast<__nv_bfloat16*>(p); p += up256(nh);
  s->bar = reinterpret_cast<unsigned*>(p); p += 256;
  s->err = reinterpret_cast<unsigned*>(p); p += 256;
  s->chain[0] = p; p += up256(nchain);
  s->chain[1] = p;
  if (s->persistent) {
    std::vector<StackLayerPtrs> hp(n_layers);
    for (int l = 0; l < n_layers; ++l) {
      const moe_weights& w = layers[l];
      hp[l] = StackLayerPtrs{w.router_w, w.router_b,
                             static_cast<const __nv_bfloat16*>(w.w_gate), static_cast<const __nv_bfloat16*>(w.w_up),
                             static_cast<const __nv_bfloat16*>(w.w_down), static_cast<const __nv_bfloat16*>(w.ws_gate),
                             static_cast<const __nv_bfloat16*>(w.ws_up), static_cast<const __nv_bfloat16*>(w.ws_down)};
    }
    std::vector<CUtensorMap> maps((size_t)n_layers * kSdMaps);
    bool ok = true;
    for (int l = 0; l < n_layers && ok; ++l) ok = stack_layer_views(c, layers[l], &maps[(size_t)l * kSdMaps]);
    void* dl = nullptr;
    void* dm = nullptr;
    if (ok && (dev_malloc(&dl, sizeof(StackLayerPtrs) * n_layers) != cudaSuccess ||
               dev_malloc(&dm, sizeof(CUtensorMap) * maps.size()) != cudaSuccess)) {
      cudaGetLastError();
      if (dl) cudaFree(dl);
      free_stack(s);
      return MOE_ERR_OOM;
    }
    if (!ok) {
      s->persistent = false;                 // the per-layer path serves every T
    } else {
      s->d_layers = static_cast<StackLayerPtrs*>(dl);
      s->d_maps = static_cast<CUtensorMap*>(dm);
      if (cudaMemcpy(s->d_layers, hp.data(), sizeof(StackLayerPtrs) * n_layers, cudaMemcpyHostToDevice) !=
              cudaSuccess ||
          cudaMemcpy(s->d_maps, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice) !=
              cudaSuccess) {
        cudaGetLastError();
        free_stack(s);
        return MOE_ERR_CUDA;
      }
    }
  }
  if (!s->persistent) {
    bool q4 = true;
    s->persistent4 = stack_decode_fp4_supported(c, &q4);
    if (!q4) {
      free_stack(s);
      return MOE_ERR_CUDA;
    }
  }
  if (s->persistent4) {
    std::vector<Stack4LayerPtrs> hp(n_layers);
    std::vector<CUtensorMap> maps((size_t)n_layers * kS4Maps);
    bool ok = true;
    for (int l = 0; l < n_layers && ok; ++l) {
      const moe_weights& w = layers[l];
      hp[l] = Stack4LayerPtrs{w.router_w, w.router_b, w.t_gate, w.t_up, w.t_down, w.ts_gate, w.ts_up, w.ts_down};
      ok = stack_layer_views_fp4(c, w, &maps[(size_t)l * kS4Maps]);
    }
    if (!ok) {
      s->persistent4 = false;                // the per-layer path serves every T
    } else {
      const size_t slots = (size_t)kS4MaxT * (c.top_k + 1);
      const size_t nmaps = up256(sizeof(CUtensorMap) * maps.size()), nlp = up256(sizeof(Stack4LayerPtrs) * n_layers);
      const size_t nxh = up256((size_t)kS4MaxT * c.d * 2), nxs = up256((size_t)kS4MaxT * 4);
      const size_t nh4 = up256(slots * Fmax * 2), no4 = up256(slots * c.d * 4), ntk = up256((size_t)kS4MaxT * kMaxTopK * 4);
      if (dev_malloc(&s->block4, nmaps + nlp + nxh + nxs + nh4 + no4 + 2 * ntk) != cudaSuccess) {
        cudaGetLastError();
        s->block4 = nullptr;
        free_stack(s);
        return MOE_ERR_OOM;
      }
      uint8_t* q = static_cast<uint8_t*>(s->block4);
      s->d_maps4 = reinterpret_cast<CUtensorMap*>(q); q += nmaps;
      s->d_layers4 = reinterpret_cast<Stack4LayerPtrs*>(q); q += nlp;
      s->xh = reinterpret_cast<__half*>(q); q += nxh;
      s->xsc = reinterpret_cast<float*>(q); q += nxs;
      s->h4 = reinterpret_cast<__half*>(q); q += nh4;
      s->o4 = reinterpret_cast<float*>(q); q += no4;
      s->topk_e = reinterpret_cast<int32_t*>(q); q += ntk;
      s->topk_g = reinterpret_cast<float*>(q);
      if (cudaMemcpy(s->d_maps4, maps.data(), sizeof(CUtensorMap) * maps.size(), cudaMemcpyHostToDevice) !=
              cudaSuccess ||
          cudaMemcpy(s->d_layers4, hp.data(), sizeof(Stack4LayerPtrs) * n_layers, cudaMemcpyHostToDevice) !=
              cudaSuccess) {
        cudaGetLastError();
        free_stack(s);
        return MOE_ERR_CUDA;
      }
    }
  }
  if (cudaMemsetAsync(s->err, 0, 256, stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    free_stack(s);
    return MOE_ERR_CUDA;
  }
  *out = s;
  return MOE_OK;
}

moe_status moe_stack_destroy(moe_stack_handle h) {
  if (!h) return MOE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  free_stack(h);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int32_t moe_stack_uses_persistent(moe_stack_handle h, int32_t T) {
  if (!h || T < 1 || T > h->cfg.max_tokens) return 0;
  return ((h->persistent && T <= kSdMaxT) || (h->persistent4 && T <= kS4MaxT)) ? 1 : 0;
}

moe_status moe_stack_forward(moe_stack_handle h, const void* x, int32_t T, void* y, void* x_trace, int32_t* idx_trace,
                             float* gate_trace, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  const moe_config& c = h->cfg;
  if (T < 0 || T > c.max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (!x || !y || mis(x) || mis(y) || mis(x_trace)) return MOE_ERR_INVALID_ARG;
  if ((idx_trace == nullptr) != (gate_trace == nullptr)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx_trace) & 3u) || (reinterpret_cast<uintptr_t>(gate_trace) & 3u))
    return MOE_ERR_INVALID_ARG;
  const size_t es = c.act_dtype == MOE_F32 ? 4 : 2;
  const size_t nb = (size_t)T * c.d * es;
  {
    const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
    if (a < b + nb && b < a + nb) return MOE_ERR_INVALID_ARG;
  }
  if (h->persistent4 && !x_trace && moe_stack_uses_persistent(h, T)) {
    if (cudaMemsetAsync(h->bar, 0, 4, stream) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    Stack4Args a;
    a.layers = h->d_layers4;
    a.maps = h->d_maps4;
    a.L = h->L;
    a.x_in = static_cast<const __nv_bfloat16*>(x);
    a.y_out = static_cast<__nv_bfloat16*>(y);
    a.xbuf = h->xbuf;
    a.logits = h->logits;
    a.xh = h->xh;
    a.xsc = h->xsc;
    a.h = h->h4;
    a.o = h->o4;
    a.topk_e = h->topk_e;
    a.topk_g = h->topk_g;
    a.idx_trace = idx_trace;
    a.gate_trace = gate_trace;
    a.g_offsets = a.g_tok_of_slot = a.g_slot_of = nullptr;
    a.bar = h->bar;
    a.err = h->err;
    a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
    a.add_residual = 1;
    a.wait_ns = h->wait_ns;
    if (launch_stack_decode_fp4(a, h->num_sms, stream) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  if (h->persistent && moe_stack_uses_persistent(h, T)) {
    if (cudaMemsetAsync(h->bar, 0, 4, stream) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    StackArgs a;
    a.layers = h->d_layers;
    a.maps = h->d_maps;
    a.L = h->L;
    a.x_in = static_cast<const __nv_bfloat16*>(x);
    a.y_out = static_cast<__nv_bfloat16*>(y);
    a.xbuf = h->xbuf;
    a.logits = h->logits;
    a.h = h->h;
    a.x_trace = static_cast<__nv_bfloat16*>(x_trace);
    a.idx_trace = idx_trace;
    a.gate_trace = gate_trace;
    a.bar = h->bar;
    a.err = h->err;
    a.T = T; a.d = c.d; a.F = c.ffn; a.Fs = c.shared_ffn; a.E = c.num_experts; a.k = c.top_k;
    a.add_residual = 1;
    a.g_offsets = a.g_tok_of_slot = a.g_slot_of = nullptr;
    a.wait_ns = h->wait_ns;
    if (launch_stack_decode(a, h->num_sms, stream) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  // layer by layer: layer l reads the previous output, writes the next buffer
  uint8_t* tr = static_cast<uint8_t*>(x_trace);
  if (tr && cudaMemcpyAsync(tr, x, nb, cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  const void* cur = x;
  for (int l = 0; l < h->L; ++l) {
    void* dst = tr ? static_cast<void*>(tr + (size_t)(l + 1) * nb) : (l == h->L - 1 ? y : h->chain[l & 1]);
    int32_t* it = idx_trace ? idx_trace + (size_t)l * T * c.top_k : nullptr;
    float* gt = gate_trace ? gate_trace + (size_t)l * T * c.top_k : nullptr;
    const moe_status st = moe_forward(h->layers[l], cur, T, dst, it, gt, stream);
    if (st != MOE_OK) return st;
    cur = dst;
  }
  if (tr && cudaMemcpyAsync(y, cur, nb, cudaMemcpyDeviceToDevice, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_stack_check(moe_stack_handle h, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word && cudaMemset(h->err, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
  moe_status worst = (word & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_OK;
  for (moe_handle l : h->layers) {
    const moe_status st = moe_check(l, stream);
    if (worst == MOE_OK) worst = st;
  }
  return worst;
}

}  // extern "C"
