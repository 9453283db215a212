// Weight-streaming expert kernels for small batches (decode).
//
// Per generated token the selected experts' weights are read once, so decode
// is bound by memory bandwidth (kongchang.com, section "125+ tokens/s: The
// Practical Threshold for Local Inference").  These kernels therefore stream
// each touched expert's rows exactly once per call and apply them to every
// token routed to that expert (the grouping made by the router kernels).
//
//  * gemv_gateup: one warp per (expert, FFN row f): the gate row and the up
//    row are read with 16-byte loads, dotted with every routed token, and
//    h[slot][f] = silu(g) * u is written in fp32.  The shared expert's rows
//    come first and need no routing, so with programmatic dependent launch
//    they are streamed while the router is still running.
//  * gemv_down: one warp per (expert, 4 rows of Wd): partial outputs
//    ypart[slot][row] = Wd[row] . h[slot] in fp32.  The last warp to finish a
//    block of 32 rows (atomic counter) combines them for every token:
//    y[t][row] = sum_j gate[t][j] * ypart[slot(t, j)][row] + ypart[shared(t)][row]
//    (+ x[t][row]), always in the same order, so the result is deterministic.
//
// Weight formats: fp32 (with fp32 activations), bf16, NVFP4 (e2m1 values with
// one e4m3 scale per 16 values and an fp32 scale per matrix, decoded in
// registers; the format is named on the evermx.com review, section
// "Quantization").
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int WF> struct Fmt;
template <> struct Fmt<MOE_F32>   { static constexpr int EPC = 4;  };   // elements per 16-byte chunk
template <> struct Fmt<MOE_BF16>  { static constexpr int EPC = 8;  };
template <> struct Fmt<MOE_NVFP4> { static constexpr int EPC = 32; };

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two e2m1 codes (one byte, element 2i in the low nibble) -> two floats.
__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}
// Two e4m3 codes (low byte first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Dot of one 16-byte weight chunk with the matching activations.
// x points at the first activation of the chunk.  For NVFP4, sc holds the
// two block scales of the chunk (already decoded) and the result excludes the
// per-matrix scale.
template <int WF>
__device__ __forceinline__ float chunk_dot_x(const uint4& w, const void* x, float2 sc);

template <>
__device__ __forceinline__ float chunk_dot_x<MOE_F32>(const uint4& w, const void* x, float2) {
  const float4 xv = __ldg(reinterpret_cast<const float4*>(x));
  return __uint_as_float(w.x) * xv.x + __uint_as_float(w.y) * xv.y + __uint_as_float(w.z) * xv.z +
         __uint_as_float(w.w) * xv.w;
}
template <>
__device__ __forceinline__ float chunk_dot_x<MOE_BF16>(const uint4& w, const void* x, float2) {
  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x));
  float s = bf_lo(w.x) * bf_lo(xv.x);
  s = fmaf(bf_hi(w.x), bf_hi(xv.x), s);
  s = fmaf(bf_lo(w.y), bf_lo(xv.y), s);
  s = fmaf(bf_hi(w.y), bf_hi(xv.y), s);
  s = fmaf(bf_lo(w.z), bf_lo(xv.z), s);
  s = fmaf(bf_hi(w.z), bf_hi(xv.z), s);
  s = fmaf(bf_lo(w.w), bf_lo(xv.w), s);
  s = fmaf(bf_hi(w.w), bf_hi(xv.w), s);
  return s;
}
template <>
__device__ __forceinline__ float chunk_dot_x<MOE_NVFP4>(const uint4& w, const void* x, float2 sc) {
  const uint4* xp = reinterpret_cast<const uint4*>(x);
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float blk[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {          // two 16-value blocks per chunk
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {        // 8 values = 4 bytes of codes, 16 bytes of activations
      const uint4 xv = __ldg(xp + b * 2 + q);
      const uint32_t cw = wv[b * 2 + q];
      const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 wf = e2m1x2_to_f2((cw >> (8 * i)) & 0xFFu);
        s = fmaf(wf.x, bf_lo(xs[i]), s);
        s = fmaf(wf.y, bf_hi(xs[i]), s);
      }
    }
    blk[b] = s;
  }
  return blk[0] * sc.x + blk[1] * sc.y;
}

// Same, activations in fp32 registers-from-global (the intermediate h).
template <int WF>
__device__ __forceinline__ float chunk_dot_h(const uint4& w, const float* h, float2 sc);

template <>
__device__ __forceinline__ float chunk_dot_h<MOE_F32>(const uint4& w, const float* h, float2) {
  const float4 hv = *reinterpret_cast<const float4*>(h);
  return __uint_as_float(w.x) * hv.x + __uint_as_float(w.y) * hv.y + __uint_as_float(w.z) * hv.z +
         __uint_as_float(w.w) * hv.w;
}
template <>
__device__ __forceinline__ float chunk_dot_h<MOE_BF16>(const uint4& w, const float* h, float2) {
  const float4 a = *reinterpret_cast<const float4*>(h);
  const float4 b = *reinterpret_cast<const float4*>(h + 4);
  float s = bf_lo(w.x) * a.x;
  s = fmaf(bf_hi(w.x), a.y, s);
  s = fmaf(bf_lo(w.y), a.z, s);
  s = fmaf(bf_hi(w.y), a.w, s);
  s = fmaf(bf_lo(w.z), b.x, s);
  s = fmaf(bf_hi(w.z), b.y, s);
  s = fmaf(bf_lo(w.w), b.z, s);
  s = fmaf(bf_hi(w.w), b.w, s);
  return s;
}
template <>
__device__ __forceinline__ float chunk_dot_h<MOE_NVFP4>(const uint4& w, const float* h, float2 sc) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  float blk[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t cw = wv[b * 2 + q];
      const float4 h0 = *reinterpret_cast<const float4*>(h + b * 16 + q * 8);
      const float4 h1 = *reinterpret_cast<const float4*>(h + b * 16 + q * 8 + 4);
      const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 wf = e2m1x2_to_f2((cw >> (8 * i)) & 0xFFu);
        s = fmaf(wf.x, hv[2 * i], s);
        s = fmaf(wf.y, hv[2 * i + 1], s);
      }
    }
    blk[b] = s;
  }
  return blk[0] * sc.x + blk[1] * sc.y;
}

__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

// Row of a weight matrix in format WF: byte offset of element `col` of row `row`.
template <int WF>
__device__ __forceinline__ size_t row_bytes(int cols) {
  return WF == MOE_F32 ? (size_t)cols * 4 : WF == MOE_BF16 ? (size_t)cols * 2 : (size_t)cols / 2;
}

// ------------------------------------------------------------------ gate/up
template <int WF, int NCH>
__device__ void gateup_item(const GemvArgs& a, bool shared, int e, int f) {
  constexpr int EPC = Fmt<WF>::EPC;
  const int lane = threadIdx.x & 31;
  const int d = a.d, rowsF = shared ? a.Fs : a.F;
  const size_t rb = row_bytes<WF>(d);
  const size_t ridx = shared ? (size_t)f : (size_t)e * rowsF + f;
  const uint8_t* wg = static_cast<const uint8_t*>(shared ? a.sg : a.wg) + ridx * rb;
  const uint8_t* wu = static_cast<const uint8_t*>(shared ? a.su : a.wu) + ridx * rb;
  uint4 g[NCH], u[NCH];
  float2 sg[NCH], su[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const int col = (c * 32 + lane) * EPC;
    g[c] = make_uint4(0, 0, 0, 0);
    u[c] = make_uint4(0, 0, 0, 0);
    sg[c] = su[c] = make_float2(0.f, 0.f);
    if (col < d) {
      g[c] = __ldcs(reinterpret_cast<const uint4*>(wg) + c * 32 + lane);
      u[c] = __ldcs(reinterpret_cast<const uint4*>(wu) + c * 32 + lane);
      if (WF == MOE_NVFP4) {
        const uint8_t* scg = (shared ? a.ssc_g : a.sc_g) + ridx * (d / 16) + col / 16;
        const uint8_t* scu = (shared ? a.ssc_u : a.sc_u) + ridx * (d / 16) + col / 16;
        sg[c] = e4m3x2_to_f2(__ldcs(reinterpret_cast<const unsigned short*>(scg)));
        su[c] = e4m3x2_to_f2(__ldcs(reinterpret_cast<const unsigned short*>(scu)));
      }
    }
  }
  float tg = 1.f, tu = 1.f;
  if (WF == MOE_NVFP4) {
    tg = shared ? a.tss_g[0] : a.ts_g[e];
    tu = shared ? a.tss_u[0] : a.ts_u[e];
  }
  const int n = shared ? a.T : a.ws.counts[e];
  const int off = shared ? 0 : a.ws.offsets[e];
  const int Fmax = max(a.F, a.Fs);
  const size_t xes = WF == MOE_F32 ? 4 : 2;
  for (int i = 0; i < n; ++i) {
    const int t = shared ? i : a.ws.tok_of_slot[off + i];
    const int slot = shared ? a.T * a.k + i : off + i;
    const uint8_t* xt = static_cast<const uint8_t*>(a.x) + (size_t)t * d * xes;
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
      const int col = (c * 32 + lane) * EPC;
      if (col < d) {
        ag += chunk_dot_x<WF>(g[c], xt + (size_t)col * xes, sg[c]);
        au += chunk_dot_x<WF>(u[c], xt + (size_t)col * xes, su[c]);
      }
    }
    // two-value reduction: lanes 0-15 end with sum(ag), 16-31 with sum(au)
    const bool hi = lane & 16;
    float v = (hi ? au : ag) + __shfl_xor_sync(0xFFFFFFFFu, hi ? ag : au, 16);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    const float su_ = __shfl_sync(0xFFFFFFFFu, v, 16);
    if (lane == 0) a.ws.h32[(size_t)slot * Fmax + f] = silu(v * tg) * (su_ * tu);
  }
}

template <int WF, int NCH>
__global__ void __launch_bounds__(kThreads) gemv_gateup_kernel(GemvArgs a) {
  pdl_launch_dependents();
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), nw = gridDim.x * kWarps;
  const int n_sh = a.Fs;
  int g = gw;
  for (; g < n_sh; g += nw) gateup_item<WF, NCH>(a, true, 0, g);
  pdl_wait();
  const int n_act = a.ws.active[a.E];
  const int total = n_sh + n_act * a.F;
  for (; g < total; g += nw) {
    const int r = g - n_sh;
    gateup_item<WF, NCH>(a, false, a.ws.active[r / a.F], r % a.F);
  }
}

// ------------------------------------------------------------------ down + combine
template <int WF, int NCHD>
__device__ void down_item(const GemvArgs& a, bool shared, int e, int rg, int n_items_per_fin) {
  constexpr int EPC = Fmt<WF>::EPC;
  const int lane = threadIdx.x & 31;
  const int d = a.d, K = shared ? a.Fs : a.F;     // row length of Wd
  const size_t rb = row_bytes<WF>(K);
  const int cpr = K / EPC;                         // 16-byte chunks per row
  const int r0 = rg * kDownRPW;
  const size_t row0 = shared ? (size_t)r0 : (size_t)e * d + r0;
  const uint8_t* wd = static_cast<const uint8_t*>(shared ? a.sd : a.wd) + row0 * rb;
  uint4 w[NCHD];
  float2 sc[NCHD];
  int rl[NCHD], col[NCHD];
#pragma unroll
  for (int i = 0; i < NCHD; ++i) {
    const int q = i * 32 + lane;
    rl[i] = q / cpr;
    col[i] = (q % cpr) * EPC;
    w[i] = make_uint4(0, 0, 0, 0);
    sc[i] = make_float2(0.f, 0.f);
    if (rl[i] < kDownRPW) {
      w[i] = __ldcs(reinterpret_cast<const uint4*>(wd + (size_t)rl[i] * rb) + (q % cpr));
      if (WF == MOE_NVFP4) {
        const uint8_t* s = (shared ? a.ssc_d : a.sc_d) + (row0 + rl[i]) * (K / 16) + col[i] / 16;
        sc[i] = e4m3x2_to_f2(__ldcs(reinterpret_cast<const unsigned short*>(s)));
      }
    }
  }
  const float ts = WF == MOE_NVFP4 ? (shared ? a.tss_d[0] : a.ts_d[e]) : 1.f;
  const int n = shared ? a.T : a.ws.counts[e];
  const int off = shared ? 0 : a.ws.offsets[e];
  const int Fmax = max(a.F, a.Fs);
  const bool hi = lane & 16, b3 = lane & 8;
  for (int i = 0; i < n; ++i) {
    const int slot = shared ? a.T * a.k + i : off + i;
    const float* h = a.ws.h32 + (size_t)slot * Fmax;
    float acc[kDownRPW] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < NCHD; ++c) {
      if (rl[c] < kDownRPW) {
        const float s = chunk_dot_h<WF>(w[c], h + col[c], sc[c]);
        acc[0] += rl[c] == 0 ? s : 0.f;
        acc[1] += rl[c] == 1 ? s : 0.f;
        acc[2] += rl[c] == 2 ? s : 0.f;
        acc[3] += rl[c] == 3 ? s : 0.f;
      }
    }
    // four-value reduction: lane (16 h + 8 b) ends with row 2 h + b
    const float r0v = __shfl_xor_sync(0xFFFFFFFFu, hi ? acc[0] : acc[2], 16);
    const float r1v = __shfl_xor_sync(0xFFFFFFFFu, hi ? acc[1] : acc[3], 16);
    const float p0 = (hi ? acc[2] : acc[0]) + r0v;
    const float p1 = (hi ? acc[3] : acc[1]) + r1v;
    float v = (b3 ? p1 : p0) + __shfl_xor_sync(0xFFFFFFFFu, b3 ? p0 : p1, 8);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 4);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    if ((lane & 7) == 0) a.ws.ypart[(size_t)slot * d + r0 + (hi ? 2 : 0) + (b3 ? 1 : 0)] = v * ts;
  }
  // Count this item towards its 32-row block; the last one combines the block.
  __threadfence();
  __syncwarp();
  const int fb = r0 / kFinRows;
  unsigned prev = 0;
  if (lane == 0) prev = atomicAdd(&a.ws.counters[1 + fb], 1u);
  prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
  if (prev != (unsigned)n_items_per_fin - 1) return;
  __threadfence();
  const int row = fb * kFinRows + lane;
  const int T = a.T, k = a.k;
  for (int t = 0; t < T; ++t) {
    float y = 0.f;
    for (int j = 0; j < k; ++j) {
      const int s = a.ws.slot_of[t * k + j];
      y = fmaf(a.gate[t * k + j], __ldcg(a.ws.ypart + (size_t)s * d + row), y);
    }
    if (a.Fs > 0) y += __ldcg(a.ws.ypart + (size_t)(T * k + t) * d + row);
    if (a.act_bf16) {
      const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(a.x);
      if (a.add_residual) y += __bfloat162float(xb[(size_t)t * d + row]);
      static_cast<__nv_bfloat16*>(a.y)[(size_t)t * d + row] = __float2bfloat16_rn(y);
    } else {
      const float* xf = static_cast<const float*>(a.x);
      if (a.add_residual) y += xf[(size_t)t * d + row];
      static_cast<float*>(a.y)[(size_t)t * d + row] = y;
    }
  }
  if (lane == 0) a.ws.counters[1 + fb] = 0;
}

template <int WF, int NCHD>
__global__ void __launch_bounds__(kThreads) gemv_down_kernel(GemvArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5), nw = gridDim.x * kWarps;
  const int n_rg = a.d / kDownRPW;
  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_exp = a.ws.active[a.E] + has_sh;
  const int per_fin = n_exp * (kFinRows / kDownRPW);
  for (int g = gw; g < n_exp * n_rg; g += nw) {
    const int ai = g / n_rg, rg = g % n_rg;
    if (has_sh && ai == 0)
      down_item<WF, NCHD>(a, true, 0, rg, per_fin);
    else
      down_item<WF, NCHD>(a, false, a.ws.active[ai - has_sh], rg, per_fin);
  }
}

template <typename K>
cudaError_t launch_pdl(K kernel, int grid, cudaStream_t s, const GemvArgs& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int WF, int NCH, int NCHD>
cudaError_t launch_fmt(const GemvArgs& a, int num_sms, cudaStream_t s, Prof* prof) {
  static int occ_gu = 0, occ_dn = 0;
  if (!occ_gu) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_gu, gemv_gateup_kernel<WF, NCH>, kThreads, 0);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_dn, gemv_down_kernel<WF, NCHD>, kThreads, 0);
    occ_gu = occ_gu < 1 ? 1 : occ_gu;
    occ_dn = occ_dn < 1 ? 1 : occ_dn;
  }
  if (prof) prof->begin(MOE_K_GEMV_GATEUP, s);
  cudaError_t e = launch_pdl(gemv_gateup_kernel<WF, NCH>, num_sms * occ_gu, s, a);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  if (prof) prof->begin(MOE_K_GEMV_DOWN, s);
  e = launch_pdl(gemv_down_kernel<WF, NCHD>, num_sms * occ_dn, s, a);
  if (prof) prof->end(s);
  return e;
}

}  // namespace

// Chunks of 16 bytes per lane: gate/up rows hold d values, down rows hold F
// values, four rows per warp item.
cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int num_sms, cudaStream_t s, Prof* prof) {
  const int row_b = wfmt == MOE_F32 ? a.d * 4 : wfmt == MOE_BF16 ? a.d * 2 : a.d / 2;
  const int nch = (row_b + 511) / 512;
  const int kmax = a.F > a.Fs ? a.F : a.Fs;
  const int drow_b = wfmt == MOE_F32 ? kmax * 4 : wfmt == MOE_BF16 ? kmax * 2 : kmax / 2;
  const int nchd = (kDownRPW * drow_b + 511) / 512;
#define MOE_G(WF, A, B) \
  if (nch <= A && nchd <= B) return launch_fmt<WF, A, B>(a, num_sms, s, prof);
  if (wfmt == MOE_BF16) {
    MOE_G(MOE_BF16, 4, 4) MOE_G(MOE_BF16, 8, 8) MOE_G(MOE_BF16, 16, 16)
  } else if (wfmt == MOE_F32) {
    MOE_G(MOE_F32, 4, 4) MOE_G(MOE_F32, 8, 8) MOE_G(MOE_F32, 16, 16)
  } else {
    MOE_G(MOE_NVFP4, 2, 2) MOE_G(MOE_NVFP4, 4, 4) MOE_G(MOE_NVFP4, 8, 8)
  }
#undef MOE_G
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ failure-detection self-test
namespace {
__global__ void debug_wait_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);     // one arrival expected; nothing ever arrives
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl w{limit_ns, err, &abort_flag};
    (void)mbar_wait(&bar, 0, w);
  }
  __syncthreads();
}
}  // namespace

cudaError_t launch_debug_wait(unsigned int* err, uint64_t limit_ns, cudaStream_t s) {
  debug_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
