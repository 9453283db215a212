// Weight-streaming expert kernels for small batches (decode).
//
// Per generated token the selected experts' weights are read once, so decode
// is bound by memory bandwidth (kongchang.com, section "125+ tokens/s: The
// Practical Threshold for Local Inference").  These kernels stream every
// touched expert's weights exactly once per call and apply them to all the
// tokens routed to that expert (the grouping made by the router kernels).
//
// Each SM runs one persistent CTA: warp 0 streams 8 KB units of weight rows
// into a 16-stage shared-memory ring with 1-D bulk copies (cp.async.bulk,
// completion counted on an mbarrier per stage), and eight consumer warps take
// the units in turn, so up to 128 KB per SM are in flight whatever the
// compute latency.  Units are handed out in contiguous ranges per CTA.
//
//  * gemv_gateup: a unit is RG row pairs (gate row f, up row f) of one
//    expert.  For each routed token the consumer dots both rows with x and
//    writes h[slot][f] = silu(g) * u (fp32).  The shared expert's units need
//    no routing and come first, so with programmatic dependent launch they
//    stream while the router is still running.
//  * gemv_down: a unit is RD rows of Wd.  Partial outputs
//    ypart[slot][row] = Wd[row] . h[slot] (fp32); the last unit to finish a
//    block of 32 rows (atomic counter) combines them for every token:
//    y[t][row] = sum_j gate[t][j] ypart[slot(t, j)][row] + ypart[shared(t)][row]
//    (+ x[t][row]), always in that order, so the result is deterministic.
//
// Weight formats: fp32 (with fp32 activations), bf16, and NVFP4 (e2m1 codes,
// an e4m3 scale per 16 values, an fp32 scale per matrix; the format is named
// on the evermx.com review, section "Quantization").  NVFP4 runs on packed
// f16 arithmetic: each code pair is decoded exactly by cvt.rn.f16x2.e2m1x2
// and multiplied into f16 activations with fma.rn.f16x2, one 16-value block at
// a time (at most 8 products per half, magnitudes below 96), and each block
// sum is widened to fp32 and scaled by its e4m3 scale.  The activations are a
// per-token f16 copy scaled by a power of two (largest value into [1, 2),
// made by gemv_x16_kernel), the intermediate is stored in f16 as h / xs^2,
// and the exact power-of-two factors are applied to the fp32 results; an h
// beyond the f16 range saturates and sets the range bit of the error word.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumers = 8;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kStages = 16;
constexpr int kUnitBytes = 8192;                  // weight bytes per unit
constexpr int kStageBytes = kUnitBytes + 1024;    // + NVFP4 block scales
constexpr uint32_t FULLMASK = 0xFFFFFFFFu;
// Round-robin rings (unit i to consumer i % kConsumers, stage i % kStages) are
// only safe when each stage has a single consumer: its parity waits can then
// never be two phases stale.
static_assert(kStages % kConsumers == 0, "a ring stage must belong to exactly one consumer warp");

template <int WF> struct Fmt;
template <> struct Fmt<MOE_F32>   { static constexpr int EPC = 4;  static constexpr int XB = 16; };
template <> struct Fmt<MOE_NVFP4> { static constexpr int EPC = 32; static constexpr int XB = 64; };
// EPC: elements per 16-byte weight chunk; XB: bytes of activations matching one chunk
// (bf16 weights use the tensor-pipe GEMV kernels further down).

// Activations matching one weight chunk, held in registers.
template <int WF> struct XChunk { uint4 v[Fmt<WF>::XB / 16]; };

template <int WF>
__device__ __forceinline__ void load_x(XChunk<WF>& c, const uint8_t* p) {
#pragma unroll
  for (int i = 0; i < Fmt<WF>::XB / 16; ++i) c.v[i] = __ldg(reinterpret_cast<const uint4*>(p) + i);
}

// Dot of a 16-byte weight chunk with its activations.  NVFP4: sc = the two
// decoded block scales; the per-matrix scale is applied by the caller.
__device__ __forceinline__ float cdot(const uint4& w, const XChunk<MOE_F32>& x, float2) {
  const uint4 a = x.v[0];
  float s = __uint_as_float(w.x) * __uint_as_float(a.x);
  s = fmaf(__uint_as_float(w.y), __uint_as_float(a.y), s);
  s = fmaf(__uint_as_float(w.z), __uint_as_float(a.z), s);
  return fmaf(__uint_as_float(w.w), __uint_as_float(a.w), s);
}
// NVFP4: 32 codes (two 16-value blocks; sc2 = their scales as f16x2) against
// 32 f16 values (16 f16x2 words; word m holds values 2m, 2m + 1).
__device__ __forceinline__ float cdot4(const uint4& w, const XChunk<MOE_NVFP4>& x, uint32_t sc2) {
  const float2 sc = __half22float2(*reinterpret_cast<const __half2*>(&sc2));
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
  const uint32_t xv[16] = {x.v[0].x, x.v[0].y, x.v[0].z, x.v[0].w, x.v[1].x, x.v[1].y, x.v[1].z, x.v[1].w,
                           x.v[2].x, x.v[2].y, x.v[2].z, x.v[2].w, x.v[3].x, x.v[3].y, x.v[3].z, x.v[3].w};
  float r = 0.f;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    uint32_t acc = 0u;                       // f16x2 zero
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      uint32_t hq[4];
      e2m1x8_f16x2(wv[2 * b + q], hq);       // codes 8 (2b + q) + 2c, + 1
#pragma unroll
      for (int c = 0; c < 4; ++c) acc = hfma2(hq[c], xv[8 * b + 4 * q + c], acc);
    }
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&acc));
    r = fmaf(f.x + f.y, b == 0 ? sc.x : sc.y, r);
  }
  return r;
}

// Activations of a chunk taken from the fp32 intermediate h (NVFP4: f16 h / xs^2).
template <int WF> struct HChunk { float4 v[Fmt<WF>::EPC / 4]; };
template <> struct HChunk<MOE_NVFP4> { XChunk<MOE_NVFP4> c; };

template <int WF>
__device__ __forceinline__ void load_h(HChunk<WF>& c, const float* p) {
#pragma unroll
  for (int i = 0; i < Fmt<WF>::EPC / 4; ++i) c.v[i] = __ldcg(reinterpret_cast<const float4*>(p) + i);
}
__device__ __forceinline__ void load_h16(HChunk<MOE_NVFP4>& h, const __half* p) {
#pragma unroll
  for (int i = 0; i < 4; ++i) h.c.v[i] = __ldcg(reinterpret_cast<const uint4*>(p) + i);
}
// Two e4m3 codes (low byte first) -> f16x2.  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
  return h2;
}
__device__ __forceinline__ float hdot(const uint4& w, const HChunk<MOE_F32>& h, float2) {
  const float4 a = h.v[0];
  float s = __uint_as_float(w.x) * a.x;
  s = fmaf(__uint_as_float(w.y), a.y, s);
  s = fmaf(__uint_as_float(w.z), a.z, s);
  return fmaf(__uint_as_float(w.w), a.w, s);
}
__device__ __forceinline__ float silu(float z) { return z / (1.f + __expf(-z)); }

template <int WF>
__host__ __device__ __forceinline__ int row_bytes(int cols) {
  return WF == MOE_F32 ? cols * 4 : WF == MOE_BF16 ? cols * 2 : cols / 2;
}

// Contiguous share [lo, hi) of n items for CTA b of g.
__device__ __forceinline__ void share(int n, int b, int g, int& lo, int& hi) {
  lo = (int)(((long long)n * b) / g);
  hi = (int)(((long long)n * (b + 1)) / g);
}

// Units of the templated GEMV kernels, in one sequence: the shared expert's
// (if any), then each active routed expert's, upe units per expert.  A unit's
// cost is 1 + the tokens its expert serves (one weight stream, then one
// pass per token), and each CTA takes a contiguous run of units holding an
// equal share of the total cost, so a CTA whose run falls on a popular expert
// gets fewer units.  Warp-collective (one warp); *lo, *hi = the CTA's run.
__device__ void unit_range(const GemvArgs& a, int upe, int b, int G, int* lo, int* hi) {
  const int lane = threadIdx.x & 31;
  const int has_sh = a.Fs > 0 ? 1 : 0;
  const int n_seq = has_sh + a.ws.active[a.E];
  // this lane's experts s = lane * per .. lane * per + per - 1 (per <= 17 covers E + 1 <= 513)
  const int per = (n_seq + 31) / 32;
  int c[17];
  int run = 0;
#pragma unroll
  for (int i = 0; i < 17; ++i) {
    const int sq = lane * per + i;
    int v = 0;
    if (i < per && sq < n_seq)
      v = 1 + (sq < has_sh ? a.T : __ldcg(a.ws.counts + __ldcg(a.ws.active + sq - has_sh)));
    c[i] = v;
    run += v;
  }
  // exclusive scan of the lane totals
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  const long long total = (long long)__shfl_sync(0xFFFFFFFFu, incl, 31) * upe;
  const long long excl = (long long)(incl - run) * upe;
  int res[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const long long X = total * (b + w) / G;         // cost at which the run starts / ends
    int g = n_seq * upe;                             // X == total: the end
    long long st = excl;
    int found = -1;
#pragma unroll
    for (int i = 0; i < 17; ++i) {
      const long long len = (long long)c[i] * upe;
      if (found < 0 && c[i] > 0 && X >= st && X < st + len) {
        const long long j = (X - st + c[i] - 1) / c[i];     // first unit starting at or after X
        found = (lane * per + i) * upe + (int)j;
      }
      st += len;
    }
    const unsigned m = __ballot_sync(0xFFFFFFFFu, found >= 0);
    if (m) g = __shfl_sync(0xFFFFFFFFu, found, __ffs(m) - 1);
    res[w] = g;
  }
  if (lane == 0) {
    *lo = res[0];
    *hi = res[1];
  }
}

// Ring bookkeeping common to both kernels.
struct Ring {
  uint8_t* stages;
  uint64_t* full;
  uint64_t* empty;
  int* abort_flag;
};

__device__ __forceinline__ Ring ring_setup(uint8_t* dsm) {
  Ring r;
  r.stages = dsm;
  r.full = reinterpret_cast<uint64_t*>(dsm + kStages * kStageBytes);
  r.empty = r.full + kStages;
  r.abort_flag = reinterpret_cast<int*>(r.empty + kStages);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&r.full[i], 1);
      mbar_init(&r.empty[i], 1);
    }
    *r.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  return r;
}

// Consumer-side warp-uniform bounded wait on a full stage.
__device__ __forceinline__ bool warp_wait_full(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, w) ? 1 : 0;
  ok = __shfl_sync(FULLMASK, ok, 0);
  if (ok)
    while (!mbar_try_wait(bar, parity)) {
    }
  return ok != 0;
}

// Down-projection completion.  After a warp has written ypart for rows of the
// 32-row block fb for the tokens of one expert, it counts those (token, block)
// pairs; the warp that brings a pair to `target` (all of the token's experts
// done for that block) combines the block for that token, always in the
// order j = 0..k-1 then the shared expert:
//   y[t][row] = sum_j gate[t][j] ypart[slot(t, j)][row] + ypart[shared(t)][row] (+ x[t][row])
__device__ void complete_block(const GemvArgs& a, bool shared, int off, int n, int fb, int target) {
  const int lane = threadIdx.x & 31;
  const int nfb = a.d / kFinRows, T = a.T, k = a.k, d = a.d;
  __threadfence();
  __syncwarp();
  for (int q0 = 0; q0 < n; q0 += 32) {
    const int q = q0 + lane;
    int t = -1;
    bool last = false;
    if (q < n) {
      t = shared ? q : a.ws.tok_of_slot[off + q];
      last = atomicAdd(&a.ws.fin[t * nfb + fb], 1u) == (unsigned)target - 1;
    }
    unsigned m = __ballot_sync(0xFFFFFFFFu, last);
    if (m) __threadfence();
    while (m) {
      const int src = __ffs(m) - 1;
      m &= m - 1;
      const int tt = __shfl_sync(0xFFFFFFFFu, t, src);
      const int row = fb * kFinRows + lane;
      float y = 0.f;
      for (int j = 0; j < k; ++j) {
        const int sl = __ldcg(a.ws.slot_of + tt * k + j);
        y = fmaf(__ldcg(a.gate + tt * k + j), __ldcg(a.ws.ypart + (size_t)sl * d + row), y);
      }
      if (a.Fs > 0) y += __ldcg(a.ws.ypart + (size_t)(T * k + tt) * d + row);
      if (a.act_bf16) {
        if (a.add_residual) y += __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[(size_t)tt * d + row]);
        static_cast<__nv_bfloat16*>(a.y)[(size_t)tt * d + row] = __float2bfloat16_rn(y);
      } else {
        if (a.add_residual) y += static_cast<const float*>(a.x)[(size_t)tt * d + row];
        static_cast<float*>(a.y)[(size_t)tt * d + row] = y;
      }
      if (lane == 0) a.ws.fin[tt * nfb + fb] = 0;
    }
  }
}

// ------------------------------------------------------------------ gate/up
// J = 16-byte chunks per lane per row (row = d values), RG = row pairs per unit.
template <int WF, int J>
__global__ void __launch_bounds__(kThreads, 1) gemv_gateup_kernel(GemvArgs a, uint64_t wait_ns) {
  constexpr int RG = 8 / J;
  extern __shared__ __align__(128) uint8_t dsm[];
  pdl_launch_dependents();
  const Ring ring = ring_setup(dsm);
  const WaitCtl wc{wait_ns, a.ws.err, ring.abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, G = gridDim.x, b = blockIdx.x;
  const int rb = row_bytes<WF>(d);                  // bytes of one row
  const int sb = WF == MOE_NVFP4 ? d / 16 : 0;      // scale bytes of one row
  const int upe = a.F / RG;                         // units per expert (the shared expert has the routed width)
  const int has_sh = a.Fs > 0 ? 1 : 0;
  pdl_wait();
  __shared__ int s_run[2];
  if (warp == 0) unit_range(a, upe, b, G, &s_run[0], &s_run[1]);
  __syncthreads();
  const int g_lo = s_run[0], n_local = s_run[1] - s_run[0];
  // local unit i -> (shared?, expert, first row pair)
  auto unit_of = [&](int i, bool& shared, int& e, int& f0) {
    const int g = g_lo + i, sq = g / upe;
    shared = sq < has_sh;
    e = shared ? 0 : a.ws.active[sq - has_sh];
    f0 = (g % upe) * RG;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int i = 0;
    bool ok = true;
    for (; i < n_local; ++i) {
      bool shared;
      int e, f0;
      unit_of(i, shared, e, f0);
      const int s = i % kStages;
      if (!mbar_wait(&ring.empty[s], ((i / kStages) & 1) ^ 1, wc)) { ok = false; break; }
      uint8_t* st = ring.stages + s * kStageBytes;
      const size_t row0 = shared ? (size_t)f0 : (size_t)e * a.F + f0;
      const uint8_t* g = static_cast<const uint8_t*>(shared ? a.sg : a.wg) + row0 * rb;
      const uint8_t* u = static_cast<const uint8_t*>(shared ? a.su : a.wu) + row0 * rb;
      mbar_arrive_expect_tx(&ring.full[s], 2 * RG * (rb + sb));
      bulk_g2s_hint(st, g, RG * rb, &ring.full[s], pol);
      bulk_g2s_hint(st + RG * rb, u, RG * rb, &ring.full[s], pol);
      if (WF == MOE_NVFP4) {
        bulk_g2s_hint(st + 2 * RG * rb, (shared ? a.ssc_g : a.sc_g) + row0 * sb, RG * sb, &ring.full[s], pol);
        bulk_g2s_hint(st + 2 * RG * rb + RG * sb, (shared ? a.ssc_u : a.sc_u) + row0 * sb, RG * sb,
                      &ring.full[s], pol);
      }
    }
    if (!ok) {   // let the copies already issued land before the CTA leaves
      for (int j = i - kStages < 0 ? 0 : i - kStages; j < i; ++j) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&ring.full[j % kStages], (j / kStages) & 1))
          if (global_ns() - t0 > wait_ns) break;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int Fmax = max(a.F, a.Fs);
  bool range_bad = false;
  for (int i = cw; i < n_local; i += kConsumers) {
    bool shared;
    int e, f0;
    unit_of(i, shared, e, f0);
    const int s = i % kStages;
    if (!warp_wait_full(&ring.full[s], (i / kStages) & 1, wc)) break;
    const uint8_t* st = ring.stages + s * kStageBytes;
    // The unit's weights (and NVFP4 block scales, as f16x2) move to registers
    // and the stage is freed at once, so the producer refills it while the
    // tokens are computed.
    constexpr bool FP4 = WF == MOE_NVFP4;
    uint4 wg[RG][J], wu[RG][J];
    uint32_t sg[FP4 ? RG : 1][J], su[FP4 ? RG : 1][J];
#pragma unroll
    for (int p = 0; p < RG; ++p)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        wg[p][j] = reinterpret_cast<const uint4*>(st + p * rb)[j * 32 + lane];
        wu[p][j] = reinterpret_cast<const uint4*>(st + (RG + p) * rb)[j * 32 + lane];
        if constexpr (FP4) {
          const int c = j * 32 + lane;
          sg[p][j] = e4m3x2_to_h2(*reinterpret_cast<const unsigned short*>(st + 2 * RG * rb + p * sb + c * 2));
          su[p][j] = e4m3x2_to_h2(*reinterpret_cast<const unsigned short*>(st + 2 * RG * rb + (RG + p) * sb + c * 2));
        }
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[s]);
    float tg = 1.f, tu = 1.f;
    if (WF == MOE_NVFP4) {
      tg = shared ? a.tss_g[0] : a.ts_g[e];
      tu = shared ? a.tss_u[0] : a.ts_u[e];
    }
    const int n = shared ? a.T : a.ws.counts[e];
    const int off = shared ? 0 : a.ws.offsets[e];
    for (int q = 0; q < n; ++q) {
      const int t = shared ? q : a.ws.tok_of_slot[off + q];
      const int slot = shared ? a.T * a.k + q : off + q;
      const uint8_t* xt = WF == MOE_NVFP4 ? reinterpret_cast<const uint8_t*>(a.ws.xh16 + (size_t)t * d)
                                          : static_cast<const uint8_t*>(a.x) + (size_t)t * d * (WF == MOE_F32 ? 4 : 2);
      XChunk<WF> xc[J];
#pragma unroll
      for (int j = 0; j < J; ++j) load_x<WF>(xc[j], xt + (size_t)(j * 32 + lane) * Fmt<WF>::XB);
      float v[2 * RG];
#pragma unroll
      for (int p = 0; p < RG; ++p) {
        float ag = 0.f, au = 0.f;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          if constexpr (FP4) {
            ag += cdot4(wg[p][j], xc[j], sg[p][j]);
            au += cdot4(wu[p][j], xc[j], su[p][j]);
          } else {
            ag += cdot(wg[p][j], xc[j], make_float2(0.f, 0.f));
            au += cdot(wu[p][j], xc[j], make_float2(0.f, 0.f));
          }
        }
        v[2 * p] = ag * tg;
        v[2 * p + 1] = au * tu;
      }
      const float r = transpose_reduce<2 * RG, 32>(v, lane);
      // lane l holds value (l >> SH): gate of pair p at 2p, up at 2p + 1
      constexpr int SH = (2 * RG == 2) ? 4 : (2 * RG == 4) ? 3 : (2 * RG == 8) ? 2 : 1;
      const float up = __shfl_down_sync(FULLMASK, r, 1 << SH);
      const int idx = lane >> SH;
      if ((lane & ((1 << SH) - 1)) == 0 && (idx & 1) == 0) {
        if constexpr (WF == MOE_NVFP4) {
          // r, up are the products with the scaled copy x / xs: store h / xs^2
          const float xs = __ldcg(a.ws.xsc + t);
          const float hv = silu(r * xs) * up * (1.f / xs);
          range_bad |= !(fabsf(hv) <= 65504.f);
          reinterpret_cast<__half*>(a.ws.h16)[(size_t)slot * Fmax + f0 + (idx >> 1)] = __float2half_rn(fminf(fmaxf(hv, -65504.f), 65504.f));
        } else {
          a.ws.h32[(size_t)slot * Fmax + f0 + (idx >> 1)] = silu(r) * up;
        }
      }
    }
  }
  if (WF == MOE_NVFP4 && __any_sync(FULLMASK, range_bad) && lane == 0) atomicOr(a.ws.err, kErrRange);
}

// ------------------------------------------------------------------ down + combine
// CPR = 16-byte chunks per Wd row (row = F values); a unit is 512 chunks:
// RD = 512 / CPR rows.  CPR >= 32: each lane holds JD = CPR / 32 chunk columns
// of all RD rows.  CPR == 16: half-warps split the rows.
template <int WF, int CPR>
__global__ void __launch_bounds__(kThreads, 1) gemv_down_kernel(GemvArgs a, uint64_t wait_ns) {
  constexpr int RD = 512 / CPR;
  constexpr int SPLIT = CPR < 32;                    // half-warps on different rows
  constexpr int JD = SPLIT ? 1 : CPR / 32;            // chunk columns per lane
  constexpr int NR = SPLIT ? 16 : RD;                // rows per lane
  constexpr int LW = SPLIT ? 16 : 32;                // lanes sharing one row
  constexpr int EPC = Fmt<WF>::EPC;
  extern __shared__ __align__(128) uint8_t dsm[];
  pdl_launch_dependents();
  const Ring ring = ring_setup(dsm);
  const WaitCtl wc{wait_ns, a.ws.err, ring.abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F, G = gridDim.x, b = blockIdx.x;
  const int rb = row_bytes<WF>(F);
  const int sb = WF == MOE_NVFP4 ? F / 16 : 0;
  const int upe = d / RD;                            // units per expert
  const int has_sh = a.Fs > 0 ? 1 : 0;
  pdl_wait();
  __shared__ int s_run[2];
  if (warp == 0) unit_range(a, upe, b, G, &s_run[0], &s_run[1]);
  __syncthreads();
  const int g_lo = s_run[0], n_local = s_run[1] - s_run[0];
  // local unit i -> (shared?, expert, first row)
  auto unit_of = [&](int i, bool& shared, int& e, int& r0) {
    const int g = g_lo + i, sq = g / upe;
    shared = sq < has_sh;
    e = shared ? 0 : a.ws.active[sq - has_sh];
    r0 = (g % upe) * RD;
  };

  if (warp == 0) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int i = 0;
    bool ok = true;
    for (; i < n_local; ++i) {
      bool shared;
      int e, r0;
      unit_of(i, shared, e, r0);
      const size_t row0 = shared ? (size_t)r0 : (size_t)e * d + r0;
      const int s = i % kStages;
      if (!mbar_wait(&ring.empty[s], ((i / kStages) & 1) ^ 1, wc)) { ok = false; break; }
      uint8_t* st = ring.stages + s * kStageBytes;
      mbar_arrive_expect_tx(&ring.full[s], RD * (rb + sb));
      bulk_g2s_hint(st, static_cast<const uint8_t*>(shared ? a.sd : a.wd) + row0 * rb, RD * rb, &ring.full[s],
                    pol);
      if (WF == MOE_NVFP4)
        bulk_g2s_hint(st + RD * rb, (shared ? a.ssc_d : a.sc_d) + row0 * sb, RD * sb, &ring.full[s], pol);
    }
    if (!ok) {
      for (int j = i - kStages < 0 ? 0 : i - kStages; j < i; ++j) {
        const uint64_t t0 = global_ns();
        while (!mbar_try_wait(&ring.full[j % kStages], (j / kStages) & 1))
          if (global_ns() - t0 > wait_ns) break;
      }
    }
    return;
  }

  const int cw = warp - 1;
  const int Fmax = max(a.F, a.Fs);
  const int col_lane = SPLIT ? (lane & 15) : lane;   // chunk column of this lane (plus 32 j)
  const int row_lane = SPLIT ? (lane >> 4) : 0;      // first row of this lane (SPLIT: every other row)
  for (int i = cw; i < n_local; i += kConsumers) {
    bool shared;
    int e, r0;
    unit_of(i, shared, e, r0);
    const int s = i % kStages;
    if (!warp_wait_full(&ring.full[s], (i / kStages) & 1, wc)) break;
    const uint8_t* st = ring.stages + s * kStageBytes;
    constexpr bool FP4 = WF == MOE_NVFP4;      // as in gemv_gateup: weights to registers, stage freed
    uint4 w[NR][JD];
    uint32_t sc[FP4 ? NR : 1][JD];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
      for (int j = 0; j < JD; ++j) {
        const int row = SPLIT ? row_lane + 2 * r : r;
        w[r][j] = reinterpret_cast<const uint4*>(st + row * rb)[j * 32 + col_lane];
        if constexpr (FP4)
          sc[r][j] = e4m3x2_to_h2(*reinterpret_cast<const unsigned short*>(st + RD * rb + row * sb + (j * 32 + col_lane) * 2));
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[s]);
    const float ts = WF == MOE_NVFP4 ? (shared ? a.tss_d[0] : a.ts_d[e]) : 1.f;
    const int n = shared ? a.T : a.ws.counts[e];
    const int off = shared ? 0 : a.ws.offsets[e];
    for (int q = 0; q < n; ++q) {
      const int slot = shared ? a.T * a.k + q : off + q;
      HChunk<WF> hc[JD];
      float xs2 = 1.f;
      if constexpr (WF == MOE_NVFP4) {
        const int t = shared ? q : a.ws.tok_of_slot[off + q];
        const float xs = __ldcg(a.ws.xsc + t);
        xs2 = xs * xs;
        const __half* h = reinterpret_cast<const __half*>(a.ws.h16) + (size_t)slot * Fmax;
#pragma unroll
        for (int j = 0; j < JD; ++j) load_h16(hc[j], h + (j * 32 + col_lane) * EPC);
      } else {
        const float* h = a.ws.h32 + (size_t)slot * Fmax;
#pragma unroll
        for (int j = 0; j < JD; ++j) load_h<WF>(hc[j], h + (j * 32 + col_lane) * EPC);
      }
      float v[NR];
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < JD; ++j) {
          if constexpr (FP4)
            acc += cdot4(w[r][j], hc[j].c, sc[r][j]);
          else
            acc += hdot(w[r][j], hc[j], make_float2(0.f, 0.f));
        }
        v[r] = acc * ts * xs2;
      }
      const float tot = transpose_reduce<NR, LW>(v, lane);
      constexpr int SH = (LW == 32) ? (NR == 4 ? 3 : NR == 8 ? 2 : NR == 16 ? 1 : 0) : (NR == 16 ? 0 : 1);
      const int li = (lane & (LW - 1)) >> SH;         // value index held by this lane
      if ((lane & ((1 << SH) - 1)) == 0) {
        const int row = SPLIT ? row_lane + 2 * li : li;
        a.ws.ypart[(size_t)slot * d + r0 + row] = tot;
      }
    }
    // Units never straddle a 32-row block: each of a token's experts
    // contributes 32 / RD units to it.
    complete_block(a, shared, off, n, r0 / kFinRows, (a.k + has_sh) * (kFinRows / RD));
  }
}

// ------------------------------------------------------------------ bf16: tensor-core GEMV
// For bf16 weights the dot products run on the tensor pipe (mma.sync
// m16n8k16, fp32 accumulate): 16 weight rows x 16 values of A from the stage
// via ldmatrix, 8 tokens x 16 values of B from the activations, so a unit
// costs a few dozen instructions instead of several per weight.  A unit is
// 16 row segments of 256 values (512 bytes each, one bulk copy per segment,
// rows padded to 528 bytes in the stage so ldmatrix rows hit distinct banks).
// A row group (16 rows) takes K / 256 consecutive units, handed to the same
// consumer warp; the eight consumers work on eight row groups at a time with
// their units interleaved in the ring.
constexpr int kRowPad = 528;
constexpr int kKc = 256;            // values per row segment
constexpr int kMaxNT = kGemvChunkT / 8;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Row groups of one CTA: the shared expert's (round-robin over CTAs, need no
// routing) then a contiguous share of the routed ones, in batches of up to 8
// (one per consumer warp).  Units of a batch are ordered (segment, group).
struct RgSeq {
  int n_sh_local, G, b, per_exp, r_lo, r_hi;
};

// Runs the unit sequence: the producer (consumer == -1) issues each unit, a
// consumer warp c processes the row groups handed to it.  `issue(c, shared, e,
// g, kc)` issues segment kc of row group g for consumer c; `group(shared, e,
// g)` processes a whole row group.  Each consumer owns two ring stages (see
// kStagesPerConsumer), so a stage is only ever used by one consumer, in order.
template <typename Issue, typename Group>
__device__ bool rg_walk(RgSeq& q, int consumer, int KC, const GemvArgs& a, Issue&& issue, Group&& group) {
  for (int phase = 0; phase < 2; ++phase) {
    int lo, hi;
    if (phase == 0) {
      lo = 0;
      hi = q.n_sh_local;
    } else {
      pdl_wait();
      share(a.ws.active[a.E] * q.per_exp, q.b, q.G, q.r_lo, q.r_hi);
      lo = q.r_lo;
      hi = q.r_hi;
    }
    for (int bs = lo; bs < hi; bs += kConsumers) {
      const int nb = min(kConsumers, hi - bs);
      if (consumer < 0) {
        for (int kc = 0; kc < KC; ++kc)
          for (int r = 0; r < nb; ++r) {
            const int u = bs + r;
            const bool sh = phase == 0;
            const int e = sh ? 0 : a.ws.active[u / q.per_exp];
            const int g = sh ? q.b + u * q.G : u % q.per_exp;
            if (!issue(r, sh, e, g, kc)) return false;
          }
      } else if (consumer < nb) {
        const int u = bs + consumer;
        const bool sh = phase == 0;
        const int e = sh ? 0 : a.ws.active[u / q.per_exp];
        const int g = sh ? q.b + u * q.G : u % q.per_exp;
        if (!group(sh, e, g)) return false;
      }
    }
  }
  return true;
}

// Per-consumer stage ownership: consumer c uses stages 2c and 2c + 1 for its
// m-th unit alternately (stage 2c + (m & 1), phase parity (m >> 1) & 1).
constexpr int kStagesPerConsumer = kStages / kConsumers;
static_assert(kStagesPerConsumer == 2, "the ring gives each consumer warp two stages");
struct StageOwner {
  int m[kConsumers];
  uint32_t last_par[kStages];
  uint32_t used;
};
__device__ __forceinline__ void owner_init(StageOwner& o) {
  for (int c = 0; c < kConsumers; ++c) o.m[c] = 0;
  o.used = 0;
}
// Producer: wait for consumer c's next stage to be free; returns its index or -1.
__device__ __forceinline__ int owner_next(StageOwner& o, int c, uint64_t* empty, const WaitCtl& wc) {
  const int m = o.m[c]++;
  const int s = c * kStagesPerConsumer + (m & 1);
  if (!mbar_wait(&empty[s], ((m >> 1) & 1) ^ 1, wc)) return -1;
  o.last_par[s] = (m >> 1) & 1;
  o.used |= 1u << s;
  return s;
}
// Producer after an abort: let the copies already issued land.
__device__ __forceinline__ void owner_drain(const StageOwner& o, uint64_t* full, uint64_t wait_ns) {
  for (int s = 0; s < kStages; ++s)
    if (o.used & (1u << s)) {
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(&full[s], o.last_par[s]))
        if (global_ns() - t0 > wait_ns) break;
    }
}

// gate/up: row group g = gate rows 8g..8g+7 (A rows 0-7) and up rows 8g..8g+7
// (A rows 8-15); D rows 0-7 / 8-15 of the same thread are gate / up of the
// same row and token, so SwiGLU happens in registers.
__global__ void __launch_bounds__(kThreads, 1) gemv_mma_gateup_kernel(GemvArgs a, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t dsm[];
  pdl_launch_dependents();
  const Ring ring = ring_setup(dsm);
  const WaitCtl wc{wait_ns, a.ws.err, ring.abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, KC = d / kKc, G = gridDim.x, b = blockIdx.x;
  const int n_sh = a.Fs / 8;
  RgSeq q{b < n_sh ? (n_sh - b + G - 1) / G : 0, G, b, a.F / 8, 0, 0};
  if (warp == 0) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    StageOwner own;
    owner_init(own);
    auto issue = [&](int c, bool sh, int e, int g, int kc) -> bool {
      const int s = owner_next(own, c, ring.empty, wc);
      if (s < 0) return false;
      uint8_t* st = ring.stages + s * kStageBytes;
      const size_t row0 = sh ? (size_t)g * 8 : (size_t)e * a.F + (size_t)g * 8;
      const __nv_bfloat16* gw = static_cast<const __nv_bfloat16*>(sh ? a.sg : a.wg) + row0 * d + kc * kKc;
      const __nv_bfloat16* uw = static_cast<const __nv_bfloat16*>(sh ? a.su : a.wu) + row0 * d + kc * kKc;
      mbar_arrive_expect_tx(&ring.full[s], 16 * kKc * 2);
      for (int r = 0; r < 8; ++r) {
        bulk_g2s_hint(st + r * kRowPad, gw + (size_t)r * d, kKc * 2, &ring.full[s], pol);
        bulk_g2s_hint(st + (8 + r) * kRowPad, uw + (size_t)r * d, kKc * 2, &ring.full[s], pol);
      }
      return true;
    };
    auto none = [](bool, int, int) { return true; };
    if (!rg_walk(q, -1, KC, a, issue, none)) owner_drain(own, ring.full, wait_ns);
    return;
  }
  const int cw = warp - 1;
  const int Fmax = max(a.F, a.Fs);
  const uint32_t lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lcol = (lane >> 4) * 8;   // ldmatrix row / column
  auto none = [](int, bool, int, int, int) { return true; };
  int m = 0;                                   // units this consumer has taken
  auto group = [&](bool sh, int e, int g) -> bool {
    const int n = sh ? a.T : a.ws.counts[e];
    const int off = sh ? 0 : a.ws.offsets[e];
    const int ntiles = (n + 7) >> 3;
    const __nv_bfloat16* xrow[kMaxNT];
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) {
      int tok = nt * 8 + (lane >> 2);
      tok = tok < n ? tok : 0;
      const int t = sh ? tok : a.ws.tok_of_slot[off + tok];
      xrow[nt] = static_cast<const __nv_bfloat16*>(a.x) + (size_t)t * d + (lane & 3) * 2;
    }
    float acc[kMaxNT][4];
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    for (int kc = 0; kc < KC; ++kc, ++m) {
      const int s = cw * kStagesPerConsumer + (m & 1);
      if (!warp_wait_full(&ring.full[s], (m >> 1) & 1, wc)) return false;
      const uint32_t st = smem_u32(ring.stages + s * kStageBytes) + lrow * kRowPad + lcol * 2;
#pragma unroll 4
      for (int kk = 0; kk < kKc / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(st + kk * 32, af);
        const int k = kc * kKc + kk * 16;
#pragma unroll
        for (int nt = 0; nt < kMaxNT; ++nt)
          if (nt < ntiles) {
            const uint32_t b0 = __ldg(reinterpret_cast<const uint32_t*>(xrow[nt] + k));
            const uint32_t b1 = __ldg(reinterpret_cast<const uint32_t*>(xrow[nt] + k + 8));
            mma_bf16(acc[nt], af, b0, b1);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring.empty[s]);
    }
    const int f = g * 8 + (lane >> 2);
#pragma unroll
    for (int nt = 0; nt < kMaxNT; ++nt)
      if (nt < ntiles) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tok = nt * 8 + (lane & 3) * 2 + c;
          if (tok < n) {
            const int slot = sh ? a.T * a.k + tok : off + tok;
            a.ws.h16[(size_t)slot * Fmax + f] = __float2bfloat16_rn(silu(acc[nt][c]) * acc[nt][2 + c]);
          }
        }
      }
    return true;
  };
  rg_walk(q, cw, KC, a, none, group);
}

// down: row group g = Wd rows 16g..16g+15 of one expert; K = F (then F / 256
// segments); B = h (bf16) of the expert's slots.
__global__ void __launch_bounds__(kThreads, 1) gemv_mma_down_kernel(GemvArgs a, uint64_t wait_ns) {
  extern __shared__ __align__(128) uint8_t dsm[];
  pdl_launch_dependents();
  const Ring ring = ring_setup(dsm);
  const WaitCtl wc{wait_ns, a.ws.err, ring.abort_flag};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.d, F = a.F, G = gridDim.x, b = blockIdx.x;
  const int kd = F < kKc ? F : kKc, KC = F / kd, pad = kd * 2 + 16;   // segment values, segments, row pitch
  const int has_sh = a.Fs > 0 ? 1 : 0;
  pdl_wait();
  // All row groups need h, so there is no early phase: the shared expert's
  // groups join the contiguous split (routed index offset by one expert).
  const int n_exp = a.ws.active[a.E] + has_sh;
  const int total = n_exp * (d / 16);
  int lo, hi;
  share(total, b, G, lo, hi);
  auto expert_of = [&](int u, bool& sh, int& e, int& g) {
    const int ai = u / (d / 16);
    sh = has_sh && ai == 0;
    e = sh ? 0 : a.ws.active[ai - has_sh];
    g = u % (d / 16);
  };
  if (warp == 0) {
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    StageOwner own;
    owner_init(own);
    bool ok = true;
    for (int bs = lo; bs < hi && ok; bs += kConsumers) {
      const int nb = min(kConsumers, hi - bs);
      for (int kc = 0; kc < KC && ok; ++kc)
        for (int r = 0; r < nb; ++r) {
          bool sh;
          int e, g;
          expert_of(bs + r, sh, e, g);
          const int s = owner_next(own, r, ring.empty, wc);
          if (s < 0) { ok = false; break; }
          uint8_t* st = ring.stages + s * kStageBytes;
          const size_t row0 = sh ? (size_t)g * 16 : (size_t)e * d + (size_t)g * 16;
          const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(sh ? a.sd : a.wd) + row0 * F + kc * kd;
          mbar_arrive_expect_tx(&ring.full[s], 16 * kd * 2);
          for (int rr = 0; rr < 16; ++rr) bulk_g2s_hint(st + rr * pad, w + (size_t)rr * F, kd * 2, &ring.full[s], pol);
        }
    }
    if (!ok) owner_drain(own, ring.full, wait_ns);
    return;
  }
  const int cw = warp - 1;
  const int Fmax = max(a.F, a.Fs);
  const uint32_t lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lcol = (lane >> 4) * 8;
  int m = 0;                                   // units this consumer has taken
  for (int bs = lo; bs < hi; bs += kConsumers) {
    const int nb = min(kConsumers, hi - bs);
    if (cw < nb) {
      bool sh;
      int e, g;
      expert_of(bs + cw, sh, e, g);
      const int n = sh ? a.T : a.ws.counts[e];
      const int off = sh ? 0 : a.ws.offsets[e];
      const int ntiles = (n + 7) >> 3;
      const __nv_bfloat16* hrow[kMaxNT];
#pragma unroll
      for (int nt = 0; nt < kMaxNT; ++nt) {
        int tok = nt * 8 + (lane >> 2);
        tok = tok < n ? tok : 0;
        const int slot = sh ? a.T * a.k + tok : off + tok;
        hrow[nt] = a.ws.h16 + (size_t)slot * Fmax + (lane & 3) * 2;
      }
      float acc[kMaxNT][4];
#pragma unroll
      for (int nt = 0; nt < kMaxNT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      bool ok = true;
      for (int kc = 0; kc < KC; ++kc, ++m) {
        const int s = cw * kStagesPerConsumer + (m & 1);
        if (!warp_wait_full(&ring.full[s], (m >> 1) & 1, wc)) { ok = false; break; }
        const uint32_t st = smem_u32(ring.stages + s * kStageBytes) + lrow * pad + lcol * 2;
#pragma unroll 4
        for (int kk = 0; kk < kd / 16; ++kk) {
          uint32_t af[4];
          ldsm_x4(st + kk * 32, af);
          const int k = kc * kd + kk * 16;
#pragma unroll
          for (int nt = 0; nt < kMaxNT; ++nt)
            if (nt < ntiles) {
              const uint32_t b0 = __ldg(reinterpret_cast<const uint32_t*>(hrow[nt] + k));
              const uint32_t b1 = __ldg(reinterpret_cast<const uint32_t*>(hrow[nt] + k + 8));
              mma_bf16(acc[nt], af, b0, b1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[s]);
      }
      if (!ok) return;
      const int r = g * 16 + (lane >> 2);
#pragma unroll
      for (int nt = 0; nt < kMaxNT; ++nt)
        if (nt < ntiles) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tok = nt * 8 + (lane & 3) * 2 + c;
            if (tok < n) {
              const int slot = sh ? a.T * a.k + tok : off + tok;
              a.ws.ypart[(size_t)slot * d + r] = acc[nt][c];
              a.ws.ypart[(size_t)slot * d + r + 8] = acc[nt][2 + c];
            }
          }
        }
      // each of a token's experts brings two 16-row groups to a 32-row block
      complete_block(a, sh, off, n, (g * 16) / kFinRows, (a.k + has_sh) * (kFinRows / 16));
    }
  }
}

constexpr size_t kSmem = (size_t)kStages * kStageBytes + 2 * kStages * 8 + 16;

template <typename K>
cudaError_t launch_pdl(K kernel, int grid, cudaStream_t s, const GemvArgs& a, uint64_t wait_ns) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, wait_ns);
}

cudaError_t launch_mma(const GemvArgs& a, int num_sms, cudaStream_t s, Prof* prof, uint64_t wait_ns) {
  {
    cudaError_t e = ensure_smem_limit(gemv_mma_gateup_kernel, (int)kSmem);
    if (e == cudaSuccess) e = ensure_smem_limit(gemv_mma_down_kernel, (int)kSmem);
    if (e != cudaSuccess) return e;
  }
  if (prof) prof->begin(MOE_K_GEMV_GATEUP, s);
  cudaError_t e = launch_pdl(gemv_mma_gateup_kernel, num_sms, s, a, wait_ns);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  if (prof) prof->begin(MOE_K_GEMV_DOWN, s);
  e = launch_pdl(gemv_mma_down_kernel, num_sms, s, a, wait_ns);
  if (prof) prof->end(s);
  return e;
}

// f16 copy of the activations for the NVFP4 kernels: token t scaled by 2^-e
// (its largest magnitude into [1, 2)), xsc[t] = 2^e.  One warp per token.
// Needs only x, so it runs alongside the router; it waits for the router at
// the end so that a kernel waiting on this one also sees the routing.
__global__ void __launch_bounds__(256) gemv_x16_kernel(const __nv_bfloat16* __restrict__ x, __half* __restrict__ xh,
                                                       float* __restrict__ xsc, int T, int d) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t < T) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    const int n16 = d / 8;
    uint32_t mx = 0;                               // largest |x| as bits (monotone for |x|)
    for (int c = lane; c < n16; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = max(mx, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
    }
    mx = __reduce_max_sync(FULLMASK, mx);
    // 2^-e with e the exponent of the maximum (normal maxima only; a zero,
    // subnormal, infinite or NaN maximum leaves the token unscaled)
    const int eb = (int)(mx >> 23);
    const bool scaled = eb >= 2 && eb <= 252;
    const float inv = scaled ? __int_as_float((254 - eb) << 23) : 1.f;
    if (lane == 0) xsc[t] = scaled ? __int_as_float(eb << 23) : 1.f;
    uint4* dst = reinterpret_cast<uint4*>(xh + (size_t)t * d);
    for (int c = lane; c < n16; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * inv, __uint_as_float(w[i] & 0xFFFF0000u) * inv);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  pdl_wait();
}

template <int WF, int J, int CPR>
cudaError_t launch_fmt(const GemvArgs& a, int num_sms, cudaStream_t s, Prof* prof, uint64_t wait_ns) {
  {
    cudaError_t e = ensure_smem_limit(gemv_gateup_kernel<WF, J>, (int)kSmem);
    if (e == cudaSuccess) e = ensure_smem_limit(gemv_down_kernel<WF, CPR>, (int)kSmem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaSuccess;
  if (WF == MOE_NVFP4) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.T + 7) / 8);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemv_x16_kernel, static_cast<const __nv_bfloat16*>(a.x), a.ws.xh16, a.ws.xsc, a.T,
                           a.d);
    if (e != cudaSuccess) return e;
  }
  if (prof) prof->begin(MOE_K_GEMV_GATEUP, s);
  e = launch_pdl(gemv_gateup_kernel<WF, J>, num_sms, s, a, wait_ns);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  if (prof) prof->begin(MOE_K_GEMV_DOWN, s);
  e = launch_pdl(gemv_down_kernel<WF, CPR>, num_sms, s, a, wait_ns);
  if (prof) prof->end(s);
  return e;
}

}  // namespace

bool gemv_supported(int wfmt, int d, int F, int Fs) {
  if (Fs != 0 && Fs != F) return false;
  if (wfmt == MOE_BF16) return d % kKc == 0 && (F % kKc == 0 || F == 128) && d % kFinRows == 0;
  const int rb = wfmt == MOE_F32 ? d * 4 : wfmt == MOE_BF16 ? d * 2 : d / 2;
  const int fb = wfmt == MOE_F32 ? F * 4 : wfmt == MOE_BF16 ? F * 2 : F / 2;
  if (rb % 512 != 0) return false;
  const int J = rb / 512;
  if (J != 1 && J != 2 && J != 4 && J != 8) return false;
  const int cpr = fb / 16;
  if (fb % 16 != 0 || (cpr != 16 && cpr != 32 && cpr != 64 && cpr != 128)) return false;
  const int rg = 8 / J;
  if (F % rg != 0 || Fs % rg != 0 || d % (512 / cpr) != 0) return false;
  return true;
}

cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int num_sms, cudaStream_t s, Prof* prof, uint64_t wait_ns) {
  const int rb = wfmt == MOE_F32 ? a.d * 4 : wfmt == MOE_BF16 ? a.d * 2 : a.d / 2;
  const int J = rb / 512;
  const int cpr = (wfmt == MOE_F32 ? a.F * 4 : wfmt == MOE_BF16 ? a.F * 2 : a.F / 2) / 16;
#define MOE_G(WF, JJ, CC) \
  if (J == JJ && cpr == CC) return launch_fmt<WF, JJ, CC>(a, num_sms, s, prof, wait_ns);
#define MOE_GF(WF, JJ) MOE_G(WF, JJ, 16) MOE_G(WF, JJ, 32) MOE_G(WF, JJ, 64) MOE_G(WF, JJ, 128)
  if (wfmt == MOE_BF16) {
    return launch_mma(a, num_sms, s, prof, wait_ns);
  } else if (wfmt == MOE_F32) {
    MOE_GF(MOE_F32, 1) MOE_GF(MOE_F32, 2) MOE_GF(MOE_F32, 4) MOE_GF(MOE_F32, 8)
  } else {
    MOE_GF(MOE_NVFP4, 1) MOE_GF(MOE_NVFP4, 2) MOE_GF(MOE_NVFP4, 4) MOE_GF(MOE_NVFP4, 8)
  }
#undef MOE_GF
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
