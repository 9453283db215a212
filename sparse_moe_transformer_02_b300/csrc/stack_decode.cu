// Persistent decode kernel over a whole stack of MoE layers: one launch runs
// every layer for a small batch of tokens.
//
// The pages describe a decode "megakernel" that fuses the whole decode
// forward pass into one kernel (evermx.com review, Feature Overview, "Kernels
// and inference"); for the MoE layers of a stack (47 of them in Flint, joined
// by residual adds: swarmz.net, section "The architecture, in plain terms")
// this is its counterpart on B300.  Per layer and token batch (T <= 8) the
// work is a few tens of MB of weights, a few microseconds of HBM time, so a
// launch per kernel per layer would cost as much as the weight stream; here
// the layers follow each other inside one cooperative grid (one CTA per SM)
// separated by grid-wide barriers.
//
// A single layer (moe_forward with T <= 8) runs as a stack of one, with the
// residual add optional.
//
// Per layer three phases, each ending in a grid barrier:
//   A  router logits (fp32; each expert row split over 4 warps across the
//      grid, plain loads, partial sums added in a fixed order by the top-k)
//      and the shared expert's gate/up row groups (need no routing);
//   B  top-k, gates and grouping, computed by every CTA for itself from the
//      logits (identical inputs and instructions, so every CTA holds the same
//      routing), then the routed experts' gate/up row groups, split evenly
//      over the CTAs;
//   C  down projection: CTA b owns output rows [16 rb, 16 rb + 16) for
//      rb = b, b + G, ...; its consumer warps take the shared expert and the
//      active experts in turn, weight their rows by the gates and the CTA sums
//      the warps in a fixed order (deterministic), adds the residual x (in
//      a stack; optional for a single layer) and rounds to bf16.
//
// Inside a CTA one producer thread streams weights with TMA tile loads into a
// 16-stage shared-memory ring (two stages per consumer warp, each stage 16
// rows x 256 values = 8 KB in one or two loads of a 3-D box {64 values, rows,
// 4 chunks of 64} with the 128-byte swizzle; the chunk dimension is outermost
// in shared memory, so the swizzle's XOR follows the weight row and ldmatrix
// rows hit distinct banks; many small 1-D bulk copies instead left the copy
// engine, not HBM, as the limit); eight consumer warps multiply on the tensor pipe (mma.sync
// m16n8k16, bf16 in, fp32 accumulate) with the activations (x or h, staged
// once per phase in shared memory) as the 8-column B operand.  A gate/up row
// group is 8 gate rows + 8 up rows of one expert, its K segments spread over
// the consumer warps and summed through shared memory in warp order; the
// thread holding gate row f and up row f of a token applies SwiGLU.  The
// producer does not wait for barriers: it runs ahead into the next phase's
// weights as far as the ring allows (phase A needs no routing; phases B and C
// wait only for this CTA's routing), so the weights of the next phase are in
// flight while the grid synchronises.
//
// Every wait is bounded: the ring, the routing hand-off and the grid barrier
// give up after the limit, set the device error word (timeout bit) and the
// CTA unwinds, draining its bulk copies first.
#include "moe_internal.cuh"
#include "persist.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace persist;

constexpr int kSdThreads = 32 * (1 + kSdConsumers);
constexpr int kSdStages = 2 * kSdConsumers;         // two per consumer warp
constexpr int kSdSeg = 256;                         // values per row segment
constexpr int kSdRq = 4;                            // warps per router row
constexpr int kSdStageBytes = 16 * kSdSeg * 2;      // 8192 bytes: 16 rows x 4 chunks x 128 bytes

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Shared-memory layout (byte offsets), computed identically on host and device.
struct SdLayout {
  uint32_t stages, bars, route_bar, abort, xs, red, yw, rt, total;
  uint32_t x_pitch, h_pitch;
};
__host__ __device__ inline SdLayout sd_layout(int d, int Fmax, int k) {
  SdLayout L;
  L.x_pitch = (uint32_t)d * 2 + 16;
  L.h_pitch = (uint32_t)Fmax * 2 + 16;
  uint32_t o = 0;
  L.stages = o; o += kSdStages * kSdStageBytes;
  L.bars = o;   o += 2 * kSdStages * 8;
  L.route_bar = o; o += 8;
  L.abort = o;  o += 8;
  L.xs = o;                                          // x rows (phases A, B) or h rows (phase C)
  const uint32_t xsz = kSdMaxT * L.x_pitch, hsz = (uint32_t)kSdMaxT * (k + 1) * L.h_pitch;
  o += (xsz > hsz ? xsz : hsz);
  o = (o + 15) & ~15u;
  L.red = o;    o += 2 * kSdConsumers * 32 * 4 * 4;   // double-buffered partial sums of a row group
  L.yw = o;     o += kSdConsumers * 16 * kSdMaxT * 4; // per-warp down-projection sums of a row block
  L.rt = o;     o += 4096;                            // routing tables (below)
  L.total = o + 1024;                                 // slack to align the base to 1024 bytes
  return L;
}
// Routing tables inside L.rt (ints / floats):
//   sel_e[64], sel_g[64]  top-k of each token, slot s = t k + j
//   slot_tok[64], slot_gate[64]  grouped slots (experts ascending, tokens ascending)
//   act_e[65], act_off[65], n_act  active experts, first grouped slot of each
//   cnt[256], off[256]  per-expert counts / offsets (grouping scratch)
struct Rt {
  int* sel_e; float* sel_g; int* slot_tok; float* slot_gate; int* act_e; int* act_off; int* n_act;
  int* cnt; int* off;
};
__device__ __forceinline__ Rt rt_of(uint8_t* base) {
  int* p = reinterpret_cast<int*>(base);
  Rt r;
  r.sel_e = p; p += 64;
  r.sel_g = reinterpret_cast<float*>(p); p += 64;
  r.slot_tok = p; p += 64;
  r.slot_gate = reinterpret_cast<float*>(p); p += 64;
  r.act_e = p; p += 65;
  r.act_off = p; p += 65;
  r.n_act = p; p += 2;
  r.cnt = p; p += 256;
  r.off = p;
  return r;
}

// The producer's view of the ring: consumer c owns stages 2c, 2c + 1 and
// takes them alternately; its m-th stage has phase parity (m >> 1) & 1.  The
// counters live in shared memory (a local array indexed by consumer would sit
// in local memory, which this kernel's shared-memory footprint leaves
// uncached in L1).

// One CTA's walk over the stack: the producer (prod = true) issues every
// stage, the consumers process them, both in the same order.
struct SdCtx {
  const StackArgs& a;               // the kernel's __grid_constant__ parameter (no copy)
  SdLayout L;
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* route_bar;
  volatile int* abort_flag;
  Rt rt;
  WaitCtl wc;
  int G, b, warp, lane;
  int* prod_m;                      // producer: stages taken per consumer [kSdConsumers]
  uint32_t* prod_par;               // producer: phase parity last used per stage [kSdStages]
};

// ---------------------------------------------------------------- producer
// One thread issues every stage of the CTA.
struct Producer {
  SdCtx& c;
  uint64_t pol;
  uint32_t used = 0;
  __device__ __forceinline__ explicit Producer(SdCtx& ctx) : c(ctx) {
    for (int i = 0; i < kSdConsumers; ++i) c.prod_m[i] = 0;
    pol = policy_evict_first();
  }
  // Next stage of consumer w (bounded wait for it to be free); -1 on abort.
  __device__ __forceinline__ int next(int w) {
    const int m = c.prod_m[w]++;
    const int s = w * 2 + (m & 1);
    if (!mbar_wait(&c.empty[s], ((m >> 1) & 1) ^ 1, c.wc)) return -1;
    c.prod_par[s] = (m >> 1) & 1;
    used |= 1u << s;
    return s;
  }
  // Gate/up stage: gate rows [row0, row0 + 8) and up rows [row0, row0 + 8),
  // values [256 s, 256 s + 256): two 4 KB boxes.
  __device__ __forceinline__ bool issue_gu(int w, const CUtensorMap* mg, const CUtensorMap* mu, int row0, int s) {
    const int st = next(w);
    if (st < 0) return false;
    uint8_t* dst = c.smem + c.L.stages + st * kSdStageBytes;
    mbar_arrive_expect_tx(&c.full[st], kSdStageBytes);
    tma_load_3d_hint(dst, mg, 0, row0, 4 * s, &c.full[st], pol);
    tma_load_3d_hint(dst + kSdStageBytes / 2, mu, 0, row0, 4 * s, &c.full[st], pol);
    return true;
  }
  // Down stage: rows [row0, row0 + 16), values [256 s, 256 s + 256): one 8 KB box.
  __device__ __forceinline__ bool issue_dn(int w, const CUtensorMap* md, int row0, int s) {
    const int st = next(w);
    if (st < 0) return false;
    uint8_t* dst = c.smem + c.L.stages + st * kSdStageBytes;
    mbar_arrive_expect_tx(&c.full[st], kSdStageBytes);
    tma_load_3d_hint(dst, md, 0, row0, 4 * s, &c.full[st], pol);
    return true;
  }
  __device__ __forceinline__ void drain() {
    for (int s = 0; s < kSdStages; ++s)
      if (used & (1u << s)) drain_wait(&c.full[s], c.prod_par[s], c.wc.limit_ns);
  }
};

// Gate/up row group g of an expert (first row row0 = e F + 8 g, or 8 g for
// the shared expert): K segments spread over the consumers (segment s ->
// consumer s % 8).
__device__ __forceinline__ bool produce_gu(Producer& P, const CUtensorMap* mg, const CUtensorMap* mu, int row0, int d) {
  const int KC = d / kSdSeg;
  for (int s = 0; s < KC; ++s)
    if (!P.issue_gu(s % kSdConsumers, mg, mu, row0, s)) return false;
  return true;
}

__device__ __forceinline__ void run_producer(SdCtx& c) {
  const StackArgs& a = c.a;
  Producer P(c);
  const int nsh = a.Fs / 8;
  bool ok = true;
  for (int l = 0; l < a.L && ok; ++l) {
    const CUtensorMap* M = a.maps + (size_t)l * kSdMaps;
    if (l + 1 < a.L)
      for (int i = 0; i < kSdMaps; ++i) tma_prefetch_desc(M + kSdMaps + i);
    // phase A: the shared expert's row groups of this CTA
    for (int g = c.b; g < nsh && ok; g += c.G) ok = produce_gu(P, M + kMapSg, M + kMapSu, g * 8, a.d);
    if (!ok) break;
    // this CTA's routing for layer l
    if (!mbar_wait(c.route_bar, l & 1, c.wc)) { ok = false; break; }
    const int U = *c.rt.n_act;
    // phase B: routed row groups, an even share per CTA
    const int ngrp = a.F / 8, n = U * ngrp;
    const int lo = (int)(((long long)n * c.b) / c.G), hi = (int)(((long long)n * (c.b + 1)) / c.G);
    for (int u = lo; u < hi && ok; ++u) {
      const int e = c.rt.act_e[u / ngrp];
      ok = produce_gu(P, M + kMapWg, M + kMapWu, e * a.F + (u % ngrp) * 8, a.d);
    }
    // phase C: the down rows of this CTA's row blocks, unit j -> consumer j % 8
    const int has_sh = a.Fs > 0 ? 1 : 0;
    for (int rb = c.b; rb < a.d / 16 && ok; rb += c.G) {
      for (int j = 0; j < U + has_sh && ok; ++j) {
        const bool sh = has_sh && j == 0;
        const int Fe = sh ? a.Fs : a.F;
        const int row0 = sh ? rb * 16 : c.rt.act_e[j - has_sh] * a.d + rb * 16;
        for (int s = 0; s < Fe / kSdSeg && ok; ++s) ok = P.issue_dn(j % kSdConsumers, M + (sh ? kMapSd : kMapWd), row0, s);
      }
    }
  }
  if (!ok) P.drain();
}

// ---------------------------------------------------------------- consumers
// Wait for this consumer's next stage; returns its shared address or 0 on abort.
struct Cons {
  SdCtx& c;
  int m = 0;
  __device__ __forceinline__ explicit Cons(SdCtx& ctx) : c(ctx) {}
  __device__ __forceinline__ uint32_t wait() {
    const int s = c.warp - 1;
    const int st = s * 2 + (m & 1);
    int ok = 1;
    if (c.lane == 0) ok = mbar_wait(&c.full[st], (m >> 1) & 1, c.wc) ? 1 : 0;
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok) return 0;
    while (!mbar_try_wait(&c.full[st], (m >> 1) & 1)) {
    }
    cur = st;
    return smem_u32(c.smem + c.L.stages + st * kSdStageBytes);
  }
  __device__ __forceinline__ void release() {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.empty[cur]);
    ++m;
  }
  int cur = 0;
};

// acc += stage (16 rows x 256 values) x B, B row n = bidx (k offset k0, 8
// columns).  The stage holds 4 chunks of 64 values; row r of chunk c is a
// 128-byte line whose 16-byte pieces are XOR-swizzled by r & 7.  Gate/up
// stages (gu) keep rows 0-7 (gate) and 8-15 (up) in two 4 KB boxes
// [chunk][8 rows]; down stages are one 8 KB box [chunk][16 rows].
__device__ __forceinline__ void mma_stage(uint32_t st, bool gu, uint32_t bbase, uint32_t bpitch, const int (&bidx)[1],
                                          int k0, int lane, float (&acc)[4]) {
  const uint32_t lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lhi = lane >> 4;   // ldmatrix row, 8-value half
  const uint32_t rr = gu ? (lrow & 7) : lrow;
  const uint32_t rbase = st + (gu ? (lrow >> 3) * (kSdStageBytes / 2) : 0) + rr * 128;
  const uint32_t cstride = gu ? 1024 : 2048, sw = lrow & 7;
  const uint32_t b0a = bbase + (uint32_t)bidx[0] * bpitch + (uint32_t)(k0 + (lane & 3) * 2) * 2;
#pragma unroll 4
  for (int kk = 0; kk < kSdSeg / 16; ++kk) {
    uint32_t af[4];
    const uint32_t piece = ((((uint32_t)kk & 3) << 1) | lhi) ^ sw;
    ldsm_x4(rbase + (kk >> 2) * cstride + (piece << 4), af);
    const uint32_t b0 = lds32(b0a + kk * 32), b1 = lds32(b0a + kk * 32 + 16);
    mma_bf16(acc, af, b0, b1);
  }
}

// One gate/up row group: the consumer's K segments, the cross-warp sum in
// warp order, SwiGLU, h rows of the group's tokens.  rows_tok(n) = x row of
// column n (n < cnt), hslot(n) = h row to write.  rg counts row groups (for
// the double-buffered partials and the finalising warp).
template <typename Tok, typename Slot>
__device__ __forceinline__ bool consume_gu(SdCtx& c, Cons& C, int d, int g, int cnt, int rg, Tok&& rows_tok, Slot&& hslot,
                           __nv_bfloat16* h, int Fmax) {
  const int w = c.warp - 1, lane = c.lane, KC = d / kSdSeg;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  int n = lane >> 2;
  int bidx[1] = {rows_tok(n < cnt ? n : 0)};
  const uint32_t xs = smem_u32(c.smem + c.L.xs);
  // A failed wait has set the CTA's abort flag; this warp then skips its work
  // but still reaches the barrier, after which every warp leaves together
  // (a warp that left early would strand the others in bar.sync).
  for (int s = w; s < KC; s += kSdConsumers) {
    const uint32_t st = C.wait();
    if (!st) break;
    mma_stage(st, true, xs, c.L.x_pitch, bidx, s * kSdSeg, lane, acc);
    C.release();
  }
  float* red = reinterpret_cast<float*>(c.smem + c.L.red) + (size_t)(rg & 1) * kSdConsumers * 128;
  reinterpret_cast<float4*>(red)[w * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  if (named_sync_or(2, 32 * kSdConsumers, *c.abort_flag != 0)) return false;
  if (w == (rg % kSdConsumers)) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int nw = KC < kSdConsumers ? KC : kSdConsumers;
    for (int ww = 0; ww < nw; ++ww) {
      const float4 p = reinterpret_cast<const float4*>(red)[ww * 32 + lane];
      v[0] += p.x; v[1] += p.y; v[2] += p.z; v[3] += p.w;
    }
    const int f = g * 8 + (lane >> 2);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = (lane & 3) * 2 + q;
      if (col < cnt) {
        const float hv = silu_f(v[q]) * v[2 + q];
        __stcg(reinterpret_cast<unsigned short*>(h) + (size_t)hslot(col) * Fmax + f,
               __bfloat16_as_ushort(__float2bfloat16_rn(hv)));
      }
    }
  }
  return true;
}

// Grouping of the T k slots by expert (one warp): active experts ascending,
// slots of one expert in (token, j) order.
// slot_of (global memory, may be null) receives the grouped position of each
// slot t k + j.
__device__ __forceinline__ void group_slots_warp(Rt& rt, int T, int k, int E, int lane, int32_t* slot_of) {
  const int ns = T * k;
  for (int e = lane; e < 256; e += 32) rt.cnt[e] = 0;
  __syncwarp();
  const int s0 = lane, s1 = lane + 32;
  const bool v0 = s0 < ns, v1 = s1 < ns;
  const int e0 = v0 ? rt.sel_e[s0] : -1 - lane, e1 = v1 ? rt.sel_e[s1] : -100 - lane;
  const unsigned lt = (1u << lane) - 1u;
  const unsigned m0 = __match_any_sync(kFull, e0);
  const int r0 = __popc(m0 & lt);
  if (v0 && r0 == 0) rt.cnt[e0] = __popc(m0);
  __syncwarp();
  const unsigned m1 = __match_any_sync(kFull, e1);
  const int r1 = (v1 ? rt.cnt[e1] : 0) + __popc(m1 & lt);
  __syncwarp();
  if (v1 && __popc(m1 & lt) == 0) rt.cnt[e1] += __popc(m1);
  __syncwarp();
  // exclusive scans over the experts (8 per lane): slot offsets and active ranks
  int c[8], tot = 0, act = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    c[i] = e < E ? rt.cnt[e] : 0;
    tot += c[i];
    act += c[i] > 0;
  }
  int it = tot, ia = act;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, it, o), y = __shfl_up_sync(kFull, ia, o);
    if (lane >= o) { it += x; ia += y; }
  }
  int off = it - tot, rank = ia - act;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * 8 + i;
    if (e < E) {
      rt.off[e] = off;
      if (c[i] > 0) {
        rt.act_e[rank] = e;
        rt.act_off[rank] = off;
        ++rank;
      }
    }
    off += c[i];
  }
  if (lane == 31) {
    rt.act_off[ia] = ns;
    *rt.n_act = ia;
  }
  __syncwarp();
  if (v0) {
    const int p = rt.off[e0] + r0;
    rt.slot_tok[p] = s0 / k;
    rt.slot_gate[p] = rt.sel_g[s0];
    if (slot_of) slot_of[s0] = p;
  }
  if (v1) {
    const int p = rt.off[e1] + r1;
    rt.slot_tok[p] = s1 / k;
    rt.slot_gate[p] = rt.sel_g[s1];
    if (slot_of) slot_of[s1] = p;
  }
  __syncwarp();
}

__device__ __forceinline__ void run_consumers(SdCtx& c) {
  const StackArgs& a = c.a;
  Cons C(c);
  const int w = c.warp - 1, lane = c.lane, tid = threadIdx.x - 32, NT = 32 * kSdConsumers;
  const int T = a.T, d = a.d, F = a.F, Fs = a.Fs, E = a.E, k = a.k;
  const int Fmax = F > Fs ? F : Fs;
  const int has_sh = Fs > 0 ? 1 : 0;
  const int nsh = Fs / 8;
  unsigned nbar = 0;
  int rg = 0;                                  // row groups processed (partials buffer / finaliser)
  for (int l = 0; l < a.L; ++l) {
    const StackLayerPtrs& W = a.layers[l];
    const __nv_bfloat16* xcur = l == 0 ? a.x_in : a.xbuf + (size_t)((l - 1) & 1) * kSdMaxT * d;
    __nv_bfloat16* xnext = l == a.L - 1 ? a.y_out : a.xbuf + (size_t)(l & 1) * kSdMaxT * d;
    // stage x (T rows) in shared memory
    {
      uint8_t* xs = c.smem + c.L.xs;
      const int chunks = d / 8;
      stage_rows(xs, c.L.x_pitch, reinterpret_cast<const uint8_t*>(xcur), (size_t)d * 2, T, chunks, tid, NT);
      if (l == 0 && a.x_trace && c.b == 0)
        for (int i = tid; i < T * chunks; i += NT)
          __stcg(reinterpret_cast<uint4*>(a.x_trace) + i, __ldcg(reinterpret_cast<const uint4*>(a.x_in) + i));
    }
    named_sync(1, NT);
    // router: row e split into kSdRq quarter rows, task e * kSdRq + q on global
    // warp G * 8 - 1 - task (the last CTAs first); partial logits
    // part[q][t][e] are summed in q order by the top-k
    {
      const int gw = c.b * kSdConsumers + w, nw = c.G * kSdConsumers, dq = d / kSdRq;
      for (int task = nw - 1 - gw; task >= 0 && task < E * kSdRq; task += nw) {
        const int e = task / kSdRq, q = task % kSdRq;
        const float* wr = W.wr + (size_t)e * d + (size_t)q * dq;
        const float bias = (q == 0 && W.br) ? __ldg(W.br + e) : 0.f;   // quarter 0 carries the bias
        float acc[kSdMaxT];
#pragma unroll
        for (int t = 0; t < kSdMaxT; ++t) acc[t] = 0.f;
        for (int i0 = lane * 4; i0 < dq; i0 += 32 * 4 * 4) {
          float4 wv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * 128;
            wv[u] = i < dq ? __ldg(reinterpret_cast<const float4*>(wr + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * 128;
            if (i < dq) {
#pragma unroll
              for (int t = 0; t < kSdMaxT; ++t)
                if (t < T) {
                  const uint2 xv =
                      *reinterpret_cast<const uint2*>(c.smem + c.L.xs + t * c.L.x_pitch + (q * dq + i) * 2);
                  const float x0 = __uint_as_float(xv.x << 16), x1 = __uint_as_float(xv.x & 0xFFFF0000u);
                  const float x2 = __uint_as_float(xv.y << 16), x3 = __uint_as_float(xv.y & 0xFFFF0000u);
                  acc[t] = fmaf(wv[u].x, x0, fmaf(wv[u].y, x1, fmaf(wv[u].z, x2, fmaf(wv[u].w, x3, acc[t]))));
                }
            }
          }
        }
        // butterfly transpose-reduction: lanes 4 t .. 4 t + 3 end with token t's sum
        const float v = transpose_reduce<kSdMaxT, 32>(acc, lane);
        const int t = lane >> 2;
        if ((lane & 3) == 0 && t < T) __stcg(a.logits + ((size_t)q * kSdMaxT + t) * E + e, v + bias);
      }
    }
    // phase A: shared expert row groups (all T tokens)
    for (int g = c.b; g < nsh; g += c.G, ++rg)
      if (!consume_gu(c, C, d, g, T, rg, [&](int n) { return n; }, [&](int n) { return T * k + n; }, a.h, Fmax))
        return;
    if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, 32 * kSdConsumers, 32)) return;

    // routing (every CTA), then hand it to the producer
    if (w < T) topk_token(a.logits, kSdRq, kSdMaxT, E, k, w, c.rt.sel_e, c.rt.sel_g, lane);
    named_sync(1, NT);
    if (w == 0) group_slots_warp(c.rt, T, k, E, lane, c.b == 0 ? a.g_slot_of : nullptr);
    named_sync(1, NT);
    if (c.b == 0 && a.g_offsets) {             // the grouping, for a caller that asks for it
      for (int i = tid; i <= E; i += NT) a.g_offsets[i] = i < E ? c.rt.off[i] : T * k;
      for (int i = tid; i < T * k; i += NT) a.g_tok_of_slot[i] = c.rt.slot_tok[i];
    }
    if (tid == 0) mbar_arrive(c.route_bar);
    if (c.b == 0 && (a.idx_trace || a.gate_trace))
      for (int i = tid; i < T * k; i += NT) {
        if (a.idx_trace) a.idx_trace[(size_t)l * T * k + i] = c.rt.sel_e[i];
        if (a.gate_trace) a.gate_trace[(size_t)l * T * k + i] = c.rt.sel_g[i];
      }
    const int U = *c.rt.n_act;
    // phase B: routed row groups
    {
      const int ngrp = F / 8, n = U * ngrp;
      const int lo = (int)(((long long)n * c.b) / c.G), hi = (int)(((long long)n * (c.b + 1)) / c.G);
      for (int u = lo; u < hi; ++u, ++rg) {
        const int ai = u / ngrp;
        const int off = c.rt.act_off[ai], cnt = c.rt.act_off[ai + 1] - off;
        if (!consume_gu(c, C, d, u % ngrp, cnt, rg, [&](int nn) { return c.rt.slot_tok[off + nn]; },
                        [&](int nn) { return off + nn; }, a.h, Fmax))
          return;
      }
    }
    if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, 32 * kSdConsumers, 32)) return;

    // phase C: stage h (routed slots, then the shared expert's T rows) in shared memory
    const int nslots = T * k + (has_sh ? T : 0);
    {
      uint8_t* hs = c.smem + c.L.xs;
      stage_rows(hs, c.L.h_pitch, reinterpret_cast<const uint8_t*>(a.h), (size_t)Fmax * 2, nslots, Fmax / 8, tid, NT);
    }
    // CTAs that own no output rows pull the next layer's router rows into L2
    // meanwhile, so its logits do not wait on HBM latency
    if (c.b >= d / 16 && l + 1 < a.L && c.G > d / 16) {
      const size_t bytes = (size_t)E * d * 4, nidle = (size_t)(c.G - d / 16);
      const size_t per = ((bytes + nidle - 1) / nidle + 4095) & ~(size_t)4095;
      const size_t lo = per * (size_t)(c.b - d / 16), hi = lo + per < bytes ? lo + per : bytes;
      const char* base = reinterpret_cast<const char*>(a.layers[l + 1].wr);
      for (size_t o = lo + (size_t)tid * 4096; o < hi; o += (size_t)NT * 4096) {
        const uint32_t n = (uint32_t)(hi - o < 4096 ? hi - o : 4096);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(n) : "memory");
      }
    }
    float* yw = reinterpret_cast<float*>(c.smem + c.L.yw);
    for (int rb = c.b; rb < d / 16; rb += c.G) {
      for (int i = tid; i < kSdConsumers * 16 * kSdMaxT; i += NT) yw[i] = 0.f;
      named_sync(1, NT);
      for (int j = w; j < U + has_sh; j += kSdConsumers) {
        const bool sh = has_sh && j == 0;
        const int ai = j - has_sh;
        const int off = sh ? T * k : c.rt.act_off[ai];
        const int cnt = sh ? T : c.rt.act_off[ai + 1] - off;
        const int Fe = sh ? Fs : F;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int n = lane >> 2;
        int bidx[1] = {off + (n < cnt ? n : 0)};
        bool ok = true;
        for (int s = 0; s < Fe / kSdSeg; ++s) {
          const uint32_t st = C.wait();
          if (!st) { ok = false; break; }
          mma_stage(st, false, smem_u32(c.smem + c.L.xs), c.L.h_pitch, bidx, s * kSdSeg, lane, acc);
          C.release();
        }
        if (!ok) break;                        // abort: fall through to the barrier below
        const int row = lane >> 2;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int col = (lane & 3) * 2 + q;
          if (col < cnt) {
            const int t = sh ? col : c.rt.slot_tok[off + col];
            const float gsc = sh ? 1.f : c.rt.slot_gate[off + col];
            yw[(w * 16 + row) * kSdMaxT + t] += gsc * acc[q];
            yw[(w * 16 + row + 8) * kSdMaxT + t] += gsc * acc[2 + q];
          }
        }
      }
      if (named_sync_or(1, NT, *c.abort_flag != 0)) return;
      for (int i = tid; i < 16 * T; i += NT) {
        const int row = i / T, t = i % T, r = rb * 16 + row;
        float y = 0.f;
        for (int ww = 0; ww < kSdConsumers; ++ww) y += yw[(ww * 16 + row) * kSdMaxT + t];
        if (a.add_residual)
          y += __bfloat162float(
              __ushort_as_bfloat16(__ldcg(reinterpret_cast<const unsigned short*>(xcur) + (size_t)t * d + r)));
        const unsigned short ob = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        __stcg(reinterpret_cast<unsigned short*>(xnext) + (size_t)t * d + r, ob);
        if (a.x_trace)
          __stcg(reinterpret_cast<unsigned short*>(a.x_trace) + ((size_t)(l + 1) * T + t) * d + r, ob);
      }
      named_sync(1, NT);
    }
    if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, 32 * kSdConsumers, 32)) return;
  }
}

__global__ void __launch_bounds__(kSdThreads, 1) stack_decode_kernel(const __grid_constant__ StackArgs a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);   // the swizzle wants 1024-byte stages
  const int Fmax = a.F > a.Fs ? a.F : a.Fs;
  SdCtx c{a};
  c.L = sd_layout(a.d, Fmax, a.k);
  c.smem = dsm;
  c.full = reinterpret_cast<uint64_t*>(dsm + c.L.bars);
  c.empty = c.full + kSdStages;
  c.route_bar = reinterpret_cast<uint64_t*>(dsm + c.L.route_bar);
  c.abort_flag = reinterpret_cast<volatile int*>(dsm + c.L.abort);
  c.rt = rt_of(dsm + c.L.rt);
  c.prod_m = reinterpret_cast<int*>(dsm + c.L.rt + 3840);
  c.prod_par = reinterpret_cast<uint32_t*>(dsm + c.L.rt + 3840 + 4 * kSdConsumers);
  c.G = gridDim.x;
  c.b = blockIdx.x;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSdStages; ++i) {
      mbar_init(&c.full[i], 1);
      mbar_init(&c.empty[i], 1);
    }
    mbar_init(c.route_bar, 1);
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  c.wc = WaitCtl{a.wait_ns, a.err, c.abort_flag};
  if (c.warp == 0) {
    if (c.lane == 0) run_producer(c);      // one thread issues every copy
  } else {
    run_consumers(c);
  }
}

}  // namespace

size_t stack_decode_smem_bytes(int d, int F, int Fs, int k) {
  return sd_layout(d, F > Fs ? F : Fs, k).total;
}

cudaError_t launch_stack_decode(const StackArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = stack_decode_smem_bytes(a.d, a.F, a.Fs, a.k);
  cudaError_t e = ensure_smem_limit(stack_decode_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kSdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stack_decode_kernel, a);
}

}  // namespace moe
