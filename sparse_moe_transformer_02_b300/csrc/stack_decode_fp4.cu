// Persistent decode kernel for MoE layers with NVFP4 expert weights: one
// cooperative launch (one CTA per SM) runs routing, gate/up and down for a
// batch of up to 32 tokens, for one layer or a stack of them.
//
// NVFP4 (evermx.com review, section "Quantization") stores each expert weight
// as an e2m1 code with an e4m3 scale per 16 values along the reduction and one
// fp32 scale per matrix.  At decode sizes a layer is a weight stream: a routed
// expert sees one or two of the batch's tokens, so the weights are decoded
// exactly into f16 in registers (cvt e2m1x2 -> f16x2, times the block scale
// as f16x2: code x scale has at most 5 significant bits and lies in
// [2^-10, 2688]) and multiplied on the tensor pipe with mma.sync m16n8k16
// (f16 in, fp32 accumulate) against the activations.  A tcgen05 MMA would
// cover only 128 x 16 decoded weights per instruction at these token counts,
// which caps it well below the HBM rate.
//
// Activations: every token's x is scaled by a power of two 2^-e (largest
// |x| into [1, 2)) and kept as f16 (exact for every value above 2^-17 of the
// row maximum; xs = 2^e is applied to the fp32 result).  h is stored in f16
// as h / xs^2 (exact rescaling; a value beyond the f16 range saturates and
// sets the range bit of the error word).
//
// Per layer four phases, separated by grid barriers:
//   A  router logits (fp32; each expert row split into 4 parts over the
//      grid's warps; a CTA's eight warps share the part, whose slice of x is
//      staged in the stage ring, idle until the routing is known; partial
//      sums added in a fixed order by the top-k) and the f16 copy of x;
//   B  top-k and gates (up to 8 tokens: every CTA for itself, one warp per
//      token; more: one warp per token across the grid, published to global
//      memory, one more barrier), grouping and work entries computed by every
//      CTA for itself (identical inputs and instructions, so every CTA holds
//      the same routing); then the gate/up units: 32 gate + 32 up rows of one
//      entry's expert over the whole reduction, split evenly over the CTAs,
//      one unit per consumer warp at a time; SwiGLU in registers; h to global.
//      An entry is up to 16 token-slots of one expert (the shared expert's
//      rows and any crowded expert split into several), so every unit costs
//      the same: one pass over its weights with two 8-column MMA tiles;
//   C  down units: 64 output rows of one entry's expert over its F values;
//      the gate-weighted result per token-slot to global (fp32);
//   D  y = sum over the token's slots in selection order + the shared
//      expert's row (+ x), rounded to bf16: a fixed order, so the result is
//      bitwise repeatable.
// One producer thread per CTA streams the weights with TMA tile loads (64 rows
// x 256 values per stage: 8 KB of codes with the 128-byte swizzle + 1 KB of
// block scales) into a ring of two stages per consumer warp, running ahead
// into the down phase's weights while the gate/up phase finishes.  The
// activations (x, h) are read by the consumer lanes from global memory; a
// CTA's units belong to one or two experts, so their rows stay in L1.
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

constexpr int kC = kS4Consumers;
constexpr int kThreads = 32 * (1 + kC);
constexpr int kNT = 32 * kC;                          // consumer threads
constexpr int kPer = 2;                               // stages per consumer
constexpr int kStages = kC * kPer;
constexpr int kRows = 64;                             // weight rows per stage (four 16-row MMA tiles)
constexpr int kKs = 256;                              // values per stage
constexpr int kCodeBytes = kRows * kKs / 2;           // 8192
constexpr int kStageBytes = kCodeBytes + kRows * kKs / 16;   // + 1024 scale bytes = 9216
constexpr int kRpart = 512;                           // values per router part
constexpr int kNt = 2;                                // 8-column MMA tiles per unit (16 token-slots)
constexpr int kShCols = 8;                            // token-slots per work entry of the shared expert
static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment the swizzle needs");
static_assert(kNT == 256, "the grouping gives one consumer thread to each of up to 256 experts");
static_assert(kS4MaxT * (kRpart * 4 + 16) <= kStages * kStageBytes, "a router part of x fits in the stage ring");

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Shared-memory layout (byte offsets from the 1024-aligned base).  During the
// router phase the stage ring is idle (the producer waits for the routing),
// so it holds the CTA's slice of x.
constexpr uint32_t kRingBytes = kStages * kStageBytes;
constexpr uint32_t kRtBytes = 24 * 1024;
struct Layout {
  uint32_t stages, bars, route_bar, abort, rt, total;
};
__host__ __device__ constexpr Layout layout() {
  return Layout{0, kRingBytes, kRingBytes + 2 * kStages * 8, kRingBytes + 2 * kStages * 8 + 8,
                kRingBytes + 2 * kStages * 8 + 16, kRingBytes + 2 * kStages * 8 + 16 + kRtBytes + 1024};
}
constexpr int kMaxEnt = 320;   // work entries: up to 4 of the shared expert + U + T k / 16 routed
// Routing tables (ints / floats) inside Layout::rt.
struct Rt {
  int* sel_e;       // [256] selection of slot s = t k + j
  float* sel_g;     // [256] its gate
  int* pos_of;      // [256] grouped position of slot s
  int* slot_tok;    // [256] token of each grouped position
  float* slot_gate; // [256] gate of each grouped position
  int* act_e;       // [260] active experts, ascending
  int* act_off;     // [260] first grouped position of each (act_off[n_act] = T k)
  int* n_act;       // [4]
  int* cntw;        // [8][256] per-warp expert counts, then their prefix over warps
  int* off;         // [256] first grouped position of each expert
  int* wsum;        // [16] per-warp scan totals
  int* ent_e;       // [kMaxEnt] expert of each work entry (-1: the shared expert)
  int* ent_off;     // [kMaxEnt] its first grouped position (shared rows follow the T k routed slots)
  int* ent_cnt;     // [kMaxEnt] its token-slots (<= 16)
  int* n_ent;       // [4] [0] entries, [1] of the shared expert
  int* prod_m;      // [kC] producer: stages taken per consumer
  uint32_t* prod_par;   // [kStages] producer: parity last used per stage
};
__device__ __forceinline__ Rt rt_of(uint8_t* base) {
  int* p = reinterpret_cast<int*>(base);
  Rt r;
  r.sel_e = p; p += 256;
  r.sel_g = reinterpret_cast<float*>(p); p += 256;
  r.pos_of = p; p += 256;
  r.slot_tok = p; p += 256;
  r.slot_gate = reinterpret_cast<float*>(p); p += 256;
  r.act_e = p; p += 260;
  r.act_off = p; p += 260;
  r.n_act = p; p += 4;
  r.cntw = p; p += 8 * 256;
  r.off = p; p += 256;
  r.wsum = p; p += 16;
  r.ent_e = p; p += kMaxEnt;
  r.ent_off = p; p += kMaxEnt;
  r.ent_cnt = p; p += kMaxEnt;
  r.n_ent = p; p += 4;
  r.prod_m = p; p += kC;
  r.prod_par = reinterpret_cast<uint32_t*>(p); p += kStages;
  return r;   // 5468 ints = 21,872 bytes < kRtBytes
}

struct Ctx {
  const Stack4Args& a;
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* route_bar;
  volatile int* abort_flag;
  Rt rt;
  WaitCtl wc;
  int G, b, warp, lane;
};

// Even split of n units over the G CTAs: [lo, hi) for CTA b.
__device__ __forceinline__ void share(int n, int G, int b, int& lo, int& hi) {
  lo = (int)(((long long)n * b) / G);
  hi = (int)(((long long)n * (b + 1)) / G);
}

// ---------------------------------------------------------------- producer
struct Producer {
  Ctx& c;
  uint64_t pol;
  uint32_t used = 0;
  __device__ __forceinline__ explicit Producer(Ctx& ctx) : c(ctx) {
    for (int i = 0; i < kC; ++i) c.rt.prod_m[i] = 0;
    pol = policy_evict_first();
  }
  __device__ __forceinline__ int next(int w) {
    const int m = c.rt.prod_m[w]++;
    const int s = w * kPer + (m & 1);
    if (!mbar_wait(&c.empty[s], ((m >> 1) & 1) ^ 1, c.wc)) return -1;
    c.rt.prod_par[s] = (m >> 1) & 1;
    used |= 1u << s;
    return s;
  }
  // Gate/up stage: gate rows [row0, row0 + 32) and up rows [row0, row0 + 32),
  // values [256 s, 256 s + 256).
  __device__ __forceinline__ bool issue_gu(int w, const CUtensorMap* M, bool sh, int row0, int s) {
    const int st = next(w);
    if (st < 0) return false;
    uint8_t* dst = c.smem + st * kStageBytes;
    const CUtensorMap* mg = M + (sh ? 6 : 0);
    const CUtensorMap* mu = M + (sh ? 8 : 2);
    mbar_arrive_expect_tx(&c.full[st], kStageBytes);
    tma_load_2d_hint(dst, mg, s * (kKs / 2), row0, &c.full[st], pol);
    tma_load_2d_hint(dst + kCodeBytes / 2, mu, s * (kKs / 2), row0, &c.full[st], pol);
    tma_load_2d_hint(dst + kCodeBytes, mg + 1, s * (kKs / 16), row0, &c.full[st], pol);
    tma_load_2d_hint(dst + kCodeBytes + 512, mu + 1, s * (kKs / 16), row0, &c.full[st], pol);
    return true;
  }
  // Down stage: rows [row0, row0 + 64), values [256 s, 256 s + 256).
  __device__ __forceinline__ bool issue_dn(int w, const CUtensorMap* M, bool sh, int row0, int s) {
    const int st = next(w);
    if (st < 0) return false;
    uint8_t* dst = c.smem + st * kStageBytes;
    const CUtensorMap* md = M + (sh ? 10 : 4);
    mbar_arrive_expect_tx(&c.full[st], kStageBytes);
    tma_load_2d_hint(dst, md, s * (kKs / 2), row0, &c.full[st], pol);
    tma_load_2d_hint(dst + kCodeBytes, md + 1, s * (kKs / 16), row0, &c.full[st], pol);
    return true;
  }
  __device__ __forceinline__ void drain() {
    for (int s = 0; s < kStages; ++s)
      if (used & (1u << s)) drain_wait(&c.full[s], c.rt.prod_par[s], c.wc.limit_ns);
  }
};

// Work units.  Gate/up: 32 gate + 32 up rows (group) of one entry's expert;
// the shared expert's entries first.  Down: 64 output rows (block) of one
// entry's expert.  Every unit covers the entry's token-slots (<= 16) in one
// pass over its weights.
struct GuUnit { int ent, grp; };
__device__ __forceinline__ GuUnit gu_unit(const Rt& rt, int u, int gps, int gpe) {
  const int nse = rt.n_ent[1];
  if (u < nse * gps) return GuUnit{u / gps, u % gps};
  const int v = u - nse * gps;
  return GuUnit{nse + v / gpe, v % gpe};
}
__device__ __forceinline__ int gu_units(const Rt& rt, int gps, int gpe) {
  return rt.n_ent[1] * gps + (rt.n_ent[0] - rt.n_ent[1]) * gpe;
}

__device__ __forceinline__ void run_producer(Ctx& c) {
  const Stack4Args& a = c.a;
  Producer P(c);
  const int d = a.d, F = a.F, Fs = a.Fs;
  const int gpe = F / 32, gps = Fs / 32, rbn = d / kRows;
  bool ok = true;
  for (int l = 0; l < a.L && ok; ++l) {
    const CUtensorMap* M = a.maps + (size_t)l * kS4Maps;
    for (int i = 0; i < kS4Maps; ++i) tma_prefetch_desc(M + i);
    if (!mbar_wait(c.route_bar, l & 1, c.wc)) { ok = false; break; }
    // gate/up units of this CTA: rounds of up to kC units, one per consumer,
    // issued stage by stage across the consumers
    {
      int lo, hi;
      share(gu_units(c.rt, gps, gpe), c.G, c.b, lo, hi);
      const int KS = d / kKs;
      for (int r0 = lo; r0 < hi && ok; r0 += kC) {
        const int nb = hi - r0 < kC ? hi - r0 : kC;
        int row0[kC];                  // negative: the shared expert's row -row0 - 1
#pragma unroll
        for (int w = 0; w < kC; ++w)
          if (w < nb) {
            const GuUnit gu = gu_unit(c.rt, r0 + w, gps, gpe);
            const int e = c.rt.ent_e[gu.ent];
            row0[w] = e < 0 ? -(gu.grp * 32) - 1 : e * F + gu.grp * 32;
          }
        for (int s = 0; s < KS && ok; ++s)
#pragma unroll
          for (int w = 0; w < kC; ++w)
            if (w < nb && ok) ok = P.issue_gu(w, M, row0[w] < 0, row0[w] < 0 ? -row0[w] - 1 : row0[w], s);
      }
    }
    // down units
    {
      int lo, hi;
      share(c.rt.n_ent[0] * rbn, c.G, c.b, lo, hi);
      const int KSmax = (F > Fs ? F : Fs) / kKs;
      for (int r0 = lo; r0 < hi && ok; r0 += kC) {
        const int nb = hi - r0 < kC ? hi - r0 : kC;
        int row0[kC], nks[kC];         // row0 negative: the shared expert's row -row0 - 1
#pragma unroll
        for (int w = 0; w < kC; ++w)
          if (w < nb) {
            const int u = r0 + w, e = c.rt.ent_e[u / rbn], rb = u % rbn;
            row0[w] = e < 0 ? -(rb * kRows) - 1 : e * d + rb * kRows;
            nks[w] = (e < 0 ? Fs : F) / kKs;
          }
        for (int s = 0; s < KSmax && ok; ++s)
#pragma unroll
          for (int w = 0; w < kC; ++w)
            if (w < nb && ok && s < nks[w])
              ok = P.issue_dn(w, M, row0[w] < 0, row0[w] < 0 ? -row0[w] - 1 : row0[w], s);
      }
    }
  }
  if (!ok) P.drain();
}

// ---------------------------------------------------------------- consumers
struct Cons {
  Ctx& c;
  int m = 0;
  int cur = 0;
  __device__ __forceinline__ explicit Cons(Ctx& ctx) : c(ctx) {}
  __device__ __forceinline__ uint32_t wait() {
    const int st = (c.warp - 1) * kPer + (m & 1);
    int ok = 1;
    if (c.lane == 0) ok = mbar_wait(&c.full[st], (m >> 1) & 1, c.wc) ? 1 : 0;
    ok = __shfl_sync(kFull, ok, 0);
    if (!ok) return 0;
    while (!mbar_try_wait(&c.full[st], (m >> 1) & 1)) {
    }
    cur = st;
    return smem_u32(c.smem + st * kStageBytes);
  }
  __device__ __forceinline__ void release() {
    __syncwarp();
    if (c.lane == 0) mbar_arrive(&c.empty[cur]);
    ++m;
  }
};

// acc[j][n] += stage rows (tile j = rows 16 j .. 16 j + 15) x B (n-tile n,
// column g = lane / 4: the 16-bit row brow[n] of global memory, values
// k0 .. k0 + 255).  In half h of the stage, lane (g, t) takes the 32-value
// chunk c = 2 t + h: one 16-byte load per row (rows g and g + 8 of each
// tile) brings its 32 codes, one 2-byte load their two block scales, four
// 16-byte loads the same 32 values of its B row.  Each 8-code word feeds two
// MMAs; the reduction order is permuted alike in A and B, so the sum is
// unchanged.  Codes: row r is a 128-byte line whose 16-byte chunk c sits at
// c ^ (r & 7); with c = 2 t + h the eight lanes of each quarter-warp (rows g
// and g + 1) read eight distinct chunk positions, so the loads are
// conflict-free.
__device__ __forceinline__ void mma_stage(uint32_t st, const uint8_t* const (&brow)[kNt], int ntl, int k0, int lane,
                                          float (&acc)[4][kNt][4]) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t rowb = st + g * 128, scb = st + kCodeBytes + g * 16;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int cch = 2 * t + h;
    const uint32_t coff = (uint32_t)((cch ^ g) << 4);
    uint4 cw[8];                        // row 16 j + g (2 j) and 16 j + g + 8 (2 j + 1)
    uint32_t sp[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t ra = rowb + (r >> 1) * 2048 + (r & 1) * 1024 + coff;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(cw[r].x), "=r"(cw[r].y), "=r"(cw[r].z), "=r"(cw[r].w)
                   : "r"(ra));
      asm volatile("ld.shared.u16 %0, [%1];" : "=r"(sp[r]) : "r"(scb + (r >> 1) * 256 + (r & 1) * 128 + 2 * cch));
    }
    const size_t boff = (size_t)(k0 + 32 * cch) * 2;
    uint32_t slo[8], shi[8];            // the two block scales of the chunk, each as {s, s}
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      uint32_t pr;
      asm("{\n\t.reg .b16 u;\n\tcvt.u16.u32 u, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, u;\n\t}" : "=r"(pr) : "r"(sp[r]));
      slo[r] = dup_lo(pr);
      shi[r] = dup_hi(pr);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 xv[kNt];
#pragma unroll
      for (int n = 0; n < kNt; ++n)
        if (n < ntl) xv[n] = *reinterpret_cast<const uint4*>(brow[n] + boff + i * 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4& c0 = cw[2 * j];
        const uint4& c8 = cw[2 * j + 1];
        const uint32_t w0 = i == 0 ? c0.x : i == 1 ? c0.y : i == 2 ? c0.z : c0.w;
        const uint32_t w8 = i == 0 ? c8.x : i == 1 ? c8.y : i == 2 ? c8.z : c8.w;
        uint32_t d0[4], d8[4];
        e2m1x8_f16x2(w0, d0);
        e2m1x8_f16x2(w8, d8);
        const uint32_t s0 = i < 2 ? slo[2 * j] : shi[2 * j], s8 = i < 2 ? slo[2 * j + 1] : shi[2 * j + 1];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          d0[v] = hmul2(d0[v], s0);
          d8[v] = hmul2(d8[v], s8);
        }
#pragma unroll
        for (int n = 0; n < kNt; ++n)
          if (n < ntl) {
            mma_f16(acc[j][n], d0[0], d8[0], d0[1], d8[1], xv[n].x, xv[n].y);
            mma_f16(acc[j][n], d0[2], d8[2], d0[3], d8[3], xv[n].z, xv[n].w);
          }
      }
    }
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[4][kNt][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int n = 0; n < kNt; ++n) acc[j][n][0] = acc[j][n][1] = acc[j][n][2] = acc[j][n][3] = 0.f;
}

// Grouping of the T k slots by expert over the CTA's 256 consumer threads
// (warp w takes slots 32 w .. 32 w + 31): active experts ascending, the
// slots of one expert in (token, j) order.  slot_of (global, may be null)
// receives each slot's grouped position.
__device__ __forceinline__ void group_slots(Rt& rt, int T, int k, int E, int w, int lane, int tid, int32_t* slot_of) {
  const int ns = T * k;
  int* cw = rt.cntw + w * 256;
  for (int e = lane; e < 256; e += 32) cw[e] = 0;
  __syncwarp();
  const int s = w * 32 + lane;
  const bool v = s < ns;
  const int e = v ? rt.sel_e[s] : -1 - lane;
  const unsigned m = __match_any_sync(kFull, e);
  const int r = __popc(m & ((1u << lane) - 1u));
  if (v && r == 0) cw[e] = __popc(m);
  named_sync(1, kNT);
  // thread tid = expert: prefix of its counts over the warps, its total
  int cnt = 0;
  {
    const int ex = tid;
#pragma unroll
    for (int ww = 0; ww < kC; ++ww) {
      const int c = rt.cntw[ww * 256 + ex];
      rt.cntw[ww * 256 + ex] = cnt;
      cnt += c;
    }
    if (ex >= E) cnt = 0;
  }
  // exclusive scans over the experts of the counts and of the active flags
  int it = cnt, ia = cnt > 0 ? 1 : 0;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, it, o), y = __shfl_up_sync(kFull, ia, o);
    if (lane >= o) { it += x; ia += y; }
  }
  if (lane == 31) { rt.wsum[w] = it; rt.wsum[8 + w] = ia; }
  named_sync(1, kNT);
  int bo = 0, ba = 0;
  for (int ww = 0; ww < w; ++ww) { bo += rt.wsum[ww]; ba += rt.wsum[8 + ww]; }
  const int off = bo + it - cnt, rank = ba + ia - (cnt > 0 ? 1 : 0);
  if (tid < E) {
    rt.off[tid] = off;
    if (cnt > 0) {
      rt.act_e[rank] = tid;
      rt.act_off[rank] = off;
    }
  }
  if (tid == kNT - 1) {
    const int U = ba + ia;
    rt.act_off[U] = ns;
    *rt.n_act = U;
  }
  named_sync(1, kNT);
  if (v) {
    const int p = rt.off[e] + cw[e] + r;
    rt.slot_tok[p] = s / k;
    rt.slot_gate[p] = rt.sel_g[s];
    rt.pos_of[s] = p;
    if (slot_of) slot_of[s] = p;
  }
  named_sync(1, kNT);
}

// Work entries: the shared expert's rows in chunks of 8 tokens (one MMA
// column tile, so a unit's activation rows stay within L1), then every active
// expert's token-slots in chunks of 16 (almost always one chunk).
// One thread per active expert; block scan of the chunk counts.
__device__ __forceinline__ void build_entries(Rt& rt, int T, int k, int has_sh, int w, int lane, int tid) {
  const int U = *rt.n_act;
  const int nse = has_sh ? (T + kShCols - 1) / kShCols : 0;
  int cnt = 0, nch = 0;
  if (tid < U) {
    cnt = rt.act_off[tid + 1] - rt.act_off[tid];
    nch = (cnt + 15) >> 4;
  }
  int it = nch;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(kFull, it, o);
    if (lane >= o) it += x;
  }
  if (lane == 31) rt.wsum[w] = it;
  named_sync(1, kNT);
  int base = 0;
  for (int ww = 0; ww < w; ++ww) base += rt.wsum[ww];
  const int pre = base + it - nch;
  for (int i = 0; i < nch; ++i) {
    const int en = nse + pre + i;
    rt.ent_e[en] = rt.act_e[tid];
    rt.ent_off[en] = rt.act_off[tid] + 16 * i;
    rt.ent_cnt[en] = cnt - 16 * i < 16 ? cnt - 16 * i : 16;
  }
  if (tid < nse) {
    rt.ent_e[tid] = -1;
    rt.ent_off[tid] = T * k + kShCols * tid;
    rt.ent_cnt[tid] = T - kShCols * tid < kShCols ? T - kShCols * tid : kShCols;
  }
  if (tid == kNT - 1) {
    rt.n_ent[0] = nse + base + it;
    rt.n_ent[1] = nse;
  }
  named_sync(1, kNT);
}

__device__ __forceinline__ void run_consumers(Ctx& c) {
  const Stack4Args& a = c.a;
  Cons C(c);
  const int w = c.warp - 1, lane = c.lane, tid = threadIdx.x - 32;
  const int T = a.T, d = a.d, F = a.F, Fs = a.Fs, E = a.E, k = a.k;
  const int Fmax = F > Fs ? F : Fs;
  const int has_sh = Fs > 0 ? 1 : 0;
  const int gpe = F / 32, gps = Fs / 32, rbn = d / kRows;
  const int g = lane >> 2, tq = lane & 3;
  unsigned nbar = 0;
  for (int l = 0; l < a.L; ++l) {
    const Stack4LayerPtrs& W = a.layers[l];
    const __nv_bfloat16* xcur = l == 0 ? a.x_in : a.xbuf + (size_t)((l - 1) & 1) * kS4MaxT * d;
    __nv_bfloat16* xnext = l == a.L - 1 ? a.y_out : a.xbuf + (size_t)(l & 1) * kS4MaxT * d;
    const unsigned short* xb = reinterpret_cast<const unsigned short*>(xcur);

    // ---- phase A: router parts of 512 values.  Task tk: expert
    // ((tk / 8) / nq) 8 + tk % 8, part (tk / 8) % nq, so a CTA's eight warps
    // share the part, whose slice of x (all tokens, as fp32) is staged in the
    // idle stage ring.  A lane holds its 16 router values in registers, loaded
    // before the slice is staged.
    const int gw = c.b * kC + w, nw = c.G * kC, nq = (d + kRpart - 1) / kRpart;
    const int ntasks = ((E + 7) / 8) * 8 * nq;
    for (int tk0 = c.b * kC; tk0 < ntasks; tk0 += nw) {
      const int q = (tk0 >> 3) % nq, q0 = q * kRpart, dq = d - q0 < kRpart ? d - q0 : kRpart;
      const int tk = tk0 + w, e = ((tk >> 3) / nq) * 8 + (tk & 7);
      const bool mine = tk < ntasks && e < E;
      float4 wv[kRpart / 128];
#pragma unroll
      for (int u = 0; u < kRpart / 128; ++u) {
        const int i = lane * 4 + u * 128;
        wv[u] = (mine && i < dq) ? __ldg(reinterpret_cast<const float4*>(W.wr + (size_t)e * d + q0 + i))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const uint32_t pitch = (uint32_t)dq * 4 + 16;
      {
        const int per = dq / 8, n = T * per;
        for (int i0 = tid; i0 < n; i0 += 4 * kNT) {
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kNT;
            if (i < n) v[u] = __ldcg(reinterpret_cast<const uint4*>(xb + (size_t)(i / per) * d + q0) + i % per);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * kNT;
            if (i < n) {
              float4* dst = reinterpret_cast<float4*>(c.smem + (i / per) * pitch + (i % per) * 32);
              dst[0] = make_float4(__uint_as_float(v[u].x << 16), __uint_as_float(v[u].x & 0xFFFF0000u),
                                   __uint_as_float(v[u].y << 16), __uint_as_float(v[u].y & 0xFFFF0000u));
              dst[1] = make_float4(__uint_as_float(v[u].z << 16), __uint_as_float(v[u].z & 0xFFFF0000u),
                                   __uint_as_float(v[u].w << 16), __uint_as_float(v[u].w & 0xFFFF0000u));
            }
          }
        }
      }
      named_sync(1, kNT);
      if (mine) {
        const uint32_t xs0 = smem_u32(c.smem);
        const float bias = (q == 0 && W.br) ? __ldg(W.br + e) : 0.f;   // part 0 carries the bias
        constexpr int kTp = 16;        // tokens per accumulation pass (registers)
#pragma unroll
        for (int tp = 0; tp < kS4MaxT; tp += kTp) {
          if (tp >= T) break;
          float acc[kTp];
#pragma unroll
          for (int tt = 0; tt < kTp; ++tt) acc[tt] = 0.f;
#pragma unroll
          for (int u = 0; u < kRpart / 128; ++u) {
            const int i = lane * 4 + u * 128;
            if (i >= dq) break;
#pragma unroll
            for (int tt = 0; tt < kTp; ++tt)
              if (tp + tt < T) {
                float4 xv;
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(xv.x), "=f"(xv.y), "=f"(xv.z), "=f"(xv.w)
                             : "r"(xs0 + (uint32_t)(tp + tt) * pitch + (uint32_t)i * 4));
                acc[tt] = fmaf(wv[u].x, xv.x, fmaf(wv[u].y, xv.y, fmaf(wv[u].z, xv.z, fmaf(wv[u].w, xv.w, acc[tt]))));
              }
          }
          // butterfly transpose-reduction: lanes 2 i and 2 i + 1 end with token tp + i's sum
          const float v = transpose_reduce<kTp, 32>(acc, lane);
          const int tt = lane >> 1;
          if ((lane & 1) == 0 && tp + tt < T) __stcg(a.logits + ((size_t)q * kS4MaxT + tp + tt) * E + e, v + bias);
        }
      }
      named_sync(1, kNT);   // the slice is restaged by the next round
    }
    // f16 copy of x with a power-of-two scale per token (warps left without a router task)
    {
      const int spare = nw > ntasks ? nw - ntasks : nw;
      const int cw = nw > ntasks ? gw - ntasks : gw;
      for (int t = cw; cw >= 0 && t < T; t += spare) {
        const uint4* src = reinterpret_cast<const uint4*>(xb + (size_t)t * d);
        float amax = 0.f;
        for (int i = lane; i < d / 8; i += 32) {
          const uint4 v = __ldcg(src + i);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[h2] << 16)), fabsf(__uint_as_float(u[h2] & 0xFFFF0000u))));
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        int ex = amax > 0.f ? ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127) : 0;
        ex = ex < -126 ? -126 : (ex > 127 ? 127 : ex);
        const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);   // 2^-ex
        if (lane == 0) __stcg(a.xsc + t, __uint_as_float((uint32_t)(127 + ex) << 23));
        for (int i = lane; i < d / 8; i += 32) {
          const uint4 v = __ldcg(src + i);
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
          uint32_t o4[4];
#pragma unroll
          for (int h2 = 0; h2 < 4; ++h2) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(u[h2] << 16) * inv,
                                                 __uint_as_float(u[h2] & 0xFFFF0000u) * inv);
            o4[h2] = *reinterpret_cast<const uint32_t*>(&hh);
          }
          __stcg(reinterpret_cast<uint4*>(a.xh + (size_t)t * d) + i, make_uint4(o4[0], o4[1], o4[2], o4[3]));
        }
      }
    }
    if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, kNT, 32)) return;

    // ---- phase B: top-k (above 8 tokens one warp per token across the grid,
    // published, another barrier; else every CTA for itself), grouping, work
    // entries, hand-off to the producer, gate/up units
    if (T > kC) {
      const int t = c.b * kC + w;
      if (t < T) {
        topk_token(a.logits, nq, kS4MaxT, E, k, t, c.rt.sel_e, c.rt.sel_g, lane);
        __syncwarp();
        if (lane < k) {
          __stcg(a.topk_e + t * k + lane, c.rt.sel_e[t * k + lane]);
          __stcg(a.topk_g + t * k + lane, c.rt.sel_g[t * k + lane]);
        }
      }
      if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, kNT, 32)) return;
      for (int i = tid; i < T * k; i += kNT) {
        c.rt.sel_e[i] = __ldcg(a.topk_e + i);
        c.rt.sel_g[i] = __ldcg(a.topk_g + i);
      }
    } else {
      for (int t = w; t < T; t += kC) topk_token(a.logits, nq, kS4MaxT, E, k, t, c.rt.sel_e, c.rt.sel_g, lane);
    }
    named_sync(1, kNT);
    group_slots(c.rt, T, k, E, w, lane, tid, (c.b == 0 && l == 0) ? a.g_slot_of : nullptr);
    build_entries(c.rt, T, k, has_sh, w, lane, tid);
    if (tid == 0) mbar_arrive(c.route_bar);
    if (c.b == 0) {
      for (int i = tid; i < T * k; i += kNT) {
        if (a.idx_trace) a.idx_trace[(size_t)l * T * k + i] = c.rt.sel_e[i];
        if (a.gate_trace) a.gate_trace[(size_t)l * T * k + i] = c.rt.sel_g[i];
      }
      if (l == 0 && a.g_offsets) {
        for (int i = tid; i <= E; i += kNT) a.g_offsets[i] = i < E ? c.rt.off[i] : T * k;
        for (int i = tid; i < T * k; i += kNT) a.g_tok_of_slot[i] = c.rt.slot_tok[i];
      }
    }
    // ---- phases B (gate/up units) and C (down units): one loop, one copy of
    // the stage arithmetic; a grid barrier after each
    bool ok = true;
#pragma unroll 1
    for (int ph = 0; ph < 2; ++ph) {
      int lo, hi;
      share(ph == 0 ? gu_units(c.rt, gps, gpe) : c.rt.n_ent[0] * rbn, c.G, c.b, lo, hi);
      for (int u = lo + w; u < hi && ok; u += kC) {
        int ent, sub;                  // entry, and its row group (gate/up) or row block (down)
        if (ph == 0) {
          const GuUnit gu = gu_unit(c.rt, u, gps, gpe);
          ent = gu.ent;
          sub = gu.grp;
        } else {
          ent = u / rbn;
          sub = u % rbn;
        }
        const int e = c.rt.ent_e[ent], off = c.rt.ent_off[ent], cnt = c.rt.ent_cnt[ent];
        const bool sh = e < 0;
        const int ntl = (cnt + 7) >> 3;
        const uint8_t* brow[kNt];
#pragma unroll
        for (int n = 0; n < kNt; ++n) {
          const int col = n * 8 + g, cc = col < cnt ? col : 0;
          if (ph == 0) {
            const int tok = sh ? off - T * k + cc : c.rt.slot_tok[off + cc];
            brow[n] = reinterpret_cast<const uint8_t*>(a.xh + (size_t)tok * d);
          } else {
            brow[n] = reinterpret_cast<const uint8_t*>(a.h + (size_t)(off + cc) * Fmax);
          }
        }
        float acc[4][kNt][4];
        zero_acc(acc);
        const int KS = ph == 0 ? d / kKs : (sh ? Fs : F) / kKs;
        for (int s = 0; s < KS; ++s) {
          const uint32_t st = C.wait();
          if (!st) { ok = false; break; }
          mma_stage(st, brow, ntl, s * kKs, lane, acc);
          C.release();
        }
        if (!ok) break;
        asm volatile("" ::: "memory");   // keep the epilogue's loads after the loop (registers)
        if (ph == 0) {
            const float tsg = __ldg(sh ? W.tsg : W.tg + e), tsu = __ldg(sh ? W.tsu : W.tu + e);
            // h / xs^2 = silu(a) (u / xs^2) for every held (row, column), then the stores
    #pragma unroll
            for (int n = 0; n < kNt; ++n) {
              if (n >= ntl) continue;
    #pragma unroll
              for (int cix = 0; cix < 4; ++cix) {
                const int col = n * 8 + tq * 2 + (cix & 1), cc = col < cnt ? col : 0;
                const int tok = sh ? off - T * k + cc : c.rt.slot_tok[off + cc];
                const float xs = __ldcg(a.xsc + tok);
                const float ga = tsg * xs, ua = tsu / xs;
    #pragma unroll
                for (int jt = 0; jt < 2; ++jt) {
                  const float av = acc[jt][n][cix] * ga;
                  acc[jt][n][cix] = silu_f(av) * (acc[jt + 2][n][cix] * ua);
                }
              }
            }
            bool sat = false;
    #pragma unroll
            for (int n = 0; n < kNt; ++n) {
              if (n >= ntl) continue;
    #pragma unroll
              for (int cix = 0; cix < 4; ++cix) {
                const int col = n * 8 + tq * 2 + (cix & 1);
                if (col >= cnt) continue;
                __half* hr = a.h + (size_t)(off + col) * Fmax + sub * 32 + g + (cix >= 2 ? 8 : 0);
    #pragma unroll
                for (int jt = 0; jt < 2; ++jt) {
                  float hv = acc[jt][n][cix];
                  if (fabsf(hv) > 65504.f) {
                    sat = true;
                    hv = copysignf(65504.f, hv);
                  }
                  hr[jt * 16] = __float2half_rn(hv);
                }
              }
            }
            if (sat) atomicOr(a.err, kErrRange);
        } else {
          const int rb = sub;
            const float tsd = __ldg(sh ? W.tsd : W.td + e);
    #pragma unroll
            for (int n = 0; n < kNt; ++n) {
              if (n >= ntl) continue;
    #pragma unroll
              for (int cix = 0; cix < 4; ++cix) {
                const int col = n * 8 + tq * 2 + (cix & 1);
                if (col >= cnt) continue;
                const int tok = sh ? off - T * k + col : c.rt.slot_tok[off + col];
                const float xs = __ldcg(a.xsc + tok);
                const float sc = tsd * xs * xs * (sh ? 1.f : c.rt.slot_gate[off + col]);
                float* orow = a.o + (size_t)(off + col) * d + rb * kRows + g + (cix >= 2 ? 8 : 0);
    #pragma unroll
                for (int j = 0; j < 4; ++j) __stcg(orow + j * 16, acc[j][n][cix] * sc);
              }
            }
        }
      }
      if (!grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, kNT, 32)) return;
    }

    // ---- phase D: y = sum of the token's slots (selection order) + shared (+ x)
    {
      const int per = d / 4, n = T * per;
      for (int it = c.b * kNT + tid; it < n; it += c.G * kNT) {
        const int t = it / per, i = (it % per) * 4;
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o + (size_t)c.rt.pos_of[t * k + j] * d + i));
          y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
        }
        if (has_sh) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(a.o + (size_t)(T * k + t) * d + i));
          y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
        }
        if (a.add_residual) {
          const uint2 xv = __ldcg(reinterpret_cast<const uint2*>(xb + (size_t)t * d + i));
          y.x += __uint_as_float(xv.x << 16);
          y.y += __uint_as_float(xv.x & 0xFFFF0000u);
          y.z += __uint_as_float(xv.y << 16);
          y.w += __uint_as_float(xv.y & 0xFFFF0000u);
        }
        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(y.x, y.y), hi2 = __floats2bfloat162_rn(y.z, y.w);
        uint2 ov;
        ov.x = *reinterpret_cast<const uint32_t*>(&lo2);
        ov.y = *reinterpret_cast<const uint32_t*>(&hi2);
        __stcg(reinterpret_cast<uint2*>(xnext + (size_t)t * d + i), ov);
      }
    }
    if (l + 1 < a.L && !grid_sync(a.bar, (++nbar) * c.G, c.wc, c.abort_flag, kNT, 32)) return;
  }
}

__global__ void __launch_bounds__(kThreads, 1) stack_decode_fp4_kernel(const __grid_constant__ Stack4Args a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);   // the swizzle wants 1024-byte stages
  constexpr Layout L = layout();
  Ctx c{a};
  c.smem = dsm;
  c.full = reinterpret_cast<uint64_t*>(dsm + L.bars);
  c.empty = c.full + kStages;
  c.route_bar = reinterpret_cast<uint64_t*>(dsm + L.route_bar);
  c.abort_flag = reinterpret_cast<volatile int*>(dsm + L.abort);
  c.rt = rt_of(dsm + L.rt);
  c.G = gridDim.x;
  c.b = blockIdx.x;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
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

size_t stack_decode_fp4_smem_bytes() { return layout().total; }

bool stack_decode_fp4_supported(const moe_config& c, bool* query_ok) {
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
  return c.act_dtype == MOE_BF16 && c.weight_dtype == MOE_NVFP4 && c.num_experts <= 256 && c.top_k <= 8 &&
         c.d % 256 == 0 && c.ffn % 256 == 0 && c.shared_ffn % 256 == 0 && cc_major == 10 && coop &&
         stack_decode_fp4_smem_bytes() <= (size_t)smem_optin;
}

bool stack_layer_views_fp4(const moe_config& c, const moe_weights& w, CUtensorMap* m) {
  // codes [rows][K / 2] bytes, 128-byte boxes with the 128-byte swizzle;
  // block scales [rows][K / 16] bytes, 16-byte boxes
  auto codes = [](CUtensorMap* t, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    const uint64_t dims[2] = {K / 2, rows}, strides[1] = {K / 2};
    const uint32_t box[2] = {128, box_rows};
    return encode_tiled(t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  auto scales = [](CUtensorMap* t, const void* base, uint64_t rows, uint64_t K, uint32_t box_rows) {
    const uint64_t dims[2] = {K / 16, rows}, strides[1] = {K / 16};
    const uint32_t box[2] = {16, box_rows};
    return encode_tiled(t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  };
  const uint64_t E = c.num_experts, d = c.d, F = c.ffn, Fs = c.shared_ffn;
  bool ok = codes(m + 0, w.w_gate, E * F, d, 32) && scales(m + 1, w.s_gate, E * F, d, 32) &&
            codes(m + 2, w.w_up, E * F, d, 32) && scales(m + 3, w.s_up, E * F, d, 32) &&
            codes(m + 4, w.w_down, E * d, F, 64) && scales(m + 5, w.s_down, E * d, F, 64);
  if (ok && Fs > 0)
    ok = codes(m + 6, w.ws_gate, Fs, d, 32) && scales(m + 7, w.ss_gate, Fs, d, 32) &&
         codes(m + 8, w.ws_up, Fs, d, 32) && scales(m + 9, w.ss_up, Fs, d, 32) &&
         codes(m + 10, w.ws_down, d, Fs, 64) && scales(m + 11, w.ss_down, d, Fs, 64);
  return ok;
}

cudaError_t launch_stack_decode_fp4(const Stack4Args& a, int num_sms, cudaStream_t s) {
  const size_t smem = stack_decode_fp4_smem_bytes();
  cudaError_t e = ensure_smem_limit(stack_decode_fp4_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stack_decode_fp4_kernel, a);
}

}  // namespace moe
