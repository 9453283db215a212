// Sliding-window grouped-query attention for a decode step: B sequences, one
// new token each, in one cooperative launch.
//
// What it computes (swarmz.net, "Recursive Flint: 40B Open Model, 2.5B
// Active", section "The architecture, in plain terms"; futurpulse.com,
// section "How does Flint use 39.8B parameters efficiently?"): 35 of Flint's
// 49 layers attend over the current token and the 512 before it; 32 query
// heads share 4 key/value heads of dimension 128; queries and keys get a
// per-head RMSNorm; each head has a learned sink; these layers apply RoPE.
// Per sequence b at position p:
//   q = Wq x, k = Wk x, v = Wv x; q_h, k_g <- RMSNorm(.) * gamma, then RoPE(p)
//   cache[p % W] <- (bf16 k, bf16 v)
//   o_h = sum_j softmax_j(q_h . k_j / sqrt(128) ; sink_h) v_j over the window
//   y = Wo o (+ x)
// The sink is one more logit in each head's softmax denominator.
//
// Phases, separated by grid-wide barriers (bounded waits):
//   1  the q/k/v projections: rows of Wq, Wk, Wv in groups of 16, every K
//      segment of 256 values one 8 KB TMA box (3-D view {64 values, 16 rows,
//      4 chunks}, 128-byte swizzle) multiplied on the tensor pipe (mma.sync
//      m16n8k16, bf16, fp32 accumulate) against x staged in shared memory;
//      segments of a group spread over the eight consumer warps and summed in
//      warp order;
//   2  attention: work items (sequence, key/value head, window split); each
//      normalises and rotates its 8 query heads and the new key (RoPE angles
//      reduced in fp64 so large positions stay exact), the first split writes
//      the new key/value to the cache, every warp takes keys of the split and
//      keeps an online softmax per head; the splits' (max, sum, o) are
//      combined, with the sink, by the last split to finish;
//   3  the output projection (rows of Wo, K = heads x 128) against o staged
//      in shared memory, plus the residual if asked for.
// The producer thread issues the weights of phases 1 and 3 from the start
// (they depend on no data), so the output projection's first stages are in
// shared memory before phase 3 begins.
#include <new>
#include <vector>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kAtConsumers = 8;
constexpr int kAtThreads = 32 * (1 + kAtConsumers);
constexpr int kAtStages = 2 * kAtConsumers;
constexpr int kAtSeg = 256;
constexpr int kAtStageBytes = 16 * kAtSeg * 2;          // 8 KB: 4 chunks x 16 rows x 128 bytes
constexpr int kAtHd = 128;
constexpr int kAtMaxGroup = 8;                          // query heads per key/value head
constexpr int kAtMaxSplit = 64;
constexpr int kAtWp = kAtHd + 4;                        // per-warp softmax state pitch: o[128], max, sum (16-byte rows)
constexpr uint32_t kAll = 0xFFFFFFFFu;

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
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void named_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }
__device__ __forceinline__ bool named_sync_or(int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.or.pred q, 1, %1, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(n), "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Sums 8 per-lane values over the warp with 9 shuffles: afterwards lanes
// 4h .. 4h + 3 hold the total of value h (explicit registers, no indexing).
__device__ __forceinline__ float reduce8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                         float v7, int lane) {
  bool hi = (lane & 16) != 0;
  float a0 = (hi ? v4 : v0) + __shfl_xor_sync(kAll, hi ? v0 : v4, 16);
  float a1 = (hi ? v5 : v1) + __shfl_xor_sync(kAll, hi ? v1 : v5, 16);
  float a2 = (hi ? v6 : v2) + __shfl_xor_sync(kAll, hi ? v2 : v6, 16);
  float a3 = (hi ? v7 : v3) + __shfl_xor_sync(kAll, hi ? v3 : v7, 16);
  hi = (lane & 8) != 0;
  float b0 = (hi ? a2 : a0) + __shfl_xor_sync(kAll, hi ? a0 : a2, 8);
  float b1 = (hi ? a3 : a1) + __shfl_xor_sync(kAll, hi ? a1 : a3, 8);
  hi = (lane & 4) != 0;
  float c0 = (hi ? b1 : b0) + __shfl_xor_sync(kAll, hi ? b0 : b1, 4);
  c0 += __shfl_xor_sync(kAll, c0, 2);
  c0 += __shfl_xor_sync(kAll, c0, 1);
  return c0;   // lane l holds value 4 (l >> 4 & 1) + 2 (l >> 3 & 1) + (l >> 2 & 1) = l >> 2
}

struct AtLayout {
  uint32_t stages, bars, abort, prod, tab, act, red, total, x_pitch, o_pitch;
};
// Offsets from the 1024-aligned base (the allocation carries 1024 bytes of slack).
__host__ __device__ inline AtLayout at_layout(int d, int qdim) {
  AtLayout L;
  L.x_pitch = (uint32_t)d * 2 + 16;
  L.o_pitch = (uint32_t)qdim * 2 + 16;
  uint32_t o = 0;
  L.stages = o; o += kAtStages * kAtStageBytes;
  L.bars = o;   o += 2 * kAtStages * 8;
  L.abort = o;  o += 16;
  L.prod = o;   o += 4 * (kAtConsumers + kAtStages);
  o = (o + 15) & ~15u;
  L.tab = o;    o += 2 * kAtHd * 4 + (kAtHd / 2) * 8 + 64 * 4;   // q_norm, k_norm, RoPE turns, sinks (n_q <= 64)
  o = (o + 15) & ~15u;
  L.act = o;                                        // x rows (1), attention scratch (2) or o rows (3)
  const uint32_t xs = kAtMaxT * L.x_pitch, os = kAtMaxT * L.o_pitch;
  const uint32_t scratch = (kAtMaxGroup * kAtHd + 4 * kAtHd) * 4 + kAtConsumers * kAtMaxGroup * kAtWp * 4 + 256;
  uint32_t m = xs > os ? xs : os;
  m = m > scratch ? m : scratch;
  o += m;
  o = (o + 15) & ~15u;
  L.red = o;    o += 2 * kAtConsumers * 32 * 16;
  L.total = o + 1024;
  return L;
}

struct AtCtx {
  const AttnArgs& a;
  AtLayout L;
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
  WaitCtl wc;
  int G, b, warp, lane;
};

// Row groups of 16 rows of one projection.  Phase 1 enumerates the rows of
// Wq, Wk, Wv in that order; phase 3 the rows of Wo.
__device__ __forceinline__ void qkv_group(const AttnArgs& a, int rg, int& which, int& row0) {
  const int nq = a.n_q * kAtHd / 16, nk = a.n_kv * kAtHd / 16;
  if (rg < nq) { which = 0; row0 = rg * 16; }
  else if (rg < nq + nk) { which = 1; row0 = (rg - nq) * 16; }
  else { which = 2; row0 = (rg - nq - nk) * 16; }
}

__device__ __forceinline__ void share(int n, int b, int G, int& lo, int& hi) {
  lo = (int)(((long long)n * b) / G);
  hi = (int)(((long long)n * (b + 1)) / G);
}

// ---------------------------------------------------------------- producer (one thread)
__device__ __forceinline__ void run_producer(AtCtx& c) {
  const AttnArgs& a = c.a;
  int* pm = reinterpret_cast<int*>(c.smem + c.L.prod);
  uint32_t* ppar = reinterpret_cast<uint32_t*>(pm + kAtConsumers);
  for (int i = 0; i < kAtConsumers; ++i) pm[i] = 0;
  for (int i = 0; i < 4; ++i) tma_prefetch_desc(&a.tm[i]);
  const uint64_t pol = policy_evict_first();
  uint32_t used = 0;
  bool ok = true;
  auto issue = [&](int w, const CUtensorMap* m, int row0, int s) -> bool {
    const int mm = pm[w]++;
    const int st = w * 2 + (mm & 1);
    if (!mbar_wait(&c.empty[st], ((mm >> 1) & 1) ^ 1, c.wc)) return false;
    ppar[st] = (mm >> 1) & 1;
    used |= 1u << st;
    mbar_arrive_expect_tx(&c.full[st], kAtStageBytes);
    tma_load_3d_hint(c.smem + c.L.stages + st * kAtStageBytes, m, 0, row0, 4 * s, &c.full[st], pol);
    return true;
  };
  const int qdim = a.n_q * kAtHd;
  int lo, hi;
  share((qdim + 2 * a.n_kv * kAtHd) / 16, c.b, c.G, lo, hi);
  for (int rg = lo; rg < hi && ok; ++rg) {
    int which, row0;
    qkv_group(a, rg, which, row0);
    for (int s = 0; s < a.d / kAtSeg && ok; ++s) ok = issue(s % kAtConsumers, &a.tm[which], row0, s);
  }
  share(a.d / 16, c.b, c.G, lo, hi);
  for (int rg = lo; rg < hi && ok; ++rg)
    for (int s = 0; s < qdim / kAtSeg && ok; ++s) ok = issue(s % kAtConsumers, &a.tm[3], rg * 16, s);
  if (!ok)
    for (int st = 0; st < kAtStages; ++st)
      if (used & (1u << st)) drain_wait(&c.full[st], ppar[st], c.wc.limit_ns);
}

// ---------------------------------------------------------------- consumers
// One 16-row group: this warp's K segments (s = w, w + 8, ...) against the
// activation rows in shared memory (row n of B at bbase + n * bpitch), the
// warps' partial sums added in warp order by warp rg % 8, which calls
// out(row, n, value) for rows 0..15 and columns n < B.  Returns false (for
// every warp alike) if the CTA aborted.
template <typename Out>
__device__ __forceinline__ bool consume_group(AtCtx& c, int& m, int KC, uint32_t bbase, uint32_t bpitch, int B,
                                              int rg, Out&& out) {
  const int w = c.warp - 1, lane = c.lane;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t lrow = (lane & 7) + ((lane >> 3) & 1) * 8, lhi = lane >> 4, sw = lrow & 7;
  const int n = lane >> 2;
  const uint32_t b0a = bbase + (uint32_t)(n < B ? n : 0) * bpitch + (uint32_t)(lane & 3) * 4;
  for (int s = w; s < KC; s += kAtConsumers, ++m) {
    const int st = w * 2 + (m & 1);
    int good = 1;
    if (lane == 0) good = mbar_wait(&c.full[st], (m >> 1) & 1, c.wc) ? 1 : 0;
    good = __shfl_sync(kAll, good, 0);
    if (!good) break;
    while (!mbar_try_wait(&c.full[st], (m >> 1) & 1)) {
    }
    const uint32_t rbase = smem_u32(c.smem + c.L.stages + st * kAtStageBytes) + lrow * 128;
    const uint32_t bk = b0a + (uint32_t)s * kAtSeg * 2;
#pragma unroll 4
    for (int kk = 0; kk < kAtSeg / 16; ++kk) {
      uint32_t af[4];
      const uint32_t piece = ((((uint32_t)kk & 3) << 1) | lhi) ^ sw;
      ldsm_x4(rbase + (kk >> 2) * 2048 + (piece << 4), af);
      mma_bf16(acc, af, lds32(bk + kk * 32), lds32(bk + kk * 32 + 16));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.empty[st]);
  }
  float4* red = reinterpret_cast<float4*>(c.smem + c.L.red) + (rg & 1) * kAtConsumers * 32;
  red[w * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  if (named_sync_or(32 * kAtConsumers, *c.abort_flag != 0)) return false;
  if (w == rg % kAtConsumers) {
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const int nw = KC < kAtConsumers ? KC : kAtConsumers;
    for (int ww = 0; ww < nw; ++ww) {
      const float4 p = red[ww * 32 + lane];
      v[0] += p.x; v[1] += p.y; v[2] += p.z; v[3] += p.w;
    }
    const int row = lane >> 2;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = (lane & 3) * 2 + q;
      if (col < B) {
        out(row, col, v[q]);
        out(row + 8, col, v[2 + q]);
      }
    }
  }
  return true;
}

// Copy `rows` rows of `chunks` 16-byte pieces from global (src_pitch bytes)
// to shared memory (dst_pitch bytes) with asynchronous 16-byte copies
// (cp.async, L2 to shared memory, no registers held): every piece of the
// thread is in flight before it waits.  The caller synchronises the threads.
__device__ __forceinline__ void stage_rows(uint8_t* dst, uint32_t dst_pitch, const uint8_t* src, size_t src_pitch,
                                           int rows, int chunks, int tid, int nt) {
  const int n = rows * chunks;
  const uint32_t d0 = smem_u32(dst);
  for (int i = tid; i < n; i += nt) {
    const uint8_t* g = src + (size_t)(i / chunks) * src_pitch + (size_t)(i % chunks) * 16;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d0 + (uint32_t)(i / chunks) * dst_pitch +
                                                                    (uint32_t)(i % chunks) * 16),
                 "l"(g)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ bool grid_sync(AtCtx& c, unsigned target) {
  named_sync(32 * kAtConsumers);
  bool bad = false;
  if (threadIdx.x == 32 && !*c.abort_flag) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c.a.bar) : "memory");
    bool ok = ld_acquire_gpu(c.a.bar) >= target;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1; !ok; ++it) {
      ok = ld_acquire_gpu(c.a.bar) >= target;
      if (!ok && (it & 255u) == 0 && global_ns() - t0 > c.wc.limit_ns) break;
    }
    if (!ok) {
      atomicOr(c.a.err, kErrTimeout);
      *c.abort_flag = 1;
      bad = true;
    }
  }
  return !named_sync_or(32 * kAtConsumers, bad || *c.abort_flag != 0);
}

// RMSNorm with gamma, then RoPE at position pos, of one 128-value head held as
// 4 values per lane (lane l: values 2l, 2l + 1, 64 + 2l, 65 + 2l).  The angle
// of pair i is pos * f_i turns with f_i = base^(-2 i / 128) / (2 pi) stored as
// a 64-bit fraction (turns[i] = f_i 2^64, made on the host in fp64): the
// product's low 64 bits are pos * f_i mod 1 exactly, so the reduced angle
// keeps full precision at any position with integer arithmetic only.
__device__ __forceinline__ void norm_rope(float (&v)[4], const float* gamma, float eps, int pos, bool use_rope,
                                          const unsigned long long* turns, int lane) {
  float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(kAll, ss, o);
  const float r = rsqrtf(ss / (float)kAtHd + eps);
  const int i0 = 2 * lane;
  v[0] *= r * gamma[i0];
  v[1] *= r * gamma[i0 + 1];
  v[2] *= r * gamma[64 + i0];
  v[3] *= r * gamma[64 + i0 + 1];
  if (!use_rope) return;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const unsigned long long frac = (unsigned long long)(unsigned)pos * turns[i0 + j];
    // the turn as a signed fraction in [-1/2, 1/2): the angle lands in [-pi, pi),
    // where the fast sine and cosine are accurate to about 2^-21
    const float ang = (float)((long long)frac >> 40) * (6.283185307179586f / 16777216.f);
    float sn, cs;
    __sincosf(ang, &sn, &cs);
    const float x0 = v[j], x1 = v[2 + j];
    v[j] = x0 * cs - x1 * sn;
    v[2 + j] = x0 * sn + x1 * cs;
  }
}

__device__ __forceinline__ void run_consumers(AtCtx& c) {
  const AttnArgs& a = c.a;
  const int w = c.warp - 1, lane = c.lane, tid = threadIdx.x - 32, NT = 32 * kAtConsumers;
  const int B = a.B, d = a.d, qdim = a.n_q * kAtHd, kvdim = a.n_kv * kAtHd, R = qdim + 2 * kvdim;
  const int group = a.n_q / a.n_kv;
  int m = 0;
  // tables of phase 2 in shared memory (gammas, RoPE turns, sinks), and this
  // CTA's keys and values pulled into L2 while phase 1 runs
  float* tq = reinterpret_cast<float*>(c.smem + c.L.tab);
  float* tk = tq + kAtHd;
  unsigned long long* tt = reinterpret_cast<unsigned long long*>(tk + kAtHd);
  float* tsk = reinterpret_cast<float*>(tt + kAtHd / 2);
  for (int i = tid; i < kAtHd; i += NT) {
    tq[i] = __ldg(a.q_norm + i);
    tk[i] = __ldg(a.k_norm + i);
    if (i < kAtHd / 2) tt[i] = __ldg(a.rope_turns + i);
    if (i < a.n_q) tsk[i] = __ldg(a.sinks + i);
  }
  {
    const int S = a.splits, n_items = B * a.n_kv * S;
    for (int item = c.b; item < n_items; item += c.G) {
      const int bq = item / (a.n_kv * S), g = (item / S) % a.n_kv, sp = item % S;
      const int pos = max(__ldg(a.pos + bq), 0), W = a.window;
      const int n_keys = pos + 1 < W ? pos + 1 : W, first = pos + 1 - n_keys;
      const int j0 = (int)(((long long)n_keys * sp) / S), j1 = (int)(((long long)n_keys * (sp + 1)) / S);
      for (int j = j0 + tid; j < j1; j += NT) {
        const size_t sl = (((size_t)bq * W + ((first + j) % W)) * a.n_kv + g) * kAtHd;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], 256;" ::"l"(a.k_cache + sl) : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], 256;" ::"l"(a.v_cache + sl) : "memory");
      }
    }
  }
  // ---------------- phase 1: q, k, v
  {
    uint8_t* xs = c.smem + c.L.act;
    stage_rows(xs, c.L.x_pitch, reinterpret_cast<const uint8_t*>(a.x), (size_t)d * 2, B, d / 8, tid, NT);
    named_sync(NT);
    int lo, hi;
    share(R / 16, c.b, c.G, lo, hi);
    for (int rg = lo; rg < hi; ++rg) {
      int which, row0;
      qkv_group(a, rg, which, row0);
      const int col0 = which == 0 ? row0 : (which == 1 ? qdim + row0 : qdim + kvdim + row0);
      if (!consume_group(c, m, d / kAtSeg, smem_u32(xs), c.L.x_pitch, B, rg,
                         [&](int row, int n, float v) { __stcg(a.qkv + (size_t)n * R + col0 + row, v); }))
        return;
    }
  }
  if (!grid_sync(c, 1u * c.G)) return;

  // ---------------- phase 2: attention items (sequence, kv head, split)
  {
    const int S = a.splits;
    const int n_items = B * a.n_kv * S;
    float* qs = reinterpret_cast<float*>(c.smem + c.L.act);            // [group][128] normalised, rotated q
    float* kn = qs + kAtMaxGroup * kAtHd;                               // [128] new key (bf16 values)
    float* vn = kn + kAtHd;                                             // [128] new value (bf16 values)
    uint16_t* knb = reinterpret_cast<uint16_t*>(vn + kAtHd);           // [128] new key, bf16 bits
    uint16_t* vnb = knb + kAtHd;                                        // [128] new value, bf16 bits
    float* wst = vn + 2 * kAtHd;                                        // [8 warps][group][kAtWp]
    const float scale = rsqrtf((float)kAtHd);
    for (int item = c.b; item < n_items; item += c.G) {
      const int bq = item / (a.n_kv * S), g = (item / S) % a.n_kv, sp = item % S;
      int pos = __ldg(a.pos + bq);
      if (pos < 0) {                               // a negative position is reported and treated as 0
        if (tid == 0) atomicOr(a.err, kErrRange);
        pos = 0;
      }
      const int W = a.window;
      const int n_keys = pos + 1 < W ? pos + 1 : W, first = pos + 1 - n_keys;
      const int j0 = (int)(((long long)n_keys * sp) / S), j1 = (int)(((long long)n_keys * (sp + 1)) / S);
      const float* qrow = a.qkv + (size_t)bq * R;
      // tasks 0 .. group - 1: query head g * group + task; task group: the new
      // key and value (task t on warp t % 8, so warp 0 also takes task 8)
      for (int task = w; task <= group; task += kAtConsumers) {
        float v[4];
        const float* src = task < group ? qrow + (g * group + task) * kAtHd : qrow + qdim + g * kAtHd;
        const int i0 = 2 * lane;
        v[0] = __ldcg(src + i0); v[1] = __ldcg(src + i0 + 1); v[2] = __ldcg(src + 64 + i0); v[3] = __ldcg(src + 65 + i0);
        norm_rope(v, task < group ? tq : tk, a.eps, pos, a.use_rope != 0, tt, lane);
        float* dst = task < group ? qs + task * kAtHd : kn;
        if (task == group) {                     // the cache holds bf16
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
        }
        dst[i0] = v[0]; dst[i0 + 1] = v[1]; dst[64 + i0] = v[2]; dst[65 + i0] = v[3];
        if (task == group) {
          knb[i0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[0]));
          knb[i0 + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(v[1]));
          knb[64 + i0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[2]));
          knb[65 + i0] = __bfloat16_as_ushort(__float2bfloat16_rn(v[3]));
          const float* vs = qrow + qdim + kvdim + g * kAtHd;
          for (int i = lane; i < kAtHd; i += 32) {
            const __nv_bfloat16 vb = __float2bfloat16_rn(__ldcg(vs + i));
            vn[i] = __bfloat162float(vb);
            vnb[i] = __bfloat16_as_ushort(vb);
          }
        }
      }
      named_sync(NT);
      const size_t slot_new = ((size_t)bq * W + (pos % W)) * a.n_kv + g;
      if (sp == 0)
        for (int i = tid; i < kAtHd; i += NT) {
          a.k_cache[slot_new * kAtHd + i] = __float2bfloat16_rn(kn[i]);
          a.v_cache[slot_new * kAtHd + i] = __float2bfloat16_rn(vn[i]);
        }
      // online softmax over this warp's keys; lane l holds dims 4l..4l+3 of every head
      float mx[kAtMaxGroup], sm[kAtMaxGroup], o[kAtMaxGroup][4];
#pragma unroll
      for (int h = 0; h < kAtMaxGroup; ++h) {
        mx[h] = -INFINITY;
        sm[h] = 0.f;
        o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;
      }
      float qv[kAtMaxGroup][4];
#pragma unroll
      for (int h = 0; h < kAtMaxGroup; ++h) {
        const float4 t4 = h < group ? *reinterpret_cast<const float4*>(qs + h * kAtHd + 4 * lane)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[h][0] = t4.x; qv[h][1] = t4.y; qv[h][2] = t4.z; qv[h][3] = t4.w;
      }
      // keys j0 + w, j0 + w + 8, ...: eight at a time, all their loads issued
      // before any of them is used (the new token's entry comes from shared
      // memory, the others from the cache)
      for (int jb = j0 + w; jb < j1; jb += 8 * kAtConsumers) {
        uint2 kbv[8], vbv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = jb + u * kAtConsumers;
          kbv[u] = make_uint2(0u, 0u);
          vbv[u] = make_uint2(0u, 0u);
          if (j < j1) {
            const int p = first + j;
            if (p == pos) {                      // shared memory
              kbv[u] = *reinterpret_cast<const uint2*>(knb + 4 * lane);
              vbv[u] = *reinterpret_cast<const uint2*>(vnb + 4 * lane);
            } else {                             // the cache, through L2
              const size_t sl = (((size_t)bq * W + (p % W)) * a.n_kv + g) * kAtHd + 4 * lane;
              kbv[u] = __ldcg(reinterpret_cast<const uint2*>(a.k_cache + sl));
              vbv[u] = __ldcg(reinterpret_cast<const uint2*>(a.v_cache + sl));
            }
          }
        }
        // all eight scores first (independent reductions), then one rescale per head for the batch
        float zs[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          float kk[4];
          kk[0] = __uint_as_float(kbv[u].x << 16); kk[1] = __uint_as_float(kbv[u].x & 0xFFFF0000u);
          kk[2] = __uint_as_float(kbv[u].y << 16); kk[3] = __uint_as_float(kbv[u].y & 0xFFFF0000u);
#define AT_DOT(h) (qv[h][0] * kk[0] + qv[h][1] * kk[1] + qv[h][2] * kk[2] + qv[h][3] * kk[3])
          zs[u] = reduce8(AT_DOT(0), AT_DOT(1), AT_DOT(2), AT_DOT(3), AT_DOT(4), AT_DOT(5), AT_DOT(6), AT_DOT(7),
                          lane);   // lane 4 h holds head h's score
#undef AT_DOT
        }
        const int nu = (j1 - jb + kAtConsumers - 1) / kAtConsumers;   // keys of this batch (>= 1)
#pragma unroll
        for (int h = 0; h < kAtMaxGroup; ++h) {
          if (h < group) {
            float z[8], mb = -INFINITY;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              z[u] = u < nu ? __shfl_sync(kAll, zs[u], 4 * h) * scale : -INFINITY;
              mb = fmaxf(mb, z[u]);
            }
            const float mn = fmaxf(mx[h], mb);
            const float f = __expf(mx[h] - mn);
            sm[h] *= f;
#pragma unroll
            for (int q = 0; q < 4; ++q) o[h][q] *= f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const float pz = __expf(z[u] - mn);       // 0 for the batch's missing keys
              sm[h] += pz;
              o[h][0] += pz * __uint_as_float(vbv[u].x << 16);
              o[h][1] += pz * __uint_as_float(vbv[u].x & 0xFFFF0000u);
              o[h][2] += pz * __uint_as_float(vbv[u].y << 16);
              o[h][3] += pz * __uint_as_float(vbv[u].y & 0xFFFF0000u);
            }
            mx[h] = mn;
          }
        }
      }
      // the warps' states to shared memory, combined by every thread for its (head, dim)
#pragma unroll
      for (int h = 0; h < kAtMaxGroup; ++h)
        if (h < group) {
          float* ws = wst + (w * kAtMaxGroup + h) * kAtWp;
          *reinterpret_cast<float4*>(ws + 4 * lane) = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
          if (lane == 0) { ws[kAtHd] = mx[h]; ws[kAtHd + 1] = sm[h]; }
        }
      named_sync(NT);
      float* part = a.part + (size_t)item * kAtMaxGroup * (kAtHd + 2);
      for (int i = tid; i < group * (kAtHd + 2); i += NT) {
        const int h = i / (kAtHd + 2), e = i % (kAtHd + 2);
        float M = -INFINITY;
        for (int ww = 0; ww < kAtConsumers; ++ww) M = fmaxf(M, wst[(ww * kAtMaxGroup + h) * kAtWp + kAtHd]);
        float acc = 0.f;
        if (M != -INFINITY) {
          for (int ww = 0; ww < kAtConsumers; ++ww) {
            const float* ws = wst + (ww * kAtMaxGroup + h) * kAtWp;
            const float wm = ws[kAtHd];
            if (wm == -INFINITY) continue;
            const float f = __expf(wm - M);
            acc += (e == kAtHd + 1 ? ws[kAtHd + 1] : (e < kAtHd ? ws[e] : 0.f)) * f;
          }
        }
        __stcg(part + h * (kAtHd + 2) + e, e == kAtHd ? M : acc);
      }
      // the last split of (sequence, kv head) to finish combines them, with the sinks
      named_sync(NT);
      __shared__ int last;
      if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(a.split_cnt + bq * a.n_kv + g, 1u);
        last = prev == (unsigned)(S - 1);
        if (last) {
          a.split_cnt[bq * a.n_kv + g] = 0;
          __threadfence();
        }
      }
      named_sync(NT);
      if (last) {
        const float* p0 = a.part + (size_t)(bq * a.n_kv + g) * S * kAtMaxGroup * (kAtHd + 2);
        // warp h: the split weights exp(m_s - M) / L of head h (sink included) into shared memory
        float* fw = wst;                                   // [group][kAtMaxSplit] (the warp states are done)
        if (w < group) {
          const float sink = tsk[g * group + w];
          float ms[2], ls[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int s2 = lane + 32 * u;
            ms[u] = s2 < S ? __ldcg(p0 + ((size_t)s2 * kAtMaxGroup + w) * (kAtHd + 2) + kAtHd) : -INFINITY;
            ls[u] = s2 < S ? __ldcg(p0 + ((size_t)s2 * kAtMaxGroup + w) * (kAtHd + 2) + kAtHd + 1) : 0.f;
          }
          float M = fmaxf(sink, fmaxf(ms[0], ms[1]));
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, o));
          float f[2], L = 0.f;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            f[u] = ms[u] == -INFINITY ? 0.f : __expf(ms[u] - M);
            L += ls[u] * f[u];
          }
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(kAll, L, o);
          L += __expf(sink - M);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (lane + 32 * u < S) fw[w * kAtMaxSplit + lane + 32 * u] = f[u] / L;
        }
        named_sync(NT);
        for (int i = tid; i < group * kAtHd; i += NT) {
          const int h = i / kAtHd, e = i % kAtHd;
          float acc = 0.f;
          // eight splits' loads in flight at a time (a loop of dependent L2 round trips would serialise them)
          for (int s0 = 0; s0 < S; s0 += 8) {
            float pv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              pv[u] = s0 + u < S ? __ldcg(p0 + ((size_t)(s0 + u) * kAtMaxGroup + h) * (kAtHd + 2) + e) : 0.f;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              if (s0 + u < S) acc += pv[u] * fw[h * kAtMaxSplit + s0 + u];
          }
          a.ob[(size_t)bq * qdim + (g * group + h) * kAtHd + e] = __float2bfloat16_rn(acc);
        }
      }
      named_sync(NT);
    }
  }
  if (!grid_sync(c, 2u * c.G)) return;

  // ---------------- phase 3: output projection
  {
    uint8_t* os = c.smem + c.L.act;
    stage_rows(os, c.L.o_pitch, reinterpret_cast<const uint8_t*>(a.ob), (size_t)qdim * 2, B, qdim / 8, tid, NT);
    named_sync(NT);
    int lo, hi;
    share(d / 16, c.b, c.G, lo, hi);
    for (int rg = lo; rg < hi; ++rg) {
      if (!consume_group(c, m, qdim / kAtSeg, smem_u32(os), c.L.o_pitch, B, rg, [&](int row, int n, float v) {
            const int r = rg * 16 + row;
            if (a.add_residual) v += __bfloat162float(a.x[(size_t)n * d + r]);
            a.y[(size_t)n * d + r] = __float2bfloat16_rn(v);
          }))
        return;
    }
  }
}

__global__ void __launch_bounds__(kAtThreads, 1) attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);
  AtCtx c{a};
  c.L = at_layout(a.d, a.n_q * kAtHd);
  c.smem = dsm;
  c.full = reinterpret_cast<uint64_t*>(dsm + c.L.bars);
  c.empty = c.full + kAtStages;
  c.abort_flag = reinterpret_cast<volatile int*>(dsm + c.L.abort);
  c.G = gridDim.x;
  c.b = blockIdx.x;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kAtStages; ++i) {
      mbar_init(&c.full[i], 1);
      mbar_init(&c.empty[i], 1);
    }
    *c.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  c.wc = WaitCtl{a.wait_ns, a.err, c.abort_flag};
  if (c.warp == 0) {
    if (c.lane == 0) run_producer(c);
  } else {
    run_consumers(c);
  }
}

}  // namespace

size_t attn_decode_smem_bytes(int d, int n_q) { return at_layout(d, n_q * kAtHd).total; }

cudaError_t launch_attn_decode(const AttnArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = attn_decode_smem_bytes(a.d, a.n_q);
  cudaError_t e = ensure_smem_limit(attn_decode_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kAtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel, a);
}

}  // namespace moe

// ---------------------------------------------------------------- C ABI
using namespace moe;

struct moe_attn {
  moe_attn_config cfg;
  moe_attn_weights w;
  int num_sms = 0;
  CUtensorMap tm[4];
  void* block = nullptr;
  float* qkv = nullptr;
  __nv_bfloat16* ob = nullptr;
  float* part = nullptr;
  unsigned* split_cnt = nullptr;
  unsigned* bar = nullptr;
  unsigned* err = nullptr;
  unsigned long long* turns = nullptr;   // [64] RoPE frequencies as 64-bit fractions of a turn
  uint64_t wait_ns = 0;
};

extern "C" {

moe_status moe_attn_create(const moe_attn_config* cfg, const moe_attn_weights* w, moe_attn_handle* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w || !w->wq || !w->wk || !w->wv || !w->wo || !w->q_norm || !w->k_norm || !w->sinks)
    return MOE_ERR_INVALID_ARG;
  const moe_attn_config& c = *cfg;
  if (c.d <= 0 || c.n_q <= 0 || c.n_kv <= 0 || c.head_dim <= 0 || c.window <= 0 || c.max_batch <= 0 ||
      c.wait_timeout_ms < 0 || !(c.eps >= 0.f) || !(c.rope_base > 0.f))
    return MOE_ERR_INVALID_ARG;
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis(w->wq) || mis(w->wk) || mis(w->wv) || mis(w->wo) || (reinterpret_cast<uintptr_t>(w->q_norm) & 3u) ||
      (reinterpret_cast<uintptr_t>(w->k_norm) & 3u) || (reinterpret_cast<uintptr_t>(w->sinks) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (c.head_dim != kAtHd || c.n_q % c.n_kv != 0 || c.n_q / c.n_kv > kAtMaxGroup || c.d % kAtSeg != 0 ||
      c.max_batch > kAtMaxT || c.n_kv * kAtMaxT > 240 || c.n_q > 64)
    return MOE_ERR_UNSUPPORTED;
  moe_attn* h = new (std::nothrow) moe_attn();
  if (!h) return MOE_ERR_OOM;
  h->cfg = c;
  h->w = *w;
  int dev = 0, coop = 0, cc = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&cc, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_CUDA;
  }
  if (!coop || cc != 10 || attn_decode_smem_bytes(c.d, c.n_q) > (size_t)optin) {
    delete h;
    return MOE_ERR_UNSUPPORTED;
  }
  const uint64_t qdim = (uint64_t)c.n_q * kAtHd, kvdim = (uint64_t)c.n_kv * kAtHd, d = c.d;
  auto view = [](CUtensorMap* m, const void* base, uint64_t rows, uint64_t K) {
    const uint64_t dims[3] = {64, rows, K / 64}, strides[2] = {K * 2, 128};
    const uint32_t box[3] = {64, 16, 4};
    return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  if (!view(&h->tm[0], w->wq, qdim, d) || !view(&h->tm[1], w->wk, kvdim, d) || !view(&h->tm[2], w->wv, kvdim, d) ||
      !view(&h->tm[3], w->wo, d, qdim)) {
    delete h;
    return MOE_ERR_CUDA;
  }
  const size_t B = kAtMaxT, R = qdim + 2 * kvdim;
  if ((c.window + 63) / 64 > kAtMaxSplit) {
    delete h;
    return MOE_ERR_UNSUPPORTED;
  }
  const size_t n_part = B * c.n_kv * kAtMaxSplit * kAtMaxGroup * (kAtHd + 2);
  const size_t bytes = ((B * R * 4 + 255) & ~(size_t)255) + ((B * qdim * 2 + 255) & ~(size_t)255) +
                       ((n_part * 4 + 255) & ~(size_t)255) + 1024 + 512;
  if (dev_malloc(&h->block, bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  uint8_t* p = static_cast<uint8_t*>(h->block);
  h->qkv = reinterpret_cast<float*>(p); p += (B * R * 4 + 255) & ~(size_t)255;
  h->ob = reinterpret_cast<__nv_bfloat16*>(p); p += (B * qdim * 2 + 255) & ~(size_t)255;
  h->part = reinterpret_cast<float*>(p); p += (n_part * 4 + 255) & ~(size_t)255;
  h->split_cnt = reinterpret_cast<unsigned*>(p);       // [B * n_kv] (at most 256 words with the bar and err)
  h->bar = h->split_cnt + 240;
  h->err = h->split_cnt + 248;
  h->turns = reinterpret_cast<unsigned long long*>(p + 1024);
  {
    // f_i = base^(-2 i / 128) / (2 pi) turns per position, as f_i 2^64 (f_i < 1)
    unsigned long long t[kAtHd / 2];
    for (int i = 0; i < kAtHd / 2; ++i) {
      const double f = pow((double)c.rope_base, -2.0 * i / kAtHd) / 6.283185307179586476925286766559;
      t[i] = (unsigned long long)ldexp(f, 64);
    }
    if (cudaMemcpy(h->turns, t, sizeof(t), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(h->block);
      delete h;
      return MOE_ERR_CUDA;
    }
  }
  if (cudaMemset(h->split_cnt, 0, 1024) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->block);
    delete h;
    return MOE_ERR_CUDA;
  }
  h->wait_ns = (uint64_t)(c.wait_timeout_ms > 0 ? c.wait_timeout_ms : 2000) * 1000000ull;
  *out = h;
  return MOE_OK;
}

moe_status moe_attn_decode(moe_attn_handle h, const void* x, int32_t B, const int32_t* pos, void* k_cache,
                           void* v_cache, void* y, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (B < 0 || B > h->cfg.max_batch) return MOE_ERR_INVALID_ARG;
  if (B == 0) return MOE_OK;
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (!x || !pos || !k_cache || !v_cache || !y || mis(x) || mis(y) || mis(k_cache) || mis(v_cache) ||
      (reinterpret_cast<uintptr_t>(pos) & 3u))
    return MOE_ERR_INVALID_ARG;
  const moe_attn_config& c = h->cfg;
  const size_t nb = (size_t)B * c.d * 2;
  {
    const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
    if (a < b + nb && b < a + nb) return MOE_ERR_INVALID_ARG;
  }
  if (cudaMemsetAsync(h->bar, 0, 4, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  AttnArgs a;
  for (int i = 0; i < 4; ++i) a.tm[i] = h->tm[i];
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.y = static_cast<__nv_bfloat16*>(y);
  a.pos = pos;
  a.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  a.q_norm = h->w.q_norm;
  a.k_norm = h->w.k_norm;
  a.sinks = h->w.sinks;
  a.qkv = h->qkv;
  a.ob = h->ob;
  a.part = h->part;
  a.split_cnt = h->split_cnt;
  a.bar = h->bar;
  a.err = h->err;
  a.B = B;
  a.d = c.d;
  a.n_q = c.n_q;
  a.n_kv = c.n_kv;
  a.window = c.window;
  a.use_rope = c.use_rope;
  a.add_residual = c.add_residual;
  a.eps = c.eps;
  a.rope_turns = h->turns;
  // window splits per (sequence, kv head): at most 64 keys each, so every
  // warp takes a single batch of 8 keys and the combine reads few partials
  int S = (c.window + 63) / 64;
  S = S < 1 ? 1 : (S > kAtMaxSplit ? kAtMaxSplit : S);
  a.splits = S;
  a.wait_ns = h->wait_ns;
  if (launch_attn_decode(a, h->num_sms, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status moe_attn_check(moe_attn_handle h, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word && cudaMemset(h->err, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
  if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
  return (word & kErrRange) ? MOE_ERR_RANGE : MOE_OK;
}

moe_status moe_attn_destroy(moe_attn_handle h) {
  if (!h) return MOE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  const cudaError_t f = cudaFree(h->block);
  delete h;
  return (e == cudaSuccess && f == cudaSuccess) ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
