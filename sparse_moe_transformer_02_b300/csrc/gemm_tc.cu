// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// for batches large enough that each expert sees many tokens (prefill).
//
// The layer is y_t = sum_j g_j E_{idx_j}(x_t) + S(x_t) with SwiGLU experts
// (readings of the evermx.com review, section "Sparse architecture").  After
// grouping, the token-slots of expert e are contiguous, so each expert is a
// small dense GEMM whose weights are read from HBM once per call.
//
// Tiles put the weights on the MMA's M side (128 weight rows per tile) and
// the tokens on the N side (up to 128 tokens, rounded up to 16), so an
// expert's ~100 tokens are not padded to 128 rows of wasted A traffic.
//
//  * pass 1 (gate/up): D_g = Wg[rows] . X^T and D_u = Wu[rows] . X^T into two
//    TMEM accumulators; the epilogue writes h = silu(D_g) * D_u (bf16) per
//    slot.  The routed slots read a slot-ordered copy of x (made by a small
//    gather kernel) with plain tiled TMA loads; the shared expert reads x.
//  * pass 2 (down): D = Wd[rows] . H^T; the epilogue multiplies by the
//    slot's gate and adds into an fp32 accumulator y_acc[t][row] with
//    red.global.add (order of the adds is not fixed: the fp32 sum is
//    deterministic up to rounding order).
//  * pass 2 for large batches (token-major): A = h of 128 slots, B = 256 rows
//    of Wd, D[slot][row]; each epilogue thread owns one slot (one (token,
//    gate) lookup per tile) and the warp passes each 32 x 32 chunk of its
//    gated outputs through a shared-memory tile, so that every
//    red.global.add.v4.f32 instruction adds 4 token rows x 128 contiguous
//    bytes (one instruction per row would touch 32 rows x 16 bytes; the
//    transposed form also beat bulk reductions from shared memory
//    (cp.reduce.async.bulk) at 16384 tokens: 404 against 491 us).
//  * finalise: y = bf16(y_acc (+ x)).
//
// One persistent CTA per SM, 6 warps: warp 0 issues TMA into a ring of
// shared-memory stages, warp 1 (one thread) issues tcgen05.mma and commits to
// mbarriers, warps 2-5 drain TMEM (double-buffered accumulators) while the
// next tile's MMAs run.  Every wait is bounded (see ptx.cuh).
#include <utility>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "units.cuh"

namespace moe {
namespace {

constexpr int kThreadsTc = 192;
// Down pass: units are claimed from a grid-wide counter (a CTA that started
// late, after a long gate/up tile, takes fewer of them) and handed from the
// producer warp to the MMA thread and the epilogue warps through a ring of
// kRing entries in shared memory.
constexpr int kRing = 8;

template <int MODE> struct TcCfg;

template <int MODE> struct TcStaging { static constexpr int BYTES = 0; };
constexpr int kTpPitch = 36;     // token-major red epilogue: floats per row of a warp's 32 x 32 transpose tile
template <> struct TcStaging<2> { static constexpr int BYTES = 4 * 32 * kTpPitch * 4; };    // one tile per warp

template <> struct TcCfg<0> {     // gate/up: A_g + A_u + B per stage
  static constexpr int STAGES = 4;
  static constexpr int STAGE_BYTES = 2 * kTcBM * 128 + kTcBN * 128;
  static constexpr int ACC_COLS = 2 * kTcBN;          // per buffer: gate then up
  static constexpr int TMEM_COLS = 2 * ACC_COLS;      // two buffers
};
template <> struct TcCfg<1> {     // down, weight-major: A (128 Wd rows) + B (h of <= 128 slots)
  static constexpr int STAGES = 6;
  static constexpr int STAGE_BYTES = kTcBM * 128 + kTcBN * 128;
  static constexpr int ACC_COLS = kTcBN;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
};
template <> struct TcCfg<2> {     // down, token-major: A (h of 128 slots) + B (256 Wd rows); red.v4 epilogue
  static constexpr int STAGES = 4;
  static constexpr int STAGE_BYTES = kTcBM * 128 + 2 * kTcBN * 128;
  static constexpr int ACC_COLS = 2 * kTcBN;
  static constexpr int TMEM_COLS = 2 * ACC_COLS;
};

struct TcParams {
  CUtensorMap tm_a0, tm_a1;   // routed weights (pass 1: gate, up; pass 2: down)
  CUtensorMap tm_sa0, tm_sa1; // shared expert weights
  CUtensorMap tm_b;           // routed B operand: pass 1 slot-ordered x copy, pass 2 h
  CUtensorMap tm_sb;          // shared-expert B operand: pass 1 x, pass 2 h
  int T, d, F, Fs, E, k, Fmax;
  int K, Ks;                  // reduction width, routed / shared
  int mt, mt_s;               // weight-row tiles per expert, routed / shared
  int n_pre;                  // units that need no routing (shared expert, pass 1)
  const int32_t* tok_of_slot;
  const int32_t* src_of_slot;
  const float* gate;
  const TcUnit* units;
  const int32_t* n_units;
  __nv_bfloat16* h16;
  float* yacc;
  float* oslot;               // deterministic mode: per-slot rows [T (k + 1)][d] instead of y_acc, or null
  unsigned int* err;
  uint64_t wait_ns;
  // Gate/up progress, read by the down pass (see below): ready[e] counts the
  // finished (tile, epilogue warp) pairs of expert e, ready[E + 2] the
  // (CTA, epilogue warp) pairs done with all their tiles, ready[E + 1] the
  // (CTA, epilogue warp) pairs done clearing y_acc.
  unsigned int* ready;
  const int32_t* counts;        // per-expert token counts (down pass: readiness targets)
  int mt_gu, mt_gu_s;           // gate/up row tiles per routed / shared expert
  int gu_ctas;                  // CTAs of the gate/up grid
  // Small batches leave most SMs idle with one unit per (expert, row tile):
  // pass 1 then splits every tile into ksplit parts along K (consecutive
  // entries u of one tile, part u % ksplit).  Each part stores its partial
  // sums to gu_part[part]; the last part to finish a warp's rows (gu_cnt)
  // adds the parts in order (deterministic) and writes h.
  int ksplit;
  unsigned int* sched;          // down pass: next unit to claim (kept at zero between calls)
  int P;                        // rows of h (T (k + 1))
  float* gu_part;
  unsigned int* gu_cnt;
};

__device__ __forceinline__ TcUnit get_unit(const TcParams& p, int u) {
  if (u < p.n_pre) {
    const int base = u / p.ksplit, tb = base / p.mt_s, m = base % p.mt_s;
    return TcUnit{p.E, m, tb * kTcBN, min(kTcBN, p.T - tb * kTcBN)};
  }
  return p.units[u];
}

// Unit descriptors one step ahead: the entry a role needs next is loaded while
// it works on the current one, so no role stalls on that load between units.
struct UnitCursor {
  TcUnit nxt;
  int nxt_u = -1;
  __device__ __forceinline__ TcUnit get(const TcParams& p, int u, int n_total) {
    const TcUnit un = u == nxt_u ? nxt : get_unit(p, u);
    const int v = u + (int)gridDim.x;
    nxt_u = -1;
    if (v < n_total) {
      nxt = get_unit(p, v);
      nxt_u = v;
    }
    return un;
  }
};

template <int MODE>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<MODE>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = dsm;
  float* red_stage = reinterpret_cast<float*>(dsm + S * C::STAGE_BYTES);   // MODE 2: [4][32][kTpPitch]
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + S * C::STAGE_BYTES + TcStaging<MODE>::BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* col_tok = abort_flag + 3;                               // [4 warps][kTcBN] token of each column (pass 2)
  float* col_gate = reinterpret_cast<float*>(col_tok + 4 * kTcBN);   // [4 warps][kTcBN] its gate
  uint64_t* ufull = reinterpret_cast<uint64_t*>(col_gate + 4 * kTcBN);   // [kRing] unit posted (pass 2)
  uint64_t* uempty = ufull + kRing;                                        // [kRing] unit taken by all roles
  TcUnit* ring = reinterpret_cast<TcUnit*>(uempty + kRing);                // [kRing]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    if (MODE >= 1)
      for (int i = 0; i < kRing; ++i) {
        mbar_init(&ufull[i], 1);
        mbar_init(&uempty[i], 5);     // the MMA thread and the four epilogue warps
      }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_a0);
    tma_prefetch_desc(&p.tm_b);
    tma_prefetch_desc(&p.tm_sb);
    tma_prefetch_desc(&p.tm_sa0);
    if (MODE == 0) {
      tma_prefetch_desc(&p.tm_a1);
      tma_prefetch_desc(&p.tm_sa1);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{p.wait_ns, p.err, abort_flag};
  constexpr int LIST = MODE == 0 ? 0 : 1;       // unit list: gate/up or down
  // Gate/up lets the down pass launch only once routing is known complete
  // (each thread triggers right after its own grid-dependency wait), so the
  // down pass can read the grouping at once; it then waits per expert on the
  // readiness counters instead of on the whole gate/up grid, and its CTAs take
  // the SMs that gate/up's last, partial wave leaves idle.
  auto wait_routing = [] {
    pdl_wait();
    pdl_launch_dependents();
  };
  if (MODE >= 1) pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t last_par[S];
    bool issued[S];
    for (int i = 0; i < S; ++i) issued[i] = false;
    int n_total = p.n_pre;
    bool waited = MODE >= 1;
    if (MODE >= 1) n_total = __ldcg(p.n_units + LIST);
    bool ok = true;
    if (MODE >= 1) {
      // the down pass adds into y_acc: every gate/up CTA must have cleared it
      int w = 1;
      if (lane == 0) w = counter_wait(p.ready + p.E + 1, 4u * p.gu_ctas, wc) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, w, 0) != 0;
    }
    UnitCursor cur;
    bool gu_done = false;                  // down pass: every gate/up tile seen finished
    // down pass: while a unit's loads are issued, the next unit's descriptor
    // load and the claim of the one after it are in flight.  With few units
    // per CTA (small batches) a CTA claims its next unit only when it is done
    // issuing the current one, so that the first CTAs to start do not take
    // two units each while other SMs have none.
    int u = blockIdx.x, claim = 0;
    const bool ahead = n_total > 2 * (int)gridDim.x;
    TcUnit un_nx{-1, 0, 0, 0};
    if (MODE >= 1 && ok) {
      if (lane == 0) claim = (int)atomicAdd(p.sched, 1u);
      u = __shfl_sync(0xFFFFFFFFu, claim, 0);
      if (u < n_total) un_nx = get_unit(p, u);
      if (ahead && lane == 0 && u < n_total) claim = (int)atomicAdd(p.sched, 1u);
    }
    for (int it = 0; ok; ++it) {
      TcUnit un;
      if constexpr (MODE == 0) {
        if (it > 0) u += gridDim.x;
        if (u >= n_total) {
          if (waited) break;
          wait_routing();
          waited = true;
          n_total = __ldcg(p.n_units + LIST);
          if (u >= n_total) break;
        }
        un = cur.get(p, u, n_total);
      } else {
        if (it > 0 && !ahead) {
          if (lane == 0) claim = (int)atomicAdd(p.sched, 1u);
          const int u_nx = __shfl_sync(0xFFFFFFFFu, claim, 0);
          un_nx = TcUnit{-1, 0, 0, 0};
          if (u_nx < n_total) un_nx = get_unit(p, u_nx);
        }
        un = un_nx;
        // post the unit (or the end mark) to the other roles
        const int slot = it % kRing;
        if (!warp_wait(&uempty[slot], ((it / kRing) & 1) ^ 1, wc)) { ok = false; break; }
        if (lane == 0) {
          ring[slot] = un;
          mbar_arrive(&ufull[slot]);
        }
        __syncwarp();
        if (un.expert < 0) break;
        if (ahead) {
          const int u_nx = __shfl_sync(0xFFFFFFFFu, claim, 0);
          un_nx = TcUnit{-1, 0, 0, 0};
          if (u_nx < n_total) un_nx = get_unit(p, u_nx);
          if (lane == 0 && u_nx < n_total) claim = (int)atomicAdd(p.sched, 1u);
        }
        u = 0;
      }
      const bool sh = un.expert == p.E;
      const int K = sh ? p.Ks : p.K;
      const int kb = K / kTcBK, part = u % p.ksplit;
      const int kbeg = part * kb / p.ksplit * kTcBK, kend = (part + 1) * kb / p.ksplit * kTcBK;
      if (MODE >= 1 && !gu_done) {
        // this expert's h rows: all of its gate/up tiles, four epilogue warps
        // each.  Once the whole gate/up grid is seen finished, no unit waits.
        const int tiles = ((sh ? p.T : __ldcg(p.counts + un.expert)) + kTcBN - 1) / kTcBN;
        const unsigned target = 4u * (sh ? p.mt_gu_s : p.mt_gu) * tiles;
        int w = 1, all = 0;
        if (lane == 0) {
          all = ld_acquire_gpu(p.ready + p.E + 2) >= 4u * p.gu_ctas ? 1 : 0;
          if (!all) w = counter_wait(p.ready + un.expert, target, wc) ? 1 : 0;
          fence_proxy_async_global();          // h was written with plain stores; TMA reads it
        }
        if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
        gu_done = __shfl_sync(0xFFFFFFFFu, all, 0) != 0;
      }
      const int wrows = MODE >= 2 ? 2 * kTcBN : kTcBM;          // weight rows per tile
      const int arow = sh ? un.m_tile * wrows : (MODE == 0 ? un.expert * p.F : un.expert * p.d) + un.m_tile * wrows;
      const CUtensorMap* ma0 = sh ? &p.tm_sa0 : &p.tm_a0;
      const CUtensorMap* ma1 = sh ? &p.tm_sa1 : &p.tm_a1;
      const uint32_t bytes = MODE == 0 ? 2 * kTcBM * 128 + kTcBN * 128 : (uint32_t)C::STAGE_BYTES;
      const CUtensorMap* mb = sh ? &p.tm_sb : &p.tm_b;
      const int brow = (MODE >= 1 && sh) ? p.T * p.k + un.slot0 : un.slot0;
      for (int k0 = kbeg; k0 < kend; k0 += kTcBK) {
        if (!warp_wait(&empty[stage], phase ^ 1, wc)) { ok = false; break; }
        uint8_t* st = stages + stage * C::STAGE_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], bytes);
          // weights are streamed once: evict them first so that the activations,
          // h and the fp32 accumulator stay in L2
          if (MODE >= 2) {
            tma_load_2d(st, mb, k0, brow, &full[stage]);                          // h: 128 slots
            tma_load_2d_hint(st + kTcBM * 128, ma0, k0, arow, &full[stage], pol);  // Wd: 256 rows
          } else {
            tma_load_2d_hint(st, ma0, k0, arow, &full[stage], pol);
            if (MODE == 0) tma_load_2d_hint(st + kTcBM * 128, ma1, k0, arow, &full[stage], pol);
            tma_load_2d(st + (MODE == 0 ? 2 : 1) * kTcBM * 128, mb, k0, brow, &full[stage]);
          }
        }
        __syncwarp();
        issued[stage] = true;
        last_par[stage] = phase;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      for (int i = 0; i < S; ++i)
        if (issued[i]) drain_wait(&full[i], last_par[i], p.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tph[2] = {0, 0};
      int buf = 0;
      int n_total = p.n_pre;
      bool waited = MODE >= 1;
      if (MODE >= 1) n_total = __ldcg(p.n_units + LIST);
      bool ok = true;
      uint64_t* last_commit = nullptr;
      uint32_t last_commit_par = 0;
      UnitCursor cur;
      int u = blockIdx.x;
      for (int it = 0; ok; ++it) {
        TcUnit un;
        if constexpr (MODE == 0) {
          if (it > 0) u += gridDim.x;
          if (u >= n_total) {
            if (waited) break;
            wait_routing();
            waited = true;
            n_total = __ldcg(p.n_units + LIST);
            if (u >= n_total) break;
          }
          un = cur.get(p, u, n_total);
        } else {
          const int slot = it % kRing;
          if (!mbar_wait(&ufull[slot], (it / kRing) & 1, wc)) { ok = false; break; }
          un = ring[slot];
          mbar_arrive(&uempty[slot]);
          if (un.expert < 0) break;
          u = 0;
        }
        const bool sh = un.expert == p.E;
        const int n_pad = (un.n + 15) & ~15;
        const int K = sh ? p.Ks : p.K;
        const uint32_t idesc = MODE >= 2 ? idesc_bf16_f32(kTcBM, 2 * kTcBN) : idesc_bf16_f32(kTcBM, n_pad);
        const int kb = K / kTcBK, part = u % p.ksplit;
        const int kbeg = part * kb / p.ksplit * kTcBK, kend = (part + 1) * kb / p.ksplit * kTcBK;
        if (!mbar_wait(&tempty[buf], tph[buf] ^ 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::ACC_COLS;
        for (int k0 = kbeg; k0 < kend; k0 += kTcBK) {
          if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = smem_u32(stages + stage * C::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < kTcBK / 16; ++kk) {
            const uint32_t accum = (k0 > kbeg || kk > 0) ? 1u : 0u;
            if (MODE == 0) {
              const uint64_t bd = sdesc_sw128(st + 2 * kTcBM * 128 + kk * 32);
              tc_mma_f16(acc, sdesc_sw128(st + kk * 32), bd, idesc, accum);
              tc_mma_f16(acc + kTcBN, sdesc_sw128(st + kTcBM * 128 + kk * 32), bd, idesc, accum);
            } else {   // MODE 1: A = Wd rows, B = h; MODES 2, 3: A = h, B = Wd rows
              tc_mma_f16(acc, sdesc_sw128(st + kk * 32), sdesc_sw128(st + kTcBM * 128 + kk * 32), idesc, accum);
            }
          }
          tc_commit(&empty[stage]);
          last_commit = &empty[stage];
          last_commit_par = phase;
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
        tph[buf] ^= 1;
        buf ^= 1;
      }
      if (!ok && last_commit) drain_wait(last_commit, last_commit_par, p.wait_ns);
    } else if (MODE == 0) {
      wait_routing();                         // the idle lanes trigger too
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int ept = threadIdx.x - 64;        // 0..127
    if (MODE == 0) {
      // clear the fp32 accumulator of pass 2 (x-independent, needs no routing).
      // Safe ahead of the grid-dependency wait: every call starts with a router
      // that lets its dependents launch only after the previous kernel on the
      // stream has completed, so no kernel of an earlier call is still running.
      float4* ya = reinterpret_cast<float4*>(p.yacc);
      const size_t n4 = (size_t)p.T * p.d / 4;
      for (size_t i = (size_t)blockIdx.x * 128 + ept; i < n4; i += (size_t)gridDim.x * 128)
        ya[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(p.ready + p.E + 1, 1u);
      }
    }
    uint32_t tph[2] = {0, 0};
    int buf = 0;
    int n_total = p.n_pre;
    bool waited = MODE >= 1;
    if (MODE >= 1) n_total = __ldcg(p.n_units + LIST);
    UnitCursor cur;
    int u = blockIdx.x;
    for (int it = 0;; ++it) {
      TcUnit un;
      if constexpr (MODE == 0) {
        if (it > 0) u += gridDim.x;
        if (u >= n_total) {
          if (waited) break;
          wait_routing();
          waited = true;
          n_total = __ldcg(p.n_units + LIST);
          if (u >= n_total) break;
        }
        un = cur.get(p, u, n_total);
      } else {
        const int slot = it % kRing;
        if (!warp_wait(&ufull[slot], (it / kRing) & 1, wc)) break;
        un = ring[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&uempty[slot]);
        if (un.expert < 0) break;
        u = 0;
      }
      const bool sh = un.expert == p.E;
      const int n_pad = (un.n + 15) & ~15;
      if (MODE == 1) {
        // token and gate of every column of this tile, loaded once per warp into
        // its own shared-memory table (no cross-warp barrier to get stuck on)
        __syncwarp();
        for (int c = lane; c < un.n; c += 32) {
          int t;
          float g;
          if (sh) {
            t = un.slot0 + c;
            g = 1.f;
          } else {
            const int src = __ldcg(p.src_of_slot + un.slot0 + c);
            t = src / p.k;
            g = __ldcg(p.gate + src);
          }
          col_tok[q * kTcBN + c] = t;
          col_gate[q * kTcBN + c] = g;
        }
        __syncwarp();
      }
      if (MODE >= 2) {
        // this thread's slot (row of the tile): token and gate, once per tile
        const int r = q * 32 + lane;
        int t = 0;
        float g = 0.f;
        if (r < un.n) {
          if (sh) {
            t = un.slot0 + r;
            g = 1.f;
          } else {
            const int src = __ldcg(p.src_of_slot + un.slot0 + r);
            t = src / p.k;
            g = __ldcg(p.gate + src);
          }
        }
        if (!warp_wait(&tfull[buf], tph[buf], wc)) break;
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::ACC_COLS + ((uint32_t)(q * 32) << 16);
        float* yrow = p.yacc + (size_t)t * p.d + un.m_tile * (2 * kTcBN);
        {
          // 16-byte red operations, each warp instruction on 4 rows x 128
          // contiguous bytes: every 32 x 32 chunk of the warp's rows goes
          // through its own shared-memory tile, after which lane l adds
          // columns 4 (l % 8) .. + 3 of rows 4 j + l / 8 (one red instruction
          // on one row each would touch 32 rows x 16 bytes).
          (void)yrow;
          float* tile = red_stage + (size_t)q * 32 * kTpPitch;
          const int tcol = (lane & 7) * 4;
          // accumulate mode: rows of y_acc (tokens); deterministic mode: this
          // tile's rows of the per-slot buffer, each stored once
          const int orow = p.oslot ? (sh ? p.T * p.k : 0) + un.slot0 + r : t;
          int tok[8];
          unsigned valid = 0;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rr = 4 * j + (lane >> 3);
            tok[j] = __shfl_sync(0xFFFFFFFFu, orow, rr);
            if (q * 32 + rr < un.n) valid |= 1u << j;
          }
          float* ybase = (p.oslot ? p.oslot : p.yacc) + (size_t)un.m_tile * (2 * kTcBN) + tcol;
#pragma unroll 1
          for (int c0 = 0; c0 < 2 * kTcBN; c0 += 32) {
            uint32_t v0[16], v1[16];
            tmem_ld16(acc + c0, v0);
            tmem_ld16(acc + c0 + 16, v1);
            tmem_ld_wait();
            float4* trow = reinterpret_cast<float4*>(tile + lane * kTpPitch);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              trow[i] = make_float4(g * __uint_as_float(v0[4 * i]), g * __uint_as_float(v0[4 * i + 1]),
                                    g * __uint_as_float(v0[4 * i + 2]), g * __uint_as_float(v0[4 * i + 3]));
              trow[4 + i] = make_float4(g * __uint_as_float(v1[4 * i]), g * __uint_as_float(v1[4 * i + 1]),
                                        g * __uint_as_float(v1[4 * i + 2]), g * __uint_as_float(v1[4 * i + 3]));
            }
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (valid & (1u << j)) {
                const float4 x = *reinterpret_cast<const float4*>(tile + (4 * j + (lane >> 3)) * kTpPitch + tcol);
                float* dst = ybase + (size_t)tok[j] * p.d + c0;
                if (p.oslot)
                  __stcg(reinterpret_cast<float4*>(dst), x);
                else
                  red_add_v4_f32(dst, x.x, x.y, x.z, x.w);
              }
            }
            __syncwarp();
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[buf]);
        tph[buf] ^= 1;
        buf ^= 1;
        continue;
      }
      if (!warp_wait(&tfull[buf], tph[buf], wc)) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * C::ACC_COLS + ((uint32_t)(q * 32) << 16);
      const int row = un.m_tile * kTcBM + q * 32 + lane;
      if (MODE == 0 && p.ksplit > 1) {
        // one part of a split tile: store the partial sums of this warp's rows
        const int part = u % p.ksplit, brow = sh ? p.T * p.k + un.slot0 : un.slot0;
        for (int c0 = 0; c0 < n_pad; c0 += 16) {
          uint32_t g[16], v[16];
          tmem_ld16(acc + c0, g);
          tmem_ld16(acc + kTcBN + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c0 + i;
            if (col < un.n) {
              float* pp = p.gu_part + ((size_t)(part * p.P + brow + col) * 2) * p.Fmax + row;
              pp[0] = __uint_as_float(g[i]);
              pp[p.Fmax] = __uint_as_float(v[i]);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[buf]);
        tph[buf] ^= 1;
        buf ^= 1;
        // the last part to arrive adds the parts in order and writes h
        unsigned int* cnt = p.gu_cnt + (size_t)(u / p.ksplit) * 4 + q;
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence();
          last = atomicAdd(cnt, 1u) == (unsigned)p.ksplit - 1 ? 1 : 0;
          if (last) __threadfence();
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        __syncwarp();
        if (last) {
          for (int col = 0; col < un.n; ++col) {
            // all parts' loads issued together, then added in part order
            float pa[kMaxKSplit], pb[kMaxKSplit];
#pragma unroll
            for (int pt = 0; pt < kMaxKSplit; ++pt) {
              pa[pt] = pb[pt] = 0.f;
              if (pt < p.ksplit) {
                const float* pp = p.gu_part + ((size_t)(pt * p.P + brow + col) * 2) * p.Fmax + row;
                pa[pt] = __ldcg(pp);
                pb[pt] = __ldcg(pp + p.Fmax);
              }
            }
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int pt = 0; pt < kMaxKSplit; ++pt) {
              a += pa[pt];
              b += pb[pt];
            }
            const float h = a / (1.f + __expf(-a)) * b;
            p.h16[(size_t)(brow + col) * p.Fmax + row] = __float2bfloat16_rn(h);
          }
          __syncwarp();
          if (lane == 0) {
            *cnt = 0;                                 // ready for the next call
            __threadfence();
            atomicAdd(p.ready + un.expert, 1u);
          }
        }
        continue;
      }
      for (int c0 = 0; c0 < n_pad; c0 += 16) {
        if (MODE == 0) {
          uint32_t g[16], v[16];
          tmem_ld16(acc + c0, g);
          tmem_ld16(acc + kTcBN + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c0 + i;
            if (col < un.n) {
              const float a = __uint_as_float(g[i]);
              const float h = a / (1.f + __expf(-a)) * __uint_as_float(v[i]);
              const int hs = sh ? p.T * p.k + un.slot0 + col : un.slot0 + col;
              p.h16[(size_t)hs * p.Fmax + row] = __float2bfloat16_rn(h);
            }
          }
        } else {
          uint32_t v[16];
          tmem_ld16(acc + c0, v);
          tmem_ld_wait();
          const int* ct = col_tok + q * kTcBN;
          const float* cg = col_gate + q * kTcBN;
          if (p.oslot) {                       // fixed order: each (slot, row) stored once
            const int s0 = sh ? p.T * p.k + un.slot0 : un.slot0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + i;
              if (col < un.n) __stcg(p.oslot + (size_t)(s0 + col) * p.d + row, cg[col] * __uint_as_float(v[i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + i;
              if (col < un.n) red_add_f32(p.yacc + (size_t)ct[col] * p.d + row, cg[col] * __uint_as_float(v[i]));
            }
          }
        }
      }
      if (MODE == 0) {
        // this warp's rows of the tile are in h: publish them to the down pass
        __syncwarp();
        if (lane == 0) {
          __threadfence();
          atomicAdd(p.ready + un.expert, 1u);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
      tph[buf] ^= 1;
      buf ^= 1;
    }
    if (MODE == 0) {
      // all of this warp's tiles are published
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(p.ready + p.E + 2, 1u);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Slot-ordered copy of the routed tokens' activations, xp[slot] = x[token of
// slot], one warp per slot.  After a large-batch router (wpb > 0) the warp
// also places the slot: it computes the grouped position of slot s = (t, j)
// from the selection bitmap and writes tok_of_slot, src_of_slot and slot_of.
// First the grid writes the unit lists of both passes.
__global__ void __launch_bounds__(256) tc_gather_kernel(const __nv_bfloat16* __restrict__ x,
                                                        const int32_t* __restrict__ idx, Workspace ws, int T,
                                                        int E, int k, int d, int wpb, UnitBuild ub) {
  pdl_launch_dependents();
  pdl_wait();
  build_unit_lists(ws, ub);
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  const int per_row = d / 8;                       // 16-byte pieces per row
  for (int s = gw; s < T * k; s += nw) {
    int pos, t;
    if (wpb > 0) {
      t = s / k;
      pos = slot_position(ws, E, t, __ldg(idx + s), wpb);
      if (lane == 0) {
        ws.tok_of_slot[pos] = t;
        ws.src_of_slot[pos] = s;
        ws.slot_of[s] = pos;
      }
    } else {
      pos = s;
      t = __ldg(ws.tok_of_slot + s);
    }
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    uint4* dst = reinterpret_cast<uint4*>(ws.xp + (size_t)pos * d);
    // eight 16-byte loads in flight per lane before the stores
    for (int c0 = 0; c0 < per_row; c0 += 256) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + 32 * i + lane < per_row) v[i] = __ldg(src + c0 + 32 * i + lane);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (c0 + 32 * i + lane < per_row) dst[c0 + 32 * i + lane] = v[i];
    }
  }
}

// y = bf16(y_acc (+ x)), 8 values per thread.  Also returns the gate/up
// readiness counters to zero for the next call (the down pass, which reads
// them, has completed).
__global__ void __launch_bounds__(256) tc_finalize_kernel(const float* __restrict__ yacc,
                                                          const __nv_bfloat16* __restrict__ x,
                                                          __nv_bfloat16* __restrict__ y, size_t n8, int residual,
                                                          unsigned int* ready, int n_ready) {
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_ready; i += blockDim.x) ready[i] = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(yacc) + 2 * i);
    const float4 b = __ldcg(reinterpret_cast<const float4*>(yacc) + 2 * i + 1);
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (residual) {
      const uint4 xr = __ldg(reinterpret_cast<const uint4*>(x) + i);
      const uint32_t xs[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] += __uint_as_float(xs[j] << 16);
        v[2 * j + 1] += __uint_as_float(xs[j] & 0xFFFF0000u);
      }
    }
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      op[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    reinterpret_cast<uint4*>(y)[i] = o;
  }
}

// Deterministic mode: y[t] = bf16(sum over j < k of oslot[slot_of[t k + j]] (selection
// order) + oslot[T k + t] (the shared expert) (+ x[t])), 8 values per thread.
__global__ void __launch_bounds__(256) tc_finalize_det_kernel(const float* __restrict__ oslot,
                                                              const int32_t* __restrict__ slot_of,
                                                              const __nv_bfloat16* __restrict__ x,
                                                              __nv_bfloat16* __restrict__ y, int T, int d, int k,
                                                              int has_shared, int residual, unsigned int* ready,
                                                              int n_ready) {
  pdl_launch_dependents();
  pdl_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_ready; i += blockDim.x) ready[i] = 0;
  const int per = d / 8;
  const size_t n8 = (size_t)T * per;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / per), c = (int)(i % per) * 8;
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    auto add_row = [&](size_t r) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(oslot + r * d + c));
      const float4 b = __ldcg(reinterpret_cast<const float4*>(oslot + r * d + c) + 1);
      v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w; v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    };
    for (int j = 0; j < k; ++j) add_row((size_t)__ldcg(slot_of + (size_t)t * k + j));
    if (has_shared) add_row((size_t)T * k + t);
    if (residual) {
      const uint4 xr = __ldg(reinterpret_cast<const uint4*>(x) + i);
      const uint32_t xs[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] += __uint_as_float(xs[j] << 16);
        v[2 * j + 1] += __uint_as_float(xs[j] & 0xFFFF0000u);
      }
    }
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      op[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    reinterpret_cast<uint4*>(y)[i] = o;
  }
}

template <int MODE>
size_t tc_smem_bytes() {
  using C = TcCfg<MODE>;
  return 1024 + C::STAGES * C::STAGE_BYTES + TcStaging<MODE>::BYTES + (2 * C::STAGES + 4) * 8 + 16 + 8 * kTcBN * 4 +
         kRing * (16 + sizeof(TcUnit));
}

template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                      Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace

int tc_max_units_gu(int T, int d, int F, int Fs, int E, int k, int tile_n) {
  (void)d;
  const long long routed = (long long)(F / kTcBM) * ((long long)T * k / tile_n + E);
  const long long shared = (long long)(Fs / kTcBM) * ((T + tile_n - 1) / tile_n);
  return (int)(routed + shared);
}
int tc_max_units_dn(int T, int d, int F, int Fs, int E, int k, int tile_n) {
  (void)F;
  const long long routed = (long long)(d / kTcBM) * ((long long)T * k / tile_n + E);
  const long long shared = Fs > 0 ? (long long)(d / kTcBM) * ((T + tile_n - 1) / tile_n) : 0;
  return (int)(routed + shared);
}

cudaError_t launch_tc_finalize(const Workspace& ws, const void* x, void* y, int T, int d, int k, bool has_shared,
                               bool residual, unsigned int* ready, int n_ready, int num_sms, cudaStream_t s,
                               Prof* prof) {
  const size_t n8 = (size_t)T * d / 8;
  const int grid = (int)((n8 + 255) / 256 < (size_t)num_sms * 4 ? (n8 + 255) / 256 : (size_t)num_sms * 4);
  if (prof) prof->begin(MOE_K_TC_FINALIZE, s);
  const cudaError_t e =
      ws.oslot ? launch_ex(tc_finalize_det_kernel, grid > 0 ? grid : 1, 256, 0, s, (const float*)ws.oslot,
                           (const int32_t*)ws.slot_of, static_cast<const __nv_bfloat16*>(x),
                           static_cast<__nv_bfloat16*>(y), T, d, k, (int)has_shared, (int)residual, ready, n_ready)
               : launch_ex(tc_finalize_kernel, grid > 0 ? grid : 1, 256, 0, s, (const float*)ws.yacc,
                           static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), n8,
                           (int)residual, ready, n_ready);
  if (prof) prof->end(s);
  return e;
}

cudaError_t launch_tc(const TcArgs& a, int num_sms, cudaStream_t s, Prof* prof) {
  {
    cudaError_t e = ensure_smem_limit(tc_kernel<0>, (int)tc_smem_bytes<0>());
    if (e == cudaSuccess) e = ensure_smem_limit(tc_kernel<1>, (int)tc_smem_bytes<1>());
    if (e == cudaSuccess) e = ensure_smem_limit(tc_kernel<2>, (int)tc_smem_bytes<2>());
    if (e != cudaSuccess) return e;
  }
  const int Fmax = a.F > a.Fs ? a.F : a.Fs;
  TcParams p;
  p.T = a.T; p.d = a.d; p.F = a.F; p.Fs = a.Fs; p.E = a.E; p.k = a.k; p.Fmax = Fmax;
  p.tok_of_slot = a.ws.tok_of_slot;
  p.src_of_slot = a.ws.src_of_slot;
  p.gate = a.gate;
  p.h16 = a.ws.h16;
  p.yacc = a.ws.yacc;
  p.oslot = a.ws.oslot;
  p.err = a.ws.err;
  p.wait_ns = a.wait_ns;
  p.n_units = a.ws.n_units;
  p.ready = a.ws.ready;
  p.counts = a.ws.counts;
  p.ksplit = a.gu_split;
  p.P = a.T * (a.k + 1);
  p.gu_part = a.ws.gu_part;
  p.gu_cnt = a.ws.gu_cnt;
  p.mt_gu = a.F / kTcBM;
  p.mt_gu_s = a.Fs > 0 ? a.Fs / kTcBM : 1;
  p.sched = nullptr;
  // slot-ordered copy of the routed activations
  const int slots = a.T * a.k;
  const int gg = (slots + 7) / 8 < num_sms * 8 ? (slots + 7) / 8 : num_sms * 8;   // 8 warps per block
  UnitBuild ub;
  ub.E = a.E; ub.T = a.T; ub.tn = kTcBN;
  ub.sh_tb = a.Fs > 0 ? (a.T + kTcBN - 1) / kTcBN : 0;
  ub.mt[0] = a.F / kTcBM; ub.mt[1] = a.d / a.dn_rows;
  ub.sh_mt[0] = a.Fs > 0 ? a.Fs / kTcBM : 0; ub.sh_mt[1] = a.d / a.dn_rows;
  ub.rep[0] = a.gu_split; ub.rep[1] = 1;
  if (prof) prof->begin(MOE_K_TC_GATHER, s);
  cudaError_t e = launch_ex(tc_gather_kernel, gg > 0 ? gg : 1, 256, 0, s, static_cast<const __nv_bfloat16*>(a.x),
                            a.idx, a.ws, a.T, a.E, a.k, a.d, a.wpb, ub);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  // pass 1: gate/up
  p.tm_a0 = *a.tm_wg; p.tm_a1 = *a.tm_wu;
  if (a.Fs > 0) { p.tm_sa0 = *a.tm_sg; p.tm_sa1 = *a.tm_su; } else { p.tm_sa0 = *a.tm_wg; p.tm_sa1 = *a.tm_wu; }
  p.tm_b = *a.tm_xp;
  p.tm_sb = *a.tm_x;
  p.K = a.d; p.Ks = a.d;
  p.mt = a.F / kTcBM;
  p.mt_s = a.Fs > 0 ? a.Fs / kTcBM : 1;
  p.n_pre = a.Fs > 0 ? a.gu_split * (a.Fs / kTcBM) * ((a.T + kTcBN - 1) / kTcBN) : 0;
  p.units = a.ws.units_gu;
  const int grid1 = num_sms < a.max_units_gu ? num_sms : (a.max_units_gu > 0 ? a.max_units_gu : 1);
  p.gu_ctas = grid1;
  if (prof) prof->begin(MOE_K_TC_GATEUP, s);
  e = launch_ex(tc_kernel<0>, grid1, kThreadsTc, tc_smem_bytes<0>(), s, p);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  // pass 2: down
  const bool tok_major = a.dn_rows == 2 * kTcBN;
  const CUtensorMap* wd = tok_major ? a.tm_wd256 : a.tm_wd;
  const CUtensorMap* sd = tok_major ? a.tm_sd256 : a.tm_sd;
  p.tm_a0 = *wd; p.tm_a1 = *wd;
  p.tm_sa0 = a.Fs > 0 ? *sd : *wd; p.tm_sa1 = p.tm_sa0;
  p.tm_b = *a.tm_h;
  p.tm_sb = *a.tm_h;
  p.K = a.F; p.Ks = a.Fs > 0 ? a.Fs : a.F;
  p.mt = a.d / a.dn_rows;
  p.mt_s = a.d / a.dn_rows;
  p.n_pre = 0;
  p.ksplit = 1;
  p.sched = a.ws.ready + a.E + 3;
  p.units = a.ws.units_dn;
  const int grid2 = num_sms < a.max_units_dn ? num_sms : (a.max_units_dn > 0 ? a.max_units_dn : 1);
  if (prof) prof->begin(MOE_K_TC_DOWN, s);
  if (tok_major)
    e = launch_ex(tc_kernel<2>, grid2, kThreadsTc, tc_smem_bytes<2>(), s, p);
  else
    e = launch_ex(tc_kernel<1>, grid2, kThreadsTc, tc_smem_bytes<1>(), s, p);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  // finalise
  return launch_tc_finalize(a.ws, a.x, a.y, a.T, a.d, a.k, a.Fs > 0, a.add_residual != 0, a.ws.ready, a.E + 4,
                            num_sms, s, prof);
}

}  // namespace moe
