// Grouped expert GEMMs with NVFP4 weights on the 5th-generation tensor cores.
//
// NVFP4 (evermx.com review, section "Quantization") stores each weight as an
// e2m1 code with one e4m3 scale per 16 values along K and one fp32 scale per
// matrix.  The tensor cores have no instruction for fp4 weights times 16-bit
// activations, so the codes are decoded on the way in: q * s_b is exact in
// f16 (at most 6 significant bits, magnitudes 2^-10 .. 2688), so
// cvt.rn.f16x2.e2m1x2 followed by one f16x2 multiply by the block scale gives
// the weight exactly, and the MMA (kind::f16, f16 A and B, fp32 accumulate)
// takes A straight from tensor memory.  Decoding into tensor memory rather
// than shared memory keeps the shared-memory traffic near one byte per weight
// (the fp4 codes in, read once); a bf16 copy in shared memory would need
// about five, more than the SM's shared-memory bandwidth at the HBM rate.
//
// Activations on the f16 side: every row of the slot-ordered copy is scaled
// by a power of two 2^-e (its largest magnitude into [1, 2)), so the f16 copy
// is exact for every value above 2^-14 of the row maximum, and the scale
// xs = 2^e is applied to the fp32 result.  The intermediate h is stored in f16
// as h / xs^2 (also exact rescaling): its range then depends on the weights,
// not on the activations' magnitude.  A value that would overflow f16
// saturates and sets the range bit of the error word.
//
// Per unit (128 weight rows x up to 64 tokens), per stage of 256 K values:
// TMA brings the codes (16 KB per matrix, 128-byte swizzle), the block scales
// (2 KB per matrix) and the activation rows (f16, 16-row boxes, only as many
// as the tile has tokens).  Four converter warps (one per TMEM lane quarter)
// decode 64 (pass 1) or 128 (pass 2) K values at a time into a double-buffered
// A area of tensor memory
// (tcgen05.st), one thread issues the MMAs, four epilogue warps drain the
// double-buffered accumulators:
//  * pass 1 (gate/up): h = silu(a) * u with a = D_g s_g xs, u = D_u s_u xs;
//  * pass 2 (down): y_acc[t][row] += gate * s_d * xs^2 * D (red.global.add);
//  * finalise: y = bf16(y_acc (+ x)) (shared with the bf16 path).
#include <cuda_fp16.h>

#include <utility>

#include "moe_internal.cuh"
#include "ptx.cuh"
#include "units.cuh"

namespace moe {
namespace {

constexpr int kThreads4 = 320;                  // producer, MMA, 4 epilogue warps, 4 converter warps
constexpr int kBoxK = 64;                       // K values per activation-row box (128 bytes of f16)
constexpr int kBRows = 16;                      // activation rows per TMA box
constexpr int kBoxPerStage = kTc4KS / kBoxK;    // 4

template <int MODE> struct Tc4Cfg;
template <> struct Tc4Cfg<0> {                  // gate/up
  static constexpr int NMAT = 2;
  static constexpr int STAGES = 3;
  static constexpr int A_BYTES = 128 * kTc4KS / 2;            // codes per matrix
  static constexpr int S_BYTES = 128 * kTc4KS / 16;           // block scales per matrix
  static constexpr int B_BYTES = kBoxPerStage * kTc4BN * 128; // activation rows
  static constexpr int B_OFF = NMAT * A_BYTES;
  static constexpr int S_OFF = B_OFF + B_BYTES;
  static constexpr int STAGE_BYTES = S_OFF + NMAT * S_BYTES;
  static constexpr int ACC_COLS = NMAT * kTc4BN;              // per accumulator buffer
  static constexpr int SUB = 64;                              // K values converted per A buffer
  static constexpr int A_COLS = NMAT * SUB / 2;               // per A buffer
  static constexpr int TMEM_COLS = 512;
};
template <> struct Tc4Cfg<1> {                  // down
  static constexpr int NMAT = 1;
  static constexpr int STAGES = 4;
  static constexpr int A_BYTES = 128 * kTc4KS / 2;
  static constexpr int S_BYTES = 128 * kTc4KS / 16;
  static constexpr int B_BYTES = kBoxPerStage * kTc4BN * 128;
  static constexpr int B_OFF = NMAT * A_BYTES;
  static constexpr int S_OFF = B_OFF + B_BYTES;
  static constexpr int STAGE_BYTES = S_OFF + NMAT * S_BYTES;
  static constexpr int ACC_COLS = NMAT * kTc4BN;
  // one matrix: its 4 MMAs per 64 values finish quickly, so each converter
  // hand-off carries twice as much to halve the hand-offs per stage
  static constexpr int SUB = 128;
  static constexpr int A_COLS = NMAT * SUB / 2;
  static constexpr int TMEM_COLS = 256;
};
static_assert(Tc4Cfg<0>::STAGE_BYTES % 1024 == 0 && Tc4Cfg<1>::STAGE_BYTES % 1024 == 0, "stage alignment");
static_assert(2 * Tc4Cfg<0>::ACC_COLS + 2 * Tc4Cfg<0>::A_COLS <= Tc4Cfg<0>::TMEM_COLS, "tensor memory budget");
static_assert(2 * Tc4Cfg<1>::ACC_COLS + 2 * Tc4Cfg<1>::A_COLS <= Tc4Cfg<1>::TMEM_COLS, "tensor memory budget");

struct Tc4Params {
  CUtensorMap q[2], sc[2];      // routed codes / block scales (pass 1: gate, up; pass 2: down)
  CUtensorMap sq[2], ssc[2];    // shared expert
  CUtensorMap tm_b;             // B rows: pass 1 f16 activations, pass 2 f16 h
  const float* ts[2];           // routed per-matrix scales [E]
  const float* tss[2];          // shared per-matrix scales [1]
  const float* xs;              // [rows of xp] power-of-two activation scales
  int T, E, k, d, Fmax;
  int rows_e;                   // weight rows per routed expert (pass 1: F, pass 2: d)
  int K, Ks;                    // reduction width, routed / shared
  int mt_s;                     // shared-expert weight-row tiles
  int n_pre;                    // units that need no routing (shared expert, pass 1)
  const int32_t* src_of_slot;
  const float* gate;
  const TcUnit* units;
  const int32_t* n_units;
  __half* h16;
  float* yacc;
  float* oslot;               // deterministic mode: per-slot rows [T (k + 1)][d] instead of y_acc, or null
  unsigned int* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ TcUnit get_unit4(const Tc4Params& p, int u) {
  if (u < p.n_pre) {
    const int tb = u / p.mt_s, m = u % p.mt_s;
    return TcUnit{p.E, m, tb * kTc4BN, min(kTc4BN, p.T - tb * kTc4BN)};
  }
  return p.units[u];
}

// The unit sequence every role of a CTA walks: n_pre units that need no
// routing, then (after the grid-dependency wait) the routed list.
struct UnitWalk {
  int u, n_total;
  bool waited;
  __device__ UnitWalk(const Tc4Params& p, int list, bool wait_first) : u(blockIdx.x), waited(wait_first) {
    n_total = wait_first ? __ldcg(p.n_units + list) : p.n_pre;
  }
  // Returns false when the sequence is over.  `before_wait` runs once, just
  // ahead of the grid-dependency wait.
  template <typename F>
  __device__ bool next(const Tc4Params& p, int list, F&& before_wait) {
    if (u < n_total) return true;
    if (waited) return false;
    before_wait();
    pdl_wait();
    waited = true;
    n_total = __ldcg(p.n_units + list);
    return u < n_total;
  }
};

template <int MODE>
__global__ void __launch_bounds__(kThreads4, 1) tc4_kernel(const __grid_constant__ Tc4Params p) {
  using C = Tc4Cfg<MODE>;
  constexpr int S = C::STAGES, NM = C::NMAT;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = dsm;
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + S * C::STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* afull = empty + S;      // [2] converted A buffer ready
  uint64_t* aempty = afull + 2;     // [2] converted A buffer consumed by the MMAs
  uint64_t* tfull = aempty + 2;     // [2] accumulator ready
  uint64_t* tempty = tfull + 2;     // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* col_tok = abort_flag + 3;                                   // [4 warps][kTc4BN]
  float* col_f = reinterpret_cast<float*>(col_tok + 4 * kTc4BN);   // [4 warps][kTc4BN]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&afull[i], 128);
      mbar_init(&aempty[i], 1);
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int m = 0; m < NM; ++m) {
      tma_prefetch_desc(&p.q[m]);
      tma_prefetch_desc(&p.sc[m]);
    }
    tma_prefetch_desc(&p.tm_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_a = tmem + 2 * C::ACC_COLS;   // converted A buffers
  pdl_launch_dependents();
  const WaitCtl wc{p.wait_ns, p.err, abort_flag};
  constexpr bool kWaitFirst = MODE == 1;
  if (kWaitFirst) pdl_wait();
  auto nothing = [] {};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t last_par[S];
    bool issued[S];
    for (int i = 0; i < S; ++i) issued[i] = false;
    bool ok = true;
    for (UnitWalk w(p, MODE, kWaitFirst); ok && w.next(p, MODE, nothing); w.u += gridDim.x) {
      const TcUnit un = get_unit4(p, w.u);
      const bool sh = un.expert == p.E;
      const int K = sh ? p.Ks : p.K;
      const int arow = (sh ? 0 : un.expert * p.rows_e) + un.m_tile * 128;
      const int brow = sh ? p.T * p.k + un.slot0 : un.slot0;
      const int nbox = (un.n + kBRows - 1) / kBRows;
      const uint32_t bytes = NM * (C::A_BYTES + C::S_BYTES) + kBoxPerStage * nbox * kBRows * 128;
      for (int k0 = 0; k0 < K; k0 += kTc4KS) {
        if (!warp_wait(&empty[stage], phase ^ 1, wc)) { ok = false; break; }
        uint8_t* st = stages + stage * C::STAGE_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
          for (int m = 0; m < NM; ++m) {
            tma_load_2d_hint(st + m * C::A_BYTES, sh ? &p.sq[m] : &p.q[m], k0 / 2, arow, &full[stage], pol);
            tma_load_2d_hint(st + C::S_OFF + m * C::S_BYTES, sh ? &p.ssc[m] : &p.sc[m], k0 / 16, arow,
                             &full[stage], pol);
          }
          for (int j = 0; j < kBoxPerStage; ++j)
            for (int rb = 0; rb < nbox; ++rb)
              tma_load_2d(st + C::B_OFF + j * (kTc4BN * 128) + rb * (kBRows * 128), &p.tm_b, k0 + j * kBoxK,
                          brow + rb * kBRows, &full[stage]);
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
      uint32_t phase = 0, tph[2] = {0, 0};
      int buf = 0, g = 0;
      bool ok = true;
      uint64_t* last_commit = nullptr;
      uint32_t last_commit_par = 0;
      for (UnitWalk w(p, MODE, kWaitFirst); ok && w.next(p, MODE, nothing); w.u += gridDim.x) {
        const TcUnit un = get_unit4(p, w.u);
        const bool sh = un.expert == p.E;
        const int K = sh ? p.Ks : p.K;
        const uint32_t idesc = idesc_f16_f32(128, (un.n + 15) & ~15);
        if (!mbar_wait(&tempty[buf], tph[buf] ^ 1, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + buf * C::ACC_COLS;
        for (int k0 = 0; k0 < K && ok; k0 += kTc4KS) {
          if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
          const uint32_t sb = smem_u32(stages + stage * C::STAGE_BYTES + C::B_OFF);
          for (int j = 0; j < kTc4KS / C::SUB; ++j, ++g) {
            const int ab = g & 1;
            if (!mbar_wait(&afull[ab], (g >> 1) & 1, wc)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < C::SUB / 16; ++kk) {
              // values j SUB + 16 kk .. + 15: box (j SUB + 16 kk) / 64 of the stage, 32 bytes per 16 values
              const int kv = j * C::SUB + kk * 16;
              const uint64_t bd = sdesc_sw128(sb + (kv / kBoxK) * (kTc4BN * 128) + (kv % kBoxK) * 2);
              const uint32_t accum = (k0 > 0 || kv > 0) ? 1u : 0u;
#pragma unroll
              for (int m = 0; m < NM; ++m)
                tc_mma_f16_ts(acc + m * kTc4BN, tmem_a + ab * C::A_COLS + m * (C::SUB / 2) + kk * 8, bd, idesc, accum);
            }
            tc_commit(&aempty[ab]);
            last_commit = &aempty[ab];
            last_commit_par = (g >> 1) & 1;
          }
          if (!ok) break;
          tc_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
        tph[buf] ^= 1;
        buf ^= 1;
      }
      if (!ok && last_commit) drain_wait(last_commit, last_commit_par, p.wait_ns);
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ converters (warps 6-9)
    const int q = warp & 3;                  // TMEM lane quarter
    const int r = q * 32 + lane;             // row of the 128-row weight tile
    int stage = 0, g = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (UnitWalk w(p, MODE, kWaitFirst); ok && w.next(p, MODE, nothing); w.u += gridDim.x) {
      const TcUnit un = get_unit4(p, w.u);
      const int K = un.expert == p.E ? p.Ks : p.K;
      for (int k0 = 0; k0 < K; k0 += kTc4KS) {
        if (!warp_wait(&full[stage], phase, wc)) { ok = false; break; }
        const uint8_t* st = stages + stage * C::STAGE_BYTES;
        for (int j = 0; j < kTc4KS / C::SUB; ++j, ++g) {
          const int ab = g & 1;
          if (!warp_wait(&aempty[ab], ((g >> 1) & 1) ^ 1, wc)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int m = 0; m < NM; ++m) {
#pragma unroll
            for (int c64 = 0; c64 < C::SUB / 64; ++c64) {
              // this row's 64 codes of values 64 q64 .. + 63 (q64 = j SUB / 64 + c64
              // of the stage): 16-byte pieces 2 q64 and 2 q64 + 1, stored at
              // piece ^ (r % 8) by the 128-byte swizzle
              const int q64 = j * (C::SUB / 64) + c64;
              const uint8_t* rowp = st + m * C::A_BYTES + r * 128;
              const uint4 c0 = *reinterpret_cast<const uint4*>(rowp + (((2 * q64) ^ (r & 7)) << 4));
              const uint4 c1 = *reinterpret_cast<const uint4*>(rowp + (((2 * q64 + 1) ^ (r & 7)) << 4));
              const uint32_t sw =
                  *reinterpret_cast<const uint32_t*>(st + C::S_OFF + m * C::S_BYTES + r * 16 + 4 * q64);
              uint32_t s01, s23;
              e4m3x4_f16x2(sw, s01, s23);
              const uint32_t sb4[4] = {dup_lo(s01), dup_hi(s01), dup_lo(s23), dup_hi(s23)};
              const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
              uint32_t v[32];
#pragma unroll
              for (int i = 0; i < 8; ++i) {          // word i: codes 8i .. 8i + 7, block i / 2
                uint32_t h[4];
                e2m1x8_f16x2(cw[i], h);
#pragma unroll
                for (int c = 0; c < 4; ++c) v[4 * i + c] = hmul2(h[c], sb4[i >> 1]);
              }
              tmem_st32(tmem_a + ((uint32_t)(q * 32) << 16) + ab * C::A_COLS + m * (C::SUB / 2) + c64 * 32, v);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&afull[ab]);
        }
        if (!ok) break;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;
    if (MODE == 0) {
      // clear the fp32 accumulator of pass 2 (x-independent, needs no routing).
      // Safe ahead of the grid-dependency wait: every call starts with a router
      // that lets its dependents launch only after the previous kernel on the
      // stream has completed, so no kernel of an earlier call is still running.
      const int ept = threadIdx.x - 64;
      float4* ya = reinterpret_cast<float4*>(p.yacc);
      const size_t n4 = (size_t)p.T * p.d / 4;
      for (size_t i = (size_t)blockIdx.x * 128 + ept; i < n4; i += (size_t)gridDim.x * 128)
        ya[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int* ct = col_tok + q * kTc4BN;
    float* cf = col_f + q * kTc4BN;
    uint32_t tph[2] = {0, 0};
    int buf = 0;
    bool range_bad = false;
    for (UnitWalk w(p, MODE, kWaitFirst); w.next(p, MODE, nothing); w.u += gridDim.x) {
      const TcUnit un = get_unit4(p, w.u);
      const bool sh = un.expert == p.E;
      const int brow = sh ? p.T * p.k + un.slot0 : un.slot0;
      // per-column tables of this warp: pass 1 the activation scale, pass 2
      // the token and gate * s_d * xs^2
      __syncwarp();
      const float tsd = MODE == 1 ? (sh ? __ldg(p.tss[0]) : __ldg(p.ts[0] + un.expert)) : 0.f;
      for (int c = lane; c < un.n; c += 32) {
        const float x_s = __ldcg(p.xs + brow + c);
        if (MODE == 0) {
          cf[c] = x_s;
        } else if (sh) {
          ct[c] = un.slot0 + c;
          cf[c] = tsd * x_s * x_s;
        } else {
          const int src = __ldcg(p.src_of_slot + un.slot0 + c);
          ct[c] = src / p.k;
          cf[c] = __ldcg(p.gate + src) * tsd * x_s * x_s;
        }
      }
      __syncwarp();
      if (!warp_wait(&tfull[buf], tph[buf], wc)) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * C::ACC_COLS + ((uint32_t)(q * 32) << 16);
      const int row = un.m_tile * 128 + q * 32 + lane;
      const int n_pad = (un.n + 15) & ~15;
      if (MODE == 0) {
        const float tg = sh ? __ldg(p.tss[0]) : __ldg(p.ts[0] + un.expert);
        const float tu = sh ? __ldg(p.tss[1]) : __ldg(p.ts[1] + un.expert);
        for (int c0 = 0; c0 < n_pad; c0 += 16) {
          uint32_t gv[16], uv[16];
          tmem_ld16(acc + c0, gv);
          tmem_ld16(acc + kTc4BN + c0, uv);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c0 + i;
            if (col < un.n) {
              const float x_s = cf[col];
              const float a = __uint_as_float(gv[i]) * tg * x_s;
              // h / xs^2 = silu(a) * (D_u s_u) / xs
              const float hv = a / (1.f + __expf(-a)) * (__uint_as_float(uv[i]) * tu) * (1.f / x_s);
              range_bad |= !(fabsf(hv) <= 65504.f);
              p.h16[(size_t)(brow + col) * p.Fmax + row] = __float2half_rn(fminf(fmaxf(hv, -65504.f), 65504.f));
            }
          }
        }
      } else {
        for (int c0 = 0; c0 < n_pad; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(acc + c0, v);
          tmem_ld_wait();
          if (p.oslot) {                       // fixed order: each (slot, row) stored once
            const int s0 = sh ? p.T * p.k + un.slot0 : un.slot0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + i;
              if (col < un.n) __stcg(p.oslot + (size_t)(s0 + col) * p.d + row, cf[col] * __uint_as_float(v[i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + i;
              if (col < un.n) red_add_f32(p.yacc + (size_t)ct[col] * p.d + row, cf[col] * __uint_as_float(v[i]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
      tph[buf] ^= 1;
      buf ^= 1;
    }
    if (MODE == 0 && __any_sync(0xFFFFFFFFu, range_bad) && lane == 0) atomicOr(p.err, kErrRange);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// f16 activation rows for the tensor cores: row s < T k is the x row of
// grouped slot s, row T k + t is token t (the shared expert's operand).  Each
// row is scaled by 2^-e (its largest magnitude into [1, 2)) and xs[row] = 2^e.
// One warp per row.  After a large-batch router (wpb > 0) the warp also places
// the slot (tok_of_slot, src_of_slot, slot_of).  First the grid writes the
// unit lists of both passes.
__global__ void __launch_bounds__(256) tc4_gather_kernel(const __nv_bfloat16* __restrict__ x,
                                                         const int32_t* __restrict__ idx, Workspace ws, int T, int E,
                                                         int k, int d, int wpb, UnitBuild ub) {
  pdl_launch_dependents();
  pdl_wait();
  build_unit_lists(ws, ub);
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, nw = (gridDim.x * blockDim.x) >> 5;
  const int per_row = d / 8;                       // 16-byte pieces of bf16
  __half* xp = reinterpret_cast<__half*>(ws.xp);
  for (int s = gw; s < T * (k + 1); s += nw) {
    int pos, t;
    if (s >= T * k) {
      pos = s;
      t = s - T * k;
    } else if (wpb > 0) {
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
    uint32_t mx = 0;                               // largest |x| as bits (monotone for |x|)
    for (int c = lane; c < per_row; c += 32) {
      const uint4 v = __ldg(src + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = max(mx, max((w[i] << 16) & 0x7FFFFFFFu, w[i] & 0x7FFF0000u));
    }
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    // 2^-e with e the exponent of the row maximum (normal maxima only; a zero,
    // subnormal, infinite or NaN maximum leaves the row unscaled)
    const int eb = (int)(mx >> 23);
    const bool scaled = eb >= 2 && eb <= 252;
    const float inv = scaled ? __int_as_float((254 - eb) << 23) : 1.f;
    if (lane == 0) ws.xs[pos] = scaled ? __int_as_float(eb << 23) : 1.f;
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)pos * d);
    for (int c = lane; c < per_row; c += 32) {
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
}

template <int MODE>
size_t tc4_smem_bytes() {
  using C = Tc4Cfg<MODE>;
  return 1024 + C::STAGES * C::STAGE_BYTES + (2 * C::STAGES + 8) * 8 + 16 + 8 * kTc4BN * 4;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, Args&&... args) {
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

cudaError_t launch_tc4(const Tc4Args& a, int num_sms, cudaStream_t s, Prof* prof) {
  {
    cudaError_t e = ensure_smem_limit(tc4_kernel<0>, (int)tc4_smem_bytes<0>());
    if (e == cudaSuccess) e = ensure_smem_limit(tc4_kernel<1>, (int)tc4_smem_bytes<1>());
    if (e != cudaSuccess) return e;
  }
  // f16 activation rows (and slot placement after a large-batch router)
  const int rows = a.T * (a.k + 1);
  const int gg = (rows + 7) / 8 < num_sms * 8 ? (rows + 7) / 8 : num_sms * 8;   // 8 warps per block
  UnitBuild ub;   // NVFP4 tiles: 128 weight rows, kTc4BN tokens, no split
  ub.E = a.E; ub.T = a.T; ub.tn = kTc4BN;
  ub.sh_tb = a.Fs > 0 ? (a.T + kTc4BN - 1) / kTc4BN : 0;
  ub.mt[0] = a.F / 128; ub.mt[1] = a.d / 128;
  ub.sh_mt[0] = a.Fs > 0 ? a.Fs / 128 : 0; ub.sh_mt[1] = a.d / 128;
  ub.rep[0] = 1; ub.rep[1] = 1;
  if (prof) prof->begin(MOE_K_TC_GATHER, s);
  cudaError_t e = launch_pdl(tc4_gather_kernel, gg > 0 ? gg : 1, 256, 0, s,
                             static_cast<const __nv_bfloat16*>(a.x), a.idx, a.ws, a.T, a.E, a.k, a.d, a.wpb, ub);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;

  Tc4Params p;
  p.T = a.T; p.E = a.E; p.k = a.k; p.d = a.d;
  p.Fmax = a.F > a.Fs ? a.F : a.Fs;
  p.xs = a.ws.xs;
  p.src_of_slot = a.ws.src_of_slot;
  p.gate = a.gate;
  p.n_units = a.ws.n_units;
  p.h16 = reinterpret_cast<__half*>(a.ws.h16);
  p.yacc = a.ws.yacc;
  p.oslot = a.ws.oslot;
  p.err = a.ws.err;
  p.wait_ns = a.wait_ns;
  const bool has_sh = a.Fs > 0;
  // pass 1: gate/up
  for (int m = 0; m < 2; ++m) {
    p.q[m] = *a.q[m];
    p.sc[m] = *a.sc[m];
    p.sq[m] = has_sh ? *a.sq[m] : *a.q[m];
    p.ssc[m] = has_sh ? *a.ssc[m] : *a.sc[m];
    p.ts[m] = a.ts[m];
    p.tss[m] = has_sh ? a.tss[m] : a.ts[m];
  }
  p.tm_b = *a.tm_xp;
  p.rows_e = a.F;
  p.K = a.d; p.Ks = a.d;
  p.mt_s = has_sh ? a.Fs / 128 : 1;
  // The shared expert's operand rows are made by the gather kernel too, so no
  // unit may start before the grid-dependency wait.
  p.n_pre = 0;
  p.units = a.ws.units_gu;
  const int grid1 = num_sms < a.max_units_gu ? num_sms : (a.max_units_gu > 0 ? a.max_units_gu : 1);
  if (prof) prof->begin(MOE_K_TC_GATEUP, s);
  e = launch_pdl(tc4_kernel<0>, grid1, kThreads4, tc4_smem_bytes<0>(), s, p);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  // pass 2: down
  p.q[0] = *a.q[2];
  p.sc[0] = *a.sc[2];
  p.sq[0] = has_sh ? *a.sq[2] : *a.q[2];
  p.ssc[0] = has_sh ? *a.ssc[2] : *a.sc[2];
  p.ts[0] = a.ts[2];
  p.tss[0] = has_sh ? a.tss[2] : a.ts[2];
  p.q[1] = p.q[0]; p.sc[1] = p.sc[0]; p.sq[1] = p.sq[0]; p.ssc[1] = p.ssc[0];
  p.ts[1] = p.ts[0]; p.tss[1] = p.tss[0];
  p.tm_b = *a.tm_h;
  p.rows_e = a.d;
  p.K = a.F; p.Ks = has_sh ? a.Fs : a.F;
  p.mt_s = a.d / 128;
  p.n_pre = 0;
  p.units = a.ws.units_dn;
  const int grid2 = num_sms < a.max_units_dn ? num_sms : (a.max_units_dn > 0 ? a.max_units_dn : 1);
  if (prof) prof->begin(MOE_K_TC_DOWN, s);
  e = launch_pdl(tc4_kernel<1>, grid2, kThreads4, tc4_smem_bytes<1>(), s, p);
  if (prof) prof->end(s);
  if (e != cudaSuccess) return e;
  return launch_tc_finalize(a.ws, a.x, a.y, a.T, a.d, a.k, a.Fs > 0, a.add_residual != 0, a.ws.ready, a.E + 3,
                            num_sms, s, prof);
}

}  // namespace moe
