// Router, top-k selection and token-slot grouping.
//
// The gating network scores each token against every routed expert and keeps
// a few of them (kongchang.com, section "Architecture: The 40B Total vs. 2.5B
// Active Trade-off"; 256 experts, 6 per token: evermx.com review, section
// "Sparse architecture").  Readings implemented here: fp32 logits
// l = x.Wr + b, selection of the k largest logits with the lower index first
// on ties, gates = softmax over the k selected logits.  The grouping puts the
// token-slots of each expert next to each other, in (token, j) order, which is
// what lets each expert's weights be streamed once per call.
//
// Two variants:
//  * route_small (T <= 64): each CTA computes the logits of eight experts for
//    eight tokens; the last CTA of each token chunk selects, the last of those
//    groups (atomic tickets).  One launch.
//  * route_large: one CTA per 32 tokens computes all E logits of its tokens
//    (fp32 SIMT tile), selects the top k and writes one selection-bitmap word
//    per expert; the last CTA scans the bitmap into the grouping.
#include <utility>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;

// Every call starts with a router.  It is launched with programmatic
// serialisation, so its launch and set-up overlap the tail of the previous
// kernel on the stream, but it waits for that kernel to complete before it
// reads x (the previous layer's output) and before it lets the next kernels
// launch: the expert kernels' work ahead of their own grid-dependency wait
// (clearing the fp32 accumulator, the shared expert's tiles) can then never
// meet a kernel of an earlier call.
__device__ __forceinline__ void route_entry() {
  pdl_wait();
  pdl_launch_dependents();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_route(void (*kernel)(KArgs...), dim3 grid, int block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
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
constexpr int kLargeBT = 32;     // tokens per CTA in route_large

__device__ __forceinline__ void load_x4(const void* x, int act_bf16, size_t off, float (&v)[4]) {
  if (act_bf16) {
    const uint2 r = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + off));
    v[0] = __uint_as_float(r.x << 16);
    v[1] = __uint_as_float(r.x & 0xFFFF0000u);
    v[2] = __uint_as_float(r.y << 16);
    v[3] = __uint_as_float(r.y & 0xFFFF0000u);
  } else {
    const float4 r = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + off));
    v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
  }
}

// Grid ticket: every CTA calls this once after writing its results; *last is
// set in the CTA that arrives n-th.  One fence by the ticket thread publishes
// the whole CTA's writes (fences are cumulative over writes ordered before
// them by the barrier) and, in the last CTA, orders the reads that follow.
__device__ __forceinline__ void ticket_last(unsigned int* counter, unsigned n, int* last) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool l = atomicAdd(counter, 1u) == n - 1;
    if (l) __threadfence();
    *last = l;
  }
  __syncthreads();
}


// Selection keys: (logit, expert) packed into 64 bits so that unsigned order
// is the selection order (larger logit first, lower index on equal logits).
// NaN counts as -inf and -0 as +0, as in the float comparison.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
  v = isnan(v) ? -INFINITY : v + 0.0f;
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint32_t)(0x7FFFFFFF - e);
}
__device__ __forceinline__ float key_value(uint64_t k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u ^ 0x80000000u) : ~u;
  return __uint_as_float(u);
}
__device__ __forceinline__ int key_index(uint64_t k) { return 0x7FFFFFFF - (int)(uint32_t)k; }
__device__ __forceinline__ void cswap(uint64_t& a, uint64_t& b) {   // a >= b afterwards
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}
// Sorts 8 keys in descending order (19-comparator network, depth 6).
__device__ __forceinline__ void sort8(uint64_t (&a)[8]) {
  cswap(a[0], a[1]); cswap(a[2], a[3]); cswap(a[4], a[5]); cswap(a[6], a[7]);
  cswap(a[0], a[2]); cswap(a[1], a[3]); cswap(a[4], a[6]); cswap(a[5], a[7]);
  cswap(a[1], a[2]); cswap(a[5], a[6]); cswap(a[0], a[4]); cswap(a[3], a[7]);
  cswap(a[1], a[5]); cswap(a[2], a[6]);
  cswap(a[1], a[4]); cswap(a[3], a[6]);
  cswap(a[2], a[4]); cswap(a[3], a[5]);
  cswap(a[3], a[4]);
}
// r = top 8 of the descending lists r and b, descending (bitonic merge).
__device__ __forceinline__ void merge_top8(uint64_t (&r)[8], const uint64_t (&b)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) r[i] = r[i] > b[7 - i] ? r[i] : b[7 - i];
#pragma unroll
  for (int dd = 4; dd >= 1; dd >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & dd) == 0) cswap(r[i], r[i + dd]);
}

// Top k of one token's E logits by one warp; row(e) returns logit e.  Lane l
// scores experts l NPL .. l NPL + NPL - 1 and keeps its best 8 as sorted keys;
// five butterfly merges then leave the warp's best 8 in every lane.  Writes
// idx/gate (and sidx, if given) for the token.
template <int NPL, typename Row>
__device__ void warp_topk(const Row& row, int E, int k, int32_t* idx_t, float* gate_t, int32_t* sidx_t) {
  static_assert(NPL == 8 || NPL == 16, "8 or 16 experts per lane");
  const int lane = threadIdx.x & 31;
  uint64_t best[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane * NPL + i;
    best[i] = e < E ? sel_key(row(e), e) : 0;             // 0 is below every real key
  }
  sort8(best);
  if (NPL == 16) {
    uint64_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * NPL + 8 + i;
      b[i] = e < E ? sel_key(row(e), e) : 0;
    }
    sort8(b);
    merge_top8(best, b);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint64_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = __shfl_xor_sync(0xFFFFFFFFu, best[i], o);
    merge_top8(best, b);
  }
  if (lane == 0) {
    float lv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) lv[j] = key_value(best[j]);
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) z += expf(lv[j] - lv[0]);
    const float inv = 1.f / z;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        const int e = key_index(best[j]);
        idx_t[j] = e;
        gate_t[j] = expf(lv[j] - lv[0]) * inv;
        if (sidx_t) sidx_t[j] = e;
      }
  }
}

// Exclusive scan of n <= 4 * blockDim ints in shared memory, in place; returns the total.
__device__ int block_exclusive_scan(int* a, int n) {
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int s = 0;
  for (int i = beg; i < end; ++i) s += a[i];
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += v;
    }
    if (lane < nwarps) warp_tot[lane] = wi - w;
    if (lane == 31) total = wi;
  }
  __syncthreads();
  int run = warp_tot[warp] + incl - s;
  for (int i = beg; i < end; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

// Everything after the counts are known: offsets, active-expert list, the
// per-expert first entries of the tcgen05 unit lists.  cnt: smem [E] counts; offs: smem [E + 1].  Runs in one CTA.
__device__ void finish_grouping(const RouteArgs& a, int* cnt, int* offs, int* scratch) {
  const int E = a.E, tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) offs[e] = cnt[e];
  __syncthreads();
  const int total = block_exclusive_scan(offs, E);
  if (tid == 0) offs[E] = total;
  // active experts
  for (int e = tid; e < E; e += blockDim.x) scratch[e] = cnt[e] > 0 ? 1 : 0;
  __syncthreads();
  const int n_act = block_exclusive_scan(scratch, E);
  for (int e = tid; e < E; e += blockDim.x) {
    if (cnt[e] > 0) a.ws.active[scratch[e]] = e;
    a.ws.counts[e] = cnt[e];
    a.ws.offsets[e] = offs[e];
    if (a.counts_out) a.counts_out[e] = cnt[e];
  }
  if (tid == 0) {
    a.ws.active[E] = n_act;
    a.ws.offsets[E] = total;
    a.ws.counts[E] = a.T;
  }
  __syncthreads();
  if (!a.build_tc_units) return;
  // tcgen05 unit lists: per list, the first entry of every routed expert
  // after the shared expert's entries (the gather kernel writes the entries)
  const int mt_gu = a.F / kTcBM, mt_dn = a.d / a.dn_rows, tn = a.tile_n;
  const int sh_tb = a.has_shared ? (a.T + tn - 1) / tn : 0;
  const int sh_mt_gu = a.has_shared ? a.Fs / kTcBM : 0;
  for (int pass = 0; pass < 2; ++pass) {
    const int mt = pass == 0 ? mt_gu : mt_dn;
    const int sh_mt = pass == 0 ? sh_mt_gu : mt_dn;
    const int rep = pass == 0 ? a.gu_split : 1;   // gate/up tiles split along K: one entry per part
    for (int e = tid; e < E; e += blockDim.x) scratch[e] = rep * mt * ((cnt[e] + tn - 1) / tn);
    __syncthreads();
    const int n_routed = block_exclusive_scan(scratch, E);
    for (int e = tid; e < E; e += blockDim.x) a.ws.uprefix[pass * (E + 1) + e] = scratch[e];
    if (tid == 0) {
      a.ws.uprefix[pass * (E + 1) + E] = n_routed;
      a.ws.n_units[pass] = rep * sh_mt * sh_tb + n_routed;
    }
    __syncthreads();
  }
}

// Grouping from per-block counts.  Tokens come in blocks of 32 * wpb tokens
// (wpb selection-bitmap words per expert and block; sel[w][e] bit t % 32 is
// set when token 32 w + t % 32 chose expert e) and bcnt[b][e] is block b's
// count for expert e.  One CTA turns the counts into offsets, the active list
// and the unit-list prefixes, and stores the exclusive prefix of the block counts in
// bpref[b][e]; the per-slot placement (slot_position) runs afterwards, in
// parallel, in whichever kernel needs it.
__device__ void group_from_counts(const RouteArgs& a, int nblk) {
  __shared__ int cnt[kMaxExperts], offs[kMaxExperts + 1], scratch[kMaxExperts];
  const int E = a.E, tid = threadIdx.x, nth = blockDim.x;
  for (int ee = tid; ee < E; ee += nth) {
    int run = 0;
    for (int b0 = 0; b0 < nblk; b0 += 32) {
      int c[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) c[i] = b0 + i < nblk ? __ldcg(a.ws.bcnt + (size_t)(b0 + i) * E + ee) : 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (b0 + i < nblk) a.ws.bpref[(size_t)(b0 + i) * E + ee] = run;
        run += c[i];
      }
    }
    cnt[ee] = run;
  }
  __syncthreads();
  finish_grouping(a, cnt, offs, scratch);
  if (tid == 0) a.ws.counters[0] = 0;
}

// ------------------------------------------------------------------ small T
// grid (ceil(E / 8), ceil(T / 8)): CTA (bx, by) scores experts 8 bx .. 8 bx + 7
// against tokens 8 by .. 8 by + 7, whose activations are staged in shared
// memory as fp32.  Warp w takes four of the experts (w % 2) and a quarter of
// the reduction (w / 2); each step a lane loads four router values of each of
// its experts and four activations of each token and does 128 FMAs with them
// (about one instruction per FMA).  The four quarters are added in a fixed
// order through shared memory.
constexpr int kSmallTok = 8;
static_assert(kSmallTok * 4 * kMaxHidden <= kRouteSmallSmem, "router staging must fit its shared-memory limit");
constexpr int kSmallExp = 4;       // experts per warp
constexpr int kSmallKq = 4;        // parts of the reduction per CTA

__global__ void __launch_bounds__(kRouteThreads) route_small_kernel(RouteArgs a) {
  route_entry();
  extern __shared__ __align__(16) float xs[];       // [8][d] fp32 activations
  __shared__ float part[kSmallKq][2 * kSmallExp * kSmallTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, d = a.d, T = a.T, k = a.k;
  const int t0 = blockIdx.y * kSmallTok;
  const int nt = min(kSmallTok, T - t0);
  if (a.act_bf16) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.x) + (size_t)t0 * d);
    const int n16 = nt * d / 8;
    for (int i = threadIdx.x; i < n16; i += kRouteThreads) {
      const uint4 v = __ldg(src + i);
      float4* dst = reinterpret_cast<float4*>(xs) + 2 * i;
      dst[0] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                           __uint_as_float(v.y & 0xFFFF0000u));
      dst[1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w << 16),
                           __uint_as_float(v.w & 0xFFFF0000u));
    }
  } else {
    const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(a.x) + (size_t)t0 * d);
    const int n4 = nt * d / 4;
    for (int i = threadIdx.x; i < n4; i += kRouteThreads) reinterpret_cast<float4*>(xs)[i] = __ldg(src + i);
  }
  __syncthreads();
  const int eg = warp & 1, kq = warp >> 1;
  const int e0 = blockIdx.x * 2 * kSmallExp + eg * kSmallExp;
  const int kd = d / kSmallKq, kbeg = kq * kd;       // d / 4 is a multiple of 16 values
  {
    float acc[kSmallExp * kSmallTok];                   // [expert j][token t]
#pragma unroll
    for (int i = 0; i < kSmallExp * kSmallTok; ++i) acc[i] = 0.f;
    for (int c = kbeg + lane * 4; c < kbeg + kd; c += 128) {
      float4 wr[kSmallExp];
#pragma unroll
      for (int j = 0; j < kSmallExp; ++j)
        wr[j] = e0 + j < E ? __ldg(reinterpret_cast<const float4*>(a.Wr + (size_t)(e0 + j) * d + c))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int t = 0; t < kSmallTok; ++t) {
        if (t < nt) {
          const float4 xv = *reinterpret_cast<const float4*>(xs + (size_t)t * d + c);
#pragma unroll
          for (int j = 0; j < kSmallExp; ++j) {
            float& r = acc[j * kSmallTok + t];
            r = fmaf(wr[j].x, xv.x, r);
            r = fmaf(wr[j].y, xv.y, r);
            r = fmaf(wr[j].z, xv.z, r);
            r = fmaf(wr[j].w, xv.w, r);
          }
        }
      }
    }
    const float tot = transpose_reduce<kSmallExp * kSmallTok, 32>(acc, lane);   // lane l: expert l / 8, token l % 8
    part[kq][eg * kSmallExp * kSmallTok + lane] = tot;
  }
  __syncthreads();
  if (threadIdx.x < 2 * kSmallExp * kSmallTok) {
    const int v = threadIdx.x;                          // (expert group, expert, token)
    const float tot = ((part[0][v] + part[1][v]) + part[2][v]) + part[3][v];
    const int e = blockIdx.x * 2 * kSmallExp + (v >> 3), tt = v & 7;
    if (e < E && tt < nt) a.ws.logits[(size_t)(t0 + tt) * E + e] = tot + (a.b ? a.b[e] : 0.f);
  }
  // Two-level tail.  The last of the expert-chunk CTAs of this token chunk
  // selects the chunk's tokens (one warp per token); the last of those does
  // the grouping for all tokens.
  __shared__ int s_last;
  ticket_last(&a.ws.counters[1 + blockIdx.y], gridDim.x, &s_last);
  if (!s_last) return;
  if (warp < nt) {
    const int t = t0 + warp;
    const float* lrow = a.ws.logits + (size_t)t * E;
    auto row = [lrow](int e) { return __ldcg(lrow + e); };
    if (E <= 256)
      warp_topk<8>(row, E, k, a.idx + (size_t)t * k, a.gate + (size_t)t * k, nullptr);
    else
      warp_topk<16>(row, E, k, a.idx + (size_t)t * k, a.gate + (size_t)t * k, nullptr);
  }
  if (threadIdx.x == 0) a.ws.counters[1 + blockIdx.y] = 0;
  ticket_last(&a.ws.counters[0], gridDim.y, &s_last);
  if (!s_last) return;

  __shared__ int32_t s_idx[kSmallT * kMaxTopK];
  __shared__ int cnt[kMaxExperts], offs[kMaxExperts + 1], scratch[kMaxExperts];
  __shared__ uint32_t bm[kMaxExperts][2];
  for (int i = threadIdx.x; i < E; i += blockDim.x) { cnt[i] = 0; bm[i][0] = 0; bm[i][1] = 0; }
  for (int s = threadIdx.x; s < T * k; s += blockDim.x) s_idx[s] = __ldcg(a.idx + s);
  __syncthreads();
  for (int s = threadIdx.x; s < T * k; s += blockDim.x) {
    const int ee = s_idx[s], t = s / k;
    atomicAdd(&cnt[ee], 1);
    atomicOr(&bm[ee][t >> 5], 1u << (t & 31));
  }
  __syncthreads();
  finish_grouping(a, cnt, offs, scratch);
  for (int s = threadIdx.x; s < T * k; s += blockDim.x) {
    const int ee = s_idx[s], t = s / k, wd = t >> 5;
    const int rank = (wd ? __popc(bm[ee][0]) : 0) + __popc(bm[ee][wd] & ((1u << (t & 31)) - 1u));
    const int slot = offs[ee] + rank;
    a.ws.tok_of_slot[slot] = t;
    a.ws.src_of_slot[slot] = s;
    a.ws.slot_of[s] = slot;
  }
  if (threadIdx.x == 0) a.ws.counters[0] = 0;
}

// ------------------------------------------------------------------ large T
// Logit tile of 32 tokens x E experts: thread (ty, tx) owns tokens 4 ty .. 4 ty + 3
// and experts 4 tx + 128 j .. + 3 for j < E / 128.
template <int EJ>
__global__ void __launch_bounds__(kRouteThreads) route_large_kernel(RouteArgs a) {
  route_entry();
  extern __shared__ __align__(16) float dsm[];
  const int E = a.E, d = a.d, T = a.T, k = a.k;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int t0 = blockIdx.x * kLargeBT;
  const int Ep = EJ * 128;                  // E rounded up to 128
  float* xs = dsm;                          // [32 tok][32 kk]
  float* wsT = dsm + 32 * 32;               // [32 kk][Ep]
  const int ty = tid >> 5, tx = tid & 31;
  float acc[4][EJ][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.f;

  for (int k0 = 0; k0 < d; k0 += 32) {
    // x tile: 32 tokens x 32 values
    for (int i = tid; i < 32 * 8; i += kRouteThreads) {
      const int tt = i >> 3, c4 = (i & 7) * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t0 + tt < T) load_x4(a.x, a.act_bf16, (size_t)(t0 + tt) * d + k0 + c4, v);
      *reinterpret_cast<float4*>(xs + tt * 32 + c4) = make_float4(v[0], v[1], v[2], v[3]);
    }
    // router tile, transposed: wsT[kk][e]
    for (int i = tid; i < Ep * 8; i += kRouteThreads) {
      const int ee = i >> 3, c4 = (i & 7) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ee < E) v = __ldg(reinterpret_cast<const float4*>(a.Wr + (size_t)ee * d + k0 + c4));
      wsT[(c4 + 0) * Ep + ee] = v.x;
      wsT[(c4 + 1) * Ep + ee] = v.y;
      wsT[(c4 + 2) * Ep + ee] = v.z;
      wsT[(c4 + 3) * Ep + ee] = v.w;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < 32; ++kk) {
      float xv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) xv[i] = xs[(ty * 4 + i) * 32 + kk];
#pragma unroll
      for (int j = 0; j < EJ; ++j) {
        const float4 wv = *reinterpret_cast<const float4*>(wsT + kk * Ep + 128 * j + 4 * tx);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][j][0] = fmaf(xv[i], wv.x, acc[i][j][0]);
          acc[i][j][1] = fmaf(xv[i], wv.y, acc[i][j][1]);
          acc[i][j][2] = fmaf(xv[i], wv.z, acc[i][j][2]);
          acc[i][j][3] = fmaf(xv[i], wv.w, acc[i][j][3]);
        }
      }
    }
    __syncthreads();
  }
  // logits to shared memory [32][Ep] (reuses the router tile space)
  float* lg = wsT;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ee = 128 * j + 4 * tx + q;
        lg[(ty * 4 + i) * Ep + ee] = acc[i][j][q] + ((ee < E && a.b) ? a.b[ee] : 0.f);
      }
  __shared__ uint32_t word[kMaxExperts];
  __shared__ int32_t s_idx[kLargeBT * kMaxTopK];
  for (int i = tid; i < E; i += kRouteThreads) word[i] = 0;
  __syncthreads();
  for (int tt = warp; tt < kLargeBT; tt += kRouteThreads / 32) {
    const int t = t0 + tt;
    if (t >= T) break;
    const float* lrow = lg + tt * Ep;
    auto row = [lrow](int e) { return lrow[e]; };
    if (E <= 256)
      warp_topk<8>(row, E, k, a.idx + (size_t)t * k, a.gate + (size_t)t * k, s_idx + tt * k);
    else
      warp_topk<16>(row, E, k, a.idx + (size_t)t * k, a.gate + (size_t)t * k, s_idx + tt * k);
  }
  __syncthreads();
  for (int s = tid; s < kLargeBT * k; s += kRouteThreads) {
    const int tt = s / k;
    if (t0 + tt < T) atomicOr(&word[s_idx[s]], 1u << tt);
  }
  __syncthreads();
  for (int i = tid; i < E; i += kRouteThreads) {
    a.ws.sel[(size_t)blockIdx.x * E + i] = word[i];
    a.ws.bcnt[(size_t)blockIdx.x * E + i] = __popc(word[i]);
  }

  // Last CTA: counts, word prefixes, offsets, slots.
  __shared__ int s_last;
  ticket_last(&a.ws.counters[0], gridDim.x, &s_last);
  if (!s_last) return;
  group_from_counts(a, gridDim.x);
}

// ------------------------------------------------------------------ large T, tensor cores
// With bf16 activations (exact in bf16) and the fp32 router weights split once
// into three bf16 parts w = hi + mid + lo (to within 2^-24 of w), three bf16
// MMAs accumulating in fp32 give the logits to within fp32 rounding, on the
// tensor pipe.  CTA (es, tb): 128 tokens x 64 experts, K = d.  Each CTA keeps
// the top 8 of its 64 experts per token (ordered by logit, then lower index);
// the last CTA of a token block merges the slices (the global top k lies in
// the union of the slices' top k) and writes the token block's bitmap words;
// the last token block groups all tokens.
constexpr int kRtStages = 4;
constexpr int kRtA = 128 * 128;                // x tile: 128 tokens x 64 values
constexpr int kRtB = 64 * 128;                 // router tile: 64 experts x 64 values (one split)
constexpr int kRtStageBytes = kRtA + 3 * kRtB;

struct RouteTcParams {
  CUtensorMap tm_x;        // x [T][d] bf16, box {64, 128}
  CUtensorMap tm_wr;       // split router weights [3 E][d] bf16, box {64, 64}
  RouteArgs a;
  uint64_t* cand;          // [T][E / 64][kMaxTopK] per-slice selection keys
  uint64_t wait_ns;
};

__global__ void __launch_bounds__(192, 1) route_tc_kernel(const __grid_constant__ RouteTcParams p) {
  const RouteArgs& a = p.a;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + kRtStages * kRtStageBytes);
  uint64_t* empty = full + kRtStages;
  uint64_t* tfull = empty + kRtStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int E = a.E, T = a.T, k = a.k, d = a.d;
  const int es = blockIdx.x, nsl = gridDim.x, tb = blockIdx.y, t0 = tb * 128;
  if (tid == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  route_entry();
  const WaitCtl wc{p.wait_ns, a.ws.err, abort_flag};
  const int nkb = d / 64;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_x);
    tma_prefetch_desc(&p.tm_wr);
    int issued = 0;
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kRtStages;
      if (!mbar_wait(&empty[s], ((kb / kRtStages) & 1) ^ 1, wc)) { ok = false; break; }
      uint8_t* st = dsm + s * kRtStageBytes;
      mbar_arrive_expect_tx(&full[s], kRtStageBytes);
      tma_load_2d(st, &p.tm_x, kb * 64, t0, &full[s]);
#pragma unroll
      for (int sp = 0; sp < 3; ++sp) tma_load_2d(st + kRtA + sp * kRtB, &p.tm_wr, kb * 64, sp * E + es * 64, &full[s]);
      issued = kb + 1;
    }
    if (!ok)
      for (int j = issued - kRtStages < 0 ? 0 : issued - kRtStages; j < issued; ++j) {
        const uint64_t ts = global_ns();
        while (!mbar_try_wait(&full[j % kRtStages], (j / kRtStages) & 1))
          if (global_ns() - ts > p.wait_ns) break;
      }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, 64);
    bool ok = true;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kRtStages;
      if (!mbar_wait(&full[s], (kb / kRtStages) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      const uint32_t st = smem_u32(dsm + s * kRtStageBytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int sp = 0; sp < 3; ++sp)
          tc_mma_f16(tmem, sdesc_sw128(st + kk * 32), sdesc_sw128(st + kRtA + sp * kRtB + kk * 32), idesc,
                     (kb > 0 || kk > 0 || sp > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    if (ok) tc_commit(tfull);
    else if (nkb > 0) {
      const uint64_t ts = global_ns();
      while (!mbar_try_wait(&empty[(nkb - 1) % kRtStages], ((nkb - 1) / kRtStages) & 1))
        if (global_ns() - ts > p.wait_ns) break;
    }
  } else if (warp >= 2) {
    // epilogue: TMEM lane quarter q holds tokens 32 q .. 32 q + 31
    const int q = warp & 3, r = q * 32 + lane, t = t0 + r;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(tfull, 0, wc) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (ok) {
      while (!mbar_try_wait(tfull, 0)) {
      }
      tc_fence_after();
      uint64_t best[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) best[j] = 0;          // below every real key
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint64_t g[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = es * 64 + c0 + 8 * h + i;
            g[i] = sel_key(__uint_as_float(v[8 * h + i]) + (a.b ? __ldg(a.b + e) : 0.f), e);
          }
          sort8(g);
          merge_top8(best, g);
        }
      }
      // static indices only: a runtime index would put the list in local memory
      if (t < T) {
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
          if (j < k) p.cand[((size_t)t * nsl + es) * kMaxTopK + j] = best[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if (*abort_flag) return;

  // ---- merge the slices of this token block (last slice CTA to finish)
  __shared__ int s_last;
  ticket_last(&a.ws.counters[1 + tb], nsl, &s_last);
  if (!s_last) return;
  __shared__ uint32_t words[4][kMaxExperts];
  for (int i = tid; i < 4 * kMaxExperts; i += blockDim.x) (&words[0][0])[i] = 0;
  __syncthreads();
  for (int r = tid; r < 128; r += blockDim.x) {
    const int t = t0 + r;
    if (t >= T) continue;
    // every slice's list is already sorted: merge them pairwise
    uint64_t best[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) best[j] = 0;
#pragma unroll
    for (int sl = 0; sl < kMaxExperts / 64; ++sl) {
      if (sl >= nsl) break;
      uint64_t c[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = j < k ? __ldcg(p.cand + ((size_t)t * nsl + sl) * kMaxTopK + j) : 0;
      merge_top8(best, c);
    }
    float lv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) lv[j] = key_value(best[j]);
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) z += expf(lv[j] - lv[0]);
    const float inv = 1.f / z;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        const int e = key_index(best[j]);
        a.idx[(size_t)t * k + j] = e;
        a.gate[(size_t)t * k + j] = expf(lv[j] - lv[0]) * inv;
        atomicOr(&words[r >> 5][e], 1u << (r & 31));
      }
  }
  __syncthreads();
  const int nw = (T + 31) / 32;
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 4; ++w) {
      if (tb * 4 + w < nw) a.ws.sel[(size_t)(tb * 4 + w) * E + e] = words[w][e];
      c += __popc(words[w][e]);
    }
    a.ws.bcnt[(size_t)tb * E + e] = c;
  }
  if (tid == 0) a.ws.counters[1 + tb] = 0;

  // ---- the last token block groups everything
  ticket_last(&a.ws.counters[0], gridDim.y, &s_last);
  if (!s_last) return;
  group_from_counts(a, gridDim.y);
}

__global__ void router_split_kernel(const float* __restrict__ w, __nv_bfloat16* __restrict__ out, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    out[i] = hi;
    out[n + i] = mid;
    out[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

}  // namespace

// Grouped position of every slot (t, j): tok_of_slot, src_of_slot, slot_of.
__global__ void __launch_bounds__(256) place_kernel(const int32_t* __restrict__ idx, Workspace ws, int T, int E, int k,
                                                    int wpb) {
  pdl_launch_dependents();
  pdl_wait();
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < T * k; s += gridDim.x * blockDim.x) {
    const int t = s / k, e = __ldg(idx + s);
    const int pos = slot_position(ws, E, t, e, wpb);
    ws.tok_of_slot[pos] = t;
    ws.src_of_slot[pos] = s;
    ws.slot_of[s] = pos;
  }
}

cudaError_t launch_place(const int32_t* idx, const Workspace& ws, int T, int E, int k, int wpb, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((T * k + 255) / 256 < 1024 ? (T * k + 255) / 256 : 1024);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, place_kernel, idx, ws, T, E, k, wpb);
}

cudaError_t launch_router_split(const float* w, __nv_bfloat16* out, size_t n, cudaStream_t s) {
  router_split_kernel<<<256, 256, 0, s>>>(w, out, n);
  return cudaGetLastError();
}

cudaError_t launch_route_tc(const RouteArgs& a, const CUtensorMap* tm_x, const CUtensorMap* tm_wr, uint64_t* cand,
                            uint64_t wait_ns, cudaStream_t s, Prof* prof) {
  const size_t smem = 1024 + (size_t)kRtStages * kRtStageBytes + (2 * kRtStages + 1) * 8 + 16;
  {
    const cudaError_t e = ensure_smem_limit(route_tc_kernel, (int)smem);
    if (e != cudaSuccess) return e;
  }
  RouteTcParams p;
  p.tm_x = *tm_x;
  p.tm_wr = *tm_wr;
  p.a = a;
  p.cand = cand;
  p.wait_ns = wait_ns;
  if (prof) prof->begin(MOE_K_ROUTE, s);
  const cudaError_t e = launch_pdl_route(route_tc_kernel, dim3(a.E / 64, (a.T + 127) / 128), 192, smem, s, p);
  if (prof) prof->end(s);
  return e;
}

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s, Prof* prof) {
  (void)num_sms;
  if (prof) prof->begin(MOE_K_ROUTE, s);
  if (a.T <= kSmallT) {
    const size_t smem = (size_t)kSmallTok * a.d * 4;
    if (a.d > kMaxHidden) return cudaErrorInvalidValue;
    {
      const cudaError_t e0 = ensure_smem_limit(route_small_kernel, kRouteSmallSmem);
      if (e0 != cudaSuccess) return e0;
    }
    const int epc = 2 * kSmallExp;   // experts per CTA
    const dim3 grid((a.E + epc - 1) / epc, (a.T + kSmallTok - 1) / kSmallTok);
    const cudaError_t e = launch_pdl_route(route_small_kernel, grid, kRouteThreads, smem, s, a);
    if (prof) prof->end(s);
    return e;
  }
  const int grid = (a.T + kLargeBT - 1) / kLargeBT;
  const int ej = (a.E + 127) / 128;
  const size_t smem = (32 * 32 + 32 * ej * 128) * sizeof(float);
  switch (ej) {
#define MOE_RL(N)                                                                                   \
  case N: {                                                                                         \
    {                                                                                               \
      const cudaError_t e0 = ensure_smem_limit(route_large_kernel<N>,                               \
                                               (int)((32 * 32 + 32 * N * 128) * sizeof(float)));    \
      if (e0 != cudaSuccess) return e0;                                                             \
    }                                                                                               \
    const cudaError_t e = launch_pdl_route(route_large_kernel<N>, dim3(grid), kRouteThreads, smem, s, a); \
    if (e != cudaSuccess) return e;                                                                 \
    break;                                                                                          \
  }
    MOE_RL(1) MOE_RL(2) MOE_RL(3) MOE_RL(4)
#undef MOE_RL
    default:
      return cudaErrorInvalidValue;
  }
  if (prof) prof->end(s);
  return cudaGetLastError();
}

}  // namespace moe
