// Device helpers shared by the persistent (one CTA per SM, cooperative)
// decode kernels: named barriers, the bounded grid barrier, row staging and
// the per-token top-k.
#pragma once
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace persist {

constexpr uint32_t kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// Named barrier that also ORs a flag over the participating threads: every
// thread gets the same answer, so a decision taken on it is uniform even if
// the abort flag changes meanwhile (the producer warp may set it at any time).
__device__ __forceinline__ bool named_sync_or(int id, int n, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.or.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(n), "r"((uint32_t)v)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Grid barrier over the nthreads consumer threads of every CTA (named barrier
// 1): thread `leader` arrives on the counter (release) and waits for the
// target (acquire), polling without sleeping (the barrier is on the critical
// path), bounded in time.  Returns false (every thread alike) on a timeout or
// an abort.
__device__ __forceinline__ bool grid_sync(unsigned* ctr, unsigned target, const WaitCtl& wc, volatile int* abort_flag,
                                          int nthreads, int leader) {
  named_sync(1, nthreads);
  bool bad = false;
  if ((int)threadIdx.x == leader) {
    if (!*abort_flag) {
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
      bool ok = ld_acquire_gpu(ctr) >= target;
      if (!ok) {
        const uint64_t t0 = global_ns();
        for (uint32_t it = 1; !ok; ++it) {
          ok = ld_acquire_gpu(ctr) >= target;
          if (!ok && (it & 255u) == 0 && global_ns() - t0 > wc.limit_ns) break;
        }
      }
      if (!ok) {
        atomicOr(wc.err, kErrTimeout);
        *abort_flag = 1;
        bad = true;
      }
    }
  }
  return !named_sync_or(1, nthreads, bad || *abort_flag != 0);
}

// Copy `rows` rows of `chunks` 16-byte pieces from global (src_pitch bytes)
// to shared memory (dst_pitch bytes) with asynchronous 16-byte copies
// (cp.async, L2 to shared memory, no registers held): every piece of the
// thread is in flight before it waits, so the copy costs about one L2 round
// trip.  The caller synchronises the threads afterwards.
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

// Top-k of token t (one warp) from nq partial logit rows part[q][t][e]
// (stride maxT rows per part, added in q order): larger logit first, lower
// expert index first on equal logits; gates = softmax of the selected
// logits.  Writes sel_e[t k + j] and sel_g[t k + j] (shared memory).  E <= 256.
__device__ __forceinline__ void topk_token(const float* part, int nq, int maxT, int E, int k, int t, int* sel_e,
                                           float* sel_g, int lane) {
  float lg[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) lg[i] = 0.f;
  // parts in groups of four, every load of a group in flight before the adds
  for (int q0 = 0; q0 < nq; q0 += 4) {
    float v[4][8];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        v[qq][i] = (q0 + qq < nq && e < E) ? __ldcg(part + ((size_t)(q0 + qq) * maxT + t) * E + e) : 0.f;
      }
#pragma unroll
    for (int qq = 0; qq < 4; ++qq)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (q0 + qq < nq) lg[i] += v[qq][i];
  }
  // order-preserving 32-bit keys of the logits (0 = taken or absent)
  uint32_t key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t u = __float_as_uint(lg[i]);
    key[i] = (lane + 32 * i < E) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
  // k rounds: the warp's largest key (redux max), then the lowest expert
  // index holding it (redux min); the winner goes straight to shared memory
  // (its logit parked in sel_g until the gates)
  for (int j = 0; j < k; ++j) {
    uint32_t lm = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) lm = key[i] > lm ? key[i] : lm;
    const uint32_t wm = __reduce_max_sync(kFull, lm);
    uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (key[i] == wm) cand = min(cand, (uint32_t)(lane + 32 * i));
    const uint32_t win = __reduce_min_sync(kFull, cand);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((uint32_t)(lane + 32 * i) == win) key[i] = 0;
    if (lane == 0) {
      const uint32_t u = (wm & 0x80000000u) ? (wm & 0x7FFFFFFFu) : ~wm;
      sel_e[t * k + j] = (int)win;
      sel_g[t * k + j] = __uint_as_float(u);
    }
  }
  __syncwarp();
  // gates: softmax of the k selected logits (lane j holds selection j)
  const float l0 = sel_g[t * k];
  const float lj = lane < k ? sel_g[t * k + lane] : l0;
  const float ej = lane < k ? expf(lj - l0) : 0.f;
  float sum = ej;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  __syncwarp();
  if (lane < k) sel_g[t * k + lane] = ej / sum;
}

}  // namespace persist
}  // namespace moe
