// The 4-bit output layer (lm_head): logits[t][v] = sum_i x[t][i] W[v][i] for
// a small batch of tokens, W stored as NVFP4 (e2m1 codes, an e4m3 scale per
// 16 values, an fp32 scale for the matrix).
//
// The pages say the output layer was quantised to 4 bits because it is a
// large share of the weights read for each token (evermx.com review, Feature
// Overview, "Quantization").  At decode sizes the head is a pure weight
// stream: every code is read once per call and used for at most 8 tokens, so
// the kernel is built to stream at the HBM rate.
//
// One CTA per SM takes a contiguous range of 64-row blocks of W.  A producer
// thread copies each block in segments of 256 values with two TMA tile loads
// per stage (64 rows x 128 code bytes, 128-byte swizzle; 64 rows x 16 scale
// bytes) into a ring where every consumer warp owns two stages; eight
// consumer warps each take whole row blocks (four 16-row tiles).  A consumer
// decodes codes exactly into f16 in registers (cvt e2m1x2 -> f16x2, times the
// block scale as f16x2: code x scale has at most 5 significant bits and lies
// in [2^-10, 2688], so the product is exact) and multiplies them on the tensor
// pipe (mma.sync m16n8k16, f16 in, fp32 accumulate) against the activations,
// which every CTA converts once to f16 with an exact power-of-two scale per
// token (largest |x| into [1, 2)).  The reduction order is permuted the same
// way in A and B so that a lane decodes one 32-bit word of 8 codes per row
// (one block, one scale) and loads its 8 activations with one 16-byte load,
// shared by the four tiles; the sum over the block is unchanged.  The fp32
// result is multiplied by the matrix scale and the token's power of two.
// (Copying the rows with many small 1-D bulk copies instead left the copy
// engine, not HBM, as the limit: about 40 ns per copy whatever its size.)
//
// Every wait is bounded: on expiry the kernel records the timeout in the error
// word, drains its copies and returns.
#include <new>

#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kHdThreads = 32 * (1 + kHdConsumers);
constexpr int kHdPer = 2;                                // stages per consumer
constexpr int kHdStages = kHdConsumers * kHdPer;
constexpr int kHdRows = 64;                              // rows per block
constexpr int kHdKs = 256;                               // values per segment
constexpr int kHdCodeBytes = kHdRows * kHdKs / 2;        // 8192: 64 rows x 128 bytes, 128-byte swizzle
constexpr int kHdStageBytes = kHdCodeBytes + kHdRows * kHdKs / 16;   // + 64 rows x 16 scale bytes = 9216
constexpr uint32_t kAll = 0xFFFFFFFFu;
static_assert(kHdStageBytes % 1024 == 0, "stages keep the 1024-byte alignment the swizzle needs");

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// One e4m3 code -> {s, s} as f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3_dup_f16x2(uint32_t byte) {
  uint32_t h2;
  const uint32_t two = byte | (byte << 8);
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two));
  return h2;
}

struct HdLayout {
  uint32_t stages, bars, abort, xs, xscale, total, x_pitch;
};
// Offsets from the 1024-aligned base (the allocation has 1024 bytes of slack).
__host__ __device__ inline HdLayout hd_layout(int d) {
  HdLayout L;
  L.x_pitch = (uint32_t)d * 2 + 64;   // 16-byte loads of 8 rows x 4 lanes hit distinct bank groups
  uint32_t o = 0;
  L.stages = o; o += kHdStages * kHdStageBytes;
  L.bars = o;   o += 2 * kHdStages * 8;
  L.abort = o;  o += 16;
  L.xs = o;     o += kHdMaxT * L.x_pitch;
  L.xscale = o; o += kHdMaxT * 4;
  L.total = ((o + 15) & ~15u) + 1024;
  return L;
}

__global__ void __launch_bounds__(kHdThreads, 1) lm_head_kernel(const __grid_constant__ HeadArgs a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  uint8_t* dsm = dsm_raw + ((1024 - (smem_u32(dsm_raw) & 1023)) & 1023);
  const HdLayout L = hd_layout(a.d);
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + L.bars);
  uint64_t* empty = full + kHdStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(dsm + L.abort);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kHdStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{a.wait_ns, a.err, abort_flag};
  const int G = gridDim.x, b = blockIdx.x, d = a.d, KS = d / kHdKs;
  const int nblk = a.V / kHdRows;
  const int lo = (int)(((long long)nblk * b) / G), hi = (int)(((long long)nblk * (b + 1)) / G);

  if (warp == 0) {
    // producer (one thread): block lo + i goes to consumer i % 8
    if (lane != 0) return;
    tma_prefetch_desc(&a.tm_codes);
    tma_prefetch_desc(&a.tm_scales);
    const uint64_t pol = policy_evict_first();
    int m[kHdConsumers];
    for (int i = 0; i < kHdConsumers; ++i) m[i] = 0;
    uint32_t used = 0, last_par[kHdStages];
    bool ok = true;
    // Rounds of up to 8 blocks, one per consumer; within a round the segments
    // go out segment by segment across the consumers, so every consumer's two
    // stages stay filled (issuing a whole block before the next would stall
    // on the first consumer's ring while the others sit empty).
    for (int r0 = lo; r0 < hi && ok; r0 += kHdConsumers) {
      const int nb = hi - r0 < kHdConsumers ? hi - r0 : kHdConsumers;
      for (int s = 0; s < KS && ok; ++s)
        for (int w = 0; w < nb; ++w) {
          const int rb = r0 + w;
          const int mm = m[w]++;
          const int st = w * kHdPer + (mm % kHdPer);
          const uint32_t par = (mm / kHdPer) & 1;
          if (!mbar_wait(&empty[st], par ^ 1, wc)) { ok = false; break; }
          last_par[st] = par;
          used |= 1u << st;
          uint8_t* sp = dsm + L.stages + st * kHdStageBytes;
          mbar_arrive_expect_tx(&full[st], kHdStageBytes);
          tma_load_2d_hint(sp, &a.tm_codes, s * (kHdKs / 2), rb * kHdRows, &full[st], pol);
          tma_load_2d_hint(sp + kHdCodeBytes, &a.tm_scales, s * (kHdKs / 16), rb * kHdRows, &full[st], pol);
        }
    }
    if (!ok)
      for (int st = 0; st < kHdStages; ++st)
        if (used & (1u << st)) drain_wait(&full[st], last_par[st], a.wait_ns);
    return;
  }

  // consumers: stage x as f16 with a power-of-two scale per token
  const int w = warp - 1, NT = 32 * kHdConsumers;
  const int T = a.T;
  uint8_t* xs = dsm + L.xs;
  float* xscale = reinterpret_cast<float*>(dsm + L.xscale);
  if (w < T) {
    float amax = 0.f;
    for (int i = lane; i < d; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(a.x[(size_t)w * d + i])));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kAll, amax, o));
    // 2^-e with e = floor(log2 amax): the row's largest value lands in [1, 2)
    const int e = amax > 0.f ? ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127) : 0;
    if (lane == 0) xscale[w] = exp2f((float)e);
    const float inv = exp2f((float)-e);
    for (int i = lane * 2; i < d; i += 64) {
      const float x0 = __bfloat162float(a.x[(size_t)w * d + i]) * inv;
      const float x1 = __bfloat162float(a.x[(size_t)w * d + i + 1]) * inv;
      *reinterpret_cast<__half2*>(xs + w * L.x_pitch + i * 2) = __floats2half2_rn(x0, x1);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NT) : "memory");

  const int g = lane >> 2, t = lane & 3;
  const uint32_t xrow = smem_u32(xs) + (uint32_t)(g < T ? g : 0) * L.x_pitch + (uint32_t)t * 16;
  int mm = 0;
  for (int rb = lo + w; rb < hi; rb += kHdConsumers) {
    float acc[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    bool ok = true;
    for (int s = 0; s < KS; ++s, ++mm) {
      const int st = w * kHdPer + (mm % kHdPer);
      const uint32_t par = (mm / kHdPer) & 1;
      int good = 1;
      if (lane == 0) good = mbar_wait(&full[st], par, wc) ? 1 : 0;
      good = __shfl_sync(kAll, good, 0);
      if (!good) { ok = false; break; }
      while (!mbar_try_wait(&full[st], par)) {
      }
      const uint32_t sp = smem_u32(dsm + L.stages + st * kHdStageBytes);
      // row 16 j + g (and + 8) of the block: codes line r * 128 with 16-byte
      // chunk q stored at q ^ (r & 7) = q ^ g; scales 16 bytes per row
      const uint32_t cbase = sp + g * 128 + t * 4, sbase = sp + kHdCodeBytes + g * 16 + (t >> 1);
      const uint32_t xk = xrow + (uint32_t)s * kHdKs * 2;
#pragma unroll 2
      for (int q = 0; q < kHdKs / 32; ++q) {
        uint4 xv;
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(xv.x), "=r"(xv.y), "=r"(xv.z), "=r"(xv.w)
                     : "r"(xk + q * 64));
        const uint32_t coff = (uint32_t)((q ^ g) << 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t w0, w8, s0, s8;
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w0) : "r"(cbase + j * 2048 + coff));
          asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w8) : "r"(cbase + j * 2048 + 1024 + coff));
          asm volatile("ld.shared.u8 %0, [%1];" : "=r"(s0) : "r"(sbase + j * 256 + q * 2));
          asm volatile("ld.shared.u8 %0, [%1];" : "=r"(s8) : "r"(sbase + j * 256 + 128 + q * 2));
          uint32_t d0[4], d8[4];
          e2m1x8_f16x2(w0, d0);
          e2m1x8_f16x2(w8, d8);
          const uint32_t sc0 = e4m3_dup_f16x2(s0), sc8 = e4m3_dup_f16x2(s8);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            d0[i] = hmul2(d0[i], sc0);
            d8[i] = hmul2(d8[i], sc8);
          }
          mma_f16(acc[j], d0[0], d8[0], d0[1], d8[1], xv.x, xv.y);
          mma_f16(acc[j], d0[2], d8[2], d0[3], d8[3], xv.z, xv.w);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!ok) return;
    const float ts = __ldg(a.tscale);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int row = rb * kHdRows + j * 16 + g;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = t * 2 + q;
        if (n < T) {
          const float f = ts * xscale[n];
          a.logits[(size_t)n * a.V + row] = acc[j][q] * f;
          a.logits[(size_t)n * a.V + row + 8] = acc[j][2 + q] * f;
        }
      }
    }
  }
}

}  // namespace

size_t lm_head_smem_bytes(int d) { return hd_layout(d).total; }

cudaError_t launch_lm_head(const HeadArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = lm_head_smem_bytes(a.d);
  cudaError_t e = ensure_smem_limit(lm_head_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kHdThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  return cudaLaunchKernelEx(&cfg, lm_head_kernel, a);
}

}  // namespace moe

// ---------------------------------------------------------------- C ABI
using namespace moe;

struct moe_head {
  CUtensorMap tm_codes, tm_scales;
  int d = 0, V = 0, max_tokens = 0, num_sms = 0;
  const uint8_t* codes = nullptr;
  const uint8_t* scales = nullptr;
  const float* tscale = nullptr;
  unsigned* err = nullptr;
  uint64_t wait_ns = 0;
};

extern "C" {

moe_status moe_head_create(int32_t d, int32_t vocab, int32_t max_tokens, const uint8_t* codes, const uint8_t* scales,
                           const float* tscale, int32_t wait_timeout_ms, moe_head_handle* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  auto mis = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (d <= 0 || vocab <= 0 || max_tokens <= 0 || wait_timeout_ms < 0) return MOE_ERR_INVALID_ARG;
  if (!codes || !scales || !tscale || mis(codes) || mis(scales) || (reinterpret_cast<uintptr_t>(tscale) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (d % kHdKs != 0 || vocab % kHdRows != 0) return MOE_ERR_UNSUPPORTED;
  moe_head* h = new (std::nothrow) moe_head();
  if (!h) return MOE_ERR_OOM;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_CUDA;
  }
  if (lm_head_smem_bytes(d) > (size_t)optin) {
    delete h;
    return MOE_ERR_UNSUPPORTED;
  }
  void* e = nullptr;
  if (dev_malloc(&e, 256) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_OOM;
  }
  if (cudaMemset(e, 0, 256) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(e);
    delete h;
    return MOE_ERR_CUDA;
  }
  {
    const uint64_t cd[2] = {(uint64_t)d / 2, (uint64_t)vocab}, cs[1] = {(uint64_t)d / 2};
    const uint32_t cb[2] = {kHdKs / 2, kHdRows};
    const uint64_t sd[2] = {(uint64_t)d / 16, (uint64_t)vocab}, ss[1] = {(uint64_t)d / 16};
    const uint32_t sb[2] = {kHdKs / 16, kHdRows};
    if (!encode_tiled(&h->tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, codes, cd, cs, cb, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&h->tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, scales, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      cudaFree(e);
      delete h;
      return MOE_ERR_CUDA;
    }
  }
  h->err = static_cast<unsigned*>(e);
  h->d = d;
  h->V = vocab;
  h->max_tokens = max_tokens;
  h->codes = codes;
  h->scales = scales;
  h->tscale = tscale;
  h->wait_ns = (uint64_t)(wait_timeout_ms > 0 ? wait_timeout_ms : 2000) * 1000000ull;
  *out = h;
  return MOE_OK;
}

moe_status moe_head_forward(moe_head_handle h, const void* x, int32_t T, float* logits, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > h->max_tokens) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !logits || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(logits) & 15u))
    return MOE_ERR_INVALID_ARG;
  for (int t0 = 0; t0 < T; t0 += kHdMaxT) {
    HeadArgs a;
    a.tm_codes = h->tm_codes;
    a.tm_scales = h->tm_scales;
    a.codes = h->codes;
    a.scales = h->scales;
    a.tscale = h->tscale;
    a.x = static_cast<const __nv_bfloat16*>(x) + (size_t)t0 * h->d;
    a.logits = logits + (size_t)t0 * h->V;
    a.T = T - t0 < kHdMaxT ? T - t0 : kHdMaxT;
    a.d = h->d;
    a.V = h->V;
    a.err = h->err;
    a.wait_ns = h->wait_ns;
    if (launch_lm_head(a, h->num_sms, stream) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

moe_status moe_head_check(moe_head_handle h, cudaStream_t stream) {
  if (!h) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word && cudaMemset(h->err, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
  return (word & kErrTimeout) ? MOE_ERR_TIMEOUT : MOE_OK;
}

moe_status moe_head_destroy(moe_head_handle h) {
  if (!h) return MOE_OK;
  const cudaError_t e = cudaDeviceSynchronize();
  const cudaError_t f = cudaFree(h->err);
  delete h;
  return (e == cudaSuccess && f == cudaSuccess) ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
