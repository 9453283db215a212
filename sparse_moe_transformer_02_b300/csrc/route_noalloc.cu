// moe_route_noalloc: routing (router logits, top-k, renormalised gates,
// per-expert counts) for callers that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not available or not
// allowed -- plugins whose host process owns every device allocation, runtimes
// that forbid allocation after start-up, or latency-critical paths that must
// not call an allocator (cudaMalloc may synchronise the device).  Such callers
// cannot create a handle (moe_create allocates the workspace), so this entry
// point takes the router weights directly and keeps its scratch in one
// fixed-size array that lives in the library's own device image.
//
// The scratch array is shared by every call on a device and keeps the
// previous call's contents; the words that must start at zero (the routing
// kernel's tickets) are cleared by each call.  Calls that overlap
// on the GPU (different streams, or several host threads) race on it and must
// be serialised by the caller.
//
// It launches the same small-batch routing kernel as moe_route, with its
// workspace pointers aimed into the static array.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kNoAllocMaxT = kSmallT;   // 64 tokens per call
constexpr size_t kAlign = 256;
constexpr size_t up(size_t n) { return (n + kAlign - 1) / kAlign * kAlign; }

// Layout of the scratch array (sized for the largest E, k and T accepted).
constexpr size_t kOffLogits = 0;
constexpr size_t kOffCounts = kOffLogits + up((size_t)kNoAllocMaxT * kMaxExperts * 4);
constexpr size_t kOffOffsets = kOffCounts + up((kMaxExperts + 1) * 4);
constexpr size_t kOffActive = kOffOffsets + up((kMaxExperts + 2) * 4);
constexpr size_t kOffTok = kOffActive + up((kMaxExperts + 1) * 4);
constexpr size_t kOffSrc = kOffTok + up((size_t)kNoAllocMaxT * kMaxTopK * 4);
constexpr size_t kOffSlot = kOffSrc + up((size_t)kNoAllocMaxT * kMaxTopK * 4);
constexpr size_t kOffTicket = kOffSlot + up((size_t)kNoAllocMaxT * kMaxTopK * 4);
constexpr size_t kScratchBytes = kOffTicket + kAlign;     // about 144 KiB

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

// Device address of g_route_scratch, looked up once per device.  The cache
// assumes each device's context lives as long as the process: after a
// cudaDeviceReset the module is loaded again and the array may move, so a
// process that resets a device must not call moe_route_noalloc on it again.
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_route_noalloc(const void* x, int32_t T, int32_t d, int32_t num_experts, int32_t top_k,
                                        int32_t act_dtype, const float* router_w, const float* router_b,
                                        int32_t* idx, float* gate, int32_t* counts, cudaStream_t stream) {
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !idx || !gate) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > kNoAllocMaxT) return MOE_ERR_INVALID_ARG;           // beyond the scratch array's size
  if (num_experts < 1 || num_experts > kMaxExperts || top_k < 1 || top_k > kMaxTopK || top_k > num_experts)
    return MOE_ERR_INVALID_ARG;
  if (d <= 0 || d % 64 != 0 || d > kMaxHidden) return MOE_ERR_INVALID_ARG;
  if (act_dtype != MOE_F32 && act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(router_w) & 15u) ||
      (reinterpret_cast<uintptr_t>(router_b) & 3u) || (reinterpret_cast<uintptr_t>(idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(gate) & 3u) || (reinterpret_cast<uintptr_t>(counts) & 3u))
    return MOE_ERR_INVALID_ARG;

  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  uint8_t* s = static_cast<uint8_t*>(base);
  RouteArgs a;
  a.x = x;
  a.T = T;
  a.d = d;
  a.E = num_experts;
  a.k = top_k;
  a.act_bf16 = act_dtype == MOE_BF16;
  a.Wr = router_w;
  a.b = router_b;
  a.idx = idx;
  a.gate = gate;
  a.counts_out = counts;
  a.build_tc_units = 0;
  a.dn_rows = kTcBM;
  a.tile_n = kTcBN;
  a.gu_split = 1;
  a.F = 0;
  a.Fs = 0;
  a.has_shared = 0;
  Workspace& w = a.ws;
  w = Workspace{};
  w.logits = reinterpret_cast<float*>(s + kOffLogits);
  w.counts = reinterpret_cast<int32_t*>(s + kOffCounts);
  w.offsets = reinterpret_cast<int32_t*>(s + kOffOffsets);
  w.active = reinterpret_cast<int32_t*>(s + kOffActive);
  w.tok_of_slot = reinterpret_cast<int32_t*>(s + kOffTok);
  w.src_of_slot = reinterpret_cast<int32_t*>(s + kOffSrc);
  w.slot_of = reinterpret_cast<int32_t*>(s + kOffSlot);
  w.counters = reinterpret_cast<uint32_t*>(s + kOffTicket);
  // The previous call's tickets may be anything if it was interrupted: clear
  // them (the grid ticket and one per 8-token chunk).
  if (cudaMemsetAsync(w.counters, 0, kAlign, stream) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (launch_route(a, 0, stream, nullptr) != cudaSuccess) {
    cudaGetLastError();   // leave no launch error behind for the caller's next check
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
