// Internal types shared by the host API (moe_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "moe.h"

namespace moe {

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 8;
constexpr int kSmallT = 64;          // largest T the single-kernel small-batch router handles
constexpr int kGemvChunkT = 64;      // GEMV path: tokens per pass (longer batches run in passes)
constexpr int kFinRows = 32;         // GEMV down: rows finalised together by the last contributor
constexpr int kTcBN = 128;           // tcgen05 path: largest token tile (MMA N)
constexpr int kTcBM = 128;           // tcgen05 path: weight rows per tile (MMA M)
constexpr int kTcBK = 64;            // tcgen05 path: reduction step per stage (128 bytes of bf16)
constexpr unsigned kErrTimeout = 1u << 5;

// One unit of tcgen05 work: expert (E = the shared expert), weight-row tile,
// first slot (for the shared expert: first token) and token count (<= kTcBN).
struct TcUnit {
  int32_t expert, m_tile, slot0, n;
};

// Device workspace owned by a handle.
struct Workspace {
  int32_t* idx;           // [max_T][k]   routing when the caller passes no buffer
  float* gate;            // [max_T][k]
  float* logits;          // [kSmallT][E] small-batch router scratch
  uint32_t* sel;          // [ceil(max_T/32)][E] token-selection bitmap words (large-batch router)
  int32_t* counts;        // [E + 1]
  int32_t* offsets;       // [E + 2]
  int32_t* tok_of_slot;   // [max_T * k]  token of each grouped slot
  int32_t* src_of_slot;   // [max_T * k]  original slot t * k + j of each grouped slot
  int32_t* slot_of;       // [max_T * k]
  int32_t* active;        // [E + 1] routed experts with tokens, ascending; active[E] = how many
  TcUnit* units_gu;       // tcgen05 gate/up units
  TcUnit* units_dn;       // tcgen05 down units
  int32_t* n_units;       // [2] unit counts (gate/up, down)
  float* h32;             // [min(max_T, kGemvChunkT) * (k + 1)][F_max] GEMV intermediate
  __nv_bfloat16* h16;     // [max(max_T, ...) * (k + 1)][F_max] bf16 intermediate (tcgen05 and bf16 GEMV)
  __nv_bfloat16* xp;      // [max_T * k][d] tcgen05 slot-ordered copy of the routed activations
  float* ypart;           // [min(max_T, kGemvChunkT) * (k + 1)][d] GEMV down partials
  float* yacc;            // [max_T][d] tcgen05 fp32 accumulator
  uint32_t* counters;     // router ticket
  uint32_t* fin;          // [kGemvChunkT][d / 32] GEMV down completion counts (kept at zero between calls)
  unsigned int* err;      // device error word
  void* x_stage;          // [max_T][d] moe_forward_host staging
  void* y_stage;
  size_t bytes;           // total allocated
};

// Optional per-launch timing: event pairs recorded around each kernel.
struct Prof {
  std::vector<cudaEvent_t> ev;     // pool, 2 per launch
  std::vector<int> kid;            // kernel id of each recorded pair
  int pending = -1;
  bool on() const { return !ev.empty(); }
  void begin(int id, cudaStream_t s) {
    pending = -1;
    if (!on() || 2 * (kid.size() + 1) > ev.size()) return;
    pending = id;
    cudaEventRecord(ev[2 * kid.size()], s);
  }
  void end(cudaStream_t s) {
    if (pending < 0) return;
    cudaEventRecord(ev[2 * kid.size() + 1], s);
    kid.push_back(pending);
    pending = -1;
  }
};

// Parameters shared by the routing kernels.
struct RouteArgs {
  const void* x;          // [T][d] f32 or bf16
  int T, d, E, k;
  int act_bf16;
  const float* Wr;        // [E][d]
  const float* b;         // [E] or nullptr
  int32_t* idx;           // [T][k]
  float* gate;            // [T][k]
  int32_t* counts_out;    // [E] or nullptr
  Workspace ws;
  int build_tc_units;     // also build tcgen05 unit lists
  int F, Fs;              // widths (for unit lists)
  int has_shared;
};

// Parameters of the GEMV expert kernels.
struct GemvArgs {
  const void* x;          // [T][d]
  void* y;                // [T][d]
  const int32_t* idx;     // [T][k] (unused by the kernels; the grouping carries it)
  const float* gate;      // [T][k]
  int T, d, F, Fs, E, k;
  int act_bf16, add_residual;
  const void* wg; const void* wu; const void* wd;       // routed stacks
  const void* sg; const void* su; const void* sd;       // shared
  const uint8_t* sc_g; const uint8_t* sc_u; const uint8_t* sc_d;   // nvfp4 block scales
  const uint8_t* ssc_g; const uint8_t* ssc_u; const uint8_t* ssc_d;
  const float* ts_g; const float* ts_u; const float* ts_d;         // nvfp4 tensor scales
  const float* tss_g; const float* tss_u; const float* tss_d;
  Workspace ws;
};

// Launchers (return the launch status).
cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s, Prof* prof);
cudaError_t launch_gemv(const GemvArgs& a, int wfmt, int num_sms, cudaStream_t s, Prof* prof, uint64_t wait_ns);
// Shapes the GEMV kernels are built for: rows of d values span 1, 2, 4 or 8
// x 512 bytes; rows of F values span 16, 32, 64 or 128 chunks of 16 bytes;
// the shared expert, if any, has the routed width.
bool gemv_supported(int wfmt, int d, int F, int Fs);
cudaError_t launch_debug_wait(unsigned int* err, uint64_t limit_ns, cudaStream_t s);

struct TcArgs {
  const CUtensorMap* tm_x;      // x [T][d] (box 64 x kTcBN)
  const CUtensorMap* tm_xp;     // slot-ordered x copy [max_T*k][d] (box 64 x kTcBN)
  const CUtensorMap* tm_wg;     // [E*F][d]
  const CUtensorMap* tm_wu;
  const CUtensorMap* tm_sg;     // [Fs][d]
  const CUtensorMap* tm_su;
  const CUtensorMap* tm_wd;     // [E*d][F]
  const CUtensorMap* tm_sd;     // [d][Fs]
  const CUtensorMap* tm_h;      // [slots][F_max] (box 64 x kTcBN)
  const void* x;
  void* y;
  const float* gate;            // [T][k]
  int T, d, F, Fs, E, k, add_residual;
  Workspace ws;
  uint64_t wait_ns;
  int max_units_gu, max_units_dn;
};
cudaError_t launch_tc(const TcArgs& a, int num_sms, cudaStream_t s, Prof* prof);
int tc_max_units_gu(int T, int d, int F, int Fs, int E, int k);
int tc_max_units_dn(int T, int d, int F, int Fs, int E, int k);

}  // namespace moe
