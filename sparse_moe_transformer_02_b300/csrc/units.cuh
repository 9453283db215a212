// Unit lists of the tensor-core expert passes, written by the gather kernel
// that runs between the router and the gate/up pass.
//
// Entry u of a list (gate/up or down) is one work item (expert, weight-row
// tile, first grouped slot, slots): the shared expert's tiles come first
// (token tile major, row tile minor, each repeated rep times for the parts of
// a tile split along K), then each routed expert's tiles in expert order
// (token tile major, row tile minor, part minor).  The router stores for each
// list the first entry of every routed expert counted after the shared ones
// (ws.uprefix[list][e]; [list][E] is their number); the entries themselves
// are independent of one another, so every thread of the gather grid writes
// some of them.
#pragma once

#include "moe_internal.cuh"

namespace moe {

struct UnitBuild {
  int E, T, tn;         // routed experts, tokens, token tile
  int sh_tb;            // token tiles of the shared expert (0 without one)
  int mt[2];            // weight-row tiles of a routed expert (gate/up, down)
  int sh_mt[2];         // the same for the shared expert
  int rep[2];           // entries per tile (parts along K)
};

// Called by every thread of every block of the grid, after the grid-dependency
// wait on the router.
__device__ inline void build_unit_lists(const Workspace& ws, const UnitBuild& b) {
  __shared__ int pref[2][kMaxExperts + 1];
  for (int i = threadIdx.x; i < 2 * (b.E + 1); i += blockDim.x) {
    const int l = i / (b.E + 1);
    pref[l][i - l * (b.E + 1)] = __ldcg(ws.uprefix + i);
  }
  __syncthreads();
  const int sh0 = b.rep[0] * b.sh_mt[0] * b.sh_tb, sh1 = b.rep[1] * b.sh_mt[1] * b.sh_tb;
  const int tot0 = sh0 + pref[0][b.E], tot = tot0 + sh1 + pref[1][b.E];
  for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < tot; g += gridDim.x * blockDim.x) {
    const int l = g < tot0 ? 0 : 1, j = l ? g - tot0 : g;
    const int sh = l ? sh1 : sh0, rep = b.rep[l];
    TcUnit un;
    if (j < sh) {
      const int base = j / rep, tb = base / b.sh_mt[l], m = base - tb * b.sh_mt[l];
      un = TcUnit{b.E, m, tb * b.tn, min(b.tn, b.T - tb * b.tn)};
    } else {
      // owner: the last expert whose first entry is <= r (experts without
      // entries share their first entry with the next expert)
      const int r = j - sh;
      int lo = 0, hi = b.E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[l][mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      const int q = (r - pref[l][lo]) / rep, tb = q / b.mt[l], m = q - tb * b.mt[l];
      const int c = __ldcg(ws.counts + lo), o = __ldcg(ws.offsets + lo);
      un = TcUnit{lo, m, o + tb * b.tn, min(b.tn, c - tb * b.tn)};
    }
    (l ? ws.units_dn : ws.units_gu)[j] = un;
  }
}

}  // namespace moe
