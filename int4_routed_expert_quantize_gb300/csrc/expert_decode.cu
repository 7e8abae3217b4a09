// Host side of the decode expert kernels: the shared-memory plans (kernels and host agree on
// the carve-up), the grid of the down kernel, and the dispatch to the kernel instances of the
// handle's weight width (expert_decode.cuh; one translation unit per width).
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_internal.h"
#include "coli_select.cuh"

namespace coli {

static inline int align16(int x) { return (x + 15) & ~15; }

static long max_union_slots(int T, int K, int E, int n_shared) {
  return (long)(T * K < E ? T * K : E) + (n_shared ? 1 : 0);
}

GateupPlan gateup_plan(int d, int f, int T, int K, int E, int n_shared, int grid, int wbits) {
  GateupPlan p;
  const int nbd = d / kQB, nhb = f / 32;
  p.stage_bytes = gu_rows_per_stage(wbits) * 2 * (d * wbits / 8);
  p.xs_bytes = align16(T * d);
  p.aux_bytes = align16(T * nbd * 8);
  p.hs_bytes = align16((wbits == 8 ? 2 : 1) * 2 * 32 * T * 4);
  // Units a CTA can receive.  The cost split hands CTA c the routed units whose cost prefix lies
  // in [t_c, t_{c+1}) plus at most one unit past it, and t_{c+1} - t_c <= (total cost)/grid + 1;
  // with gu_unit_cost(np) <= kGuCostPair*np + kGuCostBytes and at most P pairs over the slots,
  // the total cost is at most nhb*(kGuCostPair*P + kGuCostBytes*slots).  So the routed units of a
  // CTA are at most (that/grid + 2 + cost(T)) / cost(1) + 1, and its shared-expert units at most
  // ceil(nhb/grid).
  const long slots = max_union_slots(T, K, E, n_shared);
  const long P = (long)T * K + (n_shared ? T : 0);
  const long cmax = (long)nhb * (kGuCostPair * P + kGuCostBytes * slots);
  const long wmax = gu_unit_cost(T), wmin = gu_unit_cost(1);
  p.max_units = (int)((cmax / grid + 2 + wmax) / wmin + 1 + (nhb + grid - 1) / grid) + 2;
  p.tab_bytes = align16(p.max_units * kGuTabBytes);
  p.sel_bytes = align16(sel_bytes(T, E));
  const int fixed =
      2 * kMaxStages * 8 + p.xs_bytes + p.aux_bytes + p.hs_bytes + p.tab_bytes + p.sel_bytes;
  int nst = (kSmemLimit - fixed) / p.stage_bytes;
  p.nst = nst > kMaxStages ? kMaxStages : nst;
  p.total = p.nst * p.stage_bytes + fixed;
  return p;
}

// per-CTA tables of the down kernel: the selection (coli_select.cuh) and the down-row scales of
// this CTA's rows for every union slot.  A ring stage holds one chunk of down rows of one union
// expert (w_bytes at most) and then the h codes, block scales and code sums of that expert's
// pairs (at most T pairs: a routed expert serves each token once, the shared one every token).
DownPlan down_plan(int d, int f, int T, int K, int E, int n_shared, int grid, int wbits) {
  DownPlan p;
  const int P = T * K + (n_shared ? T : 0);
  const int nbf = f / kQB;
  p.max_rows = (d + grid - 1) / grid;  // rows of the largest CTA range
  const int cap = dn_chunk_cap(wbits);
  const int chunk = p.max_rows < cap ? p.max_rows : cap;
  p.w_bytes = align16(chunk * (f * wbits / 8));
  p.stage_bytes = p.w_bytes + T * (f + 8 * nbf);
  p.es_bytes = align16(chunk * P * 4);
  p.max_slots = (int)max_union_slots(T, K, E, n_shared);
  p.tab_bytes = align16(p.max_slots * p.max_rows * 4);
  p.sel_bytes = align16(sel_bytes(T, E));
  const int fixed = 3 * kMaxStages * 8 + p.es_bytes + p.tab_bytes + p.sel_bytes;
  int nst = (kSmemLimit - fixed) / p.stage_bytes;
  p.nst = nst > kMaxStages ? kMaxStages : nst;
  p.total = p.nst * p.stage_bytes + fixed;
  return p;
}

int down_grid(int d, int num_sms) { return d < num_sms ? d : num_sms; }

cudaError_t configure_expert_kernels() {
  cudaError_t e = configure_gateup_kernels_wb<4>();
  if (e == cudaSuccess) e = configure_gateup_kernels_wb<8>();
  if (e == cudaSuccess) e = configure_gateup_kernels_wb<2>();
  if (e == cudaSuccess) e = configure_down_kernels_wb<4>();
  if (e == cudaSuccess) e = configure_down_kernels_wb<8>();
  if (e == cudaSuccess) e = configure_down_kernels_wb<2>();
  return e;
}

cudaError_t launch_gateup_decode(const Shape& s, const Store& st, const Work& w,
                                 const ExpertDebug& dbg, int num_sms, bool pdl,
                                 cudaStream_t stream) {
  switch (s.wbits) {
    case 4: return launch_gateup_decode_wb<4>(s, st, w, dbg, num_sms, pdl, stream);
    case 8: return launch_gateup_decode_wb<8>(s, st, w, dbg, num_sms, pdl, stream);
    case 2: return launch_gateup_decode_wb<2>(s, st, w, dbg, num_sms, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down_decode(const float* x, float* y, const Shape& s, const Store& st,
                               const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                               cudaStream_t stream) {
  switch (s.wbits) {
    case 4: return launch_down_decode_wb<4>(x, y, s, st, w, dbg, num_sms, pdl, stream);
    case 8: return launch_down_decode_wb<8>(x, y, s, st, w, dbg, num_sms, pdl, stream);
    case 2: return launch_down_decode_wb<2>(x, y, s, st, w, dbg, num_sms, pdl, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace coli
