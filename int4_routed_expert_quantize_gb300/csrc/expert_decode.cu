// Expert kernels of the decode path (a few tokens per call): the fused int4 x int8 gate/up
// projection with SwiGLU and h re-quantisation, and the down projection with the fixed-order
// routing-weighted combine.  Both are HBM-bound streams over the union experts' weights
// ("colibrì 架构概述" §5: gate/up/SiLU/down on the IDOT fast path, then the shared expert;
// README: each distinct expert of a batch is read once).
//
// Structure of both kernels: a persistent grid (one CTA per SM) splits the work into equal
// contiguous ranges; in each CTA one producer lane streams the weight rows of its range
// through a ring of shared-memory stages with bulk copies (cp.async.bulk, mbarrier
// completion, L2 evict-first), and 8 consumer warps reduce each row: lane g owns the g-th of
// 32 contiguous groups of 32-element blocks, computes exact int32 block dots with dp4a, folds
// them with fma in block order, and the warp's xor butterfly adds the 32 group partials in
// pairwise-tree order.  All waits are bounded (see coli_device.cuh).
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_select.cuh"

namespace coli {

static inline int align16(int x) { return (x + 15) & ~15; }

// per-CTA unit table of the gate/up kernel: slot, expert, first pair, pair count, the pairs'
// tokens (T at most) and the 32 gate + 32 up row scales
constexpr int kGuTabInts = 5 + kDecodeTmax;  // slot, expert, first pair, pairs, hb, tokens
constexpr int kGuTabBytes = (kGuTabInts + 64) * 4;
// Relative cost of one gate/up unit whose union slot serves np tokens: its bytes take the same
// time whatever np (kGuCostBytes), its dots grow with np (kGuCostPair each); the larger bounds
// the unit.  The routed units are split over the CTAs by this cost, not by count.  Calibrated
// on the four-token GLM layer: a four-token unit measured about 3.6 times a one-token unit, and
// the step time keeps improving up to a model ratio of about 4.4, flat beyond.
constexpr int kGuCostBytes = 20, kGuCostPair = 22;
__host__ __device__ constexpr int gu_unit_cost(int np) {
  return kGuCostPair * np > kGuCostBytes ? kGuCostPair * np : kGuCostBytes;
}

static long max_union_slots(int T, int K, int E, int n_shared) {
  return (long)(T * K < E ? T * K : E) + (n_shared ? 1 : 0);
}

GateupPlan gateup_plan(int d, int f, int T, int K, int E, int n_shared, int grid) {
  GateupPlan p;
  const int nbd = d / kQB, nhb = f / 32;
  p.stage_bytes = kGuRps * d;
  p.xs_bytes = align16(T * d);
  p.aux_bytes = align16(T * nbd * 8);
  p.hs_bytes = align16(2 * 32 * T * 4);
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
DownPlan down_plan(int d, int f, int T, int K, int E, int n_shared, int grid) {
  DownPlan p;
  const int P = T * K + (n_shared ? T : 0);
  const int nbf = f / kQB;
  p.max_rows = (d + grid - 1) / grid;  // rows of the largest CTA range
  const int chunk = p.max_rows < kDownChunk ? p.max_rows : kDownChunk;
  p.w_bytes = align16(chunk * (f / 2));
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

struct GateupArgs {
  Shape s;
  Store st;
  Work w;
  ExpertDebug dbg;
  GateupPlan pl;
};

struct DownArgs {
  Shape s;
  Store st;
  Work w;
  ExpertDebug dbg;
  DownPlan pl;
  const float* x;
  float* y;
};

// ------------------------------------------------------------------ gate/up + SwiGLU ------
// Work unit = (union slot, 32-row block of h): 32 row pairs [gate row | up row] of one expert,
// streamed as 4 stages of 8 row pairs, which yields one int8 block of h for every token of the
// slot's bucket.  The units are split evenly over the CTAs with the shared expert's units first
// in every CTA that has some: those are known before routing, so they are prefetched before
// the kernel waits for the routing grid.  Warp w reduces row pair w of every stage; when a
// unit's 32 rows are done the CTA re-quantises them (one warp per token).
// One gate/up row pair of one stage dotted with NP tokens' codes (the union slot's bucket):
// each of the warp's G blocks is loaded and split into nibble halves once for all tokens.
struct GuRow {
  const uint8_t* grow;  // the row pair in the stage: gate row, then up row (d/2 bytes each)
  const uint8_t* xs;    // the tokens' codes in lane-group order
  const float* dxs;
  const int* nsx;
  int d, nbd, A, lane;
  float sg, su;  // the row's gate and up scales
  int row, f, p0;
  float* hrow;   // h of this row for the slot's tokens (stride 1)
  ExpertDebug dbg;
};

template <int G, int NP, bool DBG>
__device__ __forceinline__ void gu_multi(const GuRow& r, const int (&toks)[kDecodeTmax]) {
  float pg[NP], pu[NP];
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    pg[q] = 0.0f;
    pu[q] = 0.0f;
  }
  const bool on = r.lane < r.A;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    uint4 wg = make_uint4(0, 0, 0, 0), wu = make_uint4(0, 0, 0, 0);
    if (on) {
      const int off = store_chunk(r.lane, i, G) * 16;
      wg = *reinterpret_cast<const uint4*>(r.grow + off);
      wu = *reinterpret_cast<const uint4*>(r.grow + r.d / 2 + off);
    }
    uint32_t gl[4], gh[4], ul[4], uh[4];
    split_nibbles(wg, gl, gh);
    split_nibbles(wu, ul, uh);
#pragma unroll
    for (int q = 0; q < NP; ++q) {
      const int t = toks[q];
      uint32_t xq[8];
      float dq = 0.0f;
      int nq = 0;
      if (on) {
        const uint8_t* base = r.xs + (long)t * r.d + (i * r.A + r.lane) * 16;
        const uint4 v0 = *reinterpret_cast<const uint4*>(base);
        const uint4 v1 = *reinterpret_cast<const uint4*>(base + r.nbd * 16);
        xq[0] = v0.x; xq[1] = v0.y; xq[2] = v0.z; xq[3] = v0.w;
        xq[4] = v1.x; xq[5] = v1.y; xq[6] = v1.z; xq[7] = v1.w;
        dq = r.dxs[t * r.nbd + r.lane * G + i];
        nq = r.nsx[t * r.nbd + r.lane * G + i];
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xq[k] = 0u;
      }
      const int ag = block_dot_split(gl, gh, xq, nq);
      const int au = block_dot_split(ul, uh, xq, nq);
      pg[q] = __fmaf_rn(dq, __int2float_rn(ag), pg[q]);
      pu[q] = __fmaf_rn(dq, __int2float_rn(au), pu[q]);
      if (DBG && r.dbg.Ag != nullptr && on) {
        const long o = ((long)(r.p0 + q) * r.f + r.row) * r.nbd + r.lane * G + i;
        r.dbg.Ag[o] = ag;
        r.dbg.Au[o] = au;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    const float tg = warp_tree_sum(pg[q]), tuu = warp_tree_sum(pu[q]);
    const float g = __fmul_rn(r.sg, tg), u = __fmul_rn(r.su, tuu);
    if (r.lane == 0) {
      r.hrow[q] = canon_silu_mul(g, u);
      if (DBG && r.dbg.g != nullptr) {
        r.dbg.g[(long)(r.p0 + q) * r.f + r.row] = g;
        r.dbg.u[(long)(r.p0 + q) * r.f + r.row] = u;
      }
    }
  }
}

template <int G, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) gateup_decode_kernel(const GateupArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  const int d = a.s.d, f = a.s.f, T = a.s.T;
  const int nbd = d >> 5, A = nbd / G, nhb = f >> 5;
  const GateupPlan& pl = a.pl;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.nst * pl.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint8_t* xs = reinterpret_cast<uint8_t*>(empty + kMaxStages);  // [T][2 halves][chunks][16]
  float* dxs = reinterpret_cast<float*>(xs + pl.xs_bytes);         // [T][nbd]
  int* nsx = reinterpret_cast<int*>(dxs + T * nbd);                // [T][nbd]  -8*sum(codes)
  float* hs = reinterpret_cast<float*>(xs + pl.xs_bytes + pl.aux_bytes);  // [2][32][T]
  int* tab = reinterpret_cast<int*>(xs + pl.xs_bytes + pl.aux_bytes + pl.hs_bytes);
  Sel sel = sel_carve(xs + pl.xs_bytes + pl.aux_bytes + pl.hs_bytes + pl.tab_bytes, T, a.s.E);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int SPU = 32 / kGuRps;
  const int G_ = gridDim.x, c = blockIdx.x;

  // shared-expert units of this CTA: [a0, a1) of the nhb units of store slot E
  const int UA = a.s.n_shared ? nhb : 0;
  const int a0 = (int)((long)UA * c / G_), a1 = (int)((long)UA * (c + 1) / G_);
  const int na = a1 - a0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < pl.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNW);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t pol = l2_evict_first_policy();
  const bool producer = (warp == kNW && lane == 0);
  int issued = 0;
  if (producer) {
    for (; issued < na * SPU && issued < pl.nst; ++issued) {
      const int unit = a0 + issued / SPU;
      const int sub = issued % SPU;
      const uint8_t* src = a.st.wgu + ((long)a.s.E * f + unit * 32 + sub * kGuRps) * (long)d;
      mbar_expect_tx(&full[issued], (uint32_t)pl.stage_bytes);
      bulk_g2s(ring + issued * pl.stage_bytes, src, (uint32_t)pl.stage_bytes, &full[issued], pol);
    }
  }
  // the selection bias does not depend on the routing grid
  if (a.st.bias)
    for (int i = threadIdx.x; i < a.s.E; i += blockDim.x) sel.bias[i] = a.st.bias[i];
  // the routing grid is complete and its results visible from here on
  griddep_wait();
  griddep_launch_dependents();

  // Every CTA selects the experts itself from the router's scores: the score loads are issued
  // first (plain loads: the bulk-copy queue still holds the shared expert's prefetch), the
  // token codes are staged meanwhile, then top-K and union run in shared memory.  CTA 0 also
  // publishes the selection for the down grid and the debug dumps.
  const int TE = T * a.s.E;
  float sreg[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < TE) sreg[k] = __ldcg(a.w.scores + i);
  }
  // every token's codes, with block b = g*G + i at chunk i*A + g; the two 16-byte halves of a
  // chunk live in separate planes so a warp's 16-byte loads are consecutive.  Each thread
  // issues the loads of 4 blocks before storing any.
  for (int i0 = threadIdx.x; i0 < T * nbd; i0 += 4 * blockDim.x) {
    uint4 q0[4], q1[4];
    float dv[4];
    int sv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = i0 + k * blockDim.x;
      if (idx < T * nbd) {
        const int t = idx / nbd, b = idx - t * nbd;
        const uint4* src = reinterpret_cast<const uint4*>(a.w.qx + (long)t * d + b * 32);
        q0[k] = __ldcg(src);
        q1[k] = __ldcg(src + 1);
        dv[k] = __ldcg(a.w.dx + (long)t * nbd + b);
        sv[k] = __ldcg(a.w.sx + (long)t * nbd + b);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int idx = i0 + k * blockDim.x;
      if (idx < T * nbd) {
        const int t = idx / nbd, b = idx - t * nbd;
        const int g = b / G, i = b - g * G;
        uint8_t* base = xs + (long)t * d + (i * A + g) * 16;
        *reinterpret_cast<uint4*>(base) = q0[k];
        *reinterpret_cast<uint4*>(base + nbd * 16) = q1[k];
        dxs[idx] = dv[k];
        nsx[idx] = -8 * sv[k];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < TE) sel.sc[i] = sreg[k];
  }
  for (int i = threadIdx.x + 4 * blockDim.x; i < TE; i += blockDim.x) sel.sc[i] = __ldcg(a.w.scores + i);
  __syncthreads();
  select_union(a.s, sel, a.st.bias != nullptr);
  if (blockIdx.x == 0) sel_publish(a.s, sel, a.w);
  const int nu = *sel.nu;

  // routed units of this CTA: the routed units (slot-major, union order) are split by cost
  // (gu_unit_cost of the slot's pairs).  CTA c's share ends where the cost prefix of all units,
  // shared ones included, reaches c+1 G-ths of the total; when one CTA's shared units could
  // outweigh an average share (so the ranges might not increase with c) the routed units alone
  // are split by cost.
  const int nr = nu - (a.s.n_shared ? 1 : 0), UB = nr * nhb;
  const long wsh = a.s.n_shared ? gu_unit_cost(sel.u_off[nu] - sel.u_off[nu - 1]) : 0;
  long cr = 0;  // cost of all routed units
  for (int sl = 0; sl < nr; ++sl) cr += (long)nhb * gu_unit_cost(sel.u_off[sl + 1] - sel.u_off[sl]);
  const long call = cr + (long)UA * wsh;
  const long na_max = (UA + G_ - 1) / G_;
  const bool with_shared = call >= (long)G_ * (na_max * wsh + 1);
  // first routed unit whose cost prefix reaches cost target t
  auto first_at = [&](long t) -> int {
    if (t <= 0) return 0;
    long acc = 0;
    for (int sl = 0; sl < nr; ++sl) {
      const long w = gu_unit_cost(sel.u_off[sl + 1] - sel.u_off[sl]);
      if (acc + w * nhb >= t) return sl * nhb + (int)((t - acc + w - 1) / w);
      acc += w * nhb;
    }
    return UB;
  };
  auto target = [&](int cc) -> long {
    if (!with_shared) return cr * cc / G_;
    const long as = (long)UA * cc / G_;  // shared units of CTAs before cc
    return call * cc / G_ - as * wsh;
  };
  const int b0 = first_at(target(c)), b1 = first_at(target(c + 1));
  const int nunit = na + (b1 - b0);
  const int nstage = nunit * SPU;

  // local unit index -> (union slot, 32-row block)
  auto unit_of = [&](int lu, int& slot, int& hb) {
    if (lu < na) {
      slot = nu - 1;
      hb = a0 + lu;
    } else {
      const int r = b0 + (lu - na);
      slot = r / nhb;
      hb = r - slot * nhb;
    }
  };

  if (warp == kNW) {
    // ---------------- producer: one lane streams the remaining stages
    if (producer) {
      int s = issued % pl.nst;
      uint32_t ph = (uint32_t)((issued / pl.nst) & 1);
      for (int it = issued; it < nstage; ++it) {
        if (it >= pl.nst && !mbar_wait_bounded(&empty[s], ph ^ 1u, &abort_flag, a.w.status)) break;
        int slot, hb;
        unit_of(it / SPU, slot, hb);
        const uint8_t* src =
            a.st.wgu + ((long)sel.u_ids[slot] * f + hb * 32 + (it % SPU) * kGuRps) * (long)d;
        mbar_expect_tx(&full[s], (uint32_t)pl.stage_bytes);
        bulk_g2s(ring + (long)s * pl.stage_bytes, src, (uint32_t)pl.stage_bytes, &full[s], pol);
        issued = it + 1;
        if (++s == pl.nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (abort_flag) drain_fills(full, pl.nst, issued);
    }
  } else {
    // unit table: every value a stage needs, loaded once (one round of memory latency)
    for (int lu = warp; lu < nunit && lu < pl.max_units; lu += kNW) {
      int slot, hb;
      unit_of(lu, slot, hb);
      int* tu = tab + lu * (kGuTabInts + 64);
      const int ex = sel.u_ids[slot];
      const int p0 = sel.u_off[slot];
      const int np = sel.u_off[slot + 1] - p0;
      if (lane == 0) {
        tu[0] = slot;
        tu[1] = ex;
        tu[2] = p0;
        tu[3] = np;
        tu[4] = hb;
      }
      if (lane < np && lane < kDecodeTmax) tu[5 + lane] = sel.p_tok[p0 + lane];
      const float* scx = a.st.sc + (long)ex * (2 * f + d);
      float* tsc = reinterpret_cast<float*>(tu + kGuTabInts);
      tsc[lane] = scx[hb * 32 + lane];
      tsc[32 + lane] = scx[f + hb * 32 + lane];
    }
    named_bar_sync(1, kNW * 32);

    // ---------------- consumers: warp `warp` takes row pair `warp` of every stage
    uint32_t xr[G][8];
    float dr[G];
    int nr[G];
    int cached_tok = -1;
    int s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nstage; ++it) {
      const int lu = it / SPU;
      const int sub = it % SPU;
      const int* tu = tab + lu * (kGuTabInts + 64);
      const int hb = tu[4];
      const int p0 = tu[2], np = tu[3];
      mbar_wait_bounded(&full[s], ph, &abort_flag, a.w.status);
      const int rr = sub * kGuRps + warp;
      const int row = hb * 32 + rr;
      const uint8_t* grow = ring + (long)s * pl.stage_bytes + (long)warp * d;
      const float* tsc = reinterpret_cast<const float*>(tu + kGuTabInts);
      const float sg = tsc[rr], su = tsc[32 + rr];
      if (np == 1) {
        // one token: its codes stay in registers while consecutive units serve the same token
        const int p = p0;
        const int t = tu[5];
        if (t != cached_tok) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            if (lane < A) {
              const uint8_t* base = xs + (long)t * d + (i * A + lane) * 16;
              const uint4 v0 = *reinterpret_cast<const uint4*>(base);
              const uint4 v1 = *reinterpret_cast<const uint4*>(base + nbd * 16);
              xr[i][0] = v0.x; xr[i][1] = v0.y; xr[i][2] = v0.z; xr[i][3] = v0.w;
              xr[i][4] = v1.x; xr[i][5] = v1.y; xr[i][6] = v1.z; xr[i][7] = v1.w;
              dr[i] = dxs[t * nbd + lane * G + i];
              nr[i] = nsx[t * nbd + lane * G + i];
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) xr[i][k] = 0u;
              dr[i] = 0.0f;
              nr[i] = 0;
            }
          }
          cached_tok = t;
        }
        float pg = 0.0f, pu = 0.0f;
#pragma unroll
        for (int i = 0; i < G; ++i) {
          uint4 wg = make_uint4(0, 0, 0, 0), wu = make_uint4(0, 0, 0, 0);
          if (lane < A) {
            const int off = store_chunk(lane, i, G) * 16;
            wg = *reinterpret_cast<const uint4*>(grow + off);
            wu = *reinterpret_cast<const uint4*>(grow + d / 2 + off);
          }
          const int ag = block_dot(wg, xr[i], nr[i]);
          const int au = block_dot(wu, xr[i], nr[i]);
          pg = __fmaf_rn(dr[i], __int2float_rn(ag), pg);
          pu = __fmaf_rn(dr[i], __int2float_rn(au), pu);
          if (DBG && a.dbg.Ag != nullptr && lane < A) {
            const long o = ((long)p * f + row) * nbd + lane * G + i;
            a.dbg.Ag[o] = ag;
            a.dbg.Au[o] = au;
          }
        }
        pg = warp_tree_sum(pg);
        pu = warp_tree_sum(pu);
        const float g = __fmul_rn(sg, pg), u = __fmul_rn(su, pu);
        if (lane == 0) {
          hs[((lu & 1) * 32 + rr) * T] = canon_silu_mul(g, u);
          if (DBG && a.dbg.g != nullptr) {
            a.dbg.g[(long)p * f + row] = g;
            a.dbg.u[(long)p * f + row] = u;
          }
        }
      } else {
        // several tokens: each block's weights are loaded and split into nibble halves once,
        // then dotted with every token's codes of that block; each token keeps its own fma
        // chain over the blocks in order (the token count is a template argument, so the
        // tokens' chains interleave with no branch between them)
        cached_tok = -1;
        int toks[kDecodeTmax];
#pragma unroll
        for (int q = 0; q < kDecodeTmax; ++q) toks[q] = q < np ? tu[5 + q] : 0;
        const GuRow r{grow, xs, dxs, nsx, d, nbd, A, lane, sg, su, row, f, p0,
                      hs + ((lu & 1) * 32 + rr) * T, DBG ? a.dbg : ExpertDebug{}};
        switch (np) {
          case 2: gu_multi<G, 2, DBG>(r, toks); break;
          case 3: gu_multi<G, 3, DBG>(r, toks); break;
          case 4: gu_multi<G, 4, DBG>(r, toks); break;
          case 5: gu_multi<G, 5, DBG>(r, toks); break;
          case 6: gu_multi<G, 6, DBG>(r, toks); break;
          case 7: gu_multi<G, 7, DBG>(r, toks); break;
          default: gu_multi<G, 8, DBG>(r, toks); break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with its row pair
      if (++s == pl.nst) {
        s = 0;
        ph ^= 1u;
      }
      if (sub == SPU - 1) {
        // the unit's 32 rows of h are complete: quantise one int8 block per token
        named_bar_sync(1, kNW * 32);
        for (int q = warp; q < np; q += kNW) {
          const float hv = hs[((lu & 1) * 32 + lane) * T + q];
          const float dd = __fdiv_rn(warp_max(fabsf(hv)), 127.0f);
          const int code = q8_code(hv, dd);
          const int p = p0 + q;
          a.w.hf[(long)p * f + hb * 32 + lane] = hv;
          a.w.qh[(long)p * f + hb * 32 + lane] = (int8_t)code;
          const int sq = warp_isum(code);
          if (lane == 0) {
            a.w.dh[(long)p * nhb + hb] = dd;
            a.w.sh[(long)p * nhb + hb] = sq;
          }
        }
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ down + combine --------
// CTA c owns the output rows [d*c/grid, d*(c+1)/grid) -- about d/grid rows, so every CTA streams
// the same number of bytes -- cut into chunks of at most kDownChunk rows.  A stage is one chunk
// of one union expert's down matrix (one contiguous bulk copy) followed by the h codes, block
// scales and code sums of that expert's pairs (three more copies, issued once the gate/up grid
// is complete).  The union is known when this grid starts (the router finished before the
// gate/up grid let it launch), so the weights of the first stages and the tables are loaded
// before waiting for the h codes.  Warp w owns rows w, w+8, ... of the chunk: every lane folds
// its group's block dots for up to 8 rows, and one transposed butterfly adds the 32 group
// partials of all 8 rows (the same pairwise tree per row as the single-row butterfly).  Once a
// chunk has seen every union expert the warp combines its rows for every token in the fixed
// order: shared expert first, then ranks 0..K-1.

__host__ __device__ inline int down_rows_begin(int d, int c, int grid) {
  return (int)((long)d * c / grid);
}

// The down rows of one stage (warp `warp`'s rows of the chunk) dotted with the h codes of NP
// consecutive pairs of the stage's union expert: each row block's weights are loaded and split
// once for all of them.
struct DnRows {
  const uint8_t* sbase;  // the warp's first row in the stage
  const uint8_t* hq;     // [np][f] h codes of the stage's pairs
  const float* hd;       // [np][nbf] their block scales
  const int* hsum;       // [np][nbf] their code sums
  const float* sdx;      // the warp's first down-row scale of the chunk (stride kNW)
  float* es;             // [chunk row][P] expert outputs
  int f, nbf, A, lane, warp, nj, jl, P, d, row0c;  // row0c: first output row of the chunk
  bool dry;
  ExpertDebug dbg;
};

// q: the first of the NP pairs within the stage, p: its index among all pairs
template <int GF, int NP, bool DBG>
__device__ __forceinline__ void dn_rows(const DnRows& r, int q, int p) {
  const bool on = r.lane < r.A;
  const int rb = r.f >> 1;
  uint32_t hr[NP][GF][8];
  float hdr[NP][GF];
  int hnr[NP][GF];
#pragma unroll
  for (int k = 0; k < NP; ++k) {
#pragma unroll
    for (int i = 0; i < GF; ++i) {
      if (on) {
        const uint8_t* base = r.hq + (long)(q + k) * r.f + (r.lane * GF + i) * 32;
        const uint4 v0 = *reinterpret_cast<const uint4*>(base);
        const uint4 v1 = *reinterpret_cast<const uint4*>(base + 16);
        hr[k][i][0] = v0.x; hr[k][i][1] = v0.y; hr[k][i][2] = v0.z; hr[k][i][3] = v0.w;
        hr[k][i][4] = v1.x; hr[k][i][5] = v1.y; hr[k][i][6] = v1.z; hr[k][i][7] = v1.w;
        hdr[k][i] = r.hd[(q + k) * r.nbf + r.lane * GF + i];
        hnr[k][i] = -8 * r.hsum[(q + k) * r.nbf + r.lane * GF + i];
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) hr[k][i][t] = 0u;
        hdr[k][i] = 0.0f;
        hnr[k][i] = 0;
      }
    }
  }
  float acc[NP][kDownRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kDownRowsPerWarp; ++j) {
#pragma unroll
    for (int k = 0; k < NP; ++k) acc[k][j] = 0.0f;
    if (j < r.nj) {
      const uint8_t* srow = r.sbase + (long)j * kNW * rb;
#pragma unroll
      for (int i = 0; i < GF; ++i) {
        uint4 wv = make_uint4(0, 0, 0, 0);
        if (on) wv = *reinterpret_cast<const uint4*>(srow + store_chunk(r.lane, i, GF) * 16);
        uint32_t lo[4], hi[4];
        split_nibbles(wv, lo, hi);
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int ai = block_dot_split(lo, hi, hr[k][i], hnr[k][i]);
          acc[k][j] = __fmaf_rn(hdr[k][i], __int2float_rn(ai), acc[k][j]);
          if (DBG && !r.dry && r.dbg.Ad != nullptr && on)
            r.dbg.Ad[((long)(p + k) * r.d + r.row0c + j * kNW + r.warp) * r.nbf + r.lane * GF + i] = ai;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const float v = warp_tree_sum8(acc[k], r.lane);
    if (!r.dry && r.lane < kDownRowsPerWarp && r.jl < r.nj) {
      const float e = __fmul_rn(r.sdx[r.jl * kNW], v);
      r.es[(r.jl * kNW + r.warp) * r.P + p + k] = e;
      if (DBG && r.dbg.e != nullptr) r.dbg.e[(long)(p + k) * r.d + r.row0c + r.jl * kNW + r.warp] = e;
    }
  }
}

template <int GF, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) down_decode_kernel(const DownArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  __shared__ __align__(8) uint64_t selbar;
  const int d = a.s.d, f = a.s.f, T = a.s.T, K = a.s.K;
  const int nbf = f >> 5, A = nbf / GF, rb = f >> 1;
  const DownPlan& pl = a.pl;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.nst * pl.stage_bytes);  // weights in
  uint64_t* hfull = full + kMaxStages;                                            // h inputs in
  uint64_t* empty = hfull + kMaxStages;
  float* es = reinterpret_cast<float*>(empty + kMaxStages);  // [chunk row][P]
  float* t_sd = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(es) + pl.es_bytes);
  Sel sel = sel_carve(reinterpret_cast<uint8_t*>(t_sd) + pl.tab_bytes, T, a.s.E);
  const int* t_ex = sel.u_ids;   // [slot] expert
  const int* t_off = sel.u_off;  // [slot] first pair
  const float* t_w = sel.wt;     // [T*K] routing weights
  const int* t_inv = sel.inv;    // [T*K] pair of (token, rank)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int row0 = down_rows_begin(d, blockIdx.x, gridDim.x);
  const int nrow = down_rows_begin(d, blockIdx.x + 1, gridDim.x) - row0;
  const int nch = (nrow + kDownChunk - 1) / kDownChunk;
  auto chunk = [&](int ci, int& c0, int& cn) {
    c0 = nrow * ci / nch;
    cn = nrow * (ci + 1) / nch - c0;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < pl.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&hfull[i], 1);
      mbar_init(&empty[i], kNW);
    }
    mbar_init(&selbar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // The router finished before the gate/up grid let this grid start.  If the gate/up grid has
  // published its selection already (one look at its flag, no waiting), load it; otherwise
  // select the experts from the router's scores here (the same selection every CTA of both
  // expert kernels makes).
  __shared__ int published;
  if (threadIdx.x == 0) published = sel_published(a.w);
  __syncthreads();
  const int TE = T * a.s.E;
  if (published) {
    sel_load_published(a.s, sel, a.w);
  } else if ((a.s.E % 4) == 0) {
    if (threadIdx.x == 0) {
      const uint64_t keep = l2_evict_last_policy();
      mbar_expect_tx(&selbar, (uint32_t)((TE + (a.st.bias ? a.s.E : 0)) * 4));
      bulk_g2s(sel.sc, a.w.scores, (uint32_t)TE * 4u, &selbar, keep);
      if (a.st.bias) bulk_g2s(sel.bias, a.st.bias, (uint32_t)a.s.E * 4u, &selbar, keep);
    }
    mbar_wait_bounded(&selbar, 0u, &abort_flag, a.w.status);
  } else {
    for (int i = threadIdx.x; i < TE; i += blockDim.x) sel.sc[i] = __ldcg(a.w.scores + i);
    if (a.st.bias)
      for (int i = threadIdx.x; i < a.s.E; i += blockDim.x) sel.bias[i] = a.st.bias[i];
  }
  if (!published) {
    __syncthreads();
    select_union(a.s, sel, a.st.bias != nullptr);
  }
  const int nu = *sel.nu;
  const int P = t_off[nu];
  const int nstage = nch * nu;
  const uint64_t pol = l2_evict_first_policy();
  const bool producer = (warp == kNW && lane == 0);
  const int nthr = kNW * 32;

  if (warp == kNW) {
    if (producer) {
      // stage it = (row chunk it / nu, union slot it % nu)
      auto issue_w = [&](int s, int it) {
        int c0, cn;
        chunk(it / nu, c0, cn);
        const uint8_t* src = a.st.wd + ((long)t_ex[it % nu] * d + row0 + c0) * (long)rb;
        mbar_expect_tx(&full[s], (uint32_t)(cn * rb));
        bulk_g2s(ring + (long)s * pl.stage_bytes, src, (uint32_t)(cn * rb), &full[s], pol);
      };
      // the slot's pairs are consecutive, so their h codes, scales and code sums are three
      // contiguous ranges of the workspace
      auto issue_h = [&](int s, int it) {
        const int slot = it % nu, p0 = t_off[slot], np = t_off[slot + 1] - p0;
        uint8_t* dst = ring + (long)s * pl.stage_bytes + pl.w_bytes;
        const uint32_t qb = (uint32_t)(np * f), sb = (uint32_t)(np * nbf * 4);
        mbar_expect_tx(&hfull[s], qb + 2 * sb);
        bulk_g2s(dst, a.w.qh + (long)p0 * f, qb, &hfull[s], pol);
        bulk_g2s(dst + qb, a.w.dh + (long)p0 * nbf, sb, &hfull[s], pol);
        bulk_g2s(dst + qb + sb, a.w.sh + (long)p0 * nbf, sb, &hfull[s], pol);
      };
      // the first stages' weights before the wait for the gate/up grid, their h inputs after it
      const int first = nstage < pl.nst ? nstage : pl.nst;
      for (int it = 0; it < first; ++it) issue_w(it, it);
      griddep_wait();  // gate/up grid complete: its h codes are visible from here on
      for (int it = 0; it < first; ++it) issue_h(it, it);
      int issued = first;
      int s = first % pl.nst;
      uint32_t ph = (uint32_t)((first / pl.nst) & 1);
      for (int it = first; it < nstage; ++it) {
        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, &abort_flag, a.w.status)) break;
        issue_w(s, it);
        issue_h(s, it);
        issued = it + 1;
        if (++s == pl.nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (abort_flag) {
        drain_fills(full, pl.nst, issued);
        drain_fills(hfull, pl.nst, issued);
      }
    }
  } else {
    // this CTA's down-row scales for every union slot (they do not depend on the gate/up grid)
    for (int i = threadIdx.x; i < nu * nrow; i += nthr) {
      const int sl = i / nrow, r = i - sl * nrow;
      t_sd[sl * pl.max_rows + r] = a.st.sc[(long)t_ex[sl] * (2 * f + d) + 2 * f + row0 + r];
    }
    named_bar_sync(1, nthr);
    int s = 0, ci = 0, slot = 0, c0 = 0, cn = 0;
    uint32_t ph = 0;
    chunk(0, c0, cn);
    // rows of this warp in the current chunk: w, w+8, ... below cn
    int nj = cn > warp ? (cn - warp + kNW - 1) / kNW : 0;
    const int jl = 4 * (lane & 1) + 2 * ((lane >> 1) & 1) + ((lane >> 2) & 1);  // row of the sum
    // Iteration -1 is a dry run of the stage code on whatever stage 0 holds (no wait, no result,
    // no arrival): it brings the loop's instructions into the SM's caches while the CTA would
    // otherwise wait for the gate/up grid, so the first real stage does not pay for fetching them.
#pragma unroll 1
    for (int it = -1; it < nstage; ++it) {
      const bool dry = it < 0;
      const int p0 = t_off[slot], np = dry ? 1 : t_off[slot + 1] - p0;
      if (!dry) {
        mbar_wait_bounded(&full[s], ph, &abort_flag, a.w.status);
        mbar_wait_bounded(&hfull[s], ph, &abort_flag, a.w.status);
      }
      const uint8_t* stage = ring + (long)s * pl.stage_bytes;
      const uint8_t* hq = stage + pl.w_bytes;
      const float* hd = reinterpret_cast<const float*>(hq + np * f);
      const int* hsum = reinterpret_cast<const int*>(hd + np * nbf);
      const float* sdx = t_sd + slot * pl.max_rows + c0 + warp;
      // pairs two at a time (the pair count is a template argument, so both pairs' chains
      // interleave with no branch between them); each row block's weights are loaded and split
      // into nibble halves once for both
      const DnRows r{stage + (long)warp * rb, hq, hd, hsum, sdx, es, f, nbf, A, lane, warp, nj, jl, P,
                     d, row0 + c0, dry, DBG ? a.dbg : ExpertDebug{}};
      for (int q = 0; q < np;) {
        if (np - q >= 2) {
          dn_rows<GF, 2, DBG>(r, q, p0 + q);
          q += 2;
        } else {
          dn_rows<GF, 1, DBG>(r, q, p0 + q);
          q += 1;
        }
      }
      __syncwarp();
      if (dry) continue;
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == pl.nst) {
        s = 0;
        ph ^= 1u;
      }
      if (slot == nu - 1) {
        // every union expert of this chunk is in: combine this warp's rows, one (row, token)
        // per lane
        const int j = lane & 7, t = lane >> 3;
        for (int tt = t; tt < T; tt += 4) {
          if (j < nj) {
            const float* er = es + (j * kNW + warp) * P;
            float y = a.s.n_shared ? er[T * K + tt] : 0.0f;
            for (int k = 0; k < K; ++k) y = __fmaf_rn(t_w[tt * K + k], er[t_inv[tt * K + k]], y);
            const long o = (long)tt * d + row0 + c0 + j * kNW + warp;
            if (a.s.has_norm) y = __fadd_rn(a.x[o], y);
            a.y[o] = y;
          }
        }
        __syncwarp();
        slot = 0;
        if (++ci < nch) {
          chunk(ci, c0, cn);
          nj = cn > warp ? (cn - warp + kNW - 1) / kNW : 0;
        }
      } else {
        ++slot;
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------ launchers -------------
template <class Args>
static cudaError_t launch_ex(void (*kern)(const Args), const Args& args, int grid, int smem,
                             bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args);
}

int down_grid(int d, int num_sms) { return d < num_sms ? d : num_sms; }

cudaError_t configure_expert_kernels() {
  cudaError_t e = cudaSuccess;
#define COLI_SET(KERN)                                                                      \
  if (e == cudaSuccess)                                                                     \
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
#define COLI_SET2(TMPL, N) COLI_SET((TMPL<N, false>)) COLI_SET((TMPL<N, true>))
  COLI_SET2(gateup_decode_kernel, 1) COLI_SET2(gateup_decode_kernel, 2)
  COLI_SET2(gateup_decode_kernel, 3) COLI_SET2(gateup_decode_kernel, 4)
  COLI_SET2(gateup_decode_kernel, 5) COLI_SET2(gateup_decode_kernel, 6)
  COLI_SET2(gateup_decode_kernel, 7) COLI_SET2(gateup_decode_kernel, 8)
  COLI_SET2(down_decode_kernel, 1) COLI_SET2(down_decode_kernel, 2)
  COLI_SET2(down_decode_kernel, 3) COLI_SET2(down_decode_kernel, 4)
  COLI_SET2(down_decode_kernel, 5) COLI_SET2(down_decode_kernel, 6)
  COLI_SET2(down_decode_kernel, 7) COLI_SET2(down_decode_kernel, 8)
#undef COLI_SET2
#undef COLI_SET
  return e;
}

// kernel instance for N blocks per lane group, with or without the debug stores
#define COLI_PICK(TMPL, N, DBG, OUT)                                \
  switch (N) {                                                     \
    case 1: OUT = DBG ? TMPL<1, true> : TMPL<1, false>; break;     \
    case 2: OUT = DBG ? TMPL<2, true> : TMPL<2, false>; break;     \
    case 3: OUT = DBG ? TMPL<3, true> : TMPL<3, false>; break;     \
    case 4: OUT = DBG ? TMPL<4, true> : TMPL<4, false>; break;     \
    case 5: OUT = DBG ? TMPL<5, true> : TMPL<5, false>; break;     \
    case 6: OUT = DBG ? TMPL<6, true> : TMPL<6, false>; break;     \
    case 7: OUT = DBG ? TMPL<7, true> : TMPL<7, false>; break;     \
    case 8: OUT = DBG ? TMPL<8, true> : TMPL<8, false>; break;     \
    default: return cudaErrorInvalidValue;                         \
  }

cudaError_t launch_gateup_decode(const Shape& s, const Store& st, const Work& w,
                                 const ExpertDebug& dbg, int num_sms, bool pdl,
                                 cudaStream_t stream) {
  // the unit count depends on the union size, known only on the device: size the grid for
  // the largest possible union (CTAs without work exit)
  long grid = max_union_slots(s.T, s.K, s.E, s.n_shared) * (s.f / 32);
  if (grid > num_sms) grid = num_sms;
  GateupArgs args{s, st, w, dbg, gateup_plan(s.d, s.f, s.T, s.K, s.E, s.n_shared, (int)grid)};
  const int G = (s.d / kQB + 31) / 32;
  const bool dbg_on = dbg.g || dbg.Ag;
  void (*k)(const GateupArgs) = nullptr;
  COLI_PICK(gateup_decode_kernel, G, dbg_on, k)
  return launch_ex(k, args, (int)grid, args.pl.total, pdl, stream);
}

cudaError_t launch_down_decode(const float* x, float* y, const Shape& s, const Store& st,
                               const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                               cudaStream_t stream) {
  const int grid = down_grid(s.d, num_sms);
  DownArgs args{s, st, w, dbg, down_plan(s.d, s.f, s.T, s.K, s.E, s.n_shared, grid), x, y};
  const int GF = (s.f / kQB + 31) / 32;
  const bool dbg_on = dbg.e || dbg.Ad;
  void (*k)(const DownArgs) = nullptr;
  COLI_PICK(down_decode_kernel, GF, dbg_on, k)
  return launch_ex(k, args, (int)grid, args.pl.total, pdl, stream);
}

}  // namespace coli
