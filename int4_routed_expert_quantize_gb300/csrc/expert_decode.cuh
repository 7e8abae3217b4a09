// Expert kernels of the decode path (a few tokens per call): the fused gate/up projection with
// SwiGLU and h re-quantisation, and the down projection with the fixed-order routing-weighted
// combine, for expert rows of 4, 8 or 2 bits per weight against int8 activation codes.  Both
// are HBM-bound streams over the union experts' weights ("colibrì 架构概述" §5: gate/up/SiLU/
// down on the IDOT fast path, then the shared expert; §3.1: int4 experts, int8 rows
// (quantize_rows, dot_i8i8) and int2 packed rows (pack_int2, matmul_i2); README: each distinct
// expert of a batch is read once).
//
// Structure of both kernels: a persistent grid (one CTA per SM) splits the work into equal
// contiguous ranges; in each CTA one producer lane streams the weight rows of its range
// through a ring of shared-memory stages with bulk copies (cp.async.bulk, mbarrier
// completion, L2 evict-first), and 8 consumer warps reduce each row: lane g owns the g-th of
// 32 contiguous groups of 32-element blocks, computes exact int32 block dots with dp4a, folds
// them with fma in block order, and the warp's xor butterfly adds the 32 group partials in
// pairwise-tree order.  All waits are bounded (see coli_device.cuh).
//
// The kernels are templates on the weight width WB; each (kernel, width) is instantiated in a
// translation unit of its own (gateup_w4.cu, down_w4.cu, ...), so the build compiles them in
// parallel.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_select.cuh"

namespace coli {

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
// streamed as 32/R stages of R row pairs, which yields one int8 block of h for every token of
// the slot's bucket.  The units are split over the CTAs with the shared expert's units first in
// every CTA that has some: those are known before routing, so they are prefetched before the
// kernel waits for the routing grid.  When a unit's 32 rows are done the CTA re-quantises them
// (one warp per token).
//
// NM rows of one stage (NM = 2: a row pair, gate then up; NM = 1: one matrix row) dotted with
// NP tokens' codes (the union slot's bucket): each of the warp's G blocks is loaded and prepared
// once for all tokens.
struct GuRow {
  const uint8_t* row;   // the warp's first row in the stage; a second one rbytes after it
  const uint8_t* xs;    // the tokens' codes in lane-group order
  const float* dxs;
  const int* nsx;       // -off * sum(codes) per token block
  int d, nbd, A, lane, rbytes;
  float sc[2];          // the rows' scales
  int row_i, f, p0;     // row index within the matrix, f, first pair of the slot
  float* out;           // per token: h (NM = 2) or the projection (NM = 1)
  int32_t* dA[2];       // debug block dots per matrix (may be null)
  float* dv[2];         // debug projections per matrix (may be null)
};

template <int G, int WB, int NM, int NP, bool DBG>
__device__ __forceinline__ void gu_multi(const GuRow& r, const int* toks) {
  float acc[NM][NP];
#pragma unroll
  for (int m = 0; m < NM; ++m)
#pragma unroll
    for (int q = 0; q < NP; ++q) acc[m][q] = 0.0f;
  const bool on = r.lane < r.A;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    uint32_t w[NM][8];
#pragma unroll
    for (int m = 0; m < NM; ++m) wload<WB>(r.row + m * r.rbytes, r.lane, i, G, r.nbd, on, w[m]);
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
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        const int a = wdot<WB>(w[m], xq, nq);
        acc[m][q] = __fmaf_rn(dq, __int2float_rn(a), acc[m][q]);
        if (DBG && r.dA[m] != nullptr && on)
          r.dA[m][((long)(r.p0 + q) * r.f + r.row_i) * r.nbd + r.lane * G + i] = a;
      }
    }
  }
#pragma unroll
  for (int q = 0; q < NP; ++q) {
    float v[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) v[m] = __fmul_rn(r.sc[m], warp_tree_sum(acc[m][q]));
    if (r.lane == 0) {
      r.out[q] = NM == 2 ? canon_silu_mul(v[0], v[NM - 1]) : v[0];
#pragma unroll
      for (int m = 0; m < NM; ++m)
        if (DBG && r.dv[m] != nullptr) r.dv[m][(long)(r.p0 + q) * r.f + r.row_i] = v[m];
    }
  }
}

// the same for one token whose codes the warp keeps in registers across stages
template <int G, int WB, int NM, bool DBG>
__device__ __forceinline__ void gu_one(const GuRow& r, const uint32_t (&xr)[G][8], const float (&dr)[G],
                                       const int (&nr)[G]) {
  float acc[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) acc[m] = 0.0f;
  const bool on = r.lane < r.A;
#pragma unroll
  for (int i = 0; i < G; ++i) {
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      uint32_t w[8];
      wload<WB>(r.row + m * r.rbytes, r.lane, i, G, r.nbd, on, w);
      const int a = wdot<WB>(w, xr[i], nr[i]);
      acc[m] = __fmaf_rn(dr[i], __int2float_rn(a), acc[m]);
      if (DBG && r.dA[m] != nullptr && on)
        r.dA[m][((long)r.p0 * r.f + r.row_i) * r.nbd + r.lane * G + i] = a;
    }
  }
  float v[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) v[m] = __fmul_rn(r.sc[m], warp_tree_sum(acc[m]));
  if (r.lane == 0) {
    r.out[0] = NM == 2 ? canon_silu_mul(v[0], v[NM - 1]) : v[0];
#pragma unroll
    for (int m = 0; m < NM; ++m)
      if (DBG && r.dv[m] != nullptr) r.dv[m][(long)r.p0 * r.f + r.row_i] = v[m];
  }
}

template <int G, int WB, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) gateup_decode_kernel(const GateupArgs a) {
  constexpr int R = gu_rows_per_stage(WB);  // row pairs per stage
  constexpr int SPU = 32 / R;               // stages per unit
  constexpr int NM = R == kNW ? 2 : 1;      // rows per warp and stage: a pair, or one matrix row
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  const int d = a.s.d, f = a.s.f, T = a.s.T;
  const int nbd = d >> 5, A = nbd / G, nhb = f >> 5;
  const int rbytes = d * WB / 8, rpb = 2 * rbytes;  // bytes of a matrix row, of a row pair
  const GateupPlan& pl = a.pl;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.nst * pl.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint8_t* xs = reinterpret_cast<uint8_t*>(empty + kMaxStages);  // [T][2 halves][chunks][16]
  float* dxs = reinterpret_cast<float*>(xs + pl.xs_bytes);         // [T][nbd]
  int* nsx = reinterpret_cast<int*>(dxs + T * nbd);                // [T][nbd]  -off*sum(codes)
  // [2][32][T] h of the current and the previous unit, or with one matrix row per warp
  // [2][2 (gate, up)][32][T] the projections
  float* hs = reinterpret_cast<float*>(xs + pl.xs_bytes + pl.aux_bytes);
  int* tab = reinterpret_cast<int*>(xs + pl.xs_bytes + pl.aux_bytes + pl.hs_bytes);
  Sel sel = sel_carve(xs + pl.xs_bytes + pl.aux_bytes + pl.hs_bytes + pl.tab_bytes, T, a.s.E);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
      const uint8_t* src =
          a.st.wgu + (store_slot(a.st, a.s.E, a.w.status) * f + unit * 32 + sub * R) * (long)rpb;
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
        nsx[idx] = -Wfmt<WB>::off * sv[k];
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
            a.st.wgu + (store_slot(a.st, sel.u_ids[slot], a.w.status) * f + hb * 32 + (it % SPU) * R) * (long)rpb;
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
      const float* scx = a.st.sc + store_slot(a.st, ex, a.w.status) * (2 * f + d);
      float* tsc = reinterpret_cast<float*>(tu + kGuTabInts);
      tsc[lane] = scx[hb * 32 + lane];
      tsc[32 + lane] = scx[f + hb * 32 + lane];
    }
    named_bar_sync(1, kNW * 32);

    // ---------------- consumers: warp `warp` takes row pair `warp` of every stage (NM = 2), or
    // row (warp / 4) of pair warp % 4 (NM = 1)
    const int rp = NM == 2 ? warp : (warp & 3);  // the warp's row pair in the stage
    const int mat = NM == 2 ? 0 : (warp >> 2);   // its matrix (0 gate, 1 up) with one row
    uint32_t xr[G][8];
    float dr[G];
    int nr_[G];
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
      const int rr = sub * R + rp;
      const float* tsc = reinterpret_cast<const float*>(tu + kGuTabInts);
      GuRow r;
      r.row = ring + (long)s * pl.stage_bytes + (long)rp * rpb + mat * rbytes;
      r.xs = xs;
      r.dxs = dxs;
      r.nsx = nsx;
      r.d = d;
      r.nbd = nbd;
      r.A = A;
      r.lane = lane;
      r.rbytes = rbytes;
      r.sc[0] = tsc[mat * 32 + rr];
      r.sc[1] = tsc[32 + rr];
      r.row_i = hb * 32 + rr;
      r.f = f;
      r.p0 = p0;
      r.out = NM == 2 ? hs + ((lu & 1) * 32 + rr) * T : hs + (((lu & 1) * 2 + mat) * 32 + rr) * T;
      r.dA[0] = DBG ? (mat ? a.dbg.Au : a.dbg.Ag) : nullptr;
      r.dA[1] = DBG ? a.dbg.Au : nullptr;
      r.dv[0] = DBG ? (mat ? a.dbg.u : a.dbg.g) : nullptr;
      r.dv[1] = DBG ? a.dbg.u : nullptr;
      if (np == 1) {
        // one token: its codes stay in registers while consecutive units serve the same token
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
              nr_[i] = nsx[t * nbd + lane * G + i];
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k) xr[i][k] = 0u;
              dr[i] = 0.0f;
              nr_[i] = 0;
            }
          }
          cached_tok = t;
        }
        gu_one<G, WB, NM, DBG>(r, xr, dr, nr_);
      } else {
        // several tokens: each block's weights are loaded and prepared once, then dotted with
        // every token's codes of that block; each token keeps its own fma chain over the blocks
        // in order (the token count is a template argument, so the tokens' chains interleave
        // with no branch between them)
        // with 8, 4, 2 or 1 tokens at a time (a token's chain does not depend on the others;
        // the debug build takes them one at a time)
        cached_tok = -1;
        for (int q0 = 0; q0 < np;) {
          const int rem = np - q0;
          GuRow rq = r;
          rq.p0 = p0 + q0;
          rq.out = r.out + q0;
          const int* tq = tu + 5 + q0;
          if (!DBG && rem >= 8) {
            gu_multi<G, WB, NM, 8, DBG>(rq, tq);
            q0 += 8;
          } else if (!DBG && rem >= 4) {
            gu_multi<G, WB, NM, 4, DBG>(rq, tq);
            q0 += 4;
          } else if (!DBG && rem >= 2) {
            gu_multi<G, WB, NM, 2, DBG>(rq, tq);
            q0 += 2;
          } else {
            gu_multi<G, WB, NM, 1, DBG>(rq, tq);
            q0 += 1;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with its rows
      if (++s == pl.nst) {
        s = 0;
        ph ^= 1u;
      }
      if (sub == SPU - 1) {
        // the unit's 32 rows of h are complete: quantise one int8 block per token
        named_bar_sync(1, kNW * 32);
        for (int q = warp; q < np; q += kNW) {
          const float hv = NM == 2 ? hs[((lu & 1) * 32 + lane) * T + q]
                                   : canon_silu_mul(hs[(((lu & 1) * 2 + 0) * 32 + lane) * T + q],
                                                    hs[(((lu & 1) * 2 + 1) * 32 + lane) * T + q]);
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
// the same number of bytes -- cut into chunks of at most dn_chunk_cap rows.  A stage is one chunk
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
// consecutive pairs of the stage's union expert: each row block's weights are loaded and
// prepared once for all of them.
struct DnRows {
  const uint8_t* sbase;  // the warp's first row in the stage
  const uint8_t* hq;     // [np][f] h codes of the stage's pairs
  const float* hd;       // [np][nbf] their block scales
  const int* hsum;       // [np][nbf] their code sums
  const float* sdx;      // the warp's first down-row scale of the chunk (stride kNW)
  float* es;             // [chunk row][P] expert outputs
  int f, nbf, A, lane, warp, nj, jl, P, d, row0c, rb;  // row0c: first output row of the chunk
  bool dry;
  ExpertDebug dbg;
};

// q: the first of the NP pairs within the stage, p: its index among all pairs
template <int GF, int WB, int NP, bool DBG>
__device__ __forceinline__ void dn_rows(const DnRows& r, int q, int p) {
  const bool on = r.lane < r.A;
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
        hnr[k][i] = -Wfmt<WB>::off * r.hsum[(q + k) * r.nbf + r.lane * GF + i];
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
      const uint8_t* srow = r.sbase + (long)j * kNW * r.rb;
#pragma unroll
      for (int i = 0; i < GF; ++i) {
        uint32_t w[8];
        wload<WB>(srow, r.lane, i, GF, r.nbf, on, w);
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          const int ai = wdot<WB>(w, hr[k][i], hnr[k][i]);
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

template <int GF, int WB, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) down_decode_kernel(const DownArgs a) {
  constexpr int CAP = dn_chunk_cap(WB);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  __shared__ __align__(8) uint64_t selbar;
  const int d = a.s.d, f = a.s.f, T = a.s.T, K = a.s.K;
  const int nbf = f >> 5, A = nbf / GF, rb = f * WB / 8;
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
  const int nch = (nrow + CAP - 1) / CAP;
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
        const uint8_t* src = a.st.wd + (store_slot(a.st, t_ex[it % nu], a.w.status) * d + row0 + c0) * (long)rb;
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
      t_sd[sl * pl.max_rows + r] = a.st.sc[store_slot(a.st, t_ex[sl], a.w.status) * (2 * f + d) + 2 * f + row0 + r];
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
      // interleave with no branch between them); each row block's weights are loaded and
      // prepared once for both
      const DnRows r{stage + (long)warp * rb, hq, hd, hsum, sdx, es, f, nbf, A, lane, warp, nj, jl, P,
                     d, row0 + c0, rb, dry, DBG ? a.dbg : ExpertDebug{}};
      for (int q = 0; q < np;) {
        if (np - q >= 2) {
          dn_rows<GF, WB, 2, DBG>(r, q, p0 + q);
          q += 2;
        } else {
          dn_rows<GF, WB, 1, DBG>(r, q, p0 + q);
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

// kernel instance for N blocks per lane group and width WB, with or without the debug stores
#define COLI_PICK(TMPL, N, WBV, DBG, OUT)                                   \
  switch (N) {                                                             \
    case 1: OUT = DBG ? TMPL<1, WBV, true> : TMPL<1, WBV, false>; break;   \
    case 2: OUT = DBG ? TMPL<2, WBV, true> : TMPL<2, WBV, false>; break;   \
    case 3: OUT = DBG ? TMPL<3, WBV, true> : TMPL<3, WBV, false>; break;   \
    case 4: OUT = DBG ? TMPL<4, WBV, true> : TMPL<4, WBV, false>; break;   \
    case 5: OUT = DBG ? TMPL<5, WBV, true> : TMPL<5, WBV, false>; break;   \
    case 6: OUT = DBG ? TMPL<6, WBV, true> : TMPL<6, WBV, false>; break;   \
    case 7: OUT = DBG ? TMPL<7, WBV, true> : TMPL<7, WBV, false>; break;   \
    case 8: OUT = DBG ? TMPL<8, WBV, true> : TMPL<8, WBV, false>; break;   \
    default: return cudaErrorInvalidValue;                                 \
  }

template <int WB>
cudaError_t configure_gateup_kernels_wb() {
  cudaError_t e = cudaSuccess;
#define COLI_SET(KERN)                                                                      \
  if (e == cudaSuccess)                                                                     \
    e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
#define COLI_SET2(TMPL, N) COLI_SET((TMPL<N, WB, false>)) COLI_SET((TMPL<N, WB, true>))
  COLI_SET2(gateup_decode_kernel, 1) COLI_SET2(gateup_decode_kernel, 2)
  COLI_SET2(gateup_decode_kernel, 3) COLI_SET2(gateup_decode_kernel, 4)
  COLI_SET2(gateup_decode_kernel, 5) COLI_SET2(gateup_decode_kernel, 6)
  COLI_SET2(gateup_decode_kernel, 7) COLI_SET2(gateup_decode_kernel, 8)
  return e;
}

template <int WB>
cudaError_t configure_down_kernels_wb() {
  cudaError_t e = cudaSuccess;
  COLI_SET2(down_decode_kernel, 1) COLI_SET2(down_decode_kernel, 2)
  COLI_SET2(down_decode_kernel, 3) COLI_SET2(down_decode_kernel, 4)
  COLI_SET2(down_decode_kernel, 5) COLI_SET2(down_decode_kernel, 6)
  COLI_SET2(down_decode_kernel, 7) COLI_SET2(down_decode_kernel, 8)
#undef COLI_SET2
#undef COLI_SET
  return e;
}

template <int WB>
cudaError_t launch_gateup_decode_wb(const Shape& s, const Store& st, const Work& w,
                                    const ExpertDebug& dbg, int num_sms, bool pdl,
                                    cudaStream_t stream) {
  // the unit count depends on the union size, known only on the device: size the grid for
  // the largest possible union (CTAs without work exit)
  long grid = (long)((s.T * s.K < s.E ? s.T * s.K : s.E) + (s.n_shared ? 1 : 0)) * (s.f / 32);
  if (grid > num_sms) grid = num_sms;
  GateupArgs args{s, st, w, dbg, gateup_plan(s.d, s.f, s.T, s.K, s.E, s.n_shared, (int)grid, WB)};
  const int G = (s.d / kQB + 31) / 32;
  const bool dbg_on = dbg.g || dbg.Ag;
  void (*k)(const GateupArgs) = nullptr;
  COLI_PICK(gateup_decode_kernel, G, WB, dbg_on, k)
  return launch_ex(k, args, (int)grid, args.pl.total, pdl, stream);
}

template <int WB>
cudaError_t launch_down_decode_wb(const float* x, float* y, const Shape& s, const Store& st,
                                  const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                                  cudaStream_t stream) {
  const int grid = down_grid(s.d, num_sms);
  DownArgs args{s, st, w, dbg, down_plan(s.d, s.f, s.T, s.K, s.E, s.n_shared, grid, WB), x, y};
  const int GF = (s.f / kQB + 31) / 32;
  const bool dbg_on = dbg.e || dbg.Ad;
  void (*k)(const DownArgs) = nullptr;
  COLI_PICK(down_decode_kernel, GF, WB, dbg_on, k)
  return launch_ex(k, args, (int)grid, args.pl.total, pdl, stream);
}

#undef COLI_PICK

// one translation unit per width and kernel instantiates these
#define COLI_GATEUP_INSTANTIATE(WBV)                                                              \
  template cudaError_t configure_gateup_kernels_wb<WBV>();                                        \
  template cudaError_t launch_gateup_decode_wb<WBV>(const Shape&, const Store&, const Work&,      \
                                                    const ExpertDebug&, int, bool, cudaStream_t);
#define COLI_DOWN_INSTANTIATE(WBV)                                                                \
  template cudaError_t configure_down_kernels_wb<WBV>();                                          \
  template cudaError_t launch_down_decode_wb<WBV>(const float*, float*, const Shape&, const Store&, \
                                                  const Work&, const ExpertDebug&, int, bool,     \
                                                  cudaStream_t);

}  // namespace coli
