// One-token decode of the expert half in a single persistent kernel: the gate/up projection with
// SwiGLU and h re-quantisation, a grid-wide barrier (every CTA's h blocks written), then the
// down projection with the fixed-order combine ("colibrì 架构概述" §5: gate/up/SiLU/down on the
// IDOT fast path; README: each distinct expert of a batch is read once).
//
// It computes exactly what gateup_decode_kernel followed by down_decode_kernel compute (the
// same per-row arithmetic, the same selection), with three differences in how the work flows:
//  * the producer lane keeps streaming: after its CTA's last gate/up stage it issues the CTA's
//    down stages into the same ring, so they arrive while the last gate/up stages are consumed
//    and while the CTA waits at the barrier;
//  * the down phase reuses the CTA's selection (no second selection, no second launch), and
//    the CTA's down-row scales are copied asynchronously right after the selection;
//  * the down phase's buffers overlay the gate/up phase's token and table buffers.
// The barrier is a counter in the workspace (cleared by the router grid each call) that every
// CTA increments; while it waits for the others a CTA runs one dry down stage (bringing that
// loop's instructions into its caches), then polls with a bounded wait.  grid <= SM count with
// one CTA per SM, so all of its CTAs are resident together once the router grid ahead of it
// has retired.
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_select.cuh"

namespace coli {

static inline int align16f(int x) { return (x + 15) & ~15; }

constexpr int kFuTabInts = 9;                 // expert, first pair, pairs, 32-row block, spare
constexpr int kFuTabStride = kFuTabInts + 64;  // ints per unit table entry

FusedPlan fused_plan(int d, int f, int K, int E, int n_shared, int grid) {
  FusedPlan p;
  const int T = 1, nbd = d / kQB, nbf = f / kQB;
  const int P = T * K + (n_shared ? T : 0);
  p.stage_bytes = kGuRps * d;
  // gate/up phase region
  p.xs_bytes = align16f(T * d);
  p.aux_bytes = align16f(T * nbd * 8);
  p.hs_bytes = align16f(2 * 32 * T * 4);
  const long units = (long)((T * K < E ? T * K : E) + (n_shared ? 1 : 0)) * (f / 32);
  p.max_units = (int)((units + grid - 1) / grid) + 2;
  p.tab_bytes = align16f(p.max_units * kFuTabStride * 4);
  const int gu_region = p.xs_bytes + p.aux_bytes + p.hs_bytes + p.tab_bytes;
  // down phase region (overlays the gate/up region once that phase is done in the CTA)
  p.max_rows = (d + grid - 1) / grid;
  p.chunk = p.max_rows < kDownChunk ? p.max_rows : kDownChunk;
  p.max_slots = (T * K < E ? T * K : E) + (n_shared ? 1 : 0);
  p.hq_bytes = align16f(P * f);
  p.haux_bytes = 2 * align16f(P * nbf * 4);
  p.es_bytes = align16f(p.chunk * P * 4);
  p.tsd_bytes = align16f(p.max_slots * p.max_rows * 4);
  const int dn_region = p.hq_bytes + p.haux_bytes + p.es_bytes;
  p.region = gu_region > dn_region ? gu_region : dn_region;
  p.sel_bytes = align16f(sel_bytes(T, E));
  const int fixed = 2 * kMaxStages * 8 + p.region + p.tsd_bytes + p.sel_bytes;
  int nst = (kSmemLimit - fixed) / p.stage_bytes;
  p.nst = nst > kMaxStages ? kMaxStages : nst;
  // a down stage (one chunk of rows) must fit a ring slot
  if (p.chunk * (f / 2) > p.stage_bytes) p.nst = 0;
  p.total = p.nst * p.stage_bytes + fixed;
  return p;
}

struct FusedArgs {
  Shape s;
  Store st;
  Work w;
  ExpertDebug dbg;
  FusedPlan pl;
  const float* x;
  float* y;
  int skip_arrival;  // failure-path test: CTA 0 stays out of the grid barrier
};

template <int G, int GF, int RPW, bool DBG>
__global__ void __launch_bounds__(kThreads, 1) expert_fused_kernel(const FusedArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int abort_flag;
  __shared__ __align__(8) uint64_t inbar;  // the down phase's h inputs are in
  const int d = a.s.d, f = a.s.f, K = a.s.K;
  const int nbd = d >> 5, A = nbd / G, nhb = f >> 5;
  const int nbf = f >> 5, AF = nbf / GF, rb = f >> 1;
  const FusedPlan& pl = a.pl;
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + pl.nst * pl.stage_bytes);
  uint64_t* empty = full + kMaxStages;
  uint8_t* region = reinterpret_cast<uint8_t*>(empty + kMaxStages);
  // gate/up phase: the token's codes in lane-group order, scales, code sums, h rows, unit table
  uint8_t* xs = region;                                             // [2 halves][chunks][16]
  float* dxs = reinterpret_cast<float*>(xs + pl.xs_bytes);          // [nbd]
  int* nsx = reinterpret_cast<int*>(dxs + nbd);                     // [nbd]  -8*sum(codes)
  float* hs = reinterpret_cast<float*>(xs + pl.xs_bytes + pl.aux_bytes);  // [2][32]
  int* tab = reinterpret_cast<int*>(xs + pl.xs_bytes + pl.aux_bytes + pl.hs_bytes);
  // down phase, over the same bytes: h codes [P][f], block scales and code sums [P][nbf], the
  // expert outputs of a chunk [chunk row][P]; after them the down-row scales [slot][max_rows]
  uint8_t* hq = region;
  float* hd = reinterpret_cast<float*>(region + pl.hq_bytes);
  int* hsum = reinterpret_cast<int*>(region + pl.hq_bytes + pl.haux_bytes / 2);
  float* es = reinterpret_cast<float*>(region + pl.hq_bytes + pl.haux_bytes);
  float* t_sd = reinterpret_cast<float*>(region + pl.region);
  Sel sel = sel_carve(region + pl.region + pl.tsd_bytes, 1, a.s.E);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int SPU = 32 / kGuRps;
  const int G_ = gridDim.x, c = blockIdx.x;
  // the grid after this one (the copy of y to the caller, or the next forward's router) may be
  // scheduled once every CTA of this grid has started; it waits for this grid to complete
  griddep_launch_dependents();

  // shared-expert units of this CTA: [a0, a1) of the nhb units of store slot E
  const int UA = a.s.n_shared ? nhb : 0;
  const int a0 = (int)((long)UA * c / G_), a1 = (int)((long)UA * (c + 1) / G_);
  const int na = a1 - a0;
  // output rows of this CTA in the down phase, in chunks of at most kDownChunk
  const int row0 = (int)((long)d * c / G_);
  const int nrow = (int)((long)d * (c + 1) / G_) - row0;
  const int nch = (nrow + kDownChunk - 1) / kDownChunk;
  auto chunk = [&](int ci, int& c0, int& cn) {
    c0 = nrow * ci / nch;
    cn = nrow * (ci + 1) / nch - c0;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < pl.nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNW);
    }
    mbar_init(&inbar, 1);
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
          a.st.wgu + (store_slot(a.st, a.s.E, a.w.status) * f + unit * 32 + sub * kGuRps) * (long)d;
      mbar_expect_tx(&full[issued], (uint32_t)pl.stage_bytes);
      bulk_g2s(ring + issued * pl.stage_bytes, src, (uint32_t)pl.stage_bytes, &full[issued], pol);
    }
  }
  // the selection bias does not depend on the routing grid
  if (a.st.bias)
    for (int i = threadIdx.x; i < a.s.E; i += blockDim.x) sel.bias[i] = a.st.bias[i];
  // the routing grid is complete and its results visible from here on
  griddep_wait();

  // the router's scores (plain loads: the bulk-copy queue still holds the shared expert's
  // prefetch) and, meanwhile, the token's codes
  const int E = a.s.E;
  float sreg[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < E) sreg[k] = __ldcg(a.w.scores + i);
  }
  for (int i0 = threadIdx.x; i0 < nbd; i0 += 4 * blockDim.x) {
    uint4 q0[4], q1[4];
    float dv[4];
    int sv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = i0 + k * blockDim.x;
      if (b < nbd) {
        const uint4* src = reinterpret_cast<const uint4*>(a.w.qx + b * 32);
        q0[k] = __ldcg(src);
        q1[k] = __ldcg(src + 1);
        dv[k] = __ldcg(a.w.dx + b);
        sv[k] = __ldcg(a.w.sx + b);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int b = i0 + k * blockDim.x;
      if (b < nbd) {
        const int g = b / G, i = b - g * G;
        uint8_t* base = xs + (i * A + g) * 16;
        *reinterpret_cast<uint4*>(base) = q0[k];
        *reinterpret_cast<uint4*>(base + nbd * 16) = q1[k];
        dxs[b] = dv[k];
        nsx[b] = -8 * sv[k];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + k * blockDim.x;
    if (i < E) sel.sc[i] = sreg[k];
  }
  for (int i = threadIdx.x + 4 * blockDim.x; i < E; i += blockDim.x) sel.sc[i] = __ldcg(a.w.scores + i);
  __syncthreads();
  select_union(a.s, sel, a.st.bias != nullptr);
  if (blockIdx.x == 0) sel_publish(a.s, sel, a.w);
  const int nu = *sel.nu;
  const int P = sel.u_off[nu];

  // routed units of this CTA: the total U = UA + UB is split evenly (each CTA's shared units
  // count towards its share) when there are at least as many routed units as CTAs
  const int UB = (nu - (a.s.n_shared ? 1 : 0)) * nhb;
  int b0, b1;
  if (UB >= G_) {
    const long U = UA + UB;
    b0 = (int)(U * c / G_) - a0;
    b1 = (int)(U * (c + 1) / G_) - a1;
  } else {
    b0 = (int)((long)UB * c / G_);
    b1 = (int)((long)UB * (c + 1) / G_);
  }
  const int nunit = na + (b1 - b0);
  const int nst_gu = nunit * SPU;               // gate/up stages of this CTA
  const int nst_all = nst_gu + nch * nu;        // then one stage per (row chunk, union slot)

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
    // ---------------- producer: one lane streams the remaining gate/up stages, then the down
    // stages of this CTA's rows (they do not depend on h, so they fill the ring early)
    if (producer) {
      int s = issued % pl.nst;
      uint32_t ph = (uint32_t)((issued / pl.nst) & 1);
      for (int it = issued; it < nst_all; ++it) {
        if (it >= pl.nst && !mbar_wait_bounded(&empty[s], ph ^ 1u, &abort_flag, a.w.status)) break;
        const uint8_t* src;
        uint32_t bytes;
        if (it < nst_gu) {
          int slot, hb;
          unit_of(it / SPU, slot, hb);
          src = a.st.wgu +
                (store_slot(a.st, sel.u_ids[slot], a.w.status) * f + hb * 32 + (it % SPU) * kGuRps) * (long)d;
          bytes = (uint32_t)pl.stage_bytes;
        } else {
          const int j = it - nst_gu, ci = j / nu, slot = j - ci * nu;
          int c0, cn;
          chunk(ci, c0, cn);
          src = a.st.wd + (store_slot(a.st, sel.u_ids[slot], a.w.status) * d + row0 + c0) * (long)rb;
          bytes = (uint32_t)(cn * rb);
        }
        mbar_expect_tx(&full[s], bytes);
        bulk_g2s(ring + (long)s * pl.stage_bytes, src, bytes, &full[s], pol);
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
      int* tu = tab + lu * kFuTabStride;
      const int ex = sel.u_ids[slot];
      const int p0 = sel.u_off[slot];
      const int np = sel.u_off[slot + 1] - p0;
      if (lane == 0) {
        tu[1] = ex;
        tu[2] = p0;
        tu[3] = np;
        tu[4] = hb;
      }
      const float* scx = a.st.sc + store_slot(a.st, ex, a.w.status) * (2 * f + d);
      float* tsc = reinterpret_cast<float*>(tu + kFuTabInts);
      tsc[lane] = scx[hb * 32 + lane];
      tsc[32 + lane] = scx[f + hb * 32 + lane];
    }
    // this CTA's down-row scales of every union expert: asynchronous copies that land while the
    // gate/up stages run (each thread waits for its own before the grid barrier)
    for (int i = threadIdx.x; i < nu * nrow; i += kNW * 32) {
      const int sl = i / nrow, r = i - sl * nrow;
      cp_async4(t_sd + sl * pl.max_rows + r,
                a.st.sc + store_slot(a.st, sel.u_ids[sl], a.w.status) * (2 * f + d) + 2 * f + row0 + r);
    }
    named_bar_sync(1, kNW * 32);

    // ---------------- consumers, gate/up phase: warp `warp` takes row pair `warp` of every
    // stage; the one token's codes stay in registers
    uint32_t xr[G][8];
    float dr[G];
    int nr[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      if (lane < A) {
        const uint8_t* base = xs + (i * A + lane) * 16;
        const uint4 v0 = *reinterpret_cast<const uint4*>(base);
        const uint4 v1 = *reinterpret_cast<const uint4*>(base + nbd * 16);
        xr[i][0] = v0.x; xr[i][1] = v0.y; xr[i][2] = v0.z; xr[i][3] = v0.w;
        xr[i][4] = v1.x; xr[i][5] = v1.y; xr[i][6] = v1.z; xr[i][7] = v1.w;
        dr[i] = dxs[lane * G + i];
        nr[i] = nsx[lane * G + i];
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) xr[i][k] = 0u;
        dr[i] = 0.0f;
        nr[i] = 0;
      }
    }
    int s = 0;
    uint32_t ph = 0;
    for (int it = 0; it < nst_gu; ++it) {
      const int lu = it / SPU;
      const int sub = it % SPU;
      const int* tu = tab + lu * kFuTabStride;
      const int hb = tu[4];
      const int p = tu[2];
      mbar_wait_bounded(&full[s], ph, &abort_flag, a.w.status);
      const int rr = sub * kGuRps + warp;
      const int row = hb * 32 + rr;
      const uint8_t* grow = ring + (long)s * pl.stage_bytes + (long)warp * d;
      const float* tsc = reinterpret_cast<const float*>(tu + kFuTabInts);
      const float sg = tsc[rr], su = tsc[32 + rr];
      float pg = 0.0f, pu = 0.0f;
      // the row pair's weights into registers first, then the dots
      uint4 wg[G], wu[G];
#pragma unroll
      for (int i = 0; i < G; ++i) {
        wg[i] = make_uint4(0, 0, 0, 0);
        wu[i] = make_uint4(0, 0, 0, 0);
        if (lane < A) {
          const int off = store_chunk(lane, i, G) * 16;
          wg[i] = *reinterpret_cast<const uint4*>(grow + off);
          wu[i] = *reinterpret_cast<const uint4*>(grow + d / 2 + off);
        }
      }
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const int ag = block_dot(wg[i], xr[i], nr[i]);
        const int au = block_dot(wu[i], xr[i], nr[i]);
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
        hs[(lu & 1) * 32 + rr] = canon_silu_mul(g, u);
        if (DBG && a.dbg.g != nullptr) {
          a.dbg.g[(long)p * f + row] = g;
          a.dbg.u[(long)p * f + row] = u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with its row pair
      if (++s == pl.nst) {
        s = 0;
        ph ^= 1u;
      }
      if (sub == SPU - 1) {
        // the unit's 32 rows of h are complete: quantise its int8 block
        named_bar_sync(1, kNW * 32);
        if (warp == 0) {
          const float hv = hs[(lu & 1) * 32 + lane];
          const float dd = __fdiv_rn(warp_max(fabsf(hv)), 127.0f);
          const int code = q8_code(hv, dd);
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

    // ---------------- grid barrier: every CTA's h blocks are written.  Each thread fences its
    // own stores, the consumers meet, one thread counts the CTA in; it polls (bounded) until all
    // CTAs are counted at the first real down stage below.  The router grid cleared the counter
    // for this call.
    cp_async_wait_all();
    __threadfence();
    named_bar_sync(1, kNW * 32);
    int* counter = a.w.sel_flag + 1;
    if (threadIdx.x == 0 && !abort_flag && !(a.skip_arrival && blockIdx.x == 0))
      atomicAdd(counter, 1);

    // ---------------- down phase.  Warp w owns rows w, w+8, ... of each chunk: each lane folds
    // its group's block dots for up to RPW rows (rows past the warp's last one repeat it and are
    // dropped, so every load is unconditional), one transposed butterfly adds the group partials
    // of all rows; once a chunk has seen every union expert the warp combines its rows in the
    // fixed order (shared expert first, then ranks 0..K-1).
    // Iteration nst_gu - 1 is a dry run of the stage code on whatever the ring slot and the
    // buffers hold (no wait, no result, no arrival): it brings the loop's instructions into the
    // SM's caches while the CTA waits for the others at the barrier.
    const int nthr = kNW * 32;
    int ci = 0, slot = 0, c0 = 0, cn = 0;
    chunk(0, c0, cn);
    int nj = cn > warp ? (cn - warp + kNW - 1) / kNW : 0;
    const int jl = 4 * (lane & 1) + 2 * ((lane >> 1) & 1) + ((lane >> 2) & 1);  // row of the sum
#pragma unroll 1
    for (int it = nst_gu - 1; it < nst_all; ++it) {
      const bool dry = it < nst_gu;
      if (it == nst_gu) {
        // all CTAs counted (bounded wait); then the gate/up buffers are free: every pair's h
        // codes, block scales and code sums as they lie in the workspace (three bulk copies, or
        // plain loads when a size is not a multiple of 16 bytes)
        if (threadIdx.x == 0 && !abort_flag) {
          const uint64_t t0 = global_ns();
          for (uint32_t k = 1;; ++k) {
            int v;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            if (v >= (int)gridDim.x) break;
            if ((k & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) {
              abort_flag = 1;
              atomicExch(a.w.status, COLI_ETIMEOUT);
              break;
            }
          }
          // the h codes are read below by bulk copies (the async proxy)
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        named_bar_sync(1, nthr);
        const uint32_t qbytes = (uint32_t)(P * f), sbytes = (uint32_t)(P * nbf * 4);
        if ((sbytes & 15u) == 0) {
          if (threadIdx.x == 0 && !abort_flag) {
            mbar_expect_tx(&inbar, qbytes + 2 * sbytes);
            bulk_g2s(hq, a.w.qh, qbytes, &inbar, pol);
            bulk_g2s(hd, a.w.dh, sbytes, &inbar, pol);
            bulk_g2s(hsum, a.w.sh, sbytes, &inbar, pol);
          }
          mbar_wait_bounded(&inbar, 0u, &abort_flag, a.w.status);
        } else {
          for (int i = threadIdx.x; i < P * f / 16; i += nthr)
            reinterpret_cast<uint4*>(hq)[i] = __ldcg(reinterpret_cast<const uint4*>(a.w.qh) + i);
          for (int i = threadIdx.x; i < P * nbf; i += nthr) {
            hd[i] = __ldcg(a.w.dh + i);
            hsum[i] = __ldcg(a.w.sh + i);
          }
        }
        named_bar_sync(1, nthr);
      }
      const int p0 = sel.u_off[slot], np = dry ? 1 : sel.u_off[slot + 1] - p0;
      if (!dry) mbar_wait_bounded(&full[s], ph, &abort_flag, a.w.status);
      const uint8_t* sbase = ring + (long)s * pl.stage_bytes + (long)warp * rb;
      const float* sdx = t_sd + slot * pl.max_rows + c0 + warp;
      for (int q = 0; q < np; ++q) {
        const int p = p0 + q;
        uint32_t hr[GF][8];
        float hdr[GF];
        int hnr[GF];
#pragma unroll
        for (int i = 0; i < GF; ++i) {
          if (lane < AF) {
            const uint8_t* base = hq + (long)p * f + (lane * GF + i) * 32;
            const uint4 v0 = *reinterpret_cast<const uint4*>(base);
            const uint4 v1 = *reinterpret_cast<const uint4*>(base + 16);
            hr[i][0] = v0.x; hr[i][1] = v0.y; hr[i][2] = v0.z; hr[i][3] = v0.w;
            hr[i][4] = v1.x; hr[i][5] = v1.y; hr[i][6] = v1.z; hr[i][7] = v1.w;
            hdr[i] = hd[p * nbf + lane * GF + i];
            hnr[i] = -8 * hsum[p * nbf + lane * GF + i];
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) hr[i][k] = 0u;
            hdr[i] = 0.0f;
            hnr[i] = 0;
          }
        }
        float acc[kDownRowsPerWarp];
#pragma unroll
        for (int j = 0; j < kDownRowsPerWarp; ++j) acc[j] = 0.0f;
        if (nj > 0) {
          // every row's weights into registers first, then the dots
          uint4 wv[RPW][GF];
#pragma unroll
          for (int j = 0; j < RPW; ++j) {
            const int jj = j < nj ? j : nj - 1;
            const uint8_t* srow = sbase + (long)jj * kNW * rb;
#pragma unroll
            for (int i = 0; i < GF; ++i)
              wv[j][i] = lane < AF ? *reinterpret_cast<const uint4*>(srow + store_chunk(lane, i, GF) * 16)
                                   : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int j = 0; j < RPW; ++j) {
#pragma unroll
            for (int i = 0; i < GF; ++i) {
              const int ai = block_dot(wv[j][i], hr[i], hnr[i]);
              acc[j] = __fmaf_rn(hdr[i], __int2float_rn(ai), acc[j]);
              if (DBG && !dry && a.dbg.Ad != nullptr && lane < AF && j < nj)
                a.dbg.Ad[((long)p * d + row0 + c0 + j * kNW + warp) * nbf + lane * GF + i] = ai;
            }
          }
        }
        const float v = warp_tree_sum8(acc, lane);
        if (!dry && lane < kDownRowsPerWarp && jl < nj) {
          const float e = __fmul_rn(sdx[jl * kNW], v);
          es[(jl * kNW + warp) * P + p] = e;
          if (DBG && a.dbg.e != nullptr) a.dbg.e[(long)p * d + row0 + c0 + jl * kNW + warp] = e;
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
        // every union expert of this chunk is in: combine this warp's rows (one token)
        const int j = lane;
        if (j < nj) {
          const float* er = es + (j * kNW + warp) * P;
          float y = a.s.n_shared ? er[K] : 0.0f;
          for (int k = 0; k < K; ++k) y = __fmaf_rn(sel.wt[k], er[sel.inv[k]], y);
          const long o = row0 + c0 + j * kNW + warp;
          if (a.s.has_norm) y = __fadd_rn(a.x[o], y);
          a.y[o] = y;
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

// ------------------------------------------------------------------ host side --------------
// Instances built: G blocks per lane group on the gate/up side (d/32/32 rounded up), GF on the
// down side (f/32/32), and RPW down rows per warp and chunk (at least ceil(chunk rows / 8)): the
// GLM-shaped layer (d = 6144, f = 2048: 41 rows per CTA on 152 SMs) and layers with one block
// per group on both sides, each with an 8-row fallback.  Other shapes use the two-kernel path.
typedef void (*FusedKernel)(const FusedArgs);

template <int G, int GF, int RPW>
static FusedKernel pick(bool dbg) {
  return dbg ? expert_fused_kernel<G, GF, RPW, true> : expert_fused_kernel<G, GF, RPW, false>;
}

static FusedKernel fused_kernel_for(int G, int GF, int rpw, bool dbg) {
  if (G == 6 && GF == 2) return rpw <= 6 ? pick<6, 2, 6>(dbg) : pick<6, 2, 8>(dbg);
  if (G == 1 && GF == 1) return rpw <= 2 ? pick<1, 1, 2>(dbg) : pick<1, 1, 8>(dbg);
  return nullptr;
}

// rows per warp of the largest down chunk
static int fused_rpw(const FusedPlan& p) {
  const int chunk = p.max_rows < kDownChunk ? p.max_rows : kDownChunk;
  return (chunk + kNW - 1) / kNW;
}

cudaError_t configure_fused_kernels() {
  const FusedKernel ks[] = {pick<6, 2, 6>(true), pick<6, 2, 6>(false), pick<6, 2, 8>(true),
                            pick<6, 2, 8>(false), pick<1, 1, 2>(true), pick<1, 1, 2>(false),
                            pick<1, 1, 8>(true),  pick<1, 1, 8>(false)};
  for (FusedKernel k : ks) {
    const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int fused_grid(int d, int num_sms) { return d < num_sms ? d : num_sms; }

bool fused_supported(int d, int f, int K, int E, int n_shared, int num_sms) {
  const int G = (d / kQB + 31) / 32, GF = (f / kQB + 31) / 32;
  if (!fused_kernel_for(G, GF, kDownRowsPerWarp, false)) return false;
  return fused_plan(d, f, K, E, n_shared, fused_grid(d, num_sms)).nst >= 2;
}

// One launch of the fused expert kernel for one token, a programmatic dependent of the router
// grid unless events are recorded between launches.  Its CTAs wait on each other at the barrier,
// so all of them must be resident together: grid <= SM count and one CTA per SM (its shared
// memory allows no second one).  The router grid ahead of it waits on nothing, so the CTAs that
// cannot start while it holds their SMs start as soon as it retires.  (A cooperative launch
// would guarantee the same but starts no CTA before the router grid has finished.)
cudaError_t launch_expert_fused(const float* x, float* y, const Shape& s, const Store& st,
                                const Work& w, const ExpertDebug& dbg, int num_sms, bool pdl,
                                bool skip_arrival, cudaStream_t stream) {
  const int grid = fused_grid(s.d, num_sms);
  FusedArgs args{s, st, w, dbg, fused_plan(s.d, s.f, s.K, s.E, s.n_shared, grid), x, y,
                 skip_arrival ? 1 : 0};
  const int G = (s.d / kQB + 31) / 32, GF = (s.f / kQB + 31) / 32;
  const FusedKernel k = fused_kernel_for(G, GF, fused_rpw(args.pl), dbg.g || dbg.Ag || dbg.e || dbg.Ad);
  if (!k || s.T != 1) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)args.pl.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args);
}

}  // namespace coli
