// Routing half of the layer in one launch: activation preparation (optional RMSNorm,
// Q8_0-style int8 blocks of 32) and the sigmoid top-K router with the batch union.
//   "colibrì 架构概述" §3.1 (IDOT: decode activations quantised to int8), §5 (moe step:
//   sigmoid routing, top-8), the ai4coding.ru page (DeepSeek-V3-style sigmoid router,
//   Q8_0-style int8 activations) and the README's batch union (each distinct expert of a
//   batch is read once).
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_select.cuh"
#include "coli_tc.cuh"

namespace coli {

// ------------------------------------------------------------------ router ---------------
constexpr int kRouterEpc = 2;  // experts per CTA
constexpr int kMaxE = 1024;

// After a timed-out wait, wait once more (bounded, ignoring the abort flag) for the bulk copy,
// so that no copy still writes shared memory when the CTA exits.
__device__ __noinline__ void route_drain(uint64_t* bar) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, 0u))
    if (global_ns() - t0 > kWaitLimitNs / 8) break;
}

// One launch does the routing half up to the scores.  Every CTA: one bulk copy brings its
// kRouterEpc router rows into shared memory while all threads stage the tokens there (in the
// router's chunk order, kRouteTgroup tokens at a time) and the gate/up grid is let start its
// weight prefetch; then, for each group of tokens, the optional RMSNorm (one warp per token), the
// logits and sigmoid scores of its experts (one warp per (expert, token): lane g runs the fma
// chain over its d/32 contiguous elements, the butterfly adds the 32 partials) and, on the other
// warps at the same time, this CTA's share of the group's int8 activation blocks (one warp per
// block of 32).  The expert kernels select the experts from the scores themselves
// (coli_select.cuh), so no CTA here waits for another.
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ x, const Shape s,
                                                    const Store st, const Work w) {
  extern __shared__ __align__(128) float route_sm[];
  __shared__ __align__(8) uint64_t wbar;
  __shared__ float rinv[kRouteTgroup];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int d = s.d, E = s.E, T = s.T, Gd = d >> 5, nbd = d >> 5;
  const int e0 = blockIdx.x * kRouterEpc;
  const int ne = min(kRouterEpc, E - e0);
  float* wrs = route_sm;                   // [kRouterEpc][d] router rows as stored
  float* xsm = route_sm + kRouterEpc * d;  // [kRouteTgroup][d] tokens of the current group
  // launched as a programmatic dependent: the preceding grid (the previous forward, or the
  // copy of x into device memory) is complete and its writes visible from here on
  griddep_wait();
  if (threadIdx.x == 0) {
    if (blockIdx.x == 0) {  // this call's selection is not published yet; no CTA at the barrier
      w.sel_flag[0] = 0;
      w.sel_flag[1] = 0;
    }
    mbar_init(&wbar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_expect_tx(&wbar, (uint32_t)(ne * d * 4));
    const uint64_t pol = l2_evict_last_policy();
    for (int r = 0; r < ne; ++r)
      bulk_g2s(wrs + r * d, st.wr + (long)(e0 + r) * d, (uint32_t)d * 4u, &wbar, pol);
  }
  griddep_launch_dependents();
  int rows = 0;  // this warp's view of the router rows: 0 not waited for, 1 in, -1 gave up

  for (int t0 = 0; t0 < T; t0 += kRouteTgroup) {
    const int Tg = min(kRouteTgroup, T - t0);
    if (t0 > 0) __syncthreads();  // every warp is done with the previous group's tokens
    // tokens into shared memory in router order: lane g's elements g*Gd + 4*i4 .. +3 at chunk
    // i4*32 + g (conflict-free reads by lane).  Work item w of a token is (i4 = 8*(w>>8) +
    // (w&7), g = (w>>3)&31), so a warp reads four 128-byte runs of x and its shared-memory
    // stores fall in 4 bank groups; each thread issues its loads in batches of 8 before storing.
    const int n_i4 = d / 128, per_t = 256 * ((n_i4 + 7) / 8), nw = Tg * per_t;
    for (int c0 = threadIdx.x; c0 < nw; c0 += 8 * blockDim.x) {
      float4 v[8];
      int dst[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = c0 + k * blockDim.x;
        const int t = c / per_t, wi = c - t * per_t;
        const int i4 = ((wi >> 8) << 3) + (wi & 7), g = (wi >> 3) & 31;
        dst[k] = c < nw && i4 < n_i4 ? t * (d / 4) + i4 * 32 + g : -1;
        if (dst[k] >= 0)
          v[k] = __ldg(reinterpret_cast<const float4*>(x + (long)(t0 + t) * d + g * Gd + 4 * i4));
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (dst[k] >= 0) reinterpret_cast<float4*>(xsm)[dst[k]] = v[k];
    }
    __syncthreads();
    if (s.has_norm) {
      // mean of squares in the canonical order (lane g: fma chain over its d/32 elements)
      for (int t = warp; t < Tg; t += nwarp) {
        const float4* xp = reinterpret_cast<const float4*>(xsm + (long)t * d);
        float p = 0.0f;
        for (int i4 = 0; i4 < d / 128; ++i4) {
          const float4 v = xp[i4 * 32 + lane];
          p = __fmaf_rn(v.x, v.x, p);
          p = __fmaf_rn(v.y, v.y, p);
          p = __fmaf_rn(v.z, v.z, p);
          p = __fmaf_rn(v.w, v.w, p);
        }
        p = warp_tree_sum(p);
        if (lane == 0) {
          const float ms = __fdiv_rn(p, (float)d);
          rinv[t] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, s.rms_eps)));
        }
      }
      __syncthreads();
      const int n4 = Tg * (d / 4);
      for (int c0 = threadIdx.x; c0 < n4; c0 += 8 * blockDim.x) {
        float4 gm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = c0 + k * blockDim.x;
          if (c < n4) {
            const int pos = c % (d / 4);
            gm[k] = __ldg(reinterpret_cast<const float4*>(st.gamma + (pos & 31) * Gd + 4 * (pos >> 5)));
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = c0 + k * blockDim.x;
          if (c < n4) {
            const float r = rinv[c / (d / 4)];
            float4 v = reinterpret_cast<float4*>(xsm)[c];
            v.x = __fmul_rn(__fmul_rn(v.x, r), gm[k].x);
            v.y = __fmul_rn(__fmul_rn(v.y, r), gm[k].y);
            v.z = __fmul_rn(__fmul_rn(v.z, r), gm[k].z);
            v.w = __fmul_rn(__fmul_rn(v.w, r), gm[k].w);
            reinterpret_cast<float4*>(xsm)[c] = v;
          }
        }
      }
      __syncthreads();
    }

    // this CTA's share of the group's activation blocks: x_n (natural order), int8 codes,
    // scale, code sum.  The warps that compute no logits take them (while the logits run);
    // without such warps every warp takes its share first.
    const int ndot = ne * Tg;
    const int nq = ndot < nwarp ? nwarp - ndot : nwarp;
    const int qw = ndot < nwarp ? warp - ndot : warp;
    for (int b = qw >= 0 ? blockIdx.x * nq + qw : Tg * nbd; b < Tg * nbd; b += gridDim.x * nq) {
      const int tl = b / nbd, bb = b - tl * nbd, t = t0 + tl;
      const int j = bb * 32 + lane;
      const int g = j / Gd, m = j - g * Gd;
      const float v = xsm[(long)tl * d + ((m >> 2) * 32 + g) * 4 + (m & 3)];
      w.xn[(long)t * d + j] = v;
      const float dd = __fdiv_rn(warp_max(fabsf(v)), 127.0f);
      const int q = q8_code(v, dd);
      w.qx[(long)t * d + j] = (int8_t)q;
      const int sq = warp_isum(q);
      if (lane == 0) {
        w.dx[(long)t * nbd + bb] = dd;
        w.sx[(long)t * nbd + bb] = sq;
      }
    }

    // logits: router rows and tokens both in shared memory, chunk i4*32 + g for lane g
    for (int pi = warp; pi < ndot && rows >= 0; pi += nwarp) {
      if (rows == 0) {
        if (mbar_wait_bounded(&wbar, 0u, &abort_flag, w.status)) {
          rows = 1;
        } else {
          rows = -1;
          route_drain(&wbar);
          break;
        }
      }
      const int r = pi / Tg, tl = pi - r * Tg;
      const float4* wp = reinterpret_cast<const float4*>(wrs + (long)r * d);
      const float4* xp = reinterpret_cast<const float4*>(xsm + (long)tl * d);
      float p = 0.0f;
#pragma unroll 4
      for (int i4 = 0; i4 < d / 128; ++i4) {
        const float4 a4 = wp[i4 * 32 + lane];
        const float4 b4 = xp[i4 * 32 + lane];
        p = __fmaf_rn(a4.x, b4.x, p);
        p = __fmaf_rn(a4.y, b4.y, p);
        p = __fmaf_rn(a4.z, b4.z, p);
        p = __fmaf_rn(a4.w, b4.w, p);
      }
      p = warp_tree_sum(p);
      if (lane == 0) {
        w.logits[(long)(t0 + tl) * E + e0 + r] = p;
        w.scores[(long)(t0 + tl) * E + e0 + r] = canon_sigmoid(p);
      }
    }
  }
  // a warp that computed no logits never waited for the router rows: wait (bounded) so that no
  // bulk copy still writes shared memory when the CTA exits
  if (rows == 0 && !mbar_wait_bounded(&wbar, 0u, &abort_flag, w.status)) route_drain(&wbar);
}

static size_t route_smem_bytes(int d, int T) {
  return ((size_t)kRouterEpc * d + (size_t)(T < kRouteTgroup ? T : kRouteTgroup) * d) * sizeof(float);
}

cudaError_t configure_route_kernels() {
  return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)route_smem_bytes(8192, kRouteTgroup));
}

// ------------------------------------------------------------------ batched routing ------
// The same routing for batches of any size (the tensor-core expert path): one CTA per token for
// RMSNorm and the int8 blocks, a register-blocked router (each warp: 4 experts x 4 tokens, every
// logit still one canonical chain per lane group plus the butterfly), one CTA that selects the
// experts and builds the union and the per-slot tile counts, and a gather of every pair's codes
// as bf16 (exact: |q| <= 127) for the matrix engine.

__global__ void __launch_bounds__(256) prep_batch_kernel(const float* __restrict__ x, const Shape s,
                                                         const Store st, const Work w) {
  extern __shared__ __align__(16) float xs[];  // [d] natural order
  __shared__ float rinv;
  const int t = blockIdx.x, d = s.d, nbd = d >> 5, Gd = d >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const float* xt = x + (long)t * d;
  for (int j = threadIdx.x * 4; j < d; j += blockDim.x * 4)
    *reinterpret_cast<float4*>(xs + j) = *reinterpret_cast<const float4*>(xt + j);
  __syncthreads();
  if (s.has_norm) {
    if (warp == 0) {
      float p = 0.0f;
      for (int j = lane * Gd; j < lane * Gd + Gd; ++j) p = __fmaf_rn(xs[j], xs[j], p);
      p = warp_tree_sum(p);
      if (lane == 0) {
        const float ms = __fdiv_rn(p, (float)d);
        rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, s.rms_eps)));
      }
    }
    __syncthreads();
    const float r = rinv;
    for (int j = threadIdx.x; j < d; j += blockDim.x) xs[j] = __fmul_rn(__fmul_rn(xs[j], r), st.gamma[j]);
    __syncthreads();
  }
  float* xn = w.xn + (long)t * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) xn[j] = xs[j];
  float4* xp = reinterpret_cast<float4*>(w.xnp + (long)t * d);
  for (int c = threadIdx.x; c < d / 4; c += blockDim.x) {
    const int i4 = c >> 5, g = c & 31;
    const float* src = xs + g * Gd + 4 * i4;
    xp[c] = make_float4(src[0], src[1], src[2], src[3]);
  }
  for (int b = warp; b < nbd; b += nwarp) {
    const float v = xs[b * 32 + lane];
    const float dd = __fdiv_rn(warp_max(fabsf(v)), 127.0f);
    const int q = q8_code(v, dd);
    w.qx[(long)t * d + b * 32 + lane] = (int8_t)q;
    const int sq = warp_isum(q);
    if (lane == 0) {
      w.dx[(long)t * nbd + b] = dd;
      w.sx[(long)t * nbd + b] = sq;
    }
  }
}

// Router for batches: CTA tile = 16 experts x 32 tokens, K in chunks of 2 steps (256 floats of
// every row, the same lane-group chunk order as the decode router) brought into shared memory
// by 2-D tensor copies, double-buffered.  Warp w: experts 4*(w%4)..+3 x tokens 8*(w/4)..+7,
// 32 canonical chains per lane, one butterfly per logit at the end.
constexpr int kRbE = 16, kRbT = 32, kRbChunk = 256;
constexpr int kRbStage = (kRbE + kRbT) * kRbChunk * 4;  // 48 KB

__global__ void __launch_bounds__(512) router_batch_kernel(const __grid_constant__ CUtensorMap map_wr,
                                                           const __grid_constant__ CUtensorMap map_x,
                                                           const Shape s, const Work w) {
  extern __shared__ __align__(128) uint8_t rsm[];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = s.d, E = s.E, T = s.T;
  const int e0 = blockIdx.x * kRbE, t0 = blockIdx.y * kRbT;
  const int nchunk = d / kRbChunk;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int c) {
    uint8_t* st = rsm + (c & 1) * kRbStage;
    mbar_expect_tx(&bar[c & 1], (uint32_t)kRbStage);
    tma_load_2d(st, &map_wr, c * kRbChunk, e0, &bar[c & 1]);
    tma_load_2d(st + kRbE * kRbChunk * 4, &map_x, c * kRbChunk, t0, &bar[c & 1]);
  };
  if (threadIdx.x == 0) {
    issue(0);
    if (nchunk > 1) issue(1);
  }
  const int ew = (warp & 3) * 4, tw = (warp >> 2) * 8;
  float acc[4][8];
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[k][j] = 0.0f;
  for (int c = 0; c < nchunk; ++c) {
    mbar_wait_bounded(&bar[c & 1], (uint32_t)((c >> 1) & 1), &abort_flag, w.status);
    const float* wst = reinterpret_cast<const float*>(rsm + (c & 1) * kRbStage);
    const float* xst = wst + kRbE * kRbChunk;
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      float4 wv[4], xv[8];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        wv[k] = reinterpret_cast<const float4*>(wst + (ew + k) * kRbChunk + st * 128)[lane];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        xv[j] = reinterpret_cast<const float4*>(xst + (tw + j) * kRbChunk + st * 128)[lane];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float p = acc[k][j];
          p = __fmaf_rn(wv[k].x, xv[j].x, p);
          p = __fmaf_rn(wv[k].y, xv[j].y, p);
          p = __fmaf_rn(wv[k].z, xv[j].z, p);
          p = __fmaf_rn(wv[k].w, xv[j].w, p);
          acc[k][j] = p;
        }
    }
    __syncthreads();  // every warp is done with this stage
    if (threadIdx.x == 0 && c + 2 < nchunk) issue(c + 2);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p = warp_tree_sum(acc[k][j]);
      const int e = e0 + ew + k, t = t0 + tw + j;
      if (lane == 0 && e < E && t < T) {
        w.logits[(long)t * E + e] = p;
        w.scores[(long)t * E + e] = canon_sigmoid(p);
      }
    }
}

// top-K of every token: one warp per token
__global__ void __launch_bounds__(256) topk_batch_kernel(const Shape s, const Store st, const Work w) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= s.T) return;
  if (s.E <= 256)
    topk_warp<8>(w.scores + (long)t * s.E, st.bias, s.E, s.K, s.routed_scale, w.ids + t * s.K,
                 w.w + t * s.K, lane);
  else
    topk_warp<32>(w.scores + (long)t * s.E, st.bias, s.E, s.K, s.routed_scale, w.ids + t * s.K,
                  w.w + t * s.K, lane);
}

// The batch union with all 32 warps: counts per expert and the union slots (as union_bucket
// builds them), then each warp places a contiguous chunk of the pairs; a warp's first position
// for expert e is the slot start plus the pairs of e in earlier chunks (a scan over the warps'
// counts), which gives the same stable order.  Then the per-slot tile counts.
__global__ void __launch_bounds__(1024) union_batch_kernel(const Shape s, const Work w,
                                                           int32_t* tile_prefix, int tile_n) {
  extern __shared__ int wcnt[];  // [32][E]
  __shared__ int cnt[kMaxE];
  __shared__ int start[kMaxE];
  const int E = s.E, K = s.K, T = s.T, TK = T * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int chunk = (TK + 31) / 32;
  const int c0 = warp * chunk, c1 = min(TK, c0 + chunk);
  for (int base = c0; base < c1; base += 32) {
    const int i = base + lane;
    const bool valid = i < c1;
    const int e = valid ? w.ids[i] : -1 - lane;
    const unsigned peers = __match_any_sync(FULL, e);
    if (valid && (__ffs(peers) - 1) == lane) {
      wcnt[warp * E + e] += __popc(peers);
      atomicAdd(&cnt[e], __popc(peers));
    }
    __syncwarp();
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int a0 = lane * per, a1 = min(E, a0 + per);
    int nz = 0, sum = 0;
    for (int e = a0; e < a1; ++e) {
      nz += cnt[e] > 0;
      sum += cnt[e];
    }
    int nz_ex = nz, sum_ex = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int a = __shfl_up_sync(FULL, nz_ex, off), b = __shfl_up_sync(FULL, sum_ex, off);
      if (lane >= off) {
        nz_ex += a;
        sum_ex += b;
      }
    }
    const int n_routed = __shfl_sync(FULL, nz_ex, 31);
    int slot = nz_ex - nz, off = sum_ex - sum;
    for (int e = a0; e < a1; ++e) {
      start[e] = off;
      if (cnt[e] > 0) {
        w.union_ids[slot] = e;
        w.offsets[slot] = off;
        ++slot;
        off += cnt[e];
      }
    }
    if (lane == 0) {
      int nu = n_routed;
      if (s.n_shared) {
        w.union_ids[nu] = E;
        w.offsets[nu] = TK;
        ++nu;
      }
      w.offsets[nu] = TK + (s.n_shared ? T : 0);
      *w.n_union = nu;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = start[e];
    for (int ww = 0; ww < 32; ++ww) {
      const int c = wcnt[ww * E + e];
      wcnt[ww * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = c0; base < c1; base += 32) {
    const int i = base + lane;
    const bool valid = i < c1;
    const int e = valid ? w.ids[i] : -1 - lane;
    const unsigned peers = __match_any_sync(FULL, e);
    if (valid) {
      const int pos = wcnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
      w.pair_token[pos] = i / K;
      w.pair_rank[pos] = i % K;
      w.inv[i] = pos;
    }
    __syncwarp();
    if (valid && (__ffs(peers) - 1) == lane) wcnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  if (s.n_shared)
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
      w.pair_token[TK + t] = t;
      w.pair_rank[TK + t] = -1;
    }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int nu = *w.n_union;
    int acc = 0;
    for (int u = 0; u < nu; ++u) {
      tile_prefix[u] = acc;
      acc += (w.offsets[u + 1] - w.offsets[u] + tile_n - 1) / tile_n;
    }
    tile_prefix[nu] = acc;
  }
}

// one CTA per pair slot of the largest batch: the pair's token codes as bf16, and its scales
__global__ void __launch_bounds__(256) gather_pairs_kernel(const Shape s, const Work w,
                                                           __nv_bfloat16* __restrict__ xb,
                                                           float* __restrict__ dxp) {
  const int p = blockIdx.x;
  const int P = w.offsets[*w.n_union];
  if (p >= P) return;
  const int d = s.d, nbd = d >> 5;
  const int t = w.pair_token[p];
  const int8_t* q = w.qx + (long)t * d;
  __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(xb + (long)p * d);
  for (int j = threadIdx.x; j < d / 2; j += blockDim.x)
    dst[j] = __floats2bfloat162_rn((float)q[2 * j], (float)q[2 * j + 1]);
  for (int b = threadIdx.x; b < nbd; b += blockDim.x) dxp[(long)p * nbd + b] = w.dx[(long)t * nbd + b];
}

cudaError_t configure_route_batch_kernels(int E) {
  cudaError_t e = cudaFuncSetAttribute(router_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       2 * kRbStage);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(union_batch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             32 * E * 4);
  return e;
}

cudaError_t launch_route_batch(const float* x, const Shape& s, const Store& st, const Work& w,
                               const CUtensorMap& map_wr, const CUtensorMap& map_x,
                               int32_t* tile_prefix, int tile_n, __nv_bfloat16* xb, float* dxp,
                               cudaStream_t stream) {
  prep_batch_kernel<<<s.T, 256, (size_t)s.d * sizeof(float), stream>>>(x, s, st, w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  router_batch_kernel<<<dim3((s.E + kRbE - 1) / kRbE, (s.T + kRbT - 1) / kRbT), 512, 2 * kRbStage,
                        stream>>>(map_wr, map_x, s, w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  topk_batch_kernel<<<(s.T + 7) / 8, 256, 0, stream>>>(s, st, w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  union_batch_kernel<<<1, 1024, (size_t)32 * s.E * 4, stream>>>(s, w, tile_prefix, tile_n);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int Pm = s.T * s.K + (s.n_shared ? s.T : 0);
  gather_pairs_kernel<<<Pm, 256, 0, stream>>>(s, w, xb, dxp);
  return cudaGetLastError();
}

// The batch's selection published to the workspace by one CTA (top-K, weights, union and
// buckets, the same values the expert kernels compute for themselves): a tiered layer reads the
// union back to the host to place the experts before the expert kernels run.
__global__ void __launch_bounds__(kThreads) select_publish_kernel(const Shape s, const Store st,
                                                                  const Work w) {
  extern __shared__ __align__(16) uint8_t sel_sm[];
  Sel sel = sel_carve(sel_sm, s.T, s.E);
  for (int i = threadIdx.x; i < s.T * s.E; i += blockDim.x) sel.sc[i] = __ldcg(w.scores + i);
  if (st.bias)
    for (int i = threadIdx.x; i < s.E; i += blockDim.x) sel.bias[i] = st.bias[i];
  __syncthreads();
  select_union(s, sel, st.bias != nullptr);
  sel_publish(s, sel, w);
}

cudaError_t launch_select_publish(const Shape& s, const Store& st, const Work& w,
                                  cudaStream_t stream) {
  select_publish_kernel<<<1, kThreads, (size_t)sel_bytes(s.T, s.E), stream>>>(s, st, w);
  return cudaGetLastError();
}

// slot table updates of a tiered layer: slot_of[ids[i]] = slots[i] in order (-1: not resident)
__global__ void set_slots_kernel(int32_t* slot_of, const SlotUpdate u) {
  if (threadIdx.x == 0)
    for (int i = 0; i < u.n; ++i) slot_of[u.ids[i]] = u.slots[i];
}

cudaError_t launch_set_slots(int32_t* slot_of, const SlotUpdate& u, cudaStream_t stream) {
  set_slots_kernel<<<1, 32, 0, stream>>>(slot_of, u);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* x, const Shape& s, const Store& st, const Work& w,
                         cudaStream_t stream) {
  // a programmatic dependent launch: its CTAs may be scheduled while the preceding grid
  // finishes, and wait for that grid (griddepcontrol.wait) before touching anything
  const int grid = (s.E + kRouterEpc - 1) / kRouterEpc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = route_smem_bytes(s.d, s.T);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel, x, s, st, w);
}

}  // namespace coli
