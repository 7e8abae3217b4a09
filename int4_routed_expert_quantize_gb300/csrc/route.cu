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
#include "coli_tc.cuh"

namespace coli {

// ------------------------------------------------------------------ router ---------------
constexpr int kRouterEpc = 2;  // experts per CTA
constexpr int kMaxE = 1024;

// top-K of one token by (score + bias) descending, ties to the lower expert id, then weights
// renormalised over the selected scores (sum taken in rank order).  One warp per token.
// sc: the token's E scores; ids/wt: its K outputs (shared or global memory).
__device__ void topk_token(const Shape& s, const Store& st, const float* sc, int* ids, float* wt,
                           int lane) {
  const int E = s.E, K = s.K;
  uint32_t taken = 0;  // bit m: expert lane + 32*m already selected
  float sv[32], sr[32];
  const int nm = (E + 31) >> 5;
  for (int m = 0; m < nm; ++m) {
    const int e = m * 32 + lane;
    sr[m & 31] = e < E ? sc[e] : 0.0f;
    sv[m & 31] = e < E ? (st.bias ? __fadd_rn(sr[m & 31], st.bias[e]) : sr[m & 31]) : 0.0f;
  }
  float S = 0.0f;      // lane 0: sum of the selected scores in rank order
  float pick[32];      // lane 0: the selected scores
  for (int k = 0; k < K; ++k) {
    float bv = 0.0f, bs = 0.0f;
    int bi = 0x7fffffff;
    for (int m = 0; m < nm; ++m) {
      const int e = m * 32 + lane;
      if (e >= E || ((taken >> m) & 1u)) continue;
      const float v = sv[m & 31];
      if (bi == 0x7fffffff || v > bv) {  // e ascending: a tie keeps the lower id
        bv = v;
        bs = sr[m & 31];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(FULL, bv, off);
      const float os = __shfl_xor_sync(FULL, bs, off);
      const int oi = __shfl_xor_sync(FULL, bi, off);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bs = os;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      ids[k] = bi;
      pick[k & 31] = bs;
      S = k == 0 ? bs : __fadd_rn(S, bs);
    }
  }
  if (lane == 0)
    for (int k = 0; k < K; ++k) wt[k] = __fmul_rn(__fdiv_rn(pick[k & 31], S), s.routed_scale);
  __syncwarp();
}

// Batch union by one CTA: count pairs per expert, list the distinct experts in ascending id
// order with their first pair, then place the pairs stably (pair index t*K+k ascending inside
// each expert) with one warp; the shared expert becomes the last slot with every token.
__device__ void union_bucket(const Shape& s, const Work& w, const int* idsv, int* cnt, int* cursor) {
  const int E = s.E, K = s.K, T = s.T, TK = T * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < TK; i += blockDim.x) atomicAdd(&cnt[idsv[i]], 1);
  __syncthreads();
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = lane * per, e1 = min(E, e0 + per);
    int nz = 0, sum = 0;
    for (int e = e0; e < e1; ++e) {
      nz += cnt[e] > 0;
      sum += cnt[e];
    }
    int nz_ex = nz, sum_ex = sum;  // inclusive scans, made exclusive below
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
    for (int e = e0; e < e1; ++e) {
      if (cnt[e] > 0) {
        w.union_ids[slot] = e;
        w.offsets[slot] = off;
        cursor[e] = off;
        ++slot;
        off += cnt[e];
      }
    }
    __syncwarp();
    for (int base = 0; base < TK; base += 32) {
      const int i = base + lane;
      const bool valid = i < TK;
      const int e = valid ? idsv[i] : -1 - lane;
      const unsigned peers = __match_any_sync(FULL, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int pos = 0;
      if (valid) {
        pos = cursor[e] + rank;
        w.pair_token[pos] = i / K;
        w.pair_rank[pos] = i % K;
        w.inv[i] = pos;
      }
      __syncwarp();
      if (valid && (__ffs(peers) - 1) == lane) cursor[e] += __popc(peers);
      __syncwarp();
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
    if (s.n_shared)
      for (int t = lane; t < T; t += 32) {
        w.pair_token[TK + t] = t;
        w.pair_rank[TK + t] = -1;
      }
  }
}

// Order-preserving key of a float score: a larger float gives a larger unsigned key, equal
// floats equal keys.  0 is below every finite score's key and marks an empty or taken entry.
// (The scores here are sigmoids plus an optional bias: finite, never -0.)
__device__ __forceinline__ uint32_t score_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// top-K of one token with warp reductions: lane l holds the keys of experts l, l+32, ...
// (NM per lane, E <= 32*NM).  Each round takes the largest key, ties to the lower expert id
// (each lane's own scan keeps its lowest id on a tie; the warp takes the lowest id among the
// lanes holding the maximum).  sc, bias: the token's E scores and the bias, in shared memory.
// Lane 0 writes the K ids; lane k < K writes weight k (selected scores renormalised, the sum
// taken in rank order).
template <int NM>
__device__ __forceinline__ void topk_warp(const float* sc, const float* bias, int E, int K,
                                          float routed_scale, int* ids, float* wt, int lane) {
  uint32_t key[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int e = m * 32 + lane;
    key[m] = e < E ? score_key(bias ? __fadd_rn(sc[e], bias[e]) : sc[e]) : 0u;
  }
  int my = 0;  // lane k < K: the k-th selected id
  for (int k = 0; k < K; ++k) {
    uint32_t bk = 0u;
    int bm = 0;
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      const bool gt = key[m] > bk;
      bm = gt ? m : bm;
      bk = gt ? key[m] : bk;
    }
    const uint32_t top = __reduce_max_sync(FULL, bk);
    const uint32_t win = __reduce_min_sync(FULL, bk == top ? (uint32_t)(bm * 32 + lane) : 0xFFFFFFFFu);
    const int wm = (int)(win & 31u) == lane ? (int)(win >> 5) : -1;
#pragma unroll
    for (int m = 0; m < NM; ++m) key[m] = m == wm ? 0u : key[m];
    if (lane == 0) ids[k] = (int)win;
    if (lane == k) my = (int)win;
  }
  // weights: the selected scores summed in rank order (values gathered by shuffle), then every
  // lane divides its own
  const float sk = lane < K ? sc[my] : 0.0f;
  float S = __shfl_sync(FULL, sk, 0);
  for (int k = 1; k < K; ++k) S = __fadd_rn(S, __shfl_sync(FULL, sk, k));
  if (lane < K) wt[lane] = __fmul_rn(__fdiv_rn(sk, S), routed_scale);
  __syncwarp();
}

// Batch union of at most 32 (token, rank) pairs by one warp: sorting the keys id*32 + pair
// index (bitonic network over the lanes) lists the pairs grouped by expert in ascending id
// order and, inside each expert, by pair index -- the stable bucket order; the slots start
// where the id changes.  The shared expert becomes the last slot with every token.
__device__ void union_warp(const Shape& s, const Work& w, const int* idsv, int lane) {
  const int TK = s.T * s.K, T = s.T, K = s.K;
  uint32_t v = lane < TK ? ((uint32_t)idsv[lane] << 5) | (uint32_t)lane : 0xFFFFFFFFu;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(FULL, v, j);
      const bool ascending = (lane & k) == 0, lower = (lane & j) == 0;
      v = (lower == ascending) ? min(v, o) : max(v, o);
    }
  }
  const bool valid = lane < TK;
  const int e = (int)(v >> 5), i = (int)(v & 31u);
  const int prev = __shfl_up_sync(FULL, e, 1);
  const bool head = valid && (lane == 0 || e != prev);
  const uint32_t heads = __ballot_sync(FULL, head);
  const int n_routed = __popc(heads);
  if (head) {
    const int slot = __popc(heads & ((1u << lane) - 1u));
    w.union_ids[slot] = e;
    w.offsets[slot] = lane;
  }
  if (valid) {
    w.pair_token[lane] = i / K;
    w.pair_rank[lane] = i % K;
    w.inv[i] = lane;
  }
  if (lane == 0) {
    int nu = n_routed;
    if (s.n_shared) {
      w.union_ids[nu] = s.E;
      w.offsets[nu] = TK;
      ++nu;
    }
    w.offsets[nu] = TK + (s.n_shared ? T : 0);
    *w.n_union = nu;
  }
  if (s.n_shared && lane < T) {
    w.pair_token[TK + lane] = lane;
    w.pair_rank[TK + lane] = -1;
  }
}

// After a timed-out wait, wait once more (bounded, ignoring the abort flag) for the bulk copy,
// so that no copy still writes shared memory when the CTA exits.
__device__ __noinline__ void route_drain(uint64_t* bar) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, 0u))
    if (global_ns() - t0 > kWaitLimitNs / 8) break;
}

// One launch does the whole routing half.  Every CTA: one bulk copy brings its kRouterEpc
// router rows into shared memory while all threads stage the tokens there (in the router's
// chunk order) and the gate/up grid is let start its weight prefetch; then the optional
// RMSNorm (one warp per token), the logits of its experts for every token (one warp per
// (expert, token): lane g runs the fma chain over its d/32 contiguous elements, the butterfly
// adds the 32 partials) and, on the other warps at the same time, this CTA's share of the int8
// activation blocks (one warp per block of 32).  The last CTA to finish (ticket counter, no
// waiting) selects the experts and builds the union in shared memory and registers.
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ x, const Shape s,
                                                    const Store st, const Work w) {
  extern __shared__ __align__(128) float route_sm[];
  __shared__ __align__(8) uint64_t wbar;
  __shared__ float rinv[kDecodeTmax];
  __shared__ int cnt[kMaxE];
  __shared__ int cursor[kMaxE];
  __shared__ int sids[kDecodeTmax * 32];
  __shared__ float swt[kDecodeTmax * 32];
  __shared__ int is_last;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int d = s.d, E = s.E, T = s.T, Gd = d >> 5, nbd = d >> 5;
  const int e0 = blockIdx.x * kRouterEpc;
  const int ne = min(kRouterEpc, E - e0);
  float* wrs = route_sm;                   // [kRouterEpc][d] router rows as stored
  float* xsm = route_sm + kRouterEpc * d;  // [T][max(d,E)] tokens, later the scores
  float* sbias = xsm + T * max(d, E);      // [E]
  if (threadIdx.x == 0) {
    mbar_init(&wbar, 1);
    abort_flag = 0;
    fence_barrier_init();
    mbar_expect_tx(&wbar, (uint32_t)(ne * d * 4));
    const uint64_t pol = l2_evict_last_policy();
    for (int r = 0; r < ne; ++r)
      bulk_g2s(wrs + r * d, st.wr + (long)(e0 + r) * d, (uint32_t)d * 4u, &wbar, pol);
  }
  griddep_launch_dependents();

  // tokens into shared memory in router order: lane g's elements g*Gd + 4*i4 .. +3 at chunk
  // i4*32 + g (coalesced float4 loads; conflict-free reads by lane)
#pragma unroll 8
  for (int c = threadIdx.x; c < T * (d / 4); c += blockDim.x) {
    const int t = c / (d / 4), pos = c - t * (d / 4);
    const int i4 = pos >> 5, g = pos & 31;
    reinterpret_cast<float4*>(xsm + (long)t * d)[pos] =
        *reinterpret_cast<const float4*>(x + (long)t * d + g * Gd + 4 * i4);
  }
  __syncthreads();
  if (s.has_norm) {
    // mean of squares in the canonical order (lane g: fma chain over its d/32 elements)
    for (int t = warp; t < T; t += nwarp) {
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
    for (int c = threadIdx.x; c < T * (d / 4); c += blockDim.x) {
      const int t = c / (d / 4), pos = c - t * (d / 4);
      const int i4 = pos >> 5, g = pos & 31;
      const float r = rinv[t];
      const float4 gm = *reinterpret_cast<const float4*>(st.gamma + g * Gd + 4 * i4);
      float4 v = reinterpret_cast<float4*>(xsm + (long)t * d)[pos];
      v.x = __fmul_rn(__fmul_rn(v.x, r), gm.x);
      v.y = __fmul_rn(__fmul_rn(v.y, r), gm.y);
      v.z = __fmul_rn(__fmul_rn(v.z, r), gm.z);
      v.w = __fmul_rn(__fmul_rn(v.w, r), gm.w);
      reinterpret_cast<float4*>(xsm + (long)t * d)[pos] = v;
    }
    __syncthreads();
  }

  // this CTA's share of the activation blocks: x_n (natural order), int8 codes, scale, code sum.
  // The warps that compute no logits take them (while the logits run); without such warps
  // every warp takes its share first.
  const int ndot = ne * T;
  const int nq = ndot < nwarp ? nwarp - ndot : nwarp;
  const int qw = ndot < nwarp ? warp - ndot : warp;
  for (int b = qw >= 0 ? blockIdx.x * nq + qw : T * nbd; b < T * nbd; b += gridDim.x * nq) {
    const int t = b / nbd, bb = b - t * nbd;
    const int j = bb * 32 + lane;
    const int g = j / Gd, m = j - g * Gd;
    const float v = xsm[(long)t * d + ((m >> 2) * 32 + g) * 4 + (m & 3)];
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
  bool waited = false;
  for (int pi = warp; pi < ndot; pi += nwarp) {
    if (!waited) {
      waited = true;
      if (!mbar_wait_bounded(&wbar, 0u, &abort_flag, w.status)) {
        route_drain(&wbar);
        break;
      }
    }
    const int r = pi / T, t = pi - r * T;
    const float4* wp = reinterpret_cast<const float4*>(wrs + (long)r * d);
    const float4* xp = reinterpret_cast<const float4*>(xsm + (long)t * d);
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
      w.logits[(long)t * E + e0 + r] = p;
      w.scores[(long)t * E + e0 + r] = canon_sigmoid(p);
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(w.counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // the last CTA: every score (and the bias) into shared memory in one round, selection and
  // union there, then the results out to the workspace
  float* ssc = xsm;  // [T][E] (the token buffer is no longer needed)
  for (int i = threadIdx.x; i < T * E; i += blockDim.x) ssc[i] = __ldcg(w.scores + i);
  if (st.bias)
    for (int i = threadIdx.x; i < E; i += blockDim.x) sbias[i] = st.bias[i];
  __syncthreads();
  const float* bs = st.bias ? sbias : nullptr;
  for (int t = warp; t < T; t += nwarp) {
    if (E <= 256)
      topk_warp<8>(ssc + t * E, bs, E, s.K, s.routed_scale, sids + t * s.K, swt + t * s.K, lane);
    else
      topk_warp<32>(ssc + t * E, bs, E, s.K, s.routed_scale, sids + t * s.K, swt + t * s.K, lane);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < T * s.K; i += blockDim.x) {
    w.ids[i] = sids[i];
    w.w[i] = swt[i];
  }
  if (T * s.K <= 32) {
    if (warp == 0) union_warp(s, w, sids, lane);
  } else {
    union_bucket(s, w, sids, cnt, cursor);
  }
  if (threadIdx.x == 0) *w.counter = 0;  // ready for the next call
}

static size_t route_smem_bytes(int d, int E, int T) {
  return ((size_t)kRouterEpc * d + (size_t)T * (d > E ? d : E) + E) * sizeof(float);
}

cudaError_t configure_route_kernels() {
  return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)route_smem_bytes(8192, kMaxE, kDecodeTmax));
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
  topk_token(s, st, w.scores + (long)t * s.E, w.ids + t * s.K, w.w + t * s.K, lane);
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

cudaError_t launch_route(const float* x, const Shape& s, const Store& st, const Work& w,
                         cudaStream_t stream) {
  // an ordinary launch: it reads the caller's x, so it stays ordered after all earlier work
  const int grid = (s.E + kRouterEpc - 1) / kRouterEpc;
  route_kernel<<<grid, 256, route_smem_bytes(s.d, s.E, s.T), stream>>>(x, s, st, w);
  return cudaGetLastError();
}

}  // namespace coli
