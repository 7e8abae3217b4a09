// Routing half of the layer: activation preparation (optional RMSNorm, Q8_0-style int8
// blocks of 32) and the sigmoid top-K router with the batch union.
//   "colibrì 架构概述" §3.1 (IDOT: decode activations quantised to int8), §5 (moe step:
//   sigmoid routing, top-8), the ai4coding.ru page (DeepSeek-V3-style sigmoid router,
//   Q8_0-style int8 activations) and the README's batch union (each distinct expert of a
//   batch is read once).
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"

namespace coli {

// ------------------------------------------------------------------ prep -----------------
// One CTA per token: x_n = RMSNorm(x) (or x), written in natural order and in the router's
// chunk order; then int8 codes, block scales and block code sums.
__global__ void __launch_bounds__(256) prep_kernel(const float* __restrict__ x, const Shape s,
                                                   const Store st, const Work w) {
  extern __shared__ float xs[];  // [d]
  __shared__ float rinv;
  const int t = blockIdx.x, d = s.d, nbd = d >> 5, Gd = d >> 5;  // Gd: elements per lane group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const float* xt = x + (long)t * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) xs[j] = xt[j];
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
    for (int j = threadIdx.x; j < d; j += blockDim.x)
      xs[j] = __fmul_rn(__fmul_rn(xs[j], r), st.gamma[j]);
    __syncthreads();
  }
  float* xn = w.xn + (long)t * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) xn[j] = xs[j];
  // router order: lane g's elements g*Gd + 4*i4 .. +3 at 4-float chunk i4*32 + g
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

cudaError_t launch_prep(const float* x, const Shape& s, const Store& st, const Work& w,
                        cudaStream_t stream) {
  prep_kernel<<<s.T, 256, s.d * sizeof(float), stream>>>(x, s, st, w);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ router ---------------
constexpr int kRouterEpc = 2;  // experts per CTA
constexpr int kMaxE = 1024;

// top-K of one token by (score + bias) descending, ties to the lower expert id, then weights
// renormalised over the selected scores (sum taken in rank order).  One warp per token.
__device__ void topk_token(const Shape& s, const Store& st, const Work& w, int t, int lane) {
  const int E = s.E, K = s.K;
  const float* sc = w.scores + (long)t * E;
  uint32_t taken = 0;  // bit m: expert lane + 32*m already selected
  for (int k = 0; k < K; ++k) {
    float bv = 0.0f;
    int bi = 0x7fffffff;
    for (int m = 0; m * 32 + lane < E; ++m) {
      if ((taken >> m) & 1u) continue;
      const int e = m * 32 + lane;
      const float sv = __ldcg(sc + e);
      const float v = st.bias ? __fadd_rn(sv, st.bias[e]) : sv;
      if (bi == 0x7fffffff || v > bv) {  // e ascending: a tie keeps the lower id
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(FULL, bv, off);
      const int oi = __shfl_xor_sync(FULL, bi, off);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) w.ids[t * K + k] = bi;
  }
  __syncwarp();
  if (lane == 0) {
    const int* ids = w.ids + t * K;
    float S = __ldcg(sc + ids[0]);
    for (int k = 1; k < K; ++k) S = __fadd_rn(S, __ldcg(sc + ids[k]));
    for (int k = 0; k < K; ++k)
      w.w[t * K + k] = __fmul_rn(__fdiv_rn(__ldcg(sc + ids[k]), S), s.routed_scale);
  }
}

// Batch union by one CTA: count pairs per expert, list the distinct experts in ascending id
// order with their first pair, then place the pairs stably (pair index t*K+k ascending inside
// each expert) with one warp; the shared expert becomes the last slot with every token.
__device__ void union_bucket(const Shape& s, const Work& w, int* cnt, int* cursor) {
  const int E = s.E, K = s.K, T = s.T, TK = T * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < TK; i += blockDim.x) atomicAdd(&cnt[w.ids[i]], 1);
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
      const int e = valid ? w.ids[i] : -1 - lane;
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

// Each CTA computes the logits of kRouterEpc experts for every token (one warp per
// (expert, token): lane g runs the fma chain over its d/32 contiguous elements, the warp
// butterfly adds the 32 partials); the last CTA to finish selects the experts and builds
// the union (last-block pattern: fence, ticket, no waiting).
__global__ void __launch_bounds__(256) router_kernel(const Shape s, const Store st, const Work w) {
  __shared__ int cnt[kMaxE];
  __shared__ int cursor[kMaxE];
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int d = s.d, E = s.E, T = s.T;
  const int e0 = blockIdx.x * kRouterEpc;
  const int ne = min(kRouterEpc, E - e0);
  const int nchunk = d / 128;  // 4-float chunks per lane
  for (int pi = warp; pi < ne * T; pi += nwarp) {
    const int e = e0 + pi / T, t = pi % T;
    const float4* wr = reinterpret_cast<const float4*>(st.wr + (long)e * d);
    const float4* xp = reinterpret_cast<const float4*>(w.xnp + (long)t * d);
    float p = 0.0f;
    for (int i4 = 0; i4 < nchunk; ++i4) {
      const float4 a = __ldg(wr + i4 * 32 + lane);
      const float4 b = xp[i4 * 32 + lane];
      p = __fmaf_rn(a.x, b.x, p);
      p = __fmaf_rn(a.y, b.y, p);
      p = __fmaf_rn(a.z, b.z, p);
      p = __fmaf_rn(a.w, b.w, p);
    }
    p = warp_tree_sum(p);
    if (lane == 0) {
      w.logits[(long)t * E + e] = p;
      w.scores[(long)t * E + e] = canon_sigmoid(p);
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(w.counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int t = warp; t < T; t += nwarp) topk_token(s, st, w, t, lane);
  __syncthreads();
  union_bucket(s, w, cnt, cursor);
  if (threadIdx.x == 0) *w.counter = 0;  // ready for the next call
}

cudaError_t launch_router(const Shape& s, const Store& st, const Work& w, int num_sms,
                          cudaStream_t stream) {
  (void)num_sms;
  const int grid = (s.E + kRouterEpc - 1) / kRouterEpc;
  router_kernel<<<grid, 256, 0, stream>>>(s, st, w);
  return cudaGetLastError();
}

}  // namespace coli
