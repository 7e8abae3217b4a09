// Expert selection of a decode batch (T <= 8 tokens), computed inside the CTAs that need it:
// top-K per token by score + selection bias (ties to the lower expert id), the weights
// renormalised over the selected scores (summed in rank order), and the batch union -- the
// distinct experts in ascending id order, each with its bucket of (token, rank) pairs in pair
// order, the shared expert last with every token.  Every CTA that runs it from the same scores
// gets the same result, so the expert kernels can each select for themselves instead of waiting
// for one CTA to publish it.  ("colibrì 架构概述" §5: sigmoid routing, top-8; the ai4coding.ru
// page: DeepSeek-V3-style selection bias and renormalised weights; README: batch union.)
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"

namespace coli {

// Selection state in shared memory
struct Sel {
  float* sc;     // [T][E] scores
  float* bias;   // [E]
  int* ids;      // [T*K] selected experts, rank order
  float* wt;     // [T*K] their weights
  int* skey;     // [T*K] sorted pair keys (scratch)
  int* u_ids;    // [nu] expert of each union slot (the shared expert's slot holds E)
  int* u_off;    // [nu+1] first pair of each slot
  int* p_tok;    // [P] token of each pair
  int* p_rank;   // [P] rank of each pair (-1: shared expert)
  int* inv;      // [T*K] pair position of (token, rank)
  int* nu;       // [1] number of union slots
};

// ints of the selection tables of a batch of T tokens (at most 32 routed pairs per token)
__host__ __device__ inline int sel_ints(int T) {
  const int mp = T * 32, ms = mp + 1;
  return 3 * mp + ms + (ms + 1) + 2 * (mp + T) + mp + 4;
}

__host__ __device__ inline int sel_bytes(int T, int E) {
  return ((T * E + E) * 4 + 15) / 16 * 16 + sel_ints(T) * 4;
}

__device__ inline Sel sel_carve(uint8_t* base, int T, int E) {
  const int mp = T * 32, ms = mp + 1;
  Sel m;
  m.sc = reinterpret_cast<float*>(base);
  m.bias = m.sc + T * E;
  int* p = reinterpret_cast<int*>(base + ((T * E + E) * 4 + 15) / 16 * 16);
  m.ids = p;
  p += mp;
  m.wt = reinterpret_cast<float*>(p);
  p += mp;
  m.skey = p;
  p += mp;
  m.u_ids = p;
  p += ms;
  m.u_off = p;
  p += ms + 1;
  m.p_tok = p;
  p += mp + T;
  m.p_rank = p;
  p += mp + T;
  m.inv = p;
  p += mp;
  m.nu = p;
  return m;
}

// Order-preserving key of a float score: a larger float gives a larger unsigned key, equal
// floats equal keys.  (The scores here are sigmoids plus an optional bias: never -0.)
__device__ __forceinline__ uint32_t score_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// top-K of one token by one warp in K rounds of warp reductions: lane l holds the score keys of
// experts l, l+32, ... (NM per lane, E <= 32*NM); each round takes the largest key, ties to the
// lower expert id (each lane's own scan keeps its lowest id on a tie; the warp takes the lowest
// id among the lanes holding the maximum).  Lane k < K writes id k and weight k (the selected
// scores renormalised by their sum taken in rank order).  sc, bias: the token's E scores and
// the bias, in shared memory.
template <int NM>
__device__ __forceinline__ void topk_warp(const float* sc, const float* bias, int E, int K,
                                          float routed_scale, int* ids, float* wt, int lane) {
  uint32_t key[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) {
    const int e = m * 32 + lane;
    key[m] = e < E ? score_key(bias ? __fadd_rn(sc[e], bias[e]) : sc[e]) : 0u;
  }
  int my = 0;
  float mine = 0.0f, S = 0.0f;
  for (int k = 0; k < K; ++k) {
    // this lane's best key by a tree (pairs, then pairs of pairs, ...): a tie keeps the lower m
    uint32_t bk[NM];
    int bm[NM];
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      bk[m] = key[m];
      bm[m] = m;
    }
#pragma unroll
    for (int w = 1; w < NM; w <<= 1) {
#pragma unroll
      for (int m = 0; m + w < NM; m += 2 * w) {
        const bool gt = bk[m + w] > bk[m];
        bk[m] = gt ? bk[m + w] : bk[m];
        bm[m] = gt ? bm[m + w] : bm[m];
      }
    }
    const uint32_t top = __reduce_max_sync(FULL, bk[0]);
    uint32_t win = __reduce_min_sync(FULL, bk[0] == top ? (uint32_t)(bm[0] * 32 + lane) : 0xFFFFFFFFu);
    win = win < (uint32_t)E ? win : 0u;  // only scores that are not numbers could leave none
    const int wm = (int)(win & 31u) == lane ? (int)(win >> 5) : -1;
#pragma unroll
    for (int m = 0; m < NM; ++m) key[m] = m == wm ? 0u : key[m];
    // the selected scores summed in rank order as they are found
    const float v = sc[win];
    S = k == 0 ? v : __fadd_rn(S, v);
    my = lane == k ? (int)win : my;
    mine = lane == k ? v : mine;
  }
  if (lane < K) {
    ids[lane] = my;
    wt[lane] = __fmul_rn(__fdiv_rn(mine, S), routed_scale);
  }
  __syncwarp();
}

// The common decode case (E <= 256, K <= 8, one token) in one warp with no CTA barrier inside
// and no divergent branch: each of the K rounds takes every lane's best key by a depth-3 tree
// (ties keep the lower expert), the warp maximum and the lowest expert among the lanes holding
// it (two warp reductions), and clears the winner's key; the rank-order sum of the selected
// scores builds up during the rounds.  With one token the union is the K distinct experts in
// ascending order, one pair each, then the shared expert: every lane knows all K winners, so
// lane j places pair j directly.
__device__ __forceinline__ void select_t1_fast(const Shape& s, Sel& m, const float* bias,
                                               int lane) {
  const int E = s.E, K = s.K;
  const float* sc = m.sc;
  uint32_t key[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = j * 32 + lane;
    key[j] = e < E ? score_key(bias ? __fadd_rn(sc[e], bias[e]) : sc[e]) : 0u;
  }
  int wid[8];
  float S = 0.0f, mine = 0.0f;
  int my = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    wid[k] = 0x7fffffff;
    if (k < K) {
      uint32_t k4[4];
      int m4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool gt = key[2 * i + 1] > key[2 * i];
        k4[i] = gt ? key[2 * i + 1] : key[2 * i];
        m4[i] = gt ? 2 * i + 1 : 2 * i;
      }
      uint32_t k2[2];
      int m2[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool gt = k4[2 * i + 1] > k4[2 * i];
        k2[i] = gt ? k4[2 * i + 1] : k4[2 * i];
        m2[i] = gt ? m4[2 * i + 1] : m4[2 * i];
      }
      const bool gt = k2[1] > k2[0];
      const uint32_t bk = gt ? k2[1] : k2[0];
      const int bm = gt ? m2[1] : m2[0];
      const uint32_t top = __reduce_max_sync(FULL, bk);
      uint32_t win = __reduce_min_sync(FULL, bk == top ? (uint32_t)(bm * 32 + lane) : 0xFFFFFFFFu);
      win = win < (uint32_t)E ? win : 0u;  // only scores that are not numbers could leave none
      const int wm = (int)(win & 31u) == lane ? (int)(win >> 5) : -1;
#pragma unroll
      for (int j = 0; j < 8; ++j) key[j] = j == wm ? 0u : key[j];
      const float v = sc[win];
      S = k == 0 ? v : __fadd_rn(S, v);
      wid[k] = (int)win;
      my = lane == k ? (int)win : my;
      mine = lane == k ? v : mine;
    }
  }
  int slot = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) slot += wid[k] < my ? 1 : 0;
  if (lane < K) {
    m.ids[lane] = my;
    m.wt[lane] = __fmul_rn(__fdiv_rn(mine, S), s.routed_scale);
    m.u_ids[slot] = my;
    m.u_off[slot] = slot;
    m.p_tok[slot] = 0;
    m.p_rank[slot] = lane;
    m.inv[lane] = slot;
  }
  if (lane == 0) {
    int nu = K;
    if (s.n_shared) {
      m.u_ids[nu] = E;
      m.u_off[nu] = K;
      m.p_tok[K] = 0;
      m.p_rank[K] = -1;
      ++nu;
    }
    m.u_off[nu] = K + (s.n_shared ? 1 : 0);
    *m.nu = nu;
  }
}

// Batch union of at most 32 (token, rank) pairs by one warp: sorting the keys id*32 + pair
// index (bitonic network over the lanes) lists the pairs grouped by expert in ascending id
// order and, inside each expert, by pair index; the slots start where the id changes.
__device__ inline void union_warp(const Shape& s, Sel& m, int lane) {
  const int TK = s.T * s.K, T = s.T, K = s.K;
  uint32_t v = lane < TK ? ((uint32_t)m.ids[lane] << 5) | (uint32_t)lane : 0xFFFFFFFFu;
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
  if (head) {
    const int slot = __popc(heads & ((1u << lane) - 1u));
    m.u_ids[slot] = e;
    m.u_off[slot] = lane;
  }
  if (valid) {
    m.p_tok[lane] = i / K;
    m.p_rank[lane] = i % K;
    m.inv[i] = lane;
  }
  if (lane == 0) {
    int nu = __popc(heads);
    if (s.n_shared) {
      m.u_ids[nu] = s.E;
      m.u_off[nu] = TK;
      ++nu;
    }
    m.u_off[nu] = TK + (s.n_shared ? T : 0);
    *m.nu = nu;
  }
  if (s.n_shared && lane < T) {
    m.p_tok[TK + lane] = lane;
    m.p_rank[TK + lane] = -1;
  }
}

// Selection from the scores (and, with has_bias, the bias) already in m.sc / m.bias and visible
// to the whole CTA.
// Every thread of the CTA calls it (it synchronises the CTA); results are visible on return.
// The union of more than 32 pairs: pair i = t*K + k gets key (expert << 8) | i; its position in
// the sorted keys is the number of smaller keys, which groups the pairs by expert in ascending id
// and keeps pair order inside each group; a slot starts wherever the expert changes.
__device__ inline void select_union(const Shape& s, Sel& m, bool has_bias) {
  const int T = s.T, K = s.K, E = s.E, TK = T * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* bias = has_bias ? m.bias : nullptr;
  if (T == 1 && E <= 256 && K <= 8) {
    if (warp == 0) select_t1_fast(s, m, bias, lane);
    __syncthreads();
    return;
  }
  if (warp < T) {
    if (E <= 256)
      topk_warp<8>(m.sc + warp * E, bias, E, K, s.routed_scale, m.ids + warp * K, m.wt + warp * K, lane);
    else
      topk_warp<32>(m.sc + warp * E, bias, E, K, s.routed_scale, m.ids + warp * K, m.wt + warp * K, lane);
  }
  __syncthreads();
  if (TK <= 32) {
    if (warp == 0) union_warp(s, m, lane);
    __syncthreads();
    return;
  }
  for (int i = threadIdx.x; i < TK; i += blockDim.x) {
    const int key = (m.ids[i] << 8) | i;
    int pos = 0;
    for (int j = 0; j < TK; ++j) pos += ((m.ids[j] << 8) | j) < key;
    m.skey[pos] = key;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < TK; p += blockDim.x) {
    const int key = m.skey[p], e = key >> 8, i = key & 255;
    int slot = 0;  // heads before p
    for (int q = 1; q <= p; ++q) slot += (m.skey[q] >> 8) != (m.skey[q - 1] >> 8);
    if (p == 0 || (m.skey[p - 1] >> 8) != e) {
      m.u_ids[slot] = e;
      m.u_off[slot] = p;
    }
    m.p_tok[p] = i / K;
    m.p_rank[p] = i % K;
    m.inv[i] = p;
  }
  if (threadIdx.x == 0) {
    int nr = 1;
    for (int q = 1; q < TK; ++q) nr += (m.skey[q] >> 8) != (m.skey[q - 1] >> 8);
    int nu = nr;
    if (s.n_shared) {
      m.u_ids[nu] = E;
      m.u_off[nu] = TK;
      ++nu;
    }
    m.u_off[nu] = TK + (s.n_shared ? T : 0);
    *m.nu = nu;
  }
  if (s.n_shared)
    for (int t = threadIdx.x; t < T; t += blockDim.x) {
      m.p_tok[TK + t] = t;
      m.p_rank[TK + t] = -1;
    }
  __syncthreads();
}

// The selection out to the workspace, for the debug dumps and for the down grid, then the flag
// that says it is there (release: every thread fences its own stores, the CTA synchronises,
// one thread raises the flag).  Every thread of one CTA calls it.
__device__ inline void sel_publish(const Shape& s, const Sel& m, const Work& w) {
  const int TK = s.T * s.K, P = TK + (s.n_shared ? s.T : 0), nu = *m.nu;
  for (int i = threadIdx.x; i < TK; i += blockDim.x) {
    w.ids[i] = m.ids[i];
    w.w[i] = m.wt[i];
    w.inv[i] = m.inv[i];
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    w.pair_token[p] = m.p_tok[p];
    w.pair_rank[p] = m.p_rank[p];
  }
  for (int i = threadIdx.x; i <= nu; i += blockDim.x) {
    if (i < nu) w.union_ids[i] = m.u_ids[i];
    w.offsets[i] = m.u_off[i];
  }
  if (threadIdx.x == 0) *w.n_union = nu;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(w.sel_flag), "r"(1) : "memory");
}

// 1 when the gate/up grid of this call has published its selection (acquire), else 0
__device__ __forceinline__ int sel_published(const Work& w) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(w.sel_flag) : "memory");
  return v;
}

// The published selection into shared memory (every thread of the CTA calls it after one thread
// saw the flag and the CTA synchronised); the same values select_union would compute.
__device__ inline void sel_load_published(const Shape& s, Sel& m, const Work& w) {
  const int TK = s.T * s.K, P = TK + (s.n_shared ? s.T : 0);
  const int nu = __ldcg(w.n_union);
  for (int i = threadIdx.x; i < TK; i += blockDim.x) {
    m.ids[i] = __ldcg(w.ids + i);
    m.wt[i] = __ldcg(w.w + i);
    m.inv[i] = __ldcg(w.inv + i);
  }
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    m.p_tok[p] = __ldcg(w.pair_token + p);
    m.p_rank[p] = __ldcg(w.pair_rank + p);
  }
  for (int i = threadIdx.x; i <= nu; i += blockDim.x) {
    if (i < nu) m.u_ids[i] = __ldcg(w.union_ids + i);
    m.u_off[i] = __ldcg(w.offsets + i);
  }
  if (threadIdx.x == 0) *m.nu = nu;
  __syncthreads();
}

}  // namespace coli
