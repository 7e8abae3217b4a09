// Device helpers of the coli_moe kernels (sm_103a): inline PTX for the bulk-copy engine and
// mbarriers, the mixed-sign dp4a, and the canonical fp32 operations (explicitly rounded
// intrinsics, so nvcc cannot contract or reorder them).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_internal.h"

namespace coli {

constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------ canonical fp32 -------
// exp(x) = 2^k * e^r: k the nearest integer to x*log2(e) (rounded with the 1.5*2^23 shifter),
// r = x - k*ln2 by Cody-Waite reduction (ln2 = hi + lo, hi with 12 fractional bits so k*hi is
// exact), e^r by the degree-7 Taylor polynomial in Horner form, then two exact power-of-two
// multiplies (only a subnormal result rounds).  Coefficients are 1/n! rounded to fp32.
__device__ __forceinline__ float canon_exp(float x) {
  if (x != x) return __fadd_rn(x, x);
  if (x > 89.0f) return __int_as_float(0x7f800000);
  if (x < -104.0f) return 0.0f;
  const float t = __fmul_rn(x, 0x1.715476p+0f);
  const float kf = __fsub_rn(__fadd_rn(t, 12582912.0f), 12582912.0f);
  float r = __fmaf_rn(-kf, 0x1.62ep-1f, x);
  r = __fmaf_rn(-kf, 0x1.0bfbe8p-15f, r);
  float p = __fmaf_rn(0x1.a01a02p-13f, r, 0x1.6c16c2p-10f);
  p = __fmaf_rn(p, r, 0x1.111112p-7f);
  p = __fmaf_rn(p, r, 0x1.555556p-5f);
  p = __fmaf_rn(p, r, 0x1.555556p-3f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  const int k = (int)kf;
  const int k1 = k / 2, k2 = k - k1;
  return __fmul_rn(__fmul_rn(p, __int_as_float((k1 + 127) << 23)), __int_as_float((k2 + 127) << 23));
}

__device__ __forceinline__ float canon_sigmoid(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, canon_exp(-x)));
}

// SiLU(g) * u, SiLU(g) = g / (1 + exp(-g))
__device__ __forceinline__ float canon_silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, canon_exp(-g))), u);
}

// xor butterfly over the 32 lanes; every lane ends with the pairwise-tree sum of the lane
// values in lane order (fp32 addition is commutative, so both partners compute the same sum)
__device__ __forceinline__ float warp_tree_sum(float v) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) v = __fadd_rn(v, __shfl_xor_sync(FULL, v, off));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, off));
  return v;
}

__device__ __forceinline__ int warp_isum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(FULL, v, off);
  return v;
}

// Q8_0-style code of one element of a 32-block held one element per lane:
// d = max|x| / 127, q = round(x / d) (half away from zero), clamped to [-127, 127].
__device__ __forceinline__ int q8_code(float x, float d) {
  if (d == 0.0f) return 0;
  int q = (int)roundf(__fdiv_rn(x, d));
  return max(-127, min(127, q));
}

// ------------------------------------------------------------------ integer dots ---------
// a: four unsigned bytes, b: four signed bytes -> c + sum a_i*b_i
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// int32 dot of one 32-element block.  w: the block's 16 bytes in the store layout (word k
// covers elements 8k..8k+7; byte m holds element 8k+m in its low nibble and 8k+m+4 in its
// high nibble, both offset by +8).  x: the 32 int8 codes as 8 words in element order.
// neg8sx = -8 * (sum of the 32 codes) removes the +8 offset exactly.
__device__ __forceinline__ int block_dot(const uint4 w, const uint32_t (&x)[8], int neg8sx) {
  int a1 = 0, a16 = 0;
  a1 = dp4a_us(w.x & 0x0F0F0F0Fu, x[0], a1);
  a16 = dp4a_us(w.x & 0xF0F0F0F0u, x[1], a16);
  a1 = dp4a_us(w.y & 0x0F0F0F0Fu, x[2], a1);
  a16 = dp4a_us(w.y & 0xF0F0F0F0u, x[3], a16);
  a1 = dp4a_us(w.z & 0x0F0F0F0Fu, x[4], a1);
  a16 = dp4a_us(w.z & 0xF0F0F0F0u, x[5], a16);
  a1 = dp4a_us(w.w & 0x0F0F0F0Fu, x[6], a1);
  a16 = dp4a_us(w.w & 0xF0F0F0F0u, x[7], a16);
  return a1 + (a16 >> 4) + neg8sx;
}

// block_dot with the weight words already split into their low-nibble and high-nibble halves
// (lo[k] = w.k & 0x0F0F0F0F, hi[k] = w.k & 0xF0F0F0F0), for a block dotted with several tokens
__device__ __forceinline__ void split_nibbles(const uint4 w, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
  lo[0] = w.x & 0x0F0F0F0Fu; hi[0] = w.x & 0xF0F0F0F0u;
  lo[1] = w.y & 0x0F0F0F0Fu; hi[1] = w.y & 0xF0F0F0F0u;
  lo[2] = w.z & 0x0F0F0F0Fu; hi[2] = w.z & 0xF0F0F0F0u;
  lo[3] = w.w & 0x0F0F0F0Fu; hi[3] = w.w & 0xF0F0F0F0u;
}
__device__ __forceinline__ int block_dot_split(const uint32_t (&lo)[4], const uint32_t (&hi)[4],
                                               const uint32_t (&x)[8], int neg8sx) {
  int a1 = 0, a16 = 0;
  a1 = dp4a_us(lo[0], x[0], a1);
  a16 = dp4a_us(hi[0], x[1], a16);
  a1 = dp4a_us(lo[1], x[2], a1);
  a16 = dp4a_us(hi[1], x[3], a16);
  a1 = dp4a_us(lo[2], x[4], a1);
  a16 = dp4a_us(hi[2], x[5], a16);
  a1 = dp4a_us(lo[3], x[6], a1);
  a16 = dp4a_us(hi[3], x[7], a16);
  return a1 + (a16 >> 4) + neg8sx;
}

// Position, within a stored row, of block b = g*G + i (G blocks per lane group): the groups are
// contiguous and a group's blocks are rotated by one for groups 4..7 mod 8, so that the
// 16-byte loads of 8 consecutive lanes fall in distinct shared-memory banks.
__host__ __device__ __forceinline__ int store_chunk(int g, int i, int G) {
  int c = i + ((g >> 2) & 1);
  if (c >= G) c -= G;
  return g * G + c;
}

// The same for 8-byte units (int2 blocks): rotated by one for groups 8..15 mod 16, so that the
// 8-byte loads of 16 consecutive lanes fall in distinct banks.
__host__ __device__ __forceinline__ int store_chunk8(int g, int i, int G) {
  int c = i + ((g >> 3) & 1);
  if (c >= G) c -= G;
  return g * G + c;
}

__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ------------------------------------------------------------------ weight widths ---------
// One 32-element weight block of a stored row, prepared as 8 words for dp4a against the block's
// activation codes x[0..7] (x[j] = elements 4j..4j+3), for WB = 4, 8 or 2 bits per weight:
//  * int4 (store: 16 bytes, word k = elements 8k..8k+7, byte m = element 8k+m low nibble and
//    8k+m+4 high nibble, each code + 8): w[2k] = word & 0x0F0F0F0F pairs with x[2k], w[2k+1] =
//    word & 0xF0F0F0F0 (16 x code) with x[2k+1];
//  * int8 (store: the block's two 16-byte halves in two planes of the row, nb chunks apart,
//    codes as they are): w[j] = word j, signed;
//  * int2 (store: 8 bytes, word h = elements 16h..16h+15, element 16h+4k+m in bits 2k..2k+1 of
//    byte m, each code + 2): w[4h+k] = (word h >> 2k) & 0x03030303.
// The offset codes (+8, +2) are removed by the block's correction -off * sum(x).
template <int WB>
struct Wfmt {
  static constexpr int off = WB == 4 ? 8 : (WB == 2 ? 2 : 0);  // code offset in the store
  static constexpr int row_bytes(int n) { return n * WB / 8; }
};

// row: the stored row; g: the lane's group; i: block within the group; G blocks per group; nb
// blocks in the row.  Lanes outside the active groups pass on = false and get zeros.
template <int WB>
__device__ __forceinline__ void wload(const uint8_t* row, int g, int i, int G, int nb, bool on,
                                      uint32_t (&w)[8]) {
  if constexpr (WB == 4) {
    uint4 c = make_uint4(0, 0, 0, 0);
    if (on) c = *reinterpret_cast<const uint4*>(row + store_chunk(g, i, G) * 16);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[2 * k] = cw[k] & 0x0F0F0F0Fu;
      w[2 * k + 1] = cw[k] & 0xF0F0F0F0u;
    }
  } else if constexpr (WB == 8) {
    uint4 c0 = make_uint4(0, 0, 0, 0), c1 = make_uint4(0, 0, 0, 0);
    if (on) {
      const int o = store_chunk(g, i, G) * 16;
      c0 = *reinterpret_cast<const uint4*>(row + o);
      c1 = *reinterpret_cast<const uint4*>(row + nb * 16 + o);
    }
    w[0] = c0.x; w[1] = c0.y; w[2] = c0.z; w[3] = c0.w;
    w[4] = c1.x; w[5] = c1.y; w[6] = c1.z; w[7] = c1.w;
  } else {
    uint2 c = make_uint2(0, 0);
    if (on) c = *reinterpret_cast<const uint2*>(row + store_chunk8(g, i, G) * 8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[k] = (c.x >> (2 * k)) & 0x03030303u;
      w[4 + k] = (c.y >> (2 * k)) & 0x03030303u;
    }
  }
}

// exact int32 dot of a prepared weight block with the block's activation codes; corr = -off *
// (sum of the 32 activation codes)
template <int WB>
__device__ __forceinline__ int wdot(const uint32_t (&w)[8], const uint32_t (&x)[8], int corr) {
  if constexpr (WB == 4) {
    int a1 = 0, a16 = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a1 = dp4a_us(w[2 * k], x[2 * k], a1);
      a16 = dp4a_us(w[2 * k + 1], x[2 * k + 1], a16);
    }
    return a1 + (a16 >> 4) + corr;
  } else if constexpr (WB == 8) {
    int a = 0, b = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a = dp4a_ss(w[k], x[k], a);
      b = dp4a_ss(w[4 + k], x[4 + k], b);
    }
    return a + b + corr;
  } else {
    int a = 0, b = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      a = dp4a_us(w[k], x[k], a);
      b = dp4a_us(w[4 + k], x[4 + k], b);
    }
    return a + b + corr;
  }
}

// ------------------------------------------------------------------ mbarrier / bulk copy ---
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async (bulk-copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `parity` of `bar`.  Gives up after kWaitLimitNs, records
// COLI_ETIMEOUT in the device status word and raises the CTA's abort flag; once the flag is
// up every later wait returns false at once, so no thread of the CTA can block forever.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort_flag, int* status) {
  if (*abort_flag) return false;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicExch(status, COLI_ETIMEOUT);
        return false;
      }
    }
  }
}

// fast path inline (phase already complete), the bounded loop out of line
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, status);
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// one bulk copy global -> shared (the TMA engine's non-tensor form), completing on `bar`.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Two lanes of fp32 at once (sm_100 and later): each lane rounds exactly as the scalar
// fma.rn / add.rn does, so a pair of these is bit-identical to two scalar operations.
// c = a * b + c on (c0, c1)
__device__ __forceinline__ void fma2_rn(float a0, float a1, float b0, float b1, float& c0, float& c1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// c = a + c on (c0, c1)
__device__ __forceinline__ void add2_rn(float a0, float a1, float& c0, float& c1) {
  asm("{\n\t.reg .b64 a, c;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 c, {%0, %1};\n\t"
      "add.rn.f32x2 c, a, c;\n\tmov.b64 {%0, %1}, c;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1));
}

// hint: bring the 128-byte line holding p into L2
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// asynchronous 4-byte copy global -> shared through the load path (not the bulk-copy engine,
// whose queue may hold weight stages); the thread's copies are complete after
// cp_async_wait_all()
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// programmatic dependent launch: wait for the preceding grid (no-op without the attribute) /
// allow the next grid in the stream to start its prologue
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Store slot of expert `ex`: the slot table of a tiered layer, else the id itself.  An expert
// that is not resident (a forward on a tiered layer before its experts were placed) reads slot 0
// and records COLI_ESTATE in the status word, so no copy addresses outside the store.
__device__ __forceinline__ long store_slot(const Store& st, int ex, int* status) {
  if (!st.slot_of) return ex;
  const int s = __ldcg(st.slot_of + ex);
  if (s < 0) {
    atomicExch(status, COLI_ESTATE);
    return 0;
  }
  return s;
}

// ------------------------------------------------------------------ shared by the expert kernels
// Sum over the warp of 8 values per lane, one per row: the exchange at distance o keeps half
// of the rows on each side, so after distances 1, 2, 4 lane l holds one row's partial, and
// distances 8, 16 finish it.  Every row's total is the pairwise tree over lanes in lane order,
// bit-identical to warp_tree_sum.  Returns the total of row 4*(l&1) + 2*((l>>1)&1) + ((l>>2)&1)
// (the same in lanes l, l+8, l+16, l+24).
__device__ __forceinline__ float warp_tree_sum8(const float (&v)[8], int lane) {
  const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
  float u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b0 ? v[i + 4] : v[i], send = b0 ? v[i] : v[i + 4];
    u[i] = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 1));
  }
  float z[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float keep = b1 ? u[i + 2] : u[i], send = b1 ? u[i] : u[i + 2];
    z[i] = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 2));
  }
  const float keep = b2 ? z[1] : z[0], send = b2 ? z[0] : z[1];
  float r = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 4));
  r = __fadd_rn(r, __shfl_xor_sync(FULL, r, 8));
  r = __fadd_rn(r, __shfl_xor_sync(FULL, r, 16));
  return r;
}

// After an abort, wait (bounded, ignoring the abort flag) for the last fills the producer
// issued, so no bulk copy is still writing shared memory when the CTA exits.
static __device__ __noinline__ void drain_fills(uint64_t* full, int nst, long issued) {
  const long first = issued > nst ? issued - nst : 0;
  for (long it = first; it < issued; ++it) {
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(&full[it % nst], (uint32_t)((it / nst) & 1))) {
      if (global_ns() - t0 > kWaitLimitNs / 8) break;
    }
  }
}

}  // namespace coli
