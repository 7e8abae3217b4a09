// Expert kernels of the batched (prefill) path on the 5th-generation tensor cores.
//
// For a batch the union experts see many tokens each (up to a few hundred), so the expert
// projections are genuinely dense grouped GEMMs: per union slot, [rows of W] x [K] x [pairs of
// the slot's bucket].  sm_103a has no int8 MMA (ptxas refuses tcgen05.mma kind::i8 for it),
// so the int8 x int4 products run as kind::f16 with bf16 operands holding the exact integers
// (|code| <= 127, products <= 1016, a 32-term block sum < 2^24: every partial is exact in the
// f32 accumulator).  Each K-block of 32 (one activation scale) gets accumulator columns of its
// own (its two MMAs write only those, below), so the epilogue sees the exact int32 block dot
// and applies the canonical fp32 order of the decode path: an fma chain over
// the blocks of each of 32 contiguous groups (registers) and the pairwise tree over the groups
// (a 5-level stack kept in TMEM columns).  Results are therefore bit-identical to the decode
// kernels and the CPU oracle ("colibrì 架构概述" §5 gate/up/SiLU/down; README batch union).
//
// CTA: 15 warps, one tile (128 weight rows x 32 pairs) at a time, persistent over tiles:
//   warp 0      bulk-tensor copies of raw int4 weight groups (HBM stream)
//   warp 1      bulk-tensor copies of each burst's activation codes (bf16): two boxes of 64 K x
//               32 pairs with 128-byte swizzle
//   warp 2      TMEM owner (512 columns: two accumulator buffers, the tree stack) and the single
//               MMA issuer: per burst 8 MMAs (K = 16, N = 32 per block) and two commits (operand
//               stage free; accumulator ready)
//   warps 3-6   int4 -> bf16 conversion of the weight blocks into the MMA's shared layout
//   warps 7-14  epilogue: TMEM -> registers, block scales, canonical sums, SwiGLU / outputs
//               (warp w: TMEM lanes 32*(w%4).., 16 of the tile's 32 pairs)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_tc.cuh"

namespace coli {

constexpr int kPfM = 128;               // weight rows per tile
constexpr int kPfP = kPrefillTileN;     // pairs per tile
constexpr int kPfR = 4;                 // 32-element blocks per MMA burst
constexpr int kPfN = kPfR * kPfP;       // MMA width: block-diagonal columns (block, pair)
constexpr int kPfBurstK = kPfR * 32;    // K elements of a burst
constexpr int kPfOpStages = 3;          // operand stages (converted weights + activations) in flight
constexpr int kPfAccStages = 2;         // accumulator buffers in flight
constexpr int kPfRawStages = 4;         // raw int4 weight ring (one lane group of blocks each)
constexpr int kPfConv = 4;              // int4 -> bf16 converter warps
constexpr int kPfEpi0 = 3 + kPfConv;    // first epilogue warp
static_assert(kPfConv == 4 || kPfConv == 8, "converter warps: one or two per row");
constexpr int kPfEpiW = 8;              // epilogue warps: 2 per TMEM lane quadrant
constexpr int kPfEpiC = kPfP * 4 / kPfEpiW;  // pairs (accumulator columns per block) per epilogue warp
constexpr int kPfWarps = kPfEpi0 + kPfEpiW;
constexpr int kDxS = kPfP + 4;          // row stride (floats) of the staged block scales: 16-byte rows,
                                        // and 8 blocks x 4 pairs of one copy round hit 32 banks
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfAStage = kPfM * kPfBurstK * 2;   // 32 KB of bf16 weights
constexpr int kPfBStage = kPfBurstK * kPfP * 2;   // 8 KB of bf16 activations: 2 x [32 pairs][64 K], 128-byte swizzle
constexpr uint32_t kTmemCols = 512;     // accumulators 2 x 128 columns, tree stack 5 x 32
constexpr uint32_t kStackCol = kPfAccStages * kPfN;

struct PfArgs {
  Shape s;
  Store st;
  Work w;
  PrefillWork pw;
  ExpertDebug dbg;
  int down;   // 0: gate/up + SwiGLU, 1: down
  int raw_stage_bytes;
  int dx_bytes;
};

struct PfSmem {
  uint8_t* raw;
  uint8_t* a;
  uint8_t* b;
  float* dxs;  // [nb][kDxS]: block scales of the tile's pairs
  float* us;   // [kPfP][64] u values (gate/up only)
  uint64_t* raw_full;
  uint64_t* raw_empty;
  uint64_t* a_full;     // a burst's converted weights and activation blocks are in
  uint64_t* op_free;    // a burst's MMAs are complete: its operand stage is free
  uint64_t* acc_full;   // ... and its accumulator is readable
  uint64_t* acc_empty;  // the epilogue has read a burst's accumulator
  uint32_t* tmem_slot;
  int* tp;    // [nu+1] tile prefix per union slot
  int* tex;   // [nu]   expert id per union slot
  int* toff;  // [nu+1] first pair per union slot
};

__device__ __forceinline__ PfSmem pf_carve(uint8_t* smem, const PfArgs& a) {
  PfSmem m;
  uint8_t* p = smem;
  m.b = p;  // first: the swizzled activation stages need 1024-byte alignment
  p += kPfOpStages * kPfBStage;
  m.raw = p;
  p += kPfRawStages * a.raw_stage_bytes;
  m.a = p;
  p += kPfOpStages * kPfAStage;
  m.dxs = reinterpret_cast<float*>(p);
  p += a.dx_bytes;
  m.us = reinterpret_cast<float*>(p);
  p += a.down ? 0 : kPfP * 64 * 4;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  m.raw_full = bars;
  m.raw_empty = bars + kPfRawStages;
  m.a_full = m.raw_empty + kPfRawStages;
  m.op_free = m.a_full + kPfOpStages;
  m.acc_full = m.op_free + kPfOpStages;
  m.acc_empty = m.acc_full + kPfAccStages;
  m.tmem_slot = reinterpret_cast<uint32_t*>(m.acc_empty + kPfAccStages);
  m.tp = reinterpret_cast<int*>(m.tmem_slot + 4);
  m.tex = m.tp + a.s.E + 2;
  m.toff = m.tex + a.s.E + 2;
  return m;
}

int prefill_smem_bytes(int d, int f, int E, int down) {
  const int K = down ? f : d;
  const int nb = K / kQB, G = (nb + 31) / 32;
  const int raw = kPfM * G * 16;
  const int dx = nb * kDxS * 4;
  const int bars = (2 * kPfRawStages + 2 * kPfOpStages + 2 * kPfAccStages) * 8 + 16;
  const int tabs = 3 * (E + 2) * 4;
  return kPfRawStages * raw + kPfOpStages * (kPfAStage + kPfBStage) + dx + (down ? 0 : kPfP * 64 * 4) +
         bars + tabs;
}

// tile t -> (union slot, M-tile, N-tile); slots own n_mt * ntiles(slot) consecutive tiles,
// N fastest so consecutive tiles share their weight rows (L2 reuse).  prefix: shared memory.
__device__ __forceinline__ void pf_tile(const int* prefix, int nu, int n_mt, int t, int& u,
                                        int& mt, int& nt) {
  int lo = 0, hi = nu - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (n_mt * prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  u = lo;
  const int base = n_mt * prefix[u];
  const int ntu = prefix[u + 1] - prefix[u];
  const int r = t - base;
  mt = r / ntu;
  nt = r - mt * ntu;
}

// int4 chunk (store layout: word k = elements 8k..8k+7, byte m low nibble 8k+m, high 8k+m+4,
// each code + 8) -> 4 x 16 bytes of bf16 (k-core kc = elements 8kc..8kc+7 in order)
__device__ __forceinline__ void int4_chunk_to_bf16(const uint4 c, uint4 (&out)[4]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = w[k] & 0x0F0F0F0Fu, hi = (w[k] >> 4) & 0x0F0F0F0Fu;
    // 0x43vv is bf16(128 + v); subtracting 136 leaves v - 8 = the signed code exactly
    uint32_t q[4] = {__byte_perm(lo, 0x43434343u, 0x4140), __byte_perm(lo, 0x43434343u, 0x4342),
                     __byte_perm(hi, 0x43434343u, 0x4140), __byte_perm(hi, 0x43434343u, 0x4342)};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&q[j]);
      v = __hsub2(v, off);
      q[j] = *reinterpret_cast<uint32_t*>(&v);
    }
    out[k] = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

// group leaf gi complete: merge it into the pairwise-tree stack (levels in TMEM); after the last
// leaf `chain` holds the whole sum
#define COLI_PF_PUSH_GROUP()                                                   \
  {                                                                            \
    int l = 0;                                                                 \
    for (; (gi >> l) & 1; ++l) {                                               \
      float lv[kPfEpiC];                                                       \
      tmem_ld16(tl + kStackCol + l * kPfP + e8, lv);                           \
      _Pragma("unroll") for (int c = 0; c < kPfEpiC; c += 2)                   \
        add2_rn(lv[c], lv[c + 1], chain[c], chain[c + 1]);                     \
    }                                                                          \
    if (l < 5) {                                                               \
      tmem_st16(tl + kStackCol + l * kPfP + e8, chain);                        \
      _Pragma("unroll") for (int c = 0; c < kPfEpiC; ++c) chain[c] = 0.0f;    \
    }                                                                          \
    ++gi;                                                                      \
  }

// One tile = 128 weight rows x 32 pairs of one union slot, its K range walked in bursts of 4
// blocks of 32.  A burst is 8 MMAs (K = 16 each, M = 128, N = 32) into one accumulator buffer of
// 128 columns: block j of the burst accumulates into columns 32j..32j+31 only, so column
// (j, p) holds the exact int32 dot of block j with pair p.  After the burst one commit frees its
// operand stage and another hands the accumulator to the epilogue.
template <bool kDown>
__global__ void __launch_bounds__(kPfThreads, 1)
    expert_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                       const PfArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int abort_flag;
  const PfSmem m = pf_carve(smem, a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.s.d, f = a.s.f;
  constexpr bool down = kDown;
  const int K = down ? f : d;
  const int nb = K / kQB, G = (nb + 31) / 32, ngrp = nb / G;
  const int nburst = nb / kPfR;  // d and f are multiples of 128
  const int n_mt = down ? d / kPfM : f / (kPfM / 2);
  const int raw_bytes = kPfM * G * 16;
  const int nu = __ldcg(a.w.n_union);
  const int total = n_mt * __ldcg(a.pw.tile_prefix + nu);
  int* status = a.w.status;

  if ((smem_addr(m.b) & 1023u) != 0) {  // the swizzled activation stages need 1024-byte alignment
    if (threadIdx.x == 0) atomicExch(a.w.status, COLI_EUNSUPPORTED);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfRawStages; ++i) {
      mbar_init(&m.raw_full[i], 1);
      mbar_init(&m.raw_empty[i], kPfConv);
    }
    for (int i = 0; i < kPfOpStages; ++i) {
      mbar_init(&m.a_full[i], kPfConv + 1);  // the converter warps + the activation loader (expect_tx)
      mbar_init(&m.op_free[i], 1);
    }
    for (int i = 0; i < kPfAccStages; ++i) {
      mbar_init(&m.acc_full[i], 1);
      mbar_init(&m.acc_empty[i], kPfEpiW);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i <= nu; i += blockDim.x) {
    m.tp[i] = __ldcg(a.pw.tile_prefix + i);
    m.toff[i] = __ldcg(a.w.offsets + i);
    m.tex[i] = i < nu ? __ldcg(a.w.union_ids + i) : 0;
  }
  if (warp == 2) tmem_alloc(m.tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *m.tmem_slot;

  if (warp == 0) {
    // ---------------- raw int4 weight groups (128 rows x G chunks) by tensor copies
    if (lane == 0) {
      long kg = 0;
      for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
        int u, mt, nt;
        pf_tile(m.tp, nu, n_mt, t, u, mt, nt);
        const int ex = m.tex[u];
        for (int gi = 0; gi < ngrp; ++gi, ++kg) {
          const int rs = (int)(kg % kPfRawStages);
          const long n = kg / kPfRawStages;
          if (n > 0 && !mbar_wait_bounded(&m.raw_empty[rs], (uint32_t)((n - 1) & 1), &abort_flag, status))
            break;
          uint8_t* dst = m.raw + (long)rs * a.raw_stage_bytes;
          mbar_expect_tx(&m.raw_full[rs], (uint32_t)raw_bytes);
          if (down) {
            tma_load_2d(dst, &map_w, gi * G * 16, ex * d + mt * kPfM, &m.raw_full[rs]);
          } else {
            const int y = ex * f + mt * (kPfM / 2);
            tma_load_2d(dst, &map_w, gi * G * 16, y, &m.raw_full[rs]);
            tma_load_2d(dst + (kPfM / 2) * G * 16, &map_w, d / 2 + gi * G * 16, y, &m.raw_full[rs]);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- the activation blocks of every burst, each on the diagonal: block j of
    // the burst -> K rows 32j..32j+31 (core-matrix columns 4j..4j+3) x columns 32j..32j+31
    if (lane == 0) {
      long kb = 0;
      for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
        int u, mt, nt;
        pf_tile(m.tp, nu, n_mt, t, u, mt, nt);
        const int row0 = m.toff[u] + nt * kPfP;
        for (int bu = 0; bu < nburst; ++bu, ++kb) {
          const int s = (int)(kb % kPfOpStages);
          const long n = kb / kPfOpStages;
          if (n > 0 && !mbar_wait_bounded(&m.op_free[s], (uint32_t)((n - 1) & 1), &abort_flag, status))
            break;
          uint8_t* dst = m.b + (long)s * kPfBStage;
          mbar_expect_tx(&m.a_full[s], (uint32_t)kPfBStage);
          // two boxes of 64 K x 32 pairs (128-byte rows, swizzled): blocks 0-1 and 2-3
          tma_load_2d(dst, &map_x, bu * kPfBurstK, row0, &m.a_full[s]);
          tma_load_2d(dst + kPfBStage / 2, &map_x, bu * kPfBurstK + kPfBurstK / 2, row0, &m.a_full[s]);
        }
      }
    }
  } else if (warp >= 3 && warp < kPfEpi0) {
    // ---------------- int4 -> bf16: thread r owns weight row r % 128 of the tile and, with more
    // than 4 converter warps, its share of a burst's blocks (j % (kPfConv / 4) == r / 128);
    // block j of a burst goes to core-matrix columns 4j..4j+3 of the burst's weight stage.  A
    // burst's raw chunks are all read before any is converted, so the four conversions overlap.
    const int r = (threadIdx.x - 96) & (kPfM - 1);
    const int hf = (threadIdx.x - 96) >> 7;
    long kb = 0, kg = 0;  // bursts and raw groups so far
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int gi = 0, ci = 0;  // group of the next block, and its chunk within the group
      for (int bu = 0; bu < nburst; ++bu, ++kb) {
        const int s = (int)(kb % kPfOpStages);
        const long n = kb / kPfOpStages;
        if (n > 0) mbar_wait_bounded(&m.op_free[s], (uint32_t)((n - 1) & 1), &abort_flag, status);
        uint4 c[kPfR];
        int rel = 0;  // raw stages released by this burst: count, first one is (kg0 % ring)
        const long kg0 = kg;
#pragma unroll
        for (int j = 0; j < kPfR; ++j) {
          const int rs = (int)(kg % kPfRawStages);
          if (ci == 0) mbar_wait_bounded(&m.raw_full[rs], (uint32_t)((kg / kPfRawStages) & 1), &abort_flag, status);
          int cc = ci + ((gi >> 2) & 1);  // the store's chunk rotation within a group
          if (cc >= G) cc -= G;
          c[j] = make_uint4(0, 0, 0, 0);
          if (j % (kPfConv / 4) == hf)
            c[j] = *reinterpret_cast<const uint4*>(m.raw + (long)rs * a.raw_stage_bytes + (r * G + cc) * 16);
          if (++ci == G) {
            ci = 0;
            ++gi;
            ++kg;
            ++rel;
          }
        }
        uint8_t* ast = m.a + (long)s * kPfAStage;
#pragma unroll
        for (int j = 0; j < kPfR; ++j) {
          if (j % (kPfConv / 4) != hf) continue;
          uint4 o[4];
          int4_chunk_to_bf16(c[j], o);
#pragma unroll
          for (int kc = 0; kc < 4; ++kc)
            *reinterpret_cast<uint4*>(ast + ((4 * j + kc) * (kPfM / 8) + (r >> 3)) * 128 + (r & 7) * 16) = o[kc];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&m.a_full[s]);
          for (int i = 0; i < rel; ++i) mbar_arrive(&m.raw_empty[(int)((kg0 + i) % kPfRawStages)]);
        }
      }
    }
  } else if (warp == 2) {
    // ---------------- MMA issuer: one burst of 8 MMAs and one commit per 4 blocks
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPfM, kPfP);
      long kb = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        for (int bu = 0; bu < nburst; ++bu, ++kb) {
          const int s = (int)(kb % kPfOpStages), sa = (int)(kb % kPfAccStages);
          const long n = kb / kPfOpStages, na = kb / kPfAccStages;
          bool ok = mbar_wait_bounded(&m.a_full[s], (uint32_t)(n & 1), &abort_flag, status);
          if (na > 0) ok = mbar_wait_bounded(&m.acc_empty[sa], (uint32_t)((na - 1) & 1), &abort_flag, status) && ok;
          if (!ok) continue;
          tc_fence_after();
          const uint8_t* as = m.a + (long)s * kPfAStage;
          const uint8_t* bs = m.b + (long)s * kPfBStage;
#pragma unroll
          for (int ks = 0; ks < kPfBurstK / 16; ++ks) {
            const int j = ks >> 1, kk = ks & 1;  // block j of the burst -> accumulator columns 32j..
            const uint64_t da = smem_desc(as + ks * 2 * (kPfM / 8) * 128, (kPfM / 8) * 128, 128);
            const uint64_t db = smem_desc_sw128(bs + (j >> 1) * (kPfBStage / 2) + (j & 1) * 64 + kk * 32);
            tc_mma_bf16(tmem + (uint32_t)(sa * kPfN + j * kPfP), da, db, idesc, kk > 0);
          }
          tc_commit(&m.op_free[s]);
          tc_commit(&m.acc_full[sa]);
        }
      }
    }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32*(w%4).. and the columns of pairs
    // e8..e8+7 of every block
    const int q = warp & 3;
    const int e8 = ((warp - kPfEpi0) >> 2) * kPfEpiC;
    const int row = q * 32 + lane;
    const int ew = warp - kPfEpi0;
    const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
    int32_t* const Adump = down ? a.dbg.Ad : a.dbg.Ag;
    long kb = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      int u, mt, nt;
      pf_tile(m.tp, nu, n_mt, t, u, mt, nt);
      const int ex = m.tex[u];
      const int pb = m.toff[u] + nt * kPfP;  // first pair of the tile
      const int pe = m.toff[u + 1];          // end of the slot's pairs
      const int nv = min(kPfP, pe - pb);       // valid pairs of the tile
      const bool active = e8 < nv;             // this warp has columns to finish
      // this tile's activation block scales -> dxs[block][pair], all copies in flight at once: a
      // copy round is 8 consecutive blocks (32 contiguous bytes of a pair's row) x 4 pairs
      named_bar_sync(2, kPfEpiW * 32);
      {
        const float* dsrc = down ? a.w.dh : a.pw.dxp;
        const int col = (lane >> 3), bi = lane & 7;
        const int nbb = (nb + 7) >> 3;
        for (int g = ew; g < nbb * (kPfP / 4); g += kPfEpiW) {
          const int c = (g % (kPfP / 4)) * 4 + col, b = (g / (kPfP / 4)) * 8 + bi;
          if (b < nb) {
            float* dst = m.dxs + b * kDxS + c;
            if (c < nv) cp_async4(dst, dsrc + (long)(pb + c) * nb + b);
            else *dst = 0.0f;
          }
        }
        cp_async_wait_all();
      }
      named_bar_sync(2, kPfEpiW * 32);
      {
        // the next tile's block scales: pull their lines into L2 while this tile runs
        const int tn = t + gridDim.x;
        if (tn < total) {
          int un, mtn, ntn;
          pf_tile(m.tp, nu, n_mt, tn, un, mtn, ntn);
          const int pbn = m.toff[un] + ntn * kPfP;
          const int nvn = min(kPfP, m.toff[un + 1] - pbn);
          const float* dsrc = down ? a.w.dh : a.pw.dxp;
          const int lines = (nb * 4 + 127) >> 7;  // 128-byte lines per pair row (rows need not align)
          for (int i = threadIdx.x - kPfEpi0 * 32; i < nvn * (lines + 1); i += kPfEpiW * 32) {
            const int pr = i / (lines + 1), li = i - pr * (lines + 1);
            const float* row = dsrc + (long)(pbn + pr) * nb;
            prefetch_l2(reinterpret_cast<const char*>(row) + min(li * 128, nb * 4 - 4));
          }
        }
      }

      float chain[kPfEpiC];
#pragma unroll
      for (int c = 0; c < kPfEpiC; ++c) chain[c] = 0.0f;
      int gi = 0, gb = 0;  // current group and block within it
      for (int bu = 0; bu < nburst; ++bu, ++kb) {
        const int s = (int)(kb % kPfAccStages);
        const long n = kb / kPfAccStages;
        mbar_wait_bounded(&m.acc_full[s], (uint32_t)(n & 1), &abort_flag, status);
        tc_fence_after();
        // the burst's 4 blocks in one round of loads, then the accumulator goes back to the MMA
        // issuer before they are folded
        uint32_t acc4[kPfR][kPfEpiC];
        if (active) {
          const uint32_t t0 = tl + s * kPfN + e8;
          tmem_ld16x4(t0, t0 + kPfP, t0 + 2 * kPfP, t0 + 3 * kPfP, acc4);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.acc_empty[s]);
        if (!active) continue;
#pragma unroll
        for (int j = 0; j < kPfR; ++j) {
          const int b = bu * kPfR + j;
          const float4* dxb = reinterpret_cast<const float4*>(m.dxs + b * kDxS + e8);
#pragma unroll
          for (int c4 = 0; c4 < kPfEpiC / 4; ++c4) {
            const float4 dv = dxb[c4];
            fma2_rn(dv.x, dv.y, __uint_as_float(acc4[j][4 * c4 + 0]), __uint_as_float(acc4[j][4 * c4 + 1]),
                    chain[4 * c4 + 0], chain[4 * c4 + 1]);
            fma2_rn(dv.z, dv.w, __uint_as_float(acc4[j][4 * c4 + 2]), __uint_as_float(acc4[j][4 * c4 + 3]),
                    chain[4 * c4 + 2], chain[4 * c4 + 3]);
          }
          if (Adump != nullptr) {
            const int wrow = down ? mt * kPfM + row : mt * (kPfM / 2) + (row & 63);
            int32_t* dump = (!down && row >= 64) ? a.dbg.Au : Adump;
            const int nrow = down ? d : f;
#pragma unroll
            for (int c = 0; c < kPfEpiC; ++c) {
              const int p = pb + e8 + c;
              if (p < pe) dump[((long)p * nrow + wrow) * nb + b] = (int32_t)__uint_as_float(acc4[j][c]);
            }
          }
          if (++gb == G) {
            gb = 0;
            COLI_PF_PUSH_GROUP()
          }
        }
      }
      if (active) {
        // empty groups ngrp..31 are +0 leaves of the tree
        while (gi < 32) COLI_PF_PUSH_GROUP()
      }
      // chain = the canonical sum of every (row, pair) of this thread (every loop over the
      // pairs is unrolled, so chain stays in registers)
      const float* scx = a.st.sc + (long)ex * (2 * f + d);
      if (down) {
        if (!active) continue;
        const int r = mt * kPfM + row;
        const float sd = scx[2 * f + r];
#pragma unroll
        for (int c = 0; c < kPfEpiC; ++c) {
          const int p = pb + e8 + c;
          if (p < pe) a.pw.e[(long)p * d + r] = __fmul_rn(sd, chain[c]);
        }
      } else {
        const int r = mt * (kPfM / 2) + (row & 63);
        const bool is_up = row >= 64;
        const float sr = is_up ? scx[f + r] : scx[r];
#pragma unroll
        for (int c = 0; c < kPfEpiC; ++c) chain[c] = __fmul_rn(sr, chain[c]);  // the row-scaled projection
        if (a.dbg.g != nullptr && active) {
          float* dst = is_up ? a.dbg.u : a.dbg.g;
#pragma unroll
          for (int c = 0; c < kPfEpiC; ++c) {
            const int p = pb + e8 + c;
            if (p < pe) dst[(long)p * f + r] = chain[c];
          }
        }
        if (is_up && active) {
#pragma unroll
          for (int c = 0; c < kPfEpiC; ++c) m.us[(e8 + c) * 64 + (row - 64)] = chain[c];
        }
        named_bar_sync(2, kPfEpiW * 32);
        if (!is_up && active) {
          // h = SiLU(g) * u; the warp's 32 rows are one int8 block of h for each pair
          const int nhb = f >> 5, hbk = r >> 5;
#pragma unroll
          for (int c = 0; c < kPfEpiC; ++c) {
            const int p = pb + e8 + c;
            const float hv = canon_silu_mul(chain[c], m.us[(e8 + c) * 64 + row]);
            const float dd = __fdiv_rn(warp_max(fabsf(hv)), 127.0f);
            const int code = q8_code(hv, dd);
            const int sq = warp_isum(code);
            if (p < pe) {
              a.w.hf[(long)p * f + r] = hv;
              a.w.qh[(long)p * f + r] = (int8_t)code;
              a.pw.hb[(long)p * f + r] = __float2bfloat16_rn((float)code);
              if (lane == 0) {
                a.w.dh[(long)p * nhb + hbk] = dd;
                a.w.sh[(long)p * nhb + hbk] = sq;
              }
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ combine ----------------
// y[t, r] = e(shared, t)[r], then fma(w_{t,k}, e(t,k)[r], y) for k = 0..K-1, (+ x[t, r])
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ x, float* __restrict__ y,
                                                      const Shape s, const Work w, const float* __restrict__ e) {
  const int t = blockIdx.y;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= s.d) return;
  const int K = s.K, T = s.T;
  float acc = s.n_shared ? e[(long)(T * K + t) * s.d + r] : 0.0f;
  for (int k = 0; k < K; ++k)
    acc = __fmaf_rn(__ldcg(w.w + t * K + k), e[(long)__ldcg(w.inv + t * K + k) * s.d + r], acc);
  if (s.has_norm) acc = __fadd_rn(x[(long)t * s.d + r], acc);
  y[(long)t * s.d + r] = acc;
}

// ------------------------------------------------------------------ host side --------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the CUDA driver API's tensor-map encoder, looked up through the runtime (no link against libcuda)
static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over a row-major [rows][cols] array (elem_bytes 1 or 2), box {box_cols, box_rows}
static bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes,
                     uint64_t cols, uint64_t rows, uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t configure_prefill_kernels(int d, int f, int E) {
  const int need = prefill_smem_bytes(d, f, E, 0) > prefill_smem_bytes(d, f, E, 1)
                       ? prefill_smem_bytes(d, f, E, 0)
                       : prefill_smem_bytes(d, f, E, 1);
  if (need > kSmemLimit) return cudaErrorInvalidValue;
  const cudaError_t e = cudaFuncSetAttribute(expert_gemm_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(expert_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

bool prefill_make_maps(PrefillMaps* maps, const Store& st, const Work& w, const PrefillWork& pw, int d,
                       int f, int E, int slots, int prow, int tmax) {
  const int Gd = (d / kQB + 31) / 32, Gf = (f / kQB + 31) / 32;
  bool ok = make_map(&maps->wgu, st.wgu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)d,
                     (uint64_t)slots * f, (uint32_t)(Gd * 16), (uint32_t)(kPfM / 2));
  ok = ok && make_map(&maps->wd, st.wd, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)(f / 2),
                      (uint64_t)slots * d, (uint32_t)(Gf * 16), (uint32_t)kPfM);
  // activation codes: boxes of 64 bf16 (one 128-byte swizzled row) x 32 pairs
  ok = ok && make_map(&maps->xb, pw.xb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)d, (uint64_t)prow,
                      (uint32_t)(kPfBurstK / 2), (uint32_t)kPfP, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_map(&maps->hb, pw.hb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)f, (uint64_t)prow,
                      (uint32_t)(kPfBurstK / 2), (uint32_t)kPfP, CU_TENSOR_MAP_SWIZZLE_128B);
  // router rows and normalised tokens (both in the router's chunk order), 256-float boxes
  ok = ok && make_map(&maps->wr, st.wr, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)d, (uint64_t)E,
                      256u, 16u);
  ok = ok && make_map(&maps->xnp, w.xnp, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)d, (uint64_t)tmax,
                      256u, 32u);
  return ok;
}

cudaError_t launch_prefill_experts(const float* x, float* y, const Shape& s, const Store& st, const Work& w,
                                   const PrefillWork& pw, const PrefillMaps& maps, const ExpertDebug& dbg,
                                   int num_sms, cudaStream_t stream, cudaEvent_t after_gateup) {
  for (int down = 0; down < 2; ++down) {
    if (down && after_gateup) {
      const cudaError_t e = cudaEventRecord(after_gateup, stream);
      if (e != cudaSuccess) return e;
    }
    PfArgs args;
    args.s = s;
    args.st = st;
    args.w = w;
    args.pw = pw;
    args.dbg = dbg;
    args.down = down;
    const int K = down ? s.f : s.d;
    const int nb = K / kQB, G = (nb + 31) / 32;
    args.raw_stage_bytes = kPfM * G * 16;
    args.dx_bytes = nb * kDxS * 4;
    const int smem = prefill_smem_bytes(s.d, s.f, s.E, down);
    if (down)
      expert_gemm_kernel<true><<<num_sms, kPfThreads, smem, stream>>>(maps.wd, maps.hb, args);
    else
      expert_gemm_kernel<false><<<num_sms, kPfThreads, smem, stream>>>(maps.wgu, maps.xb, args);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  combine_kernel<<<dim3((s.d + 255) / 256, s.T), 256, 0, stream>>>(x, y, s, w, pw.e);
  return cudaGetLastError();
}

}  // namespace coli
