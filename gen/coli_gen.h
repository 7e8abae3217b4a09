/* Seeded synthetic input generator: counter-based, bit-identical on host and device.
 *
 * This module only makes test/benchmark inputs (weights, activations, gammas, biases).
 * It holds none of the MoE layer's arithmetic: no quantisation, no dot products, no
 * routing.  Both the CPU oracle and the CUDA path draw their inputs from it, so any
 * expert of any layer can be regenerated independently by either side.
 *
 * Definitions
 *  - splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
 *    OOPSLA 2014; the 64-bit finaliser constants are those of Vigna's public splitmix64).
 *    cg_draw(key, n) is the n-th output of a splitmix64 sequence seeded with `key`, so it
 *    can be evaluated at any n without running the sequence.
 *  - A stream key is derived by chaining draws: key = draw(draw(draw(draw(seed,0),layer),tensor),slot).
 *  - Normal(0,1) draws use the Irwin-Hall construction (sum of 12 uniforms minus 6): the
 *    12 uniforms are 16-bit fields taken from three consecutive 64-bit draws, summed as an
 *    integer, so the float result is exact before the final multiply by sigma and is the
 *    same on every machine.
 *  - Uniform [0,1) draws are the top 24 bits of one 64-bit draw times 2^-24.
 */
#ifndef COLI_GEN_H
#define COLI_GEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define CG_FN static __host__ __device__ __forceinline__
#else
#define CG_FN static inline
#endif

#define CG_GAMMA 0x9E3779B97F4A7C15ull

/* tensor ids used in stream keys */
enum {
  CG_T_X = 0,      /* activations x[t, j]                       */
  CG_T_ROUTER = 1, /* router weights W_r[e, j]                  */
  CG_T_GATE = 2,   /* expert gate weights [f, d]                */
  CG_T_UP = 3,     /* expert up weights   [f, d]                */
  CG_T_DOWN = 4,   /* expert down weights [d, f]                */
  CG_T_GAMMA = 5,  /* RMSNorm gamma [d]                         */
  CG_T_PERM = 6,   /* permutations used by routing-bias recipes */
  CG_T_PICK = 7    /* other integer picks (expert subsets)      */
};

CG_FN uint64_t cg_finalise(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* n-th output (n = 0, 1, ...) of splitmix64 seeded with key */
CG_FN uint64_t cg_draw(uint64_t key, uint64_t n) {
  return cg_finalise(key + (n + 1ull) * CG_GAMMA);
}

CG_FN uint64_t cg_key(uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t slot) {
  uint64_t k = cg_draw(seed, 0);
  k = cg_draw(k, layer);
  k = cg_draw(k, tensor);
  return cg_draw(k, slot);
}

/* Irwin-Hall integer: sum of twelve 16-bit uniforms minus 6*65535, in [-393210, 393210] */
CG_FN int32_t cg_irwin_hall12(uint64_t key, uint64_t idx) {
  int64_t s = 0;
  for (int i = 0; i < 3; ++i) {
    uint64_t z = cg_draw(key, 3ull * idx + (uint64_t)i);
    s += (int64_t)(z & 0xFFFFull) + (int64_t)((z >> 16) & 0xFFFFull) +
         (int64_t)((z >> 32) & 0xFFFFull) + (int64_t)(z >> 48);
  }
  return (int32_t)(s - 393210);
}

/* sigma * N(0,1)-like draw; the int->float conversion and the 2^-16 scaling are exact,
 * the multiply by sigma is one correctly rounded fp32 product on both sides. */
CG_FN float cg_normal(uint64_t key, uint64_t idx, float sigma) {
  float z = (float)cg_irwin_hall12(key, idx) * 0x1p-16f;
  return z * sigma;
}

/* uniform in [0,1) with 24-bit resolution (exact in fp32) */
CG_FN float cg_uniform(uint64_t key, uint64_t idx) {
  return (float)(uint32_t)(cg_draw(key, idx) >> 40) * 0x1p-24f;
}

#endif /* COLI_GEN_H */
