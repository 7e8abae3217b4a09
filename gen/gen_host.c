/* Host fill routines of the seeded input generator (see coli_gen.h).
 * Built with -ffp-contract=off so every fp32 operation rounds exactly as written. */
#include <stddef.h>
#include <stdint.h>
#include "coli_gen.h"

void cg_fill_normal_host(float* out, uint64_t n, uint64_t seed, uint32_t layer,
                         uint32_t tensor, uint32_t slot, uint64_t idx0, float sigma) {
  const uint64_t key = cg_key(seed, layer, tensor, slot);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = cg_normal(key, idx0 + (uint64_t)i, sigma);
}

/* out[i] = lo + span * u_i  (one fp32 product, then one fp32 sum) */
void cg_fill_uniform_affine_host(float* out, uint64_t n, uint64_t seed, uint32_t layer,
                                 uint32_t tensor, uint32_t slot, uint64_t idx0, float lo,
                                 float span) {
  const uint64_t key = cg_key(seed, layer, tensor, slot);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) {
    float p = span * cg_uniform(key, idx0 + (uint64_t)i);
    out[i] = lo + p;
  }
}

void cg_fill_draws_host(uint64_t* out, uint64_t n, uint64_t seed, uint32_t layer,
                        uint32_t tensor, uint32_t slot, uint64_t idx0) {
  const uint64_t key = cg_key(seed, layer, tensor, slot);
  for (uint64_t i = 0; i < n; ++i) out[i] = cg_draw(key, idx0 + i);
}

/* the n-th output of a splitmix64 sequence seeded with `key` (exposed for its published
 * test vector) */
uint64_t cg_draw_raw_host(uint64_t key, uint64_t n) { return cg_draw(key, n); }
