/* Device fill kernels of the seeded input generator (see coli_gen.h).  They produce the
 * same bits as gen_host.c; big weight sets (tens of GB) are generated here instead of on
 * the host.  Explicit-rounding intrinsics keep nvcc from contracting the affine map. */
#include <cuda_runtime.h>
#include <stdint.h>
#include "coli_gen.h"

__global__ void cg_normal_kernel(float* __restrict__ out, uint64_t n, uint64_t key,
                                 uint64_t idx0, float sigma) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float z = __int2float_rn(cg_irwin_hall12(key, idx0 + i));
    out[i] = __fmul_rn(__fmul_rn(z, 0x1p-16f), sigma);
  }
}

__global__ void cg_uniform_affine_kernel(float* __restrict__ out, uint64_t n, uint64_t key,
                                         uint64_t idx0, float lo, float span) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float u = __fmul_rn(__uint2float_rn((uint32_t)(cg_draw(key, idx0 + i) >> 40)), 0x1p-24f);
    out[i] = __fadd_rn(lo, __fmul_rn(span, u));
  }
}

static unsigned grid_for(uint64_t n) {
  uint64_t b = (n + 255) / 256;
  if (b > 152ull * 16ull) b = 152ull * 16ull;
  return (unsigned)(b ? b : 1);
}

extern "C" int cg_fill_normal_dev(float* out, uint64_t n, uint64_t seed, uint32_t layer,
                                  uint32_t tensor, uint32_t slot, uint64_t idx0, float sigma,
                                  void* stream) {
  if (n == 0) return 0;
  cg_normal_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      out, n, cg_key(seed, layer, tensor, slot), idx0, sigma);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

extern "C" int cg_fill_uniform_affine_dev(float* out, uint64_t n, uint64_t seed, uint32_t layer,
                                          uint32_t tensor, uint32_t slot, uint64_t idx0,
                                          float lo, float span, void* stream) {
  if (n == 0) return 0;
  cg_uniform_affine_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      out, n, cg_key(seed, layer, tensor, slot), idx0, lo, span);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
