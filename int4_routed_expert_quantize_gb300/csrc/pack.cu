// Format kernels: the canonical int4, int8 and int2 row packers ("colibrì 架构概述" §3.1: two
// 4-bit values per byte, one value per byte, four 2-bit values per byte; one f32 scale per
// row), the standalone Q8_0-style activation quantiser, and the load-time repack of canonical
// records into the store layout the expert kernels stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include "coli_device.cuh"
#include "coli_internal.h"

namespace coli {

// code of one weight: round(w / s) half away from zero, clamped to the symmetric [-7, 7]
__device__ __forceinline__ int i4_code(float w, float s) {
  if (s == 0.0f) return 0;
  const int q = (int)roundf(__fdiv_rn(w, s));
  return max(-7, min(7, q));
}

// one warp per row: s = max|w| / 7; byte i = code(w[2i]) | code(w[2i+1]) << 4 (two's complement)
__global__ void __launch_bounds__(256) quantize_i4_rows_kernel(const float* __restrict__ w,
                                                               long rows, int cols,
                                                               uint8_t* __restrict__ packed,
                                                               float* __restrict__ scales) {
  const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float2* wr = reinterpret_cast<const float2*>(w + row * cols);
  float amax = 0.0f;
  for (int i = lane; i < cols / 2; i += 32) {
    const float2 v = wr[i];
    amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
  }
  const float s = __fdiv_rn(warp_max(amax), 7.0f);
  uint8_t* pr = packed + row * (cols / 2);
  for (int i = lane; i < cols / 2; i += 32) {
    const float2 v = wr[i];
    pr[i] = (uint8_t)((i4_code(v.x, s) & 15) | ((i4_code(v.y, s) & 15) << 4));
  }
  if (lane == 0) scales[row] = s;
}

cudaError_t launch_quantize_i4_rows(const float* w, int64_t rows, int cols, uint8_t* packed,
                                    float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const long blocks = (rows + 7) / 8;
  quantize_i4_rows_kernel<<<(unsigned)blocks, 256, 0, stream>>>(w, rows, cols, packed, scales);
  return cudaGetLastError();
}

// int8 rows ("colibrì 架构概述" §3.1 int8, quantize_rows): one warp per row, s = max|w| / 127,
// code = round(w / s) half away from zero clamped to [-127, 127], one code per byte
__global__ void __launch_bounds__(256) quantize_i8_rows_kernel(const float* __restrict__ w,
                                                               long rows, int cols,
                                                               int8_t* __restrict__ q,
                                                               float* __restrict__ scales) {
  const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* wr = w + row * cols;
  float amax = 0.0f;
  for (int i = lane; i < cols; i += 32) amax = fmaxf(amax, fabsf(wr[i]));
  const float s = __fdiv_rn(warp_max(amax), 127.0f);
  for (int i = lane; i < cols; i += 32) {
    int v = 0;
    if (s != 0.0f) v = max(-127, min(127, (int)roundf(__fdiv_rn(wr[i], s))));
    q[row * cols + i] = (int8_t)v;
  }
  if (lane == 0) scales[row] = s;
}

// int2 rows ("colibrì 架构概述" §3.1 int2 packed, pack_int2): one warp per row, s = max|w|,
// code = round(w / s) half away from zero clamped to [-1, 1], four two's-complement 2-bit codes
// per byte with element 4i+k in bits 2k..2k+1 of byte i
__global__ void __launch_bounds__(256) quantize_i2_rows_kernel(const float* __restrict__ w,
                                                               long rows, int cols,
                                                               uint8_t* __restrict__ packed,
                                                               float* __restrict__ scales) {
  const long row = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4* wr = reinterpret_cast<const float4*>(w + row * cols);
  float amax = 0.0f;
  for (int i = lane; i < cols / 4; i += 32) {
    const float4 v = wr[i];
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
  const float s = warp_max(amax);  // max|w| / 1
  uint8_t* pr = packed + row * (cols / 4);
  for (int i = lane; i < cols / 4; i += 32) {
    const float4 v = wr[i];
    const float e[4] = {v.x, v.y, v.z, v.w};
    int byte = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int c = 0;
      if (s != 0.0f) c = max(-1, min(1, (int)roundf(__fdiv_rn(e[k], s))));
      byte |= (c & 3) << (2 * k);
    }
    pr[i] = (uint8_t)byte;
  }
  if (lane == 0) scales[row] = s;
}

cudaError_t launch_quantize_i8_rows(const float* w, int64_t rows, int cols, int8_t* q,
                                    float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  quantize_i8_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(w, rows, cols, q, scales);
  return cudaGetLastError();
}

cudaError_t launch_quantize_i2_rows(const float* w, int64_t rows, int cols, uint8_t* packed,
                                    float* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  quantize_i2_rows_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(w, rows, cols, packed, scales);
  return cudaGetLastError();
}

// one warp per block of 32: d = max|x| / 127, q = round(x / d)
__global__ void __launch_bounds__(256) quantize_q8_kernel(const float* __restrict__ x, long nblk,
                                                          int8_t* __restrict__ q,
                                                          float* __restrict__ dout) {
  const long b = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= nblk) return;
  const float v = x[b * 32 + lane];
  const float dd = __fdiv_rn(warp_max(fabsf(v)), 127.0f);
  q[b * 32 + lane] = (int8_t)q8_code(v, dd);
  if (lane == 0) dout[b] = dd;
}

cudaError_t launch_quantize_q8(const float* x, int64_t n, int8_t* q, float* d,
                               cudaStream_t stream) {
  const long nblk = n / 32;
  if (nblk <= 0) return cudaSuccess;
  quantize_q8_kernel<<<(unsigned)((nblk + 7) / 8), 256, 0, stream>>>(x, nblk, q, d);
  return cudaGetLastError();
}

// Canonical row (two's-complement nibbles, element 2m low / 2m+1 high in byte m of a block)
// -> store layout: block b = g*G + i of the row goes to chunk store_chunk(g, i, G) (groups
// contiguous, rotated inside), and inside the chunk word k byte m holds element 8k+m (low
// nibble) and 8k+m+4 (high nibble) as code + 8.
// For a 4-bit two's-complement nibble, code + 8 is the nibble with its top bit flipped.
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ src,
                                                     uint8_t* __restrict__ dst, int rows, int cols,
                                                     long dst_row_stride) {
  const int nb = cols / 32;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)rows * nb) return;
  const long r = idx / nb;
  const int b = (int)(idx - r * nb);
  const int G = (nb + 31) / 32;
  const int g = b / G, i = b - g * G;
  const uint4 c = *reinterpret_cast<const uint4*>(src + r * (cols / 2) + (long)b * 16);
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
  uint32_t nib[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const uint32_t byte = (cw[e >> 3] >> (8 * ((e >> 1) & 3))) & 0xFFu;
    nib[e] = ((e & 1) ? (byte >> 4) : (byte & 15u)) ^ 8u;
  }
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t v = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) v |= (nib[8 * k + m] | (nib[8 * k + m + 4] << 4)) << (8 * m);
    out[k] = v;
  }
  *reinterpret_cast<uint4*>(dst + r * dst_row_stride + (long)store_chunk(g, i, G) * 16) =
      make_uint4(out[0], out[1], out[2], out[3]);
}

// Canonical int8 row -> store layout: the two 16-byte halves of block b = g*G + i go to two
// planes of the row (nb chunks apart), each at chunk store_chunk(g, i, G); codes unchanged.
__global__ void __launch_bounds__(256) repack_i8_kernel(const uint8_t* __restrict__ src,
                                                        uint8_t* __restrict__ dst, int rows, int cols,
                                                        long dst_row_stride) {
  const int nb = cols / 32;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)rows * nb) return;
  const long r = idx / nb;
  const int b = (int)(idx - r * nb);
  const int G = (nb + 31) / 32;
  const int g = b / G, i = b - g * G;
  const uint4* c = reinterpret_cast<const uint4*>(src + r * cols + (long)b * 32);
  uint8_t* row = dst + r * dst_row_stride + (long)store_chunk(g, i, G) * 16;
  *reinterpret_cast<uint4*>(row) = c[0];
  *reinterpret_cast<uint4*>(row + (long)nb * 16) = c[1];
}

// Canonical int2 row (element 4i+k in bits 2k..2k+1 of byte i) -> store layout: block b = g*G +
// i (8 bytes) goes to 8-byte unit store_chunk8(g, i, G); inside it word h holds elements
// 16h..16h+15 with element 16h+4k+m in bits 2k..2k+1 of byte m, as code + 2 (for a 2-bit two's
// complement field, code + 2 is the field with its top bit flipped).
__global__ void __launch_bounds__(256) repack_i2_kernel(const uint8_t* __restrict__ src,
                                                        uint8_t* __restrict__ dst, int rows, int cols,
                                                        long dst_row_stride) {
  const int nb = cols / 32;
  const long idx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long)rows * nb) return;
  const long r = idx / nb;
  const int b = (int)(idx - r * nb);
  const int G = (nb + 31) / 32;
  const int g = b / G, i = b - g * G;
  const uint2 c = *reinterpret_cast<const uint2*>(src + r * (cols / 4) + (long)b * 8);
  const uint32_t cw[2] = {c.x, c.y};
  uint32_t out[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    // canonical: element e of the block in byte e >> 2, bits 2*(e & 3)
    const uint32_t field = (cw[e >> 4] >> (8 * ((e >> 2) & 3) + 2 * (e & 3))) & 3u;
    const int h = e >> 4, k = (e & 15) >> 2, m = e & 3;
    out[h] |= (field ^ 2u) << (8 * m + 2 * k);
  }
  *reinterpret_cast<uint2*>(dst + r * dst_row_stride + (long)store_chunk8(g, i, G) * 8) =
      make_uint2(out[0], out[1]);
}

cudaError_t launch_repack_matrix(const uint8_t* src, uint8_t* dst, int rows, int cols,
                                 int64_t dst_row_stride, cudaStream_t stream, int wbits) {
  const long n = (long)rows * (cols / 32);
  const unsigned grid = (unsigned)((n + 255) / 256);
  if (wbits == 4)
    repack_kernel<<<grid, 256, 0, stream>>>(src, dst, rows, cols, dst_row_stride);
  else if (wbits == 8)
    repack_i8_kernel<<<grid, 256, 0, stream>>>(src, dst, rows, cols, dst_row_stride);
  else if (wbits == 2)
    repack_i2_kernel<<<grid, 256, 0, stream>>>(src, dst, rows, cols, dst_row_stride);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// Host-buffer forwards: the input read from, and the output and status word written to, mapped
// pinned host memory by the GPU itself (over the host link, no copy-engine transfer).  The loads
// bypass the caches (the host rewrites the buffer between calls); the stores write through.
__global__ void __launch_bounds__(256) host_in_kernel(const float4* __restrict__ hx,
                                                      float4* __restrict__ dx, int n4) {
  griddep_launch_dependents();  // the router may be scheduled; it waits for this grid
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n4) dx[i] = __ldcv(hx + i);
}

// One CTA: y and the status word, then the completion counter (hstatus[kHostDoneWord]) one up,
// after every thread's writes are ordered before it at system scope; the host polls it.
__global__ void __launch_bounds__(1024) host_out_kernel(const float4* __restrict__ dy,
                                                        float4* __restrict__ hy, int n4,
                                                        const int* __restrict__ status,
                                                        int* __restrict__ hstatus) {
  griddep_wait();  // a programmatic dependent of the forward's last grid
  for (int i = threadIdx.x; i < n4; i += blockDim.x) __stwt(hy + i, __ldcg(dy + i));
  if (threadIdx.x == 0) __stwt(hstatus, __ldcg(status));
  __threadfence_system();
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* done = hstatus + kHostDoneWord;
    *done = *done + 1;
  }
}

cudaError_t launch_host_in(const float* hx, float* dx, int n, cudaStream_t stream) {
  const int n4 = n / 4;
  host_in_kernel<<<(n4 + 255) / 256, 256, 0, stream>>>(reinterpret_cast<const float4*>(hx),
                                                       reinterpret_cast<float4*>(dx), n4);
  return cudaGetLastError();
}

cudaError_t launch_host_out(const float* dy, float* hy, int n, const int* status, int* hstatus,
                            cudaStream_t stream) {
  const int n4 = n / 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(1024);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, host_out_kernel, reinterpret_cast<const float4*>(dy),
                            reinterpret_cast<float4*>(hy), n4, status, hstatus);
}

// router rows: lane g's contiguous elements g*(d/32) .. in 4-float chunks at i4*32 + g
__global__ void __launch_bounds__(256) permute_router_kernel(const float* __restrict__ src,
                                                             float* __restrict__ dst, int E, int d) {
  const long c = (long)blockIdx.x * blockDim.x + threadIdx.x;
  const long per_row = d / 4;
  if (c >= (long)E * per_row) return;
  const long e = c / per_row;
  const int pos = (int)(c - e * per_row);
  const int i4 = pos >> 5, g = pos & 31;
  const float4 v = *reinterpret_cast<const float4*>(src + e * d + g * (d / 32) + 4 * i4);
  reinterpret_cast<float4*>(dst + e * d)[pos] = v;
}

cudaError_t launch_permute_router(const float* src, float* dst, int E, int d, cudaStream_t stream) {
  const long n = (long)E * (d / 4);
  permute_router_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(src, dst, E, d);
  return cudaGetLastError();
}

}  // namespace coli
