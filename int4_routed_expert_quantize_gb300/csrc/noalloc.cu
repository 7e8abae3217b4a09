// Routing with no device allocation at all: the sigmoid top-K router of the layer (same
// arithmetic, bit for bit) for callers that cannot call cudaMalloc -- for example a process
// whose device memory is owned entirely by another allocator (a serving framework that
// reserves the whole device up front and hands out pieces of its own pool), where a direct
// allocation would fail or break that allocator's accounting.  The caller passes inputs and
// outputs; the scratch the kernel needs (the per-token scores and the last-CTA ticket) lives in
// the fixed array below.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "coli_device.cuh"
#include "coli_internal.h"
#include "coli_moe.h"
#include "coli_select.cuh"

namespace coli {
namespace {

constexpr int kNaMaxT = 4;             // tokens per call
constexpr int kNaMaxScores = 4096;     // T * E
constexpr int kNaMaxDevices = 64;
constexpr int kNaEpc = 2;              // experts per CTA

// scores [T][E] then the ticket counter; every device that loads the library holds it
__device__ __align__(256) float g_noalloc_scratch[kNaMaxScores + 64];

// device address of g_noalloc_scratch per device (the host-side name is only a stand-in)
float* g_scratch_ptr[kNaMaxDevices] = {};
std::mutex g_setup_mutex;

__global__ void __launch_bounds__(256) route_noalloc_kernel(const float* __restrict__ x,
                                                            const float* __restrict__ wr,
                                                            const float* __restrict__ bias,
                                                            int T, int E, int d, int K,
                                                            float routed_scale, float* scratch,
                                                            int32_t* ids_out, float* w_out) {
  extern __shared__ __align__(16) float xsm[];  // [T][d] tokens in the lane-group chunk order
  __shared__ int is_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarp = blockDim.x >> 5;
  const int Gd = d >> 5;
  float* scores = scratch;
  int* ticket = reinterpret_cast<int*>(scratch + kNaMaxScores);
  for (int c = threadIdx.x; c < T * (d / 4); c += blockDim.x) {
    const int t = c / (d / 4), pos = c - t * (d / 4);
    const int i4 = pos >> 5, g = pos & 31;
    reinterpret_cast<float4*>(xsm + (long)t * d)[pos] =
        *reinterpret_cast<const float4*>(x + (long)t * d + g * Gd + 4 * i4);
  }
  __syncthreads();
  // logits in the canonical order: lane g runs the fma chain over its d/32 contiguous elements
  // (read straight from the row-major router), the butterfly adds the 32 partials
  const int e0 = blockIdx.x * kNaEpc, ne = min(kNaEpc, E - e0);
  for (int pi = warp; pi < ne * T; pi += nwarp) {
    const int e = e0 + pi / T, t = pi % T;
    const float* row = wr + (long)e * d + lane * Gd;
    const float4* xp = reinterpret_cast<const float4*>(xsm + (long)t * d);
    float p = 0.0f;
    for (int i4 = 0; i4 < Gd / 4; ++i4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(row) + i4);
      const float4 b = xp[i4 * 32 + lane];
      p = __fmaf_rn(a.x, b.x, p);
      p = __fmaf_rn(a.y, b.y, p);
      p = __fmaf_rn(a.z, b.z, p);
      p = __fmaf_rn(a.w, b.w, p);
    }
    p = warp_tree_sum(p);
    if (lane == 0) scores[t * E + e] = canon_sigmoid(p);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(ticket, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // the last CTA: top-K per token by score + bias, ranked by the same order-preserving key as
  // the layer's selection (a taken expert's key is 0; a tie goes to the lower id, so scores that
  // are not numbers give the same ids too), weights renormalised over the selected scores summed
  // in rank order
  const int NM = E <= 256 ? 8 : 32;  // experts per lane the layer's selection scans
  for (int t = warp; t < T; t += nwarp) {
    const float* sc = scores + t * E;
    uint32_t taken = 0;
    float S = 0.0f, mine = 0.0f;
    int my = 0;
    for (int k = 0; k < K; ++k) {
      uint32_t bk = 0;
      int bm = 0;
      for (int m = 0; m < NM; ++m) {
        const int e = m * 32 + lane;
        uint32_t key = 0;
        if (e < E && !((taken >> m) & 1u)) {
          const float sv = __ldcg(sc + e);
          key = score_key(bias ? __fadd_rn(sv, bias[e]) : sv);
        }
        if (m == 0 || key > bk) {
          bk = key;
          bm = m;
        }
      }
      const uint32_t top = __reduce_max_sync(FULL, bk);
      uint32_t win = __reduce_min_sync(FULL, bk == top ? (uint32_t)(bm * 32 + lane) : 0xFFFFFFFFu);
      win = win < (uint32_t)E ? win : 0u;
      if ((int)(win & 31u) == lane) taken |= 1u << (win >> 5);
      const float v = __ldcg(sc + win);
      S = k == 0 ? v : __fadd_rn(S, v);
      my = lane == k ? (int)win : my;
      mine = lane == k ? v : mine;
    }
    if (lane < K) {
      ids_out[t * K + lane] = my;
      w_out[t * K + lane] = __fmul_rn(__fdiv_rn(mine, S), routed_scale);
    }
    __syncwarp();
  }
  if (threadIdx.x == 0) *ticket = 0;
}

// once per device, with that device current: resolve the array's device address (the first call
// on a device does this set-up, so it should come before any stream capture).  The address is
// kept for the life of the process, so calls after a cudaDeviceReset of that device (which
// unloads the module that holds the array) are not supported.
int scratch_for_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return COLI_ECUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return COLI_ECUDA;
    }
    if (cudaFuncSetAttribute(route_noalloc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kNaMaxT * 8192 * 4) != cudaSuccess)
      return COLI_ECUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return COLI_OK;
}

}  // namespace
}  // namespace coli

extern "C" int coli_route_noalloc(const float* x_dev, int T, const float* W_r_dev,
                                  const float* bias_dev, int E, int d, int K, float routed_scale,
                                  int32_t* ids_dev, float* w_dev, void* stream) {
  using namespace coli;
  if (T < 0 || T > kNaMaxT || E < 1 || E > 1024 || K < 1 || K > 32 || K > E ||
      (long)T * E > kNaMaxScores || d < 128 || d > 8192 || d % 128)
    return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x_dev || !W_r_dev || !ids_dev || !w_dev || ((uintptr_t)x_dev & 15u) || ((uintptr_t)W_r_dev & 15u))
    return COLI_EINVAL;
  float* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // the ticket must start at zero; everything else the kernel reads it has written itself
  if (cudaMemsetAsync(scratch + kNaMaxScores, 0, sizeof(int), st) != cudaSuccess) return COLI_ECUDA;
  route_noalloc_kernel<<<(E + kNaEpc - 1) / kNaEpc, 256, (size_t)T * d * sizeof(float), st>>>(
      x_dev, W_r_dev, bias_dev, T, E, d, K, routed_scale, scratch, ids_dev, w_dev);
  return cudaGetLastError() == cudaSuccess ? COLI_OK : COLI_ECUDA;
}
