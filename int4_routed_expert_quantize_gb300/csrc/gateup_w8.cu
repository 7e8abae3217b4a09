// The decode gate/up + SwiGLU kernels for int8 (one code per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_GATEUP_INSTANTIATE(8)
}  // namespace coli
