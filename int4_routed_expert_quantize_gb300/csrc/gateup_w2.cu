// The decode gate/up + SwiGLU kernels for int2 (four codes per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_GATEUP_INSTANTIATE(2)
}  // namespace coli
