// The decode gate/up + SwiGLU kernels for int4 (two codes per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_GATEUP_INSTANTIATE(4)
}  // namespace coli
