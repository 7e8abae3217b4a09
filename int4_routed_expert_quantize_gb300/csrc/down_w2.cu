// The decode down + combine kernels for int2 (four codes per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_DOWN_INSTANTIATE(2)
}  // namespace coli
