// The decode down + combine kernels for int8 (one code per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_DOWN_INSTANTIATE(8)
}  // namespace coli
