// The decode down + combine kernels for int4 (two codes per byte) expert rows.
#include "expert_decode.cuh"

namespace coli {
COLI_DOWN_INSTANTIATE(4)
}  // namespace coli
