// Status strings of the C ABI (coli_moe.h).  Host code only, so the host-only parts of the
// library (this file and the tier manager) also build without nvcc.
#include "coli_moe.h"

extern "C" const char* coli_moe_strerror(int status) {
  switch (status) {
    case COLI_OK: return "ok";
    case COLI_EINVAL: return "invalid argument";
    case COLI_ENOMEM: return "out of memory";
    case COLI_ESTATE: return "call out of order (weights not loaded, or wrong device)";
    case COLI_ECUDA: return "CUDA runtime error";
    case COLI_ETIMEOUT: return "a bounded device wait timed out";
    case COLI_EUNSUPPORTED: return "unsupported shape or request";
    case COLI_EIO: return "file input/output error";
    default: return "unknown status";
  }
}
