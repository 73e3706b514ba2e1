// Status strings of the C ABI.
#include "cpthd.h"

extern "C" const char* cpthd_status_string(int status) {
  switch (status) {
    case CPTHD_OK: return "ok";
    case CPTHD_ERR_INVALID_ARG: return "invalid argument";
    case CPTHD_ERR_NOT_DIVISIBLE: return "length not divisible (T % cp_size for NO_LOAD_BALANCE, P_j % 2*cp_size for DUAL_CHUNK_SWAP)";
    case CPTHD_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case CPTHD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CPTHD_ERR_CUDA: return "CUDA runtime error";
    case CPTHD_ERR_BAD_OFFSETS: return "offset array not starting at 0, decreasing, or not ending at T";
    case CPTHD_ERR_INDEX_RANGE: return "index out of range";
    case CPTHD_ERR_PAD_LENGTH: return "actual document length exceeds padded length";
    case CPTHD_ERR_TIMEOUT: return "pipeline wait timed out; kernel returned early";
    case CPTHD_ERR_SCRATCH_LIMIT: return "query slice too large for the built-in 32 MiB attention scratch";
    default: return "unknown status";
  }
}
