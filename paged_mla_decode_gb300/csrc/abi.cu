// abi.cu -- version and status strings of the C ABI.
#include "../../include/mla.h"

extern "C" int mla_abi_version(void) { return 1; }

extern "C" const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: null pointer, bad size or misaligned buffer";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: no kernel for this shape";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call or kernel launch failed";
    default: return "MLA_ERR_UNKNOWN";
  }
}
