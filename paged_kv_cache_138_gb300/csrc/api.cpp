// Status names and version of libpagedkv.
#include "pagedkv.h"

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID_ARG: return "invalid argument";
    case PKV_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_OUT_OF_BLOCKS: return "out of KV blocks (state unchanged)";
    case PKV_ERR_BAD_INDEX: return "unknown sequence or position outside its table";
    default: return "unknown status";
  }
}

extern "C" int pkv_version(void) { return 100; }
