// Library-wide C entry points that are not tied to one kernel.
#include "kvp.h"

extern "C" const char* kvp_status_string(int status) {
  switch (status) {
    case KVP_OK: return "ok";
    case KVP_ERR_INVALID: return "invalid argument";
    case KVP_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case KVP_ERR_CAPACITY: return "page pool, page table or reserve too small";
    case KVP_ERR_CUDA: return "CUDA runtime or launch error";
    case KVP_ERR_TIMEOUT: return "device-side wait gave up";
    case KVP_ERR_UNSUPPORTED: return "unsupported shape";
    case KVP_ERR_WORKSPACE: return "workspace missing or too small";
    case KVP_ERR_BOUNDS: return "page id or count out of range";
    default: return "unknown status";
  }
}

extern "C" int kvp_version(void) { return 100; }
