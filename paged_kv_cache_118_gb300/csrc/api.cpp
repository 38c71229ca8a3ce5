// Status strings and version of libpagedkv.
#include "pagedkv.h"

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument (null pointer, shape, dtype, size or alignment)";
    case PKV_ENOMEM: return "not enough free blocks (nothing changed)";
    case PKV_ERANGE: return "index out of range";
    case PKV_ECUDA: return "CUDA error";
    case PKV_ESTATE: return "unknown or duplicate sequence, or reference-count underflow";
    case PKV_EWORKSPACE: return "decode workspace too small";
    default: return "unknown status";
  }
}

extern "C" const char* pkv_version(void) { return "pagedkv 0.1.0 (sm_103a)"; }
