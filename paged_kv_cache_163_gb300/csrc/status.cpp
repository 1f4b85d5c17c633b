// Status strings, per-thread failure reasons and launch accounting.
#include <string>

#include "pkv.h"
#include "status.h"

namespace pkv {

static thread_local std::string t_last_error;

pkv_status fail(pkv_status s, const char *reason) {
  t_last_error = reason ? reason : "";
  return s;
}

}  // namespace pkv

extern "C" {

const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_NO_BLOCKS: return "out of KV blocks";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case PKV_ERR_DEVICE_CHECK: return "device-side check failed";
    case PKV_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char *pkv_last_error(void) { return pkv::t_last_error.c_str(); }

}  // extern "C"
