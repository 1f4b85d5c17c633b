// Element-type predicates shared by host and device code.
#pragma once

#include "pkv.h"

namespace pkv {

// One-byte cache codes with one fp32 scale per (token, KV head).
#if defined(__CUDACC__)
__host__ __device__
#endif
constexpr bool is_code8(int dt) {
  return dt == PKV_FP8_E4M3 || dt == PKV_FP8_E5M2 || dt == PKV_INT8;
}

}  // namespace pkv
