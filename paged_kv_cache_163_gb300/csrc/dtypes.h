// Element-type predicates shared by host and device code.
#pragma once

#include "pkv.h"

#if defined(__CUDACC__)
#define PKV_HD __host__ __device__
#else
#define PKV_HD
#endif

namespace pkv {

// Storage type of the V half of PKV_FP8_E4M3_INT4: symmetric 4-bit codes,
// two a byte.  Internal only; not a cache type on its own.
constexpr int kInt4 = 64;

// One-byte cache codes with one fp32 scale per (token, KV head).
PKV_HD constexpr bool is_code8(int dt) { return dt == PKV_FP8_E4M3 || dt == PKV_FP8_E5M2 || dt == PKV_INT8; }

// Storage type of the K half and of the V half of a cache type.
PKV_HD constexpr int k_part(int dt) { return dt == PKV_FP8_E4M3_INT4 ? PKV_FP8_E4M3 : dt; }
PKV_HD constexpr int v_part(int dt) { return dt == PKV_FP8_E4M3_INT4 ? kInt4 : dt; }

// A storage type whose rows carry one fp32 scale (codes times scale).
PKV_HD constexpr bool is_coded(int part) { return is_code8(part) || part == kInt4; }

// A cache type with k_scale / v_scale arrays.
PKV_HD constexpr bool has_scales(int dt) { return is_coded(k_part(dt)) || is_coded(v_part(dt)); }

// A valid cache type.
PKV_HD constexpr bool is_cache_type(int dt) {
  return dt == PKV_F16 || dt == PKV_BF16 || is_code8(dt) || dt == PKV_FP8_E4M3_INT4;
}

// Bytes of one token's row of head_dim elements in a storage type.
PKV_HD constexpr int row_bytes(int part, int head_dim) {
  return part == kInt4 ? head_dim / 2 : (is_code8(part) ? head_dim : 2 * head_dim);
}

}  // namespace pkv

#undef PKV_HD
