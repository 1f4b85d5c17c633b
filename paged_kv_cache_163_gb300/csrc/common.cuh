// Device helpers: element types, conversions, mbarrier / bulk-copy PTX.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kBS = PKV_BLOCK_SIZE;  // tokens per physical block
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
// Iteration limit of every spin on an mbarrier.  A healthy wait ends in
// microseconds; this bound (seconds) only ends a wait that would never end.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ void report(int32_t *err, int bits) {
  if (err) atomicOr(err, bits);
}

// ---- element conversions -------------------------------------------------
// Unpack a 32-bit word holding two 16-bit elements (low half first).
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w);

template <>
__device__ __forceinline__ float2 unpack2<PKV_BF16>(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<PKV_F16>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2 *>(&w);
  return __half22float2(h);
}

// Four E4M3 codes (byte 0 first) to four floats.  E4M3 values are exact in fp16.
__device__ __forceinline__ void unpack_e4m3x4(uint32_t w, float *out) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2 *>(&lo));
  float2 b = __half22float2(*reinterpret_cast<__half2 *>(&hi));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

// Unpack n bytes of cache row (n = 4, 8 or 16) into floats.
template <int DT, int NBYTES>
__device__ __forceinline__ void unpack_row(const uint8_t *src, float *out) {
  static_assert(NBYTES == 2 || NBYTES == 4 || NBYTES == 8 || NBYTES == 16, "vector width");
  if constexpr (NBYTES == 2) {  // two E4M3 codes
    static_assert(DT == PKV_FP8_E4M3, "2-byte rows are FP8 only");
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(*reinterpret_cast<const __nv_fp8x2_storage_t *>(src), __NV_E4M3);
    float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h));
    out[0] = f.x;
    out[1] = f.y;
    return;
  } else {
  uint32_t w[NBYTES / 4];
  if constexpr (NBYTES == 16) {
    uint4 v = *reinterpret_cast<const uint4 *>(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NBYTES == 8) {
    uint2 v = *reinterpret_cast<const uint2 *>(src);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t *>(src);
  }
#pragma unroll
  for (int i = 0; i < NBYTES / 4; ++i) {
    if constexpr (DT == PKV_FP8_E4M3) {
      unpack_e4m3x4(w[i], out + 4 * i);
    } else {
      float2 f = unpack2<DT>(w[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<PKV_BF16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<PKV_F16>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// ---- shared-memory barriers and bulk copies (sm_90+ PTX) -------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait: false when the iteration limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// L2 policy for data read once (streamed K/V): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Non-tensor bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

}  // namespace pkv
