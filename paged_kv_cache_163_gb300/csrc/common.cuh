// Device helpers: element types, conversions, mbarrier / bulk-copy PTX.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dtypes.h"
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

// Hardware approximations (PTX ex2.approx / rcp.approx): 2^x with relative
// error ~2^-22 (2^-inf = 0), and 1/x within 1 ulp; subnormals flush to zero.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- one-byte cache codes ----------------------------------------------------
// FP8 E4M3, FP8 E5M2 and INT8 caches store one byte per element and one
// fp32 scale per (token, KV head); the value is code value x scale.

// Largest code value R of a coded storage type: scale = amax / R.
template <int DT>
__device__ __forceinline__ float code_range() {
  static_assert(is_coded(DT), "coded storage type");
  return DT == PKV_FP8_E4M3 ? 448.f : (DT == PKV_FP8_E5M2 ? 57344.f : (DT == PKV_INT8 ? 127.f : 7.f));
}

// Four codes (byte 0 first) -> two f16x2 words (codes 0, 1 and codes 2, 3).
// Exact for all three types: every E4M3 / E5M2 value and every integer in
// [-128, 127] is a binary16 number.  INT8 codes x are stored as the byte
// x + 128 and go through the biased-exponent identity: the binary16 word
// 0x6400 | (x + 128) is 1152 + x, so one f16x2 subtraction of 1152 recovers
// x exactly.
template <int DT>
__device__ __forceinline__ void code4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  static_assert(is_code8(DT), "one-byte cache type");
  if constexpr (DT == PKV_FP8_E4M3) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else if constexpr (DT == PKV_FP8_E5M2) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, a;\n\tcvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else {
    uint32_t a, b;
    asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(w), "r"(0x64646464u));
    asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(w), "r"(0x64646464u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
  }
}

// Biased form of code4_to_f16x2 for INT8, for MMA operands whose bias the
// caller removes itself: the binary16 words 0x6400 | (x + 128), whose values
// are 1152 + x exactly (two byte permutes, no subtraction).
__device__ __forceinline__ void int8x4_to_f16x2_biased(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0x64646464u));
}
constexpr float kInt8Bias = 1152.f;

// Four codes (byte 0 first) to four floats.
template <int DT>
__device__ __forceinline__ void unpack_code4(uint32_t w, float *out) {
  uint32_t lo, hi;
  code4_to_f16x2<DT>(w, lo, hi);
  const float2 a = __half22float2(*reinterpret_cast<__half2 *>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<__half2 *>(&hi));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

// ---- 4-bit V codes (the V half of FP8_E4M3_INT4) ------------------------------
// Two codes a byte, element 2i in the low nibble of byte i; a nibble holds
// code + 8 for a code in [-7, 7].  Decoding goes through the binary16
// word 0x6400 | n, whose value is 1024 + n: one subtraction of 1032 leaves
// the code, exactly.  The high nibble is decoded in place as 0x6400 | 16 n
// = 1024 + 16 n, scaled by 1/16 and offset by -72 in one exact fused
// multiply-add.

// Bytes 0 and 2 of w (one from each of two rows) -> f16x2 words of their
// low nibbles' codes and of their high nibbles' codes.
__device__ __forceinline__ void int4_pair_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  uint32_t a, b;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(a) : "r"(w));  // (w & m) | c
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(b) : "r"(w));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64086408u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(hi) : "r"(b), "r"(0x2C002C00u), "r"(0xD480D480u));
}

// Biased form of int4_pair_to_f16x2, for MMA operands whose bias the caller
// removes itself: low nibbles n become 0x6400 | n = 1024 + n = 1032 + code,
// high nibbles 0x6400 | 16 n = 1024 + 16 n = 1152 + 16 code (exact).
__device__ __forceinline__ void int4_pair_to_f16x2_biased(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(lo) : "r"(w));  // (w & m) | c
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(hi) : "r"(w));
}
constexpr float kInt4LoBias = 1032.f;
constexpr float kInt4HiBias = 1152.f;  // on values scaled by 16

// n bytes (n = 1 or 2) of a 4-bit row -> 2 n floats, element order.
template <int NBYTES>
__device__ __forceinline__ void unpack_int4(const uint8_t *src, float *out) {
  static_assert(NBYTES == 1 || NBYTES == 2, "4-bit row slice");
  uint32_t w = NBYTES == 2 ? *reinterpret_cast<const uint16_t *>(src) : *src;
  // byte 0 stays at byte 0, byte 1 moves to byte 2
  asm("prmt.b32 %0, %1, 0, 0x4140;" : "=r"(w) : "r"(w));
  uint32_t lo, hi;
  int4_pair_to_f16x2(w, lo, hi);
  const float2 l = __half22float2(*reinterpret_cast<__half2 *>(&lo));
  const float2 h = __half22float2(*reinterpret_cast<__half2 *>(&hi));
  out[0] = l.x;
  out[1] = h.x;
  if constexpr (NBYTES == 2) {
    out[2] = l.y;
    out[3] = h.y;
  }
}

// Two float32 quotients -> two codes (a in the low byte, or the low nibble
// for 4-bit codes): nearest code, ties to even, saturating (FP8) or clamped
// to [-127, 127] (INT8) or [-7, 7] (4-bit).
template <int DT>
__device__ __forceinline__ uint32_t encode2(float a, float b) {
  static_assert(is_coded(DT), "coded storage type");
  if constexpr (DT == kInt4) {
    const int ia = min(max(__float2int_rn(a), -7), 7);
    const int ib = min(max(__float2int_rn(b), -7), 7);
    return static_cast<uint32_t>(ia + 8) | (static_cast<uint32_t>(ib + 8) << 4);
  } else if constexpr (DT == PKV_FP8_E4M3) {
    return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  } else if constexpr (DT == PKV_FP8_E5M2) {
    return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E5M2);
  } else {  // INT8: code in [-127, 127], stored as the byte code + 128
    const int ia = min(max(__float2int_rn(a), -127), 127);
    const int ib = min(max(__float2int_rn(b), -127), 127);
    return static_cast<uint32_t>(ia + 128) | (static_cast<uint32_t>(ib + 128) << 8);
  }
}

// Unpack n bytes of cache row (n = 2, 4, 8 or 16) into floats.
template <int DT, int NBYTES>
__device__ __forceinline__ void unpack_row(const uint8_t *src, float *out) {
  static_assert(NBYTES == 2 || NBYTES == 4 || NBYTES == 8 || NBYTES == 16, "vector width");
  if constexpr (NBYTES == 2) {  // two one-byte codes
    static_assert(is_code8(DT), "2-byte rows hold one-byte codes only");
    float f[4];
    unpack_code4<DT>(*reinterpret_cast<const uint16_t *>(src), f);
    out[0] = f[0];
    out[1] = f[1];
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
    if constexpr (is_code8(DT)) {
      unpack_code4<DT>(w[i], out + 4 * i);
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

// ---- reshape-and-cache of one row --------------------------------------------
// One warp encodes one (token, KV head) row of K or V: head_dim elements of
// 16-bit input into a storage type (CDT: a 16-bit type, a one-byte code
// type or kInt4).  16-bit storage keeps the bits.  Coded storage keeps
// per-row absmax codes: scale = amax / R in IEEE fp32 (1 for an all-zero
// row), code = Q(x / scale) with an IEEE fp32 division.  Lane i holds
// elements [i * D/32, (i + 1) * D/32): its slice of the cache row is
// slice_bytes bytes, returned in the low bytes of a uint2.
template <int D, int CDT>
__host__ __device__ constexpr int slice_bytes() { return row_bytes(CDT, D) / 32; }

template <int D, int IDT, int CDT>
__device__ __forceinline__ uint2 encode_slice(const uint8_t *src_row, int lane, float &scale) {
  constexpr int EPL = D / 32;  // elements per lane
  const uint8_t *src = src_row + lane * EPL * 2;
  uint2 r = make_uint2(0u, 0u);
  if constexpr (!is_coded(CDT)) {
    if constexpr (EPL == 4) {
      r = *reinterpret_cast<const uint2 *>(src);
    } else {
      r.x = *reinterpret_cast<const uint32_t *>(src);
    }
    scale = 1.f;
  } else {
    float x[EPL];
    unpack_row<IDT, EPL * 2>(src, x);
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
    const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, code_range<CDT>());
    constexpr int kBits = CDT == kInt4 ? 4 : 8;  // per element
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
      const uint32_t c2 = encode2<CDT>(__fdiv_rn(x[e], s), __fdiv_rn(x[e + 1], s));  // x[e] -> low bits
      r.x |= c2 << (kBits * e);
    }
    scale = s;
  }
  return r;
}

template <int D, int CDT>
__device__ __forceinline__ void store_slice(uint8_t *dst, uint2 r) {
  constexpr int B = slice_bytes<D, CDT>();
  if constexpr (B == 8) {
    *reinterpret_cast<uint2 *>(dst) = r;
  } else if constexpr (B == 4) {
    *reinterpret_cast<uint32_t *>(dst) = r.x;
  } else if constexpr (B == 2) {
    *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(r.x);
  } else {
    *dst = static_cast<uint8_t>(r.x);
  }
}

// Scales of coded caches: one fp32 array [blocks][heads][2][block_size],
// a (block, head)'s K scales followed by its V scales (v_scale = k_scale +
// block_size), so with 16-token blocks the K and V scales of a tile are one
// 128-byte unit.  Index, from k_scale or v_scale, of the first scale of
// 16-token tile `tile` = (block * heads + head) * tiles per block + tile in
// the block (tiles per block: 1 or 2).
__device__ __forceinline__ int64_t scale_index(int64_t tile, int tpb) {
  return tpb == 1 ? tile * 32 : (tile >> 1) * 64 + (tile & 1) * 16;
}

// Encode `src_row` and store it as cache row `row` (index into
// [blocks][heads][block_size]); lane 0 stores the scale of coded storage at
// scales[srow].
template <int D, int IDT, int CDT>
__device__ __forceinline__ void append_row(const uint8_t *src_row, uint8_t *cache, float *scales, int64_t row,
                                           int64_t srow, int lane) {
  float s;
  const uint2 r = encode_slice<D, IDT, CDT>(src_row, lane, s);
  constexpr int B = slice_bytes<D, CDT>();
  store_slice<D, CDT>(cache + row * (B * 32) + lane * B, r);
  if constexpr (is_coded(CDT)) {
    if (lane == 0) scales[srow] = s;
  }
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
