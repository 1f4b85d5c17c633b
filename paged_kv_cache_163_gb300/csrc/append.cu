// Reshape-and-cache (append) and copy-on-write block copy kernels.
//
// Append ("KV Cache 与 vLLM" (zwxr.cn) §1.3, "企业官网建设流程全解析" §3.2):
// every decode step writes the new token's K and V rows into the slot the
// block manager gave it.  With a coded cache ("KV Cache优化实战"
// §3.2-§3.3: FP8 E4M3 / E5M2, INT8, and 8-bit keys with 4-bit values) each
// (token, KV head) row is quantised with its own scale, amax / R, using IEEE
// fp32 divisions so the codes are reproducible (common.cuh: append_row).
//
// Copy ("KV Cache 与 vLLM" §3.3): a shared block that must change is
// copied whole to a fresh block before the new token lands in it.
#include <algorithm>

#include "append.h"
#include "common.cuh"

namespace pkv {

// One warp per (token, KV head, K-or-V) row.  Row = head_dim elements of
// 16-bit input; lane i handles elements [i * D/32, (i + 1) * D/32).
template <int D, int IDT, int CDT>
__global__ void __launch_bounds__(256) append_kernel(const uint8_t *__restrict__ k,
                                                     const uint8_t *__restrict__ v,
                                                     const int32_t *__restrict__ slot_mapping,
                                                     int32_t num_tokens, int32_t num_kv_heads,
                                                     uint8_t *__restrict__ k_cache,
                                                     uint8_t *__restrict__ v_cache,
                                                     float *__restrict__ k_scale,
                                                     float *__restrict__ v_scale,
                                                     int32_t num_blocks, int32_t bs, int32_t *err,
                                                     const int4 *__restrict__ meta_src,
                                                     int4 *__restrict__ meta_dst, int64_t meta_vecs) {
  // A decode launched after this kernel as a programmatic dependent may start
  // its prologue now; it waits for this grid to finish before reading K / V.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  {  // step metadata: host staging -> device (grid-stride, independent loads)
    const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
#pragma unroll 4
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < meta_vecs; i += nth)
      meta_dst[i] = meta_src[i];
  }
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads * 2;
  if (gw >= rows) return;
  const int kind = static_cast<int>(gw & 1);
  const int64_t th = gw >> 1;  // token * num_kv_heads + head
  const int64_t t = th / num_kv_heads;
  const int h = static_cast<int>(th - t * num_kv_heads);
  const int32_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * bs) {
    if (lane == 0) report(err, PKV_DEVERR_BAD_SLOT);
    return;
  }
  const int64_t blk = slot / bs;
  const int off = slot % bs;
  const int64_t row = (blk * num_kv_heads + h) * bs + off;        // index of the cache row
  const int64_t srow = (blk * num_kv_heads + h) * 2 * bs + off;  // of its scale (K and V side by side)
  if (kind)
    append_row<D, IDT, v_part(CDT)>(v + th * D * 2, v_cache, v_scale, row, srow, lane);
  else
    append_row<D, IDT, k_part(CDT)>(k + th * D * 2, k_cache, k_scale, row, srow, lane);
}

// Step metadata: page-locked host staging -> device, 16-byte vectors.  A
// decode launched after it as a programmatic dependent may start at once: it
// reads the staging itself and waits for this grid before anything else.
__global__ void __launch_bounds__(256) copy_meta_kernel(const int4 *__restrict__ src, int4 *__restrict__ dst,
                                                        int64_t vecs) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
#pragma unroll 4
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < vecs; i += nth) dst[i] = src[i];
}

// One CTA per (pair, K-or-V): copies a whole physical block (all heads, all
// slots); for coded caches the K CTA also copies the block's scales, which
// are one contiguous run (K and V scales side by side per head).
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t *k_cache, uint8_t *v_cache, float *scales,
                                                          const int32_t *__restrict__ src,
                                                          const int32_t *__restrict__ dst,
                                                          int64_t k_block_bytes, int64_t v_block_bytes,
                                                          int32_t scale_elems, int32_t num_blocks, int32_t *err) {
  const int pair = blockIdx.x;
  const int kind = blockIdx.y;
  const int32_t s = src[pair];
  const int32_t d = dst[pair];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && kind == 0) report(err, PKV_DEVERR_BAD_BLOCK);
    return;
  }
  uint8_t *base = kind ? v_cache : k_cache;
  const int64_t block_bytes = kind ? v_block_bytes : k_block_bytes;
  const uint4 *sp = reinterpret_cast<const uint4 *>(base + s * block_bytes);
  uint4 *dp = reinterpret_cast<uint4 *>(base + d * block_bytes);
  const int64_t n16 = block_bytes / 16;
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) dp[i] = sp[i];
  if (scales && kind == 0) {
    for (int i = threadIdx.x; i < scale_elems; i += blockDim.x)
      scales[static_cast<int64_t>(d) * scale_elems + i] = scales[static_cast<int64_t>(s) * scale_elems + i];
  }
}

template <int D, int IDT, int CDT>
static cudaError_t launch_append(const AppendArgs &a) {
  const int64_t rows = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads * 2;
  const int64_t threads = rows * 32;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  append_kernel<D, IDT, CDT><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
      static_cast<const uint8_t *>(a.k), static_cast<const uint8_t *>(a.v), a.slot_mapping,
      a.num_tokens, a.num_kv_heads, static_cast<uint8_t *>(a.k_cache),
      static_cast<uint8_t *>(a.v_cache), a.k_scale, a.v_scale, a.num_blocks, a.block_size, a.d_error,
      reinterpret_cast<const int4 *>(a.meta_src), reinterpret_cast<int4 *>(a.meta_dst),
      a.meta_src ? (a.meta_ints + 3) / 4 : 0);
  return cudaGetLastError();
}

template <int D, int CDT>
static cudaError_t dispatch_code8(const AppendArgs &a) {
  return a.in_dtype == PKV_BF16 ? launch_append<D, PKV_BF16, CDT>(a) : launch_append<D, PKV_F16, CDT>(a);
}

template <int D>
static cudaError_t dispatch_append_d(const AppendArgs &a) {
  switch (a.cache_dtype) {
    case PKV_FP8_E4M3: return dispatch_code8<D, PKV_FP8_E4M3>(a);
    case PKV_FP8_E5M2: return dispatch_code8<D, PKV_FP8_E5M2>(a);
    case PKV_INT8: return dispatch_code8<D, PKV_INT8>(a);
    case PKV_FP8_E4M3_INT4: return dispatch_code8<D, PKV_FP8_E4M3_INT4>(a);
    case PKV_BF16: return launch_append<D, PKV_BF16, PKV_BF16>(a);
    default: return launch_append<D, PKV_F16, PKV_F16>(a);
  }
}

cudaError_t run_append(const AppendArgs &a) {
  if (a.num_tokens == 0) return cudaSuccess;
  return a.head_dim == 128 ? dispatch_append_d<128>(a) : dispatch_append_d<64>(a);
}

// Grid-stride copy over the concatenation of the segments; vector i lies in
// the first segment whose prefix end exceeds it.
__global__ void __launch_bounds__(256) copy_segments_kernel(const CopySegs c) {
  // a decode launched after it as a programmatic dependent may start its
  // prologue (lengths and tables only); it waits for this grid before it
  // reads what this kernel writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t total = c.end[c.n - 1];
  const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int seg = 0;
#pragma unroll 4
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += nth) {
    while (i >= c.end[seg]) ++seg;  // i only grows
    const int64_t j = i - (seg ? c.end[seg - 1] : 0);
    c.dst[seg][j] = c.src[seg][j];
  }
}

cudaError_t run_copy_segments(const CopySegs &c, cudaStream_t stream) {
  if (c.n <= 0 || c.end[c.n - 1] == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((c.end[c.n - 1] + 255) / 256, 1024);
  copy_segments_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(c);
  return cudaGetLastError();
}

cudaError_t run_copy_meta(const int32_t *src, int32_t *dst, int64_t ints, cudaStream_t stream) {
  const int64_t vecs = (ints + 3) / 4;
  if (vecs <= 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((vecs + 255) / 256, 1024);
  copy_meta_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(reinterpret_cast<const int4 *>(src),
                                                                      reinterpret_cast<int4 *>(dst), vecs);
  return cudaGetLastError();
}

cudaError_t run_copy_blocks(const CopyArgs &a) {
  if (a.num_pairs == 0) return cudaSuccess;
  const bool scaled = has_scales(a.cache_dtype);
  const int64_t rows = static_cast<int64_t>(a.num_kv_heads) * a.block_size;
  const int64_t k_bytes = rows * row_bytes(k_part(a.cache_dtype), a.head_dim);
  const int64_t v_bytes = rows * row_bytes(v_part(a.cache_dtype), a.head_dim);
  const int32_t scale_elems = 2 * a.num_kv_heads * a.block_size;  // K and V scales of a block
  dim3 grid(a.num_pairs, 2);
  copy_blocks_kernel<<<grid, 256, 0, a.stream>>>(
      static_cast<uint8_t *>(a.k_cache), static_cast<uint8_t *>(a.v_cache), scaled ? a.k_scale : nullptr, a.src,
      a.dst, k_bytes, v_bytes, scale_elems, a.num_blocks, a.d_error);
  return cudaGetLastError();
}

}  // namespace pkv
