// Launch interfaces of the append and block-copy kernels (validated arguments).
#pragma once

#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

struct AppendArgs {
  const void *k, *v;
  pkv_dtype in_dtype;
  int32_t num_tokens, num_kv_heads, head_dim;
  const int32_t *slot_mapping;
  void *k_cache, *v_cache;
  pkv_dtype cache_dtype;
  float *k_scale, *v_scale;
  int32_t num_blocks;
  int32_t *d_error;
  cudaStream_t stream;
  int32_t block_size;  // 16 or 32 tokens per physical block
  // Optional: the kernel also copies meta_ints int32 from meta_src (page-locked
  // host memory, read in place) to meta_dst (device), 16-byte vectors, with
  // both pointers 16-byte aligned and room for meta_ints rounded up to 4.
  const int32_t *meta_src;
  int32_t *meta_dst;
  int64_t meta_ints;
};

struct CopyArgs {
  void *k_cache, *v_cache;
  float *k_scale, *v_scale;
  const int32_t *src, *dst;
  int32_t num_pairs, num_kv_heads, head_dim;
  pkv_dtype cache_dtype;
  int32_t num_blocks;
  int32_t *d_error;
  cudaStream_t stream;
  int32_t block_size;  // 16 or 32 tokens per physical block
};

cudaError_t run_append(const AppendArgs &a);
cudaError_t run_copy_blocks(const CopyArgs &a);
// Copy `ints` int32 (rounded up to whole 16-byte vectors) from page-locked host
// memory (device address) to device memory; both 16-byte aligned.
cudaError_t run_copy_meta(const int32_t *src, int32_t *dst, int64_t ints, cudaStream_t stream);

// Copy segments (16-byte vectors; sizes validated by the caller): one launch.
struct CopySegs {
  int4 *dst[PKV_MAX_COPY_SEGMENTS];
  const int4 *src[PKV_MAX_COPY_SEGMENTS];
  int64_t end[PKV_MAX_COPY_SEGMENTS];  // inclusive prefix sums of the segments' vector counts
  int32_t n;
};
cudaError_t run_copy_segments(const CopySegs &c, cudaStream_t stream);

// Launch with the caller's validation (the step executor's); count the launch.
pkv_status append_unchecked(const AppendArgs &a);
pkv_status copy_blocks_unchecked(const CopyArgs &a);
pkv_status copy_meta_unchecked(const int32_t *src, int32_t *dst, int64_t ints, cudaStream_t stream);

}  // namespace pkv
