// C ABI of the device calls: argument validation, launch configuration,
// workspace layout.  Kernels live in append.cu and decode_*.cu.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <cstdio>
#include <mutex>
#include <string>
#include <tuple>
#include <unordered_map>

#include "append.h"
#include "decode.h"
#include "dtypes.h"
#include "pkv.h"
#include "status.h"
#include "trace.h"

namespace pkv {
namespace {

thread_local int64_t t_launches = 0;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status cuda_fail(cudaError_t e, const char *where) {
  std::string msg = std::string(where) + ": " + cudaGetErrorString(e);
  return fail(PKV_ERR_CUDA, msg.c_str());
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

std::atomic<int> g_decode_kind{PKV_DECODE_AUTO};
std::atomic<int> g_prefix_kind{PKV_PREFIX_AUTO};
std::atomic<int> g_prefix_chunk_tiles{16};

// Per-workspace state of the split counters.  A decode call with epoch e
// counts in bank e & 1 and clears the other bank for the next call, so the
// calls on one workspace take consecutive epochs from the workspace's own
// count.  The banks sit at a shape-dependent offset: the first call on a
// workspace, and any call whose shape differs from the last call on it,
// clears them first (the kernels keep them clear from then on).  A
// forgotten workspace (the table is bounded) is cleared again on its next
// use, so its restarted count is safe.
struct WorkspaceState {
  int64_t shape = -1;
  uint32_t epoch = 0;
};

// Clear the counters if needed (on `st`) and reserve `take` consecutive
// epochs (the first returned in *epoch; take may be 0).
pkv_status prepare_counters(void *workspace, int32_t num_seqs, int32_t num_kv_heads, const void *ctr, size_t bytes,
                            cudaStream_t st, int32_t take, uint32_t *epoch) {
  static std::mutex mu;
  static std::unordered_map<uintptr_t, WorkspaceState> table;
  const int64_t shape = (static_cast<int64_t>(num_seqs) << 32) | static_cast<uint32_t>(num_kv_heads);
  std::lock_guard<std::mutex> lock(mu);
  auto it = table.find(reinterpret_cast<uintptr_t>(workspace));
  if (it == table.end() || it->second.shape != shape) {
    cudaError_t e = cudaMemsetAsync(const_cast<void *>(ctr), 0, bytes, st);
    if (e != cudaSuccess) return fail(PKV_ERR_CUDA, "paged_attention_decode: clearing the split counters failed");
    if (it == table.end()) {
      if (table.size() > 4096) table.clear();
      it = table.emplace(reinterpret_cast<uintptr_t>(workspace), WorkspaceState{}).first;
    }
    it->second.shape = shape;
  }
  if (epoch) *epoch = it->second.epoch;
  it->second.epoch += static_cast<uint32_t>(take);
  return PKV_OK;
}

using DecodeFn = cudaError_t (*)(int, int, int, const DecodeParams *, int, int64_t *, DecodeShape *);
using MmaFn = cudaError_t (*)(int, int, const DecodeParams *, const CUtensorMap *, const CUtensorMap *, int,
                              int64_t *, DecodeShape *);

MmaFn pick_mma(pkv_dtype q_dtype, pkv_dtype cache_dtype) {
  if (cache_dtype == PKV_F16 && q_dtype == PKV_F16) return decode_mma_call_f16;
  if (cache_dtype == PKV_BF16 && q_dtype == PKV_BF16) return decode_mma_call_bf16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F16) return decode_mma_call_fp8_f16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_BF16) return decode_mma_call_fp8_bf16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_F16) return decode_mma_call_e5m2_f16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_BF16) return decode_mma_call_e5m2_bf16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_F16) return decode_mma_call_int8_f16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_BF16) return decode_mma_call_int8_bf16;
  if (cache_dtype == PKV_FP8_E4M3_INT4 && q_dtype == PKV_F16) return decode_mma_call_e4m3i4_f16;
  if (cache_dtype == PKV_FP8_E4M3_INT4 && q_dtype == PKV_BF16) return decode_mma_call_e4m3i4_bf16;
  return nullptr;
}

using PrefixFn = cudaError_t (*)(int, const DecodeParams *, const PrefixParams *, const CUtensorMap *,
                                 const CUtensorMap *, int);

PrefixFn pick_prefix(pkv_dtype q_dtype, pkv_dtype cache_dtype) {
  if (cache_dtype == PKV_F16 && q_dtype == PKV_F16) return prefix_call_f16;
  if (cache_dtype == PKV_BF16 && q_dtype == PKV_BF16) return prefix_call_bf16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F16) return prefix_call_fp8_f16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_BF16) return prefix_call_fp8_bf16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_F16) return prefix_call_e5m2_f16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_BF16) return prefix_call_e5m2_bf16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_F16) return prefix_call_int8_f16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_BF16) return prefix_call_int8_bf16;
  if (cache_dtype == PKV_FP8_E4M3_INT4 && q_dtype == PKV_F16) return prefix_call_e4m3i4_f16;
  return prefix_call_e4m3i4_bf16;  // dtypes validated before
}

}  // namespace

bool prefix_uses_umma(pkv_dtype q_dtype, pkv_dtype cache_dtype) {
  return g_prefix_kind.load() == PKV_PREFIX_TCGEN05 && q_dtype == cache_dtype &&
         (cache_dtype == PKV_F16 || cache_dtype == PKV_BF16);
}

int32_t prefix_umma_chunk_tiles() { return g_prefix_chunk_tiles.load(); }

namespace {

bool use_mma(int32_t head_dim) {
  const int k = g_decode_kind.load();
  return head_dim == 128 && k != PKV_DECODE_SIMT;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2D map of one layer's K or V pool: rows of 128 elements, box [64 or 128 elements][16 rows],
// 128-byte swizzle.  Encoded maps are cached by (address, rows, element size).
pkv_status cache_tensor_map(const void *base, int64_t rows, int esz, CUtensorMap *out) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, std::pair<int64_t, CUtensorMap>> cache;
  const uint64_t key = reinterpret_cast<uint64_t>(base) ^ static_cast<uint64_t>(esz);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end() && it->second.first == rows) {
      *out = it->second.second;
      return PKV_OK;
    }
  }
  auto enc = tensor_map_encoder();
  if (!enc) return fail(PKV_ERR_CUDA, "decode: cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(128 * esz)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(esz == 1 ? 128 : 64), 16};
  const cuuint32_t elem[2] = {1, 1};
  CUtensorMap m;
  CUresult r = enc(&m, esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                   const_cast<void *>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "decode: cuTensorMapEncodeTiled rejected the cache layout");
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() > 4096) cache.clear();
  cache[key] = {rows, m};
  *out = m;
  return PKV_OK;
}

DecodeFn pick_decode(pkv_dtype q_dtype, pkv_dtype cache_dtype) {
  if (cache_dtype == PKV_F16 && q_dtype == PKV_F16) return decode_call_f16;
  if (cache_dtype == PKV_BF16 && q_dtype == PKV_BF16) return decode_call_bf16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_F16) return decode_call_fp8_f16;
  if (cache_dtype == PKV_FP8_E4M3 && q_dtype == PKV_BF16) return decode_call_fp8_bf16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_F16) return decode_call_e5m2_f16;
  if (cache_dtype == PKV_FP8_E5M2 && q_dtype == PKV_BF16) return decode_call_e5m2_bf16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_F16) return decode_call_int8_f16;
  if (cache_dtype == PKV_INT8 && q_dtype == PKV_BF16) return decode_call_int8_bf16;
  if (cache_dtype == PKV_FP8_E4M3_INT4 && q_dtype == PKV_F16) return decode_call_e4m3i4_f16;
  if (cache_dtype == PKV_FP8_E4M3_INT4 && q_dtype == PKV_BF16) return decode_call_e4m3i4_bf16;
  return nullptr;
}

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// Split counters: two banks of one per (sequence, KV head).
int64_t ctr_bytes(int32_t num_seqs, int32_t num_kv_heads) {
  return round256(2 * static_cast<int64_t>(num_seqs) * num_kv_heads * 4);
}

struct DecodeLayout {
  int64_t ctr_bytes, ml_bytes, o_bytes, pfx_ml_bytes, pfx_o_bytes, total;
  DecodeShape simt, mma;  // residency of the two kernel variants (mma: head_dim 128 only)
  int sms;
};

// Shapes and dtypes checked by the caller.  Fills the workspace layout (its
// partial slots cover every warp either variant can run at once, plus one per
// item) and the residency of each variant on this device.
pkv_status decode_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, pkv_dtype q_dtype, pkv_dtype cache_dtype,
                         DecodeLayout *lay) {
  DecodeFn fn = pick_decode(q_dtype, cache_dtype);
  if (!fn) return fail(PKV_ERR_UNSUPPORTED, "decode: unsupported q / cache dtype pair");
  const int group = num_q_heads / num_kv_heads;
  lay->simt = DecodeShape{0, 0};
  lay->mma = DecodeShape{0, 0};
  cudaError_t e = fn(head_dim, group, kDecodePrepare, nullptr, 0, nullptr, &lay->simt);
  if (e == cudaErrorNotSupported)
    return fail(PKV_ERR_UNSUPPORTED, "decode: head_dim must be 64 or 128 and group 1, 2, 4 or 8");
  if (e != cudaSuccess) return cuda_fail(e, "decode: kernel setup");
  int64_t warps_per_sm = static_cast<int64_t>(lay->simt.ctas_per_sm) * lay->simt.warps_per_cta;
  if (head_dim == 128) {  // the workspace serves either kernel variant
    e = pick_mma(q_dtype, cache_dtype)(group, kDecodePrepare, nullptr, nullptr, nullptr, 0, nullptr, &lay->mma);
    if (e != cudaSuccess) return cuda_fail(e, "decode: tensor-core kernel setup");
    warps_per_sm = std::max<int64_t>(warps_per_sm, static_cast<int64_t>(lay->mma.ctas_per_sm) * lay->mma.warps_per_cta);
  }
  lay->sms = sm_count();
  if (lay->sms <= 0) return fail(PKV_ERR_CUDA, "decode: cannot query the SM count");
  const int64_t slots = lay->sms * warps_per_sm + static_cast<int64_t>(num_seqs) * num_kv_heads;
  lay->ctr_bytes = ctr_bytes(num_seqs, num_kv_heads);
  lay->ml_bytes = round256(slots * group * 2 * 4);
  lay->o_bytes = round256(slots * group * head_dim * 4);
  // the prefix kernel's partials (cascade): up to kMaxPrefixChunks per (sequence, KV head)
  const int64_t pfx_slots = static_cast<int64_t>(std::min<int32_t>(num_seqs, kInlineLens)) * num_kv_heads *
                            kMaxPrefixChunks;
  lay->pfx_ml_bytes = head_dim == 128 ? round256(pfx_slots * group * 2 * 4) : 0;
  lay->pfx_o_bytes = head_dim == 128 ? round256(pfx_slots * group * head_dim * 4) : 0;
  lay->total = lay->ctr_bytes + lay->ml_bytes + lay->o_bytes + lay->pfx_ml_bytes + lay->pfx_o_bytes;
  return PKV_OK;
}

pkv_status check_heads(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PKV_ERR_INVALID, "num_q_heads must be a positive multiple of num_kv_heads");
  if (head_dim != 64 && head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int64_t pkv_launch_count(void) { return t_launches; }

pkv_status pkv_set_decode_kernel(pkv_decode_kernel kind) {
  if (kind != PKV_DECODE_AUTO && kind != PKV_DECODE_SIMT && kind != PKV_DECODE_MMA)
    return fail(PKV_ERR_INVALID, "pkv_set_decode_kernel: unknown kind");
  g_decode_kind.store(kind);
  return PKV_OK;
}

pkv_decode_kernel pkv_get_decode_kernel(void) { return static_cast<pkv_decode_kernel>(g_decode_kind.load()); }

pkv_status pkv_set_prefix_kernel(pkv_prefix_kernel kind, int32_t chunk_tiles) {
  if (kind != PKV_PREFIX_AUTO && kind != PKV_PREFIX_MMA_SYNC && kind != PKV_PREFIX_TCGEN05)
    return fail(PKV_ERR_INVALID, "pkv_set_prefix_kernel: unknown kind");
  if (chunk_tiles < 0 || chunk_tiles > 4096)
    return fail(PKV_ERR_INVALID, "pkv_set_prefix_kernel: chunk_tiles outside [0, 4096]");
  g_prefix_kind.store(kind);
  g_prefix_chunk_tiles.store(chunk_tiles == 0 ? 16 : chunk_tiles);
  return PKV_OK;
}

pkv_prefix_kernel pkv_get_prefix_kernel(void) { return static_cast<pkv_prefix_kernel>(g_prefix_kind.load()); }

pkv_status paged_kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                                const int32_t *src, const int32_t *dst, int32_t num_pairs,
                                int32_t num_kv_heads, int32_t head_dim, pkv_dtype cache_dtype,
                                int32_t num_blocks, int32_t block_size, int32_t *d_error, pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.copy_blocks");
  if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PKV_ERR_INVALID, "paged_kv_copy_blocks: bad sizes");
  if (block_size != PKV_BLOCK_SIZE && block_size != PKV_BLOCK_SIZE_32)
    return fail(PKV_ERR_UNSUPPORTED, "paged_kv_copy_blocks: block_size must be 16 or 32");
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "paged_kv_copy_blocks: head_dim must be 64 or 128");
  if (!is_cache_type(cache_dtype)) return fail(PKV_ERR_INVALID, "paged_kv_copy_blocks: bad cache dtype");
  if (num_pairs == 0) return PKV_OK;
  if (num_pairs > 65535) return fail(PKV_ERR_INVALID, "paged_kv_copy_blocks: at most 65535 pairs per call");
  if (!k_cache || !v_cache || !src || !dst || !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID, "paged_kv_copy_blocks: NULL or misaligned pointer");
  if (has_scales(cache_dtype) && (!k_scale || v_scale != k_scale + block_size))
    return fail(PKV_ERR_INVALID, "paged_kv_copy_blocks: a coded cache needs k_scale, and v_scale = k_scale + block_size");
  CopyArgs a{k_cache, v_cache, k_scale, v_scale, src, dst, num_pairs, num_kv_heads,
             head_dim, cache_dtype, num_blocks, d_error, reinterpret_cast<cudaStream_t>(stream), block_size};
  cudaError_t e = run_copy_blocks(a);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_copy_blocks");
  ++t_launches;
  return PKV_OK;
}

pkv_status paged_kv_append(const void *k, const void *v, pkv_dtype in_dtype, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t *slot_mapping,
                           void *k_cache, void *v_cache, pkv_dtype cache_dtype, float *k_scale,
                           float *v_scale, int32_t num_blocks, int32_t block_size, int32_t *d_error,
                           pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.append");
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0)
    return fail(PKV_ERR_INVALID, "paged_kv_append: bad sizes");
  if (block_size != PKV_BLOCK_SIZE && block_size != PKV_BLOCK_SIZE_32)
    return fail(PKV_ERR_UNSUPPORTED, "paged_kv_append: block_size must be 16 or 32");
  if (head_dim != 64 && head_dim != 128)
    return fail(PKV_ERR_UNSUPPORTED, "paged_kv_append: head_dim must be 64 or 128");
  if (in_dtype != PKV_F16 && in_dtype != PKV_BF16)
    return fail(PKV_ERR_INVALID, "paged_kv_append: input rows must be F16 or BF16");
  if (!is_cache_type(cache_dtype)) return fail(PKV_ERR_INVALID, "paged_kv_append: bad cache dtype");
  if (!has_scales(cache_dtype) && cache_dtype != in_dtype)
    return fail(PKV_ERR_UNSUPPORTED, "paged_kv_append: a 16-bit cache must match the input dtype");
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || !aligned16(k) || !aligned16(v) ||
      !aligned16(k_cache) || !aligned16(v_cache))
    return fail(PKV_ERR_INVALID, "paged_kv_append: NULL or misaligned pointer");
  if (has_scales(cache_dtype) && (!k_scale || v_scale != k_scale + block_size))
    return fail(PKV_ERR_INVALID, "paged_kv_append: a coded cache needs k_scale, and v_scale = k_scale + block_size");
  AppendArgs a{k, v, in_dtype, num_tokens, num_kv_heads, head_dim, slot_mapping, k_cache, v_cache,
               cache_dtype, k_scale, v_scale, num_blocks, d_error,
               reinterpret_cast<cudaStream_t>(stream), block_size};
  cudaError_t e = run_append(a);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_append");
  ++t_launches;
  return PKV_OK;
}

pkv_status pkv_copy_segments(const pkv_copy_segment *segs, int32_t num_segs, pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.copy_segments");
  if (num_segs < 0 || num_segs > PKV_MAX_COPY_SEGMENTS || (num_segs > 0 && !segs))
    return fail(PKV_ERR_INVALID, "pkv_copy_segments: bad segment count");
  CopySegs c{};
  int64_t run = 0;
  for (int32_t i = 0; i < num_segs; ++i) {
    const pkv_copy_segment &g = segs[i];
    if (g.bytes < 0 || (g.bytes & 15) || (g.bytes && (!g.dst || !g.src || !aligned16(g.dst) || !aligned16(g.src))))
      return fail(PKV_ERR_INVALID, "pkv_copy_segments: NULL or misaligned pointer, or a size not a multiple of 16");
    c.dst[c.n] = static_cast<int4 *>(g.dst);
    c.src[c.n] = static_cast<const int4 *>(g.src);
    run += g.bytes / 16;
    c.end[c.n] = run;
    ++c.n;
  }
  if (run == 0) return PKV_OK;
  cudaError_t e = run_copy_segments(c, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "pkv_copy_segments");
  ++t_launches;
  return PKV_OK;
}

pkv_status paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           pkv_dtype q_dtype, pkv_dtype cache_dtype,
                                           size_t *bytes) {
  if (!bytes || num_seqs < 0 || num_seqs > PKV_MAX_SEQS_PER_CALL)
    return fail(PKV_ERR_INVALID, "paged_attention_workspace_bytes: bad argument");
  pkv_status s = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (s != PKV_OK) return s;
  DecodeLayout lay;
  s = decode_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, q_dtype, cache_dtype, &lay);
  if (s != PKV_OK) return s;
  *bytes = static_cast<size_t>(lay.total);
  return PKV_OK;
}

}  // extern "C"

namespace pkv {

void add_launches(int64_t delta) { t_launches += delta; }

pkv_status take_epochs(void *workspace, int32_t num_seqs, int32_t num_kv_heads, int32_t count,
                       cudaStream_t stream, uint32_t *first) {
  const int64_t bytes = ctr_bytes(num_seqs, num_kv_heads);
  return prepare_counters(workspace, num_seqs, num_kv_heads, workspace, static_cast<size_t>(bytes), stream, count,
                          first);
}

pkv_status append_unchecked(const AppendArgs &a) {
  cudaError_t e = run_append(a);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_append");
  ++t_launches;
  return PKV_OK;
}

pkv_status copy_meta_unchecked(const int32_t *src, int32_t *dst, int64_t ints, cudaStream_t stream) {
  cudaError_t e = run_copy_meta(src, dst, ints, stream);
  if (e != cudaSuccess) return cuda_fail(e, "step metadata copy");
  ++t_launches;
  return PKV_OK;
}

pkv_status copy_blocks_unchecked(const CopyArgs &a) {
  cudaError_t e = run_copy_blocks(a);
  if (e != cudaSuccess) return cuda_fail(e, "paged_kv_copy_blocks");
  ++t_launches;
  return PKV_OK;
}

pkv_status attention_decode(int programmatic, const void *k_new, const void *v_new, void *out, pkv_dtype out_dtype,
                            const void *q, pkv_dtype q_dtype,
                            const void *k_cache, const void *v_cache, pkv_dtype cache_dtype, const float *k_scale,
                            const float *v_scale, const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                            int32_t block_size, float scale, void *workspace, size_t workspace_bytes,
                            int32_t *d_error, pkv_stream_t stream, int64_t epoch, const int32_t *host_lens,
                            const CascadePlan *plan) {
  if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS_PER_CALL)
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode: num_seqs must be in [0, 1024]");
  pkv_status s = check_heads(num_q_heads, num_kv_heads, head_dim);
  if (s != PKV_OK) return s;
  if (max_blocks_per_seq < 0 || max_context_len < 0 || num_blocks <= 0)
    return fail(PKV_ERR_INVALID, "paged_attention_decode: bad sizes");
  if (block_size != PKV_BLOCK_SIZE && block_size != PKV_BLOCK_SIZE_32)
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode: block_size must be 16 or 32");
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t(1) << 31))
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode: pool larger than 2^31 token rows");
  if (static_cast<int64_t>(num_seqs) * num_kv_heads > (1 << 24))
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode: too many (sequence, KV head) pairs");
  if (out_dtype != PKV_F32 && out_dtype != q_dtype)
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode: out_dtype must be F32 or q_dtype");
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !workspace ||
      !aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace))
    return fail(PKV_ERR_INVALID, "paged_attention_decode: NULL or misaligned pointer");
  if (has_scales(cache_dtype) && (!k_scale || !aligned16(k_scale) || v_scale != k_scale + block_size))
    return fail(PKV_ERR_INVALID,
                "paged_attention_decode: a coded cache needs an aligned k_scale, and v_scale = k_scale + block_size");
  if ((k_new != nullptr) != (v_new != nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
    return fail(PKV_ERR_INVALID, "paged_attention_decode_append: k_new and v_new must both be given, 16-byte aligned");
  DecodeLayout lay;
  s = decode_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, q_dtype, cache_dtype, &lay);
  if (s != PKV_OK) return s;
  if (workspace_bytes < static_cast<size_t>(lay.total))
    return fail(PKV_ERR_WORKSPACE, "paged_attention_decode: workspace smaller than required");

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeParams p{};
  p.out = static_cast<uint8_t *>(out);
  p.out_f32 = out_dtype == PKV_F32 ? 1 : 0;
  p.q = static_cast<const uint8_t *>(q);
  p.k_cache = static_cast<const uint8_t *>(k_cache);
  p.v_cache = static_cast<const uint8_t *>(v_cache);
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.max_context_len = max_context_len;
  p.num_seqs = num_seqs;
  p.num_kv_heads = num_kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.tiles_per_block = block_size / PKV_BLOCK_SIZE;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.ws_ctr = reinterpret_cast<uint32_t *>(ws);
  p.ws_ml = reinterpret_cast<float *>(ws + lay.ctr_bytes);
  p.ws_o = reinterpret_cast<float *>(ws + lay.ctr_bytes + lay.ml_bytes);

  p.d_error = d_error;
  p.stream = reinterpret_cast<cudaStream_t>(stream);
  p.programmatic = programmatic ? 1 : 0;
  p.early_kv = programmatic == 2 ? 1 : 0;
  p.k_new = static_cast<const uint8_t *>(k_new);
  p.v_new = static_cast<const uint8_t *>(v_new);
  if (host_lens && num_seqs <= kInlineLens) {
    std::memcpy(p.lens_inline, host_lens, sizeof(int32_t) * static_cast<size_t>(num_seqs));
    p.lens_inline_n = num_seqs;
  }
  uint32_t ep = 0;
  s = prepare_counters(workspace, num_seqs, num_kv_heads, p.ws_ctr, static_cast<size_t>(lay.ctr_bytes), p.stream,
                       epoch >= 0 ? 0 : 1, &ep);
  if (s != PKV_OK) return s;
  p.epoch = epoch >= 0 ? static_cast<uint32_t>(epoch) : ep;

  // Grid: enough warps that each gets a few tiles of the largest possible
  // share, capped at one wave of resident CTAs of the variant that runs.
  const bool mma = use_mma(head_dim);
  const DecodeShape shape = mma ? lay.mma : lay.simt;
  constexpr int64_t kMinTilesPerWarp = 4;
  const int64_t max_tiles = static_cast<int64_t>(num_seqs) * num_kv_heads *
                            ((static_cast<int64_t>(max_context_len) + PKV_BLOCK_SIZE - 1) / PKV_BLOCK_SIZE);
  const int64_t per_cta = shape.warps_per_cta * kMinTilesPerWarp;
  int64_t grid = (max_tiles + per_cta - 1) / per_cta;
  if (grid < 1) grid = 1;
  if (grid > static_cast<int64_t>(lay.sms) * shape.ctas_per_sm) grid = static_cast<int64_t>(lay.sms) * shape.ctas_per_sm;

  cudaError_t e;
  if (mma) {
    const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
    const int esz = is_code8(k_part(cache_dtype)) ? 1 : 2;
    CUtensorMap tmk, tmv;
    s = cache_tensor_map(k_cache, rows, esz, &tmk);
    if (s != PKV_OK) return s;
    if (v_part(cache_dtype) == kInt4) {
      tmv = tmk;  // not read: 4-bit V tiles arrive by plain bulk copies
    } else {
      s = cache_tensor_map(v_cache, rows, esz, &tmv);
      if (s != PKV_OK) return s;
    }
    if (plan && plan->units > 0 && num_seqs <= kInlineLens) {
      // the decode shares the GPU with the prefix grid: it takes the other SMs
      grid = std::max<int64_t>(1, std::min<int64_t>(grid, static_cast<int64_t>(lay.sms) * shape.ctas_per_sm - plan->units));
      // cascade: the prefix kernel attends the groups' shared tiles, the decode the rest
      PrefixParams pp = plan->pp;
      pp.ml = reinterpret_cast<float *>(ws + lay.ctr_bytes + lay.ml_bytes + lay.o_bytes);
      pp.o = reinterpret_cast<float *>(ws + lay.ctr_bytes + lay.ml_bytes + lay.o_bytes + lay.pfx_ml_bytes);
      p.pfx_n = num_seqs;
      std::memcpy(p.pfx_start, plan->start, sizeof(int32_t) * static_cast<size_t>(num_seqs));
      std::memcpy(p.pfx_chunks, plan->chunks, sizeof(int32_t) * static_cast<size_t>(num_seqs));
      std::memcpy(p.pfx_base, plan->pp.base, sizeof(int32_t) * static_cast<size_t>(num_seqs));
      p.pfx_ml = pp.ml;
      p.pfx_o = pp.o;
      if (plan->umma) {
        e = (cache_dtype == PKV_BF16 ? prefix_umma_call_bf16 : prefix_umma_call_f16)(num_q_heads / num_kv_heads, &p,
                                                                                    &pp, &tmk, &tmv, plan->units);
      } else {
        e = pick_prefix(q_dtype, cache_dtype)(num_q_heads / num_kv_heads, &p, &pp, &tmk, &tmv, plan->units);
      }
      if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode: prefix kernel");
      ++t_launches;
    }
    e = pick_mma(q_dtype, cache_dtype)(num_q_heads / num_kv_heads, kDecodeLaunch, &p, &tmk, &tmv,
                                       static_cast<int>(grid), &t_launches, nullptr);
  } else {
    DecodeFn fn = pick_decode(q_dtype, cache_dtype);
    e = fn(head_dim, num_q_heads / num_kv_heads, kDecodeLaunch, &p, static_cast<int>(grid), &t_launches, nullptr);
  }
  if (e != cudaSuccess) return cuda_fail(e, "paged_attention_decode");
  return PKV_OK;
}

}  // namespace pkv

extern "C" {

pkv_status paged_attention_decode(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                  const void *k_cache,
                                  const void *v_cache, pkv_dtype cache_dtype, const float *k_scale,
                                  const float *v_scale, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens,
                                  int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                  int32_t block_size, float scale, void *workspace, size_t workspace_bytes,
                                  int32_t *d_error, pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.decode");
  return pkv::attention_decode(false, nullptr, nullptr, out, out_dtype, q, q_dtype, k_cache, v_cache, cache_dtype,
                               k_scale, v_scale, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                               workspace, workspace_bytes, d_error, stream);
}

pkv_status paged_attention_decode_append(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                         const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                         pkv_dtype cache_dtype, float *k_scale, float *v_scale,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, int32_t block_size, float scale, void *workspace,
                                         size_t workspace_bytes, int32_t *d_error, pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.decode_append");
  if (num_seqs > 0 && (!k_new || !v_new))
    return fail(PKV_ERR_INVALID, "paged_attention_decode_append: NULL k_new or v_new");
  return pkv::attention_decode(false, k_new, v_new, out, out_dtype, q, q_dtype, k_cache, v_cache, cache_dtype,
                               k_scale, v_scale, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                               num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                               workspace, workspace_bytes, d_error, stream);
}

pkv_status pkv_read_device_error(int32_t *d_error, int32_t *h_error, int32_t clear,
                                 pkv_stream_t stream) {
  if (!d_error || !h_error) return fail(PKV_ERR_INVALID, "pkv_read_device_error: NULL pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h_error, d_error, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) {
    e = cudaMemsetAsync(d_error, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "pkv_read_device_error");
  if (*h_error != 0) return fail(PKV_ERR_DEVICE_CHECK, "device-side check failed");
  return PKV_OK;
}

}  // extern "C"
