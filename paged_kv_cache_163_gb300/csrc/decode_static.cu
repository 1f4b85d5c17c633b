// Decode with library-owned scratch, for callers that cannot allocate device
// memory.
//
// Some callers of this library cannot call cudaMalloc themselves. Examples:
// a plugin whose host framework owns every device allocation, or a
// latency-critical loop where an allocation could synchronise the device.
// For them, paged_attention_decode_static takes the same arguments as
// paged_attention_decode but no workspace.  The split-KV scratch it needs
// lives in a file-scope __device__ buffer of PKV_STATIC_SCRATCH_BYTES.  Each
// GPU that loads the library holds one copy until the process exits.
//
// In host code, the buffer's name is only a host-side stand-in, not a device
// address.  So the first call on each device looks the real address up with
// cudaGetSymbolAddress, with that device current, caches it, and passes it on
// as the workspace of the ordinary decode call.  Make that first call before
// any stream capture.
//
// Every call on a device shares the one buffer, and the buffer keeps the last
// call's contents.  Only the decode's split counters must start at zero;
// the partials are written before they are read.  paged_attention_decode
// keeps its counters per workspace address: the first call on an address,
// and any call whose (num_seqs, num_kv_heads) differ from the last call on
// it, clears the counter banks with cudaMemsetAsync on the caller's stream
// (prepare_counters in capi.cu), and every kernel clears the bank the next
// call uses.  So this file clears nothing itself, and the clear is ordered
// on the same stream as the decode it serves.  Calls whose kernels overlap
// on the GPU (for example on two concurrent streams) race on the buffer, so
// serialise them.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "pkv.h"
#include "status.h"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once).
pkv_status scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    std::string msg = std::string("paged_attention_decode_static: cudaGetDevice: ") + cudaGetErrorString(e);
    return fail(PKV_ERR_CUDA, msg.c_str());
  }
  if (dev < 0 || dev >= kMaxDevices)
    return fail(PKV_ERR_UNSUPPORTED, "paged_attention_decode_static: device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr) {
      std::string msg = std::string("paged_attention_decode_static: cudaGetSymbolAddress: ") +
                        cudaGetErrorString(e);
      return fail(PKV_ERR_CUDA, msg.c_str());
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status paged_attention_decode_static(
    void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype, const void *k_cache,
    const void *v_cache, pkv_dtype cache_dtype, const float *k_scale, const float *v_scale,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, int32_t *d_error,
    pkv_stream_t stream) {
  size_t need = 0;
  pkv_status s = paged_attention_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, q_dtype,
                                                 cache_dtype, &need);
  if (s != PKV_OK) return s;
  if (need > pkv::kStaticScratchBytes) {
    std::string msg = "paged_attention_decode_static: these shapes need " + std::to_string(need) +
                      " bytes of scratch, more than the " + std::to_string(pkv::kStaticScratchBytes) +
                      "-byte static buffer; call paged_attention_decode with a workspace instead";
    return pkv::fail(PKV_ERR_WORKSPACE, msg.c_str());
  }
  void *ws = nullptr;
  s = pkv::scratch_for_current_device(&ws);
  if (s != PKV_OK) return s;
  return paged_attention_decode(out, out_dtype, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                                block_tables, max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                                num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, ws,
                                pkv::kStaticScratchBytes, d_error, stream);
}
