// Decode step executor: host block manager and every layer's launches in a
// single native call, with no separate metadata transfer.
//
// The step's metadata (slot mapping, copy pairs, lengths, block tables) is
// written to page-locked host staging, which kernels read in place: the
// block copies and layer 0's decode read it directly, and with more layers
// one small kernel copies it to device memory for layers 1...  Each layer is
// one launch of the decode kernel with the append fused in.  Staging and
// device metadata are double-buffered; half h is rewritten only after the
// kernels of the step that last used it are done (one event per half).
//
// Graph mode ("KV Cache 与 vLLM" §4.2: serving engines capture the decode
// step in CUDA graphs unless run eagerly): the launches of a step without
// copy-on-write copies are captured once per metadata half into a CUDA
// graph and replayed.  The graph bakes the kernels' arguments, so the step's
// metadata keeps a layout that changes rarely (tables as wide as the next
// power of two of the longest table, the context bound that many blocks),
// and a graph is captured again when that width, the batch size or the
// caller's buffers change.  A decode call's split-counter bank is the
// parity of an epoch drawn from its workspace's own count; a graph bakes
// its layers' epochs.  Each step draws as many epochs as it has layers and
// moves to the other half, so while the stepper alone uses its workspace,
// every step that uses a half starts at the parity its graph was captured
// with; a step whose parity differs (another caller used the workspace)
// runs eagerly.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "append.h"
#include "decode.h"
#include "dtypes.h"
#include "pkv.h"
#include "status.h"
#include "trace.h"

// What a captured step graph baked in besides the stepper's own buffers.
struct GraphKey {
  int32_t n = -1, mb = 0;
  const void *k_new = nullptr, *v_new = nullptr, *q = nullptr;
  void *out = nullptr;
  int64_t kv_stride = 0, q_stride = 0, out_stride = 0;
  int32_t out_dtype = -1;
  uint32_t scale_bits = 0;
  int32_t *d_error = nullptr;
  bool same(const GraphKey &o) const {
    return n == o.n && mb == o.mb && k_new == o.k_new && v_new == o.v_new && q == o.q && out == o.out &&
           kv_stride == o.kv_stride && q_stride == o.q_stride && out_stride == o.out_stride &&
           out_dtype == o.out_dtype && scale_bits == o.scale_bits && d_error == o.d_error;
  }
};

struct pkv_stepper {
  pkv_pool_desc pool;
  int32_t max_seqs = 0, max_blocks = 0;
  int32_t *host = nullptr;        // two halves of `half_ints` int32 (host addresses)
  const int32_t *host_dev = nullptr;  // the same staging as kernels address it
  int32_t *dev = nullptr;         // two halves of `half_ints` int32
  size_t half_ints = 0;
  void *workspace = nullptr;
  size_t workspace_bytes = 0;
  cudaEvent_t used[2] = {nullptr, nullptr};   // the last step that used half h is done
  cudaStream_t used_on[2] = {nullptr, nullptr};  // stream that step ran on
  bool recorded[2] = {false, false};
  std::vector<int64_t> ids;      // scratch for the duplicate check
  int next = 0;
  bool graphs = false;
  cudaStream_t cap = nullptr;    // capture stream
  cudaGraphExec_t exec[2] = {nullptr, nullptr};  // per metadata half
  GraphKey key[2];
  uint32_t parity[2] = {0, 0};   // of the first epoch each graph was captured with
  int64_t graph_kernels[2] = {0, 0};
  int64_t replays = 0, captures = 0;
  bool cascade = true;           // plan a cascade for shared prefixes (eager steps)
  int sms = 0;
  pkv::CascadePlan plan;
  std::vector<int32_t> order;    // scratch for the cascade plan
  int64_t cascades = 0;
  std::vector<pkv_copy_segment> in_copies;  // the next step's host-input copies (pkv_stepper_copy_inputs)
};

namespace {

// Layout of one metadata half: slots[n] | cow_src[n] | cow_dst[n] | lens[n] | tables[n][mb],
// padded to whole 16-byte vectors (the append kernel copies it in vectors).
size_t meta_ints(int32_t max_seqs, int32_t max_blocks) {
  const size_t ints = static_cast<size_t>(max_seqs) * 4 + static_cast<size_t>(max_seqs) * max_blocks;
  return (ints + 3) / 4 * 4;
}


pkv_status cuda_fail(cudaError_t e, const char *where) {
  std::string msg = std::string(where) + ": " + cudaGetErrorString(e);
  return pkv::fail(PKV_ERR_CUDA, msg.c_str());
}

// Capture a step's attention launches for metadata half h into a graph.
// Nothing runs during the capture; the launch count it added is taken back
// and added again on every replay.
template <class Issue>
pkv_status capture_step(pkv_stepper *st, int h, const GraphKey &k, Issue &issue_layers, uint32_t epoch0) {
  const int64_t before = pkv_launch_count();
  cudaError_t e = cudaStreamBeginCapture(st->cap, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaStreamBeginCapture");
  pkv_status s = issue_layers(st->cap, epoch0, false);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(st->cap, &g);  // the capture always ends, also after a failed launch
  const int64_t launched = pkv_launch_count() - before;
  pkv::add_launches(-launched);
  if (s != PKV_OK) {
    if (g) cudaGraphDestroy(g);
    return s;
  }
  if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaStreamEndCapture");
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  cudaGraphDestroy(g);
  if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaGraphInstantiate");
  if (st->exec[h]) cudaGraphExecDestroy(st->exec[h]);  // freed once its last replay is done
  st->exec[h] = x;
  st->key[h] = k;
  st->parity[h] = epoch0 & 1u;
  st->graph_kernels[h] = launched;
  ++st->captures;
  return PKV_OK;
}

// Cascade plan of one step (see CascadePlan): sequences whose tables start
// with the same physical blocks form a group; its shared tiles are the
// common leading blocks that lie wholly before every member's last token.
// Groups with fewer than kMinPrefixTiles shared tiles are left out.  The
// prefix is cut into chunks so that the prefix kernel takes about 45% of the
// SMs (the best share measured for 32 forks of a 1500-token prefix); the
// decode runs on the rest meanwhile.  Returns false when no
// group qualifies.
bool plan_cascade(pkv_stepper *st, const int32_t *tables, int32_t mb, const int32_t *lens, int32_t n) {
  const pkv_pool_desc &P = st->pool;
  if (n < 2 || n > pkv::kInlineLens) return false;
  const int32_t bs = P.block_size, tpb = P.block_size / PKV_BLOCK_SIZE;
  const int32_t G = P.num_q_heads / P.num_kv_heads;
  std::vector<int32_t> &order = st->order;
  order.clear();
  for (int32_t i = 0; i < n; ++i)
    if (lens[i] > bs) order.push_back(i);
  std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    const int32_t x = tables[static_cast<int64_t>(a) * mb], y = tables[static_cast<int64_t>(b) * mb];
    return x != y ? x < y : a < b;
  });
  pkv::CascadePlan &pl = st->plan;
  pkv::PrefixParams &pp = pl.pp;
  pp.num_groups = 0;
  int32_t nmem = 0, rows_blocks = 0;
  for (size_t a = 0; a < order.size() && pp.num_groups < pkv::kMaxPrefixGroups;) {
    size_t e = a + 1;
    const int32_t first = tables[static_cast<int64_t>(order[a]) * mb];
    while (e < order.size() && tables[static_cast<int64_t>(order[e]) * mb] == first) ++e;
    if (e - a >= 2) {
      const int32_t *lead = tables + static_cast<int64_t>(order[a]) * mb;
      int32_t cap = mb;
      for (size_t k = a; k < e; ++k) cap = std::min(cap, (lens[order[k]] - 1) / bs);
      int32_t blocks = 0;
      while (blocks < cap) {
        bool same = true;
        for (size_t k = a + 1; k < e && same; ++k) same = tables[static_cast<int64_t>(order[k]) * mb + blocks] == lead[blocks];
        if (!same) break;
        ++blocks;
      }
      if (blocks * tpb >= pkv::kMinPrefixTiles) {
        pkv::PrefixGroup &g = pp.group[pp.num_groups++];
        g.lead = order[a];
        g.tiles = blocks * tpb;
        g.members = static_cast<int32_t>(e - a);
        g.member0 = nmem;
        g.row_blocks = (g.members * G + pkv::kPrefixRows - 1) / pkv::kPrefixRows;
        for (size_t k = a; k < e; ++k) pp.member[nmem++] = order[k];
        rows_blocks += g.row_blocks;
      }
    }
    a = e;
  }
  if (pp.num_groups == 0) return false;
  // mma.sync kernel: chunks so that it takes about 45% of the SMs (measured
  // best for it).  tcgen05 kernel: chunks of about chunk_tiles tiles each,
  // so it takes few SMs and the decode keeps the rest.
  pl.umma = pkv::prefix_uses_umma(P.q_dtype, P.cache_dtype) ? 1 : 0;
  const int32_t target = std::max(8, st->sms * 5 / 11);
  const int32_t want = std::max(1, (target + rows_blocks * P.num_kv_heads - 1) / (rows_blocks * P.num_kv_heads));
  const int32_t per_chunk = std::max(1, pkv::prefix_umma_chunk_tiles());
  std::fill(pl.start, pl.start + n, 0);
  std::fill(pl.chunks, pl.chunks + n, 0);
  std::fill(pp.base, pp.base + n, 0);
  int32_t units = 0, slot = 0;
  for (int32_t gi = 0; gi < pp.num_groups; ++gi) {
    pkv::PrefixGroup &g = pp.group[gi];
    g.chunks = pl.umma ? std::min(pkv::kMaxPrefixChunks, std::max(1, (g.tiles + per_chunk - 1) / per_chunk))
                       : std::min({want, pkv::kMaxPrefixChunks, std::max(1, g.tiles / 4)});
    g.unit0 = units;
    units += g.row_blocks * g.chunks * P.num_kv_heads;
    for (int32_t k = 0; k < g.members; ++k) {
      const int32_t b = pp.member[g.member0 + k];
      pl.start[b] = g.tiles;
      pl.chunks[b] = g.chunks;
      pp.base[b] = slot;
      slot += P.num_kv_heads * g.chunks;
    }
  }
  pl.units = units;
  return true;
}

void drop_graphs(pkv_stepper *st) {
  for (int h = 0; h < 2; ++h) {
    if (st->exec[h]) cudaGraphExecDestroy(st->exec[h]);
    st->exec[h] = nullptr;
    st->key[h] = GraphKey{};
  }
}

}  // namespace

extern "C" {

size_t pkv_stepper_host_bytes(int32_t max_seqs, int32_t max_blocks_per_seq) {
  if (max_seqs <= 0 || max_blocks_per_seq <= 0) return 0;
  return 2 * meta_ints(max_seqs, max_blocks_per_seq) * sizeof(int32_t);
}

size_t pkv_stepper_device_bytes(int32_t max_seqs, int32_t max_blocks_per_seq) {
  if (max_seqs <= 0 || max_blocks_per_seq <= 0) return 0;
  return 2 * meta_ints(max_seqs, max_blocks_per_seq) * sizeof(int32_t);
}

pkv_status pkv_stepper_create(const pkv_pool_desc *pool, int32_t max_seqs, int32_t max_blocks_per_seq,
                              int32_t *host_staging, size_t host_staging_bytes, int32_t *dev_meta,
                              size_t dev_meta_bytes, void *workspace, size_t workspace_bytes,
                              pkv_stepper **out) {
  if (!pool || !out || max_seqs <= 0 || max_seqs > PKV_MAX_SEQS_PER_CALL || max_blocks_per_seq <= 0)
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_create: bad argument");
  if (pool->block_size != PKV_BLOCK_SIZE && pool->block_size != PKV_BLOCK_SIZE_32)
    return pkv::fail(PKV_ERR_UNSUPPORTED, "pkv_stepper_create: block_size must be 16 or 32");
  if (pool->num_layers <= 0 || pool->num_blocks <= 0 || pool->num_kv_heads <= 0 || !pool->k_cache ||
      !pool->v_cache ||
      (pkv::has_scales(pool->cache_dtype) && (!pool->k_scale || pool->v_scale != pool->k_scale + pool->block_size)))
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_create: bad pool descriptor");
  if (!host_staging || host_staging_bytes < pkv_stepper_host_bytes(max_seqs, max_blocks_per_seq) ||
      !dev_meta || dev_meta_bytes < pkv_stepper_device_bytes(max_seqs, max_blocks_per_seq))
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_create: staging or metadata buffer too small");
  size_t need = 0;
  pkv_status s = paged_attention_workspace_bytes(max_seqs, pool->num_q_heads, pool->num_kv_heads, pool->head_dim,
                                                 pool->q_dtype, pool->cache_dtype, &need);
  if (s != PKV_OK) return s;
  if (!workspace || workspace_bytes < need)
    return pkv::fail(PKV_ERR_WORKSPACE, "pkv_stepper_create: workspace smaller than required");
  // Kernels read the staging in place: it must be page-locked host memory
  // with a device address (unified addressing makes it the host address).
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host_staging);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
    cudaGetLastError();
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_create: host_staging is not page-locked host memory");
  }
  if ((reinterpret_cast<uintptr_t>(host_staging) & 15u) || (reinterpret_cast<uintptr_t>(attr.devicePointer) & 15u) ||
      (reinterpret_cast<uintptr_t>(dev_meta) & 15u))
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_create: staging and metadata must be 16-byte aligned");
  pkv_stepper *st = new pkv_stepper();
  st->pool = *pool;
  st->max_seqs = max_seqs;
  st->max_blocks = max_blocks_per_seq;
  st->host = host_staging;
  st->host_dev = static_cast<const int32_t *>(attr.devicePointer);
  st->dev = dev_meta;
  st->half_ints = meta_ints(max_seqs, max_blocks_per_seq);
  st->workspace = workspace;
  st->workspace_bytes = workspace_bytes;
  st->ids.reserve(static_cast<size_t>(max_seqs));
  st->order.reserve(static_cast<size_t>(max_seqs));
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&st->sms, cudaDevAttrMultiProcessorCount, dev);
    if (st->sms <= 0) st->sms = 1;
  }
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&st->used[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    pkv_stepper_destroy(st);
    return cuda_fail(e, "pkv_stepper_create: event creation");
  }
  *out = st;
  return PKV_OK;
}

void pkv_stepper_destroy(pkv_stepper *st) {
  if (!st) return;
  for (auto &e : st->used)
    if (e) {
      cudaEventSynchronize(e);  // the buffers may be freed after this returns
      cudaEventDestroy(e);
    }
  drop_graphs(st);
  if (st->cap) cudaStreamDestroy(st->cap);
  delete st;
}

pkv_status pkv_stepper_copy_inputs(pkv_stepper *st, const pkv_copy_segment *segs, int32_t num_segs) {
  if (!st) return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_copy_inputs: NULL stepper");
  if (num_segs < 0 || num_segs > PKV_MAX_COPY_SEGMENTS || (num_segs > 0 && !segs))
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_copy_inputs: bad segment count");
  for (int32_t i = 0; i < num_segs; ++i) {
    const pkv_copy_segment &g = segs[i];
    const uintptr_t a = reinterpret_cast<uintptr_t>(g.dst) | reinterpret_cast<uintptr_t>(g.src);
    if (g.bytes < 0 || (g.bytes & 15) || (g.bytes && (!g.dst || !g.src || (a & 15u))))
      return pkv::fail(PKV_ERR_INVALID,
                       "pkv_stepper_copy_inputs: NULL or misaligned pointer, or a size not a multiple of 16");
  }
  st->in_copies.assign(segs, segs + num_segs);
  return PKV_OK;
}

pkv_status pkv_stepper_use_cascade(pkv_stepper *st, int32_t enable) {
  if (!st) return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_use_cascade: NULL stepper");
  st->cascade = enable != 0;
  return PKV_OK;
}

int64_t pkv_stepper_cascade_count(const pkv_stepper *st) { return st ? st->cascades : -1; }

pkv_status pkv_stepper_use_graphs(pkv_stepper *st, int32_t enable) {
  if (!st) return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_use_graphs: NULL stepper");
  if (enable && !st->cap) {
    cudaError_t e = cudaStreamCreateWithFlags(&st->cap, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_use_graphs: capture stream");
  }
  if (!enable) drop_graphs(st);
  st->graphs = enable != 0;
  return PKV_OK;
}

pkv_status pkv_stepper_graph_stats(const pkv_stepper *st, int64_t *captures, int64_t *replays) {
  if (!st || !captures || !replays) return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_graph_stats: bad argument");
  *captures = st->captures;
  *replays = st->replays;
  return PKV_OK;
}

pkv_status pkv_stepper_step(pkv_stepper *st, pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                            const void *k_new, const void *v_new, int64_t kv_layer_stride,
                            const void *q, int64_t q_layer_stride, void *out, pkv_dtype out_dtype,
                            int64_t out_layer_stride, float scale, int32_t *cow_src, int32_t *cow_dst,
                            int32_t *num_cow, int32_t *d_error, void *attn_begin, void *attn_end,
                            pkv_stream_t stream) {
  pkv::TraceRange trace("pkv.step");
  if (!st) return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: bad argument");
  // registered input copies belong to this step only, whatever becomes of it
  std::vector<pkv_copy_segment> in_copies;
  in_copies.swap(st->in_copies);
  if (!bm || n < 0 || n > st->max_seqs || (n > 0 && (!seq_ids || !k_new || !v_new || !q || !out)))
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: bad argument");
  if (pkv_bm_block_size(bm) != st->pool.block_size)
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: the block manager's block size differs from the pool's");
  if (num_cow) *num_cow = 0;
  if (n == 0) return PKV_OK;
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       static_cast<uintptr_t>(kv_layer_stride)) & 15u)
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: k_new, v_new and their layer stride must be 16-byte aligned");
  const pkv_pool_desc &P = st->pool;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // Validate before the block manager changes: distinct sequences whose
  // tables stay within max_blocks after this step's token.
  int32_t mb = 1, max_len = 0;
  st->ids.assign(seq_ids, seq_ids + n);
  std::sort(st->ids.begin(), st->ids.end());
  if (std::adjacent_find(st->ids.begin(), st->ids.end()) != st->ids.end())
    return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: a sequence appears twice in the batch");
  for (int32_t i = 0; i < n; ++i) {
    int32_t len = 0;
    pkv_status s = pkv_seq_len(bm, seq_ids[i], &len);
    if (s != PKV_OK) return s;
    const int32_t after = len + 1;
    const int32_t blocks = (after + P.block_size - 1) / P.block_size;
    if (blocks > st->max_blocks)
      return pkv::fail(PKV_ERR_INVALID, "pkv_stepper_step: a table would exceed max_blocks_per_seq");
    mb = std::max(mb, blocks);
    max_len = std::max(max_len, after);
  }
  if (st->graphs) {  // a layout that changes rarely, so that captured launches stay valid
    int32_t w = 1;
    while (w < mb) w *= 2;
    mb = std::min(w, st->max_blocks);
    max_len = mb * P.block_size;
  }
  // Half h was last used two steps ago: its kernels must be done before the
  // host rewrites the staging, and (on another stream) before this step's
  // kernels rewrite the device half.
  const int h = st->next;
  cudaError_t e = cudaSuccess;
  if (st->recorded[h]) {
    e = cudaEventQuery(st->used[h]);
    if (e == cudaErrorNotReady) e = cudaEventSynchronize(st->used[h]);
    if (e == cudaSuccess && st->used_on[h] != cs) e = cudaStreamWaitEvent(cs, st->used[h], 0);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: waiting for the metadata half");
  }
  int32_t *H = st->host + h * st->half_ints;
  int32_t *slots = H, *src = H + n, *dst = H + 2 * n, *lens = H + 3 * n, *tables = H + 4 * n;
  int32_t ncow = 0;
  pkv_status s;
  {
    pkv::TraceRange host_trace("pkv.step.block_manager");
    s = pkv_seq_append_slots(bm, seq_ids, n, slots, src, dst, &ncow);
    if (s != PKV_OK) return s;
    s = pkv_build_block_tables(bm, seq_ids, n, mb, tables, lens);
    if (s != PKV_OK) return s;
  }
  if (num_cow) *num_cow = ncow;
  if (cow_src && ncow) std::memcpy(cow_src, src, sizeof(int32_t) * ncow);
  if (cow_dst && ncow) std::memcpy(cow_dst, dst, sizeof(int32_t) * ncow);
  st->next ^= 1;
  const int64_t ints = static_cast<int64_t>(n) * 4 + static_cast<int64_t>(n) * mb;
  const int32_t *Hd = st->host_dev + h * st->half_ints;  // staging as the kernels see it
  int32_t *Dh = st->dev + h * st->half_ints;
  const int32_t *d_lens = Dh + 3 * n, *d_tables = Dh + 4 * n;

  auto layer_ptr = [](const void *base, int64_t stride, int32_t l) {
    return static_cast<uint8_t *>(const_cast<void *>(base)) + l * stride;
  };
  const int64_t v_stride = P.v_cache_layer_stride ? P.v_cache_layer_stride : P.cache_layer_stride;
  auto scale_ptr = [&](float *base, int32_t l) {
    return base ? reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(base) + l * P.scale_layer_stride) : nullptr;
  };
  if (ncow) {  // copy-on-write: every layer's shared blocks, before any append writes into the copies
    for (int32_t l = 0; l < P.num_layers; ++l) {
      pkv::CopyArgs c{layer_ptr(P.k_cache, P.cache_layer_stride, l), layer_ptr(P.v_cache, v_stride, l),
                      scale_ptr(P.k_scale, l), scale_ptr(P.v_scale, l), Hd + n, Hd + 2 * n, ncow,
                      P.num_kv_heads, P.head_dim, P.cache_dtype, P.num_blocks, d_error, cs, P.block_size};
      s = pkv::copy_blocks_unchecked(c);
      if (s != PKV_OK) return s;
    }
  }
  // Host inputs registered for this step: one copy kernel, launched only now
  // that the host work is done, so the GPU goes from it straight to the
  // attention launches.  It is an ordinary launch (it starts after every
  // kernel before it, the copy-on-write copies included) and writes no K/V
  // cache, so a one-layer step's decode may start its first cache copies
  // while it runs.
  const bool input_copy = !in_copies.empty();
  if (input_copy) {
    s = pkv_copy_segments(in_copies.data(), static_cast<int32_t>(in_copies.size()), stream);
    if (s != PKV_OK) return s;
  }
  // The step's attention launches: with more layers one small kernel first
  // copies the staging to Dh; layer 0 reads the staging in place.
  // Eager launches carry the lengths in their parameters; a captured graph
  // reads them from the staging, which every step rewrites.
  // Eager steps of the tensor-core decode attend groups' shared prefixes
  // with the prefix kernel (cascade); graph captures do not.
  const bool cascade = st->cascade && P.head_dim == 128 && pkv_get_decode_kernel() != PKV_DECODE_SIMT &&
                       plan_cascade(st, tables, mb, lens, n);
  auto issue_layers = [&](cudaStream_t ls, uint32_t epoch0, bool eager) -> pkv_status {
    if (P.num_layers > 1) {
      pkv_status r = pkv::copy_meta_unchecked(Hd, Dh, ints, ls);
      if (r != PKV_OK) return r;
    }
    for (int32_t l = 0; l < P.num_layers; ++l) {
      // Each layer is one launch: the new token's K/V rows are written by the
      // warp that owns each sequence's last tile, then the query attends.  A
      // decode reads the lengths and tables before it waits for the kernel
      // launched just before it, so it may start early (programmatic launch):
      // layer 0 reads them from the staging, later layers from Dh, which the
      // copy kernel finished before layer 0 got past its wait.
      const int32_t *t_lens = l == 0 ? Hd + 3 * n : d_lens;
      const int32_t *t_tables = l == 0 ? Hd + 4 * n : d_tables;
      // The kernel before a layer's decode writes no K/V cache memory when it
      // is the previous layer's decode (other layers' rows), this step's
      // metadata copy or its host-input copy (both launched after the
      // copy-on-write copies), so the decode may start its first cache copies
      // before waiting for it.  (A graph replay carries the launches as
      // captured; its first kernel follows the input copy in stream order.)
      const int programmatic = (l > 0 || P.num_layers > 1 || (eager && input_copy)) ? 2 : 1;
      pkv_status r = pkv::attention_decode(
          programmatic, layer_ptr(k_new, kv_layer_stride, l), layer_ptr(v_new, kv_layer_stride, l),
          layer_ptr(out, out_layer_stride, l), out_dtype, layer_ptr(q, q_layer_stride, l), P.q_dtype,
          layer_ptr(P.k_cache, P.cache_layer_stride, l), layer_ptr(P.v_cache, v_stride, l), P.cache_dtype,
          scale_ptr(P.k_scale, l), scale_ptr(P.v_scale, l), t_tables, mb, t_lens, max_len, n, P.num_q_heads,
          P.num_kv_heads, P.head_dim, P.num_blocks, P.block_size, scale, st->workspace, st->workspace_bytes,
          d_error, reinterpret_cast<pkv_stream_t>(ls), static_cast<int64_t>(epoch0 + static_cast<uint32_t>(l)),
          eager ? lens : nullptr, eager && cascade ? &st->plan : nullptr);
      if (r != PKV_OK) return r;
    }
    return PKV_OK;
  };
  // The step's decode calls take consecutive epochs of the workspace (the
  // counters are cleared first if these shapes are new to it); a graph
  // replays only from an epoch of the parity it was captured with.
  uint32_t epoch0 = 0;
  s = pkv::take_epochs(st->workspace, n, P.num_kv_heads, P.num_layers, cs, &epoch0);
  if (s != PKV_OK) return s;
  bool replay = st->graphs && ncow == 0;
  if (replay) {
    GraphKey k;
    k.n = n;
    k.mb = mb;
    k.k_new = k_new;
    k.v_new = v_new;
    k.q = q;
    k.out = out;
    k.kv_stride = kv_layer_stride;
    k.q_stride = q_layer_stride;
    k.out_stride = out_layer_stride;
    k.out_dtype = out_dtype;
    std::memcpy(&k.scale_bits, &scale, sizeof(scale));
    k.d_error = d_error;
    if (!st->exec[h] || !st->key[h].same(k)) {
      s = capture_step(st, h, k, issue_layers, epoch0);
      if (s != PKV_OK) return s;
    } else if (st->parity[h] != (epoch0 & 1u)) {
      replay = false;  // another caller used the workspace in between: this step runs eagerly
    }
  }
  if (attn_begin) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(attn_begin), cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaEventRecord");
  }
  if (replay) {
    e = cudaGraphLaunch(st->exec[h], cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaGraphLaunch");
    pkv::add_launches(st->graph_kernels[h]);
    ++st->replays;
  } else {
    s = issue_layers(cs, epoch0, true);
    if (cascade) ++st->cascades;
    if (s != PKV_OK) return s;
  }
  if (attn_end) {
    e = cudaEventRecord(static_cast<cudaEvent_t>(attn_end), cs);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaEventRecord");
  }
  e = cudaEventRecord(st->used[h], cs);
  if (e != cudaSuccess) return cuda_fail(e, "pkv_stepper_step: cudaEventRecord");
  st->used_on[h] = cs;
  st->recorded[h] = true;
  return PKV_OK;
}

}  // extern "C"
