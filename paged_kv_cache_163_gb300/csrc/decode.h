// Launch interface of the decode kernels (arguments already validated).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Residency of one decode kernel instance: CTAs per SM and warps per CTA.
struct DecodeShape {
  int ctas_per_sm;
  int warps_per_cta;
};

// Context lengths a launch can carry in its parameters (for batches up to
// this size): the prologue then reads no lengths from memory.
constexpr int kInlineLens = 128;

struct DecodeParams {
  uint8_t *out;
  int32_t out_f32;   // 1: out is float32, 0: out has the query's 16-bit type
  const uint8_t *q;
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_tables;
  const int32_t *context_lens;
  int32_t max_blocks_per_seq;
  int32_t max_context_len;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t num_blocks;
  int32_t block_size;       // tokens per physical block: 16 or 32
  int32_t tiles_per_block;  // 16-token tiles per physical block: 1 or 2
  float scale_log2;  // scale * log2(e)
  uint32_t *ws_ctr;  // [2][num_seqs * num_kv_heads] partials stored per item; bank epoch & 1
  uint32_t epoch;    // one value per decode call; consecutive calls alternate banks
  float *ws_ml;      // [slots][G][2] partial (max, sum), base-2 domain
  float *ws_o;       // [slots][G][head_dim] partial unnormalised outputs
  int32_t *d_error;
  cudaStream_t stream;
  int32_t programmatic;  // 1: launch as a programmatic dependent of the stream's previous kernel
  // 1: that kernel writes no K/V cache or scale memory, so the first tiles'
  // cache copies may start before the wait for it (queries and new rows after)
  int32_t early_kv;
  // Optional fused append: row (b, kvh) of k_new / v_new ([num_seqs][num_kv_heads][head_dim] in the
  // query dtype) is written at position context_lens[b] - 1 before that tile is read.  NULL: none.
  const uint8_t *k_new;
  const uint8_t *v_new;
  // 0, or num_seqs: lens_inline[b] == context_lens[b] for every b (read instead of memory)
  int32_t lens_inline_n;
  int32_t lens_inline[kInlineLens];
  // Cascade (0, or num_seqs): sequence b's first pfx_start[b] 16-token tiles
  // were attended by the prefix kernel, which left pfx_chunks[b] partials per
  // KV head at slots pfx_base[b] + kvh * pfx_chunks[b] of pfx_ml / pfx_o
  // (same layout as ws_ml / ws_o); this call attends the rest and merges them in.
  int32_t pfx_n;
  int32_t pfx_start[kInlineLens];
  int32_t pfx_chunks[kInlineLens];
  int32_t pfx_base[kInlineLens];
  const float *pfx_ml;
  const float *pfx_o;
};

// Cascade: groups of sequences whose first tiles are the same physical
// blocks, attended once for all members by the prefix kernel
// (decode_prefix.cuh).
constexpr int kMaxPrefixGroups = 16;
constexpr int kPrefixRows = 128;  // query rows a CTA attends: 8 warps x 16

struct PrefixGroup {
  int32_t lead;        // batch index of a member (its table row holds the shared blocks)
  int32_t tiles;       // shared 16-token tiles
  int32_t chunks;      // tile ranges the prefix is split into
  int32_t members;     // members in the group
  int32_t member0;     // offset of the members in PrefixParams::member
  int32_t row_blocks;  // ceil(members * G / 128)
  int32_t unit0;       // first CTA of the group; CTAs [unit0, unit0 + row_blocks * chunks * Hkv)
};

struct PrefixParams {
  int32_t num_groups;
  PrefixGroup group[kMaxPrefixGroups];
  int32_t member[kInlineLens];  // batch indices, group after group
  int32_t base[kInlineLens];    // per batch index: first partial slot ([KV head][chunk] from there)
  float *ml;                    // [slots][G][2] (max, sum), base-2 domain
  float *o;                     // [slots][G][head_dim] unnormalised outputs
};

// Up to this many chunks of a prefix (and partials per member and KV head).
constexpr int kMaxPrefixChunks = 16;
// Fewer shared tiles than this are left to the decode kernel.
constexpr int kMinPrefixTiles = 16;

// A step's cascade, planned on the host from its block tables (batches of up
// to kInlineLens sequences): the prefix kernel's groups, and per batch index
// the tiles it attends (start), its partials per KV head (chunks) and their
// first slot (pp.base).  attention_decode fills in pp.ml / pp.o.
struct CascadePlan {
  PrefixParams pp;
  int32_t units;  // prefix kernel CTAs
  int32_t umma;   // 1: the tcgen05 prefix kernel runs (its chunking), 0: the mma.sync one
  int32_t start[kInlineLens];
  int32_t chunks[kInlineLens];
};

// Launch `kernel` on `stream`; with programmatic != 0 the launch may begin
// before the previous kernel on the stream has finished (the kernel waits on
// griddepcontrol.wait before it reads what that kernel writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_decode(void (*kernel)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                          int programmatic, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

enum DecodeOp { kDecodePrepare = 0, kDecodeLaunch = 1 };

// op == kDecodePrepare: *shape = the instance's resident CTAs per SM and warps per CTA.
// op == kDecodeLaunch: launch the decode kernel on `grid` CTAs (it merges split items itself).
// Returns cudaErrorNotSupported when (head_dim, group) has no instance.
cudaError_t decode_call_f16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                            int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                             int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_fp8_f16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_fp8_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                 int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_e5m2_f16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                 int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_e5m2_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                 int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_int8_f16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                 int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_int8_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                 int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_e4m3i4_f16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                   int64_t *launches, DecodeShape *shape);
cudaError_t decode_call_e4m3i4_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                                    int64_t *launches, DecodeShape *shape);

// Tensor-core variant (head_dim 128 only); tmk / tmv map the K and V pools as
// 2D [rows = num_blocks * num_kv_heads * block_size][128 elements] with
// 128-byte swizzle (a 4-bit V pool is read by plain bulk copies; its tmv is
// not used).
cudaError_t decode_mma_call_f16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                 const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_fp8_f16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                    const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_fp8_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                     const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_e5m2_f16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                     const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_e5m2_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                     const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_int8_f16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                     const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_int8_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                     const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_e4m3i4_f16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                       const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);
cudaError_t decode_mma_call_e4m3i4_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                                        const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape);

// Prefix kernel (head_dim 128): grid = the groups' units; tmk / tmv as for the tensor-core decode.
#define PKV_PREFIX_DECL(SUF)                                                                        \
  cudaError_t prefix_call_##SUF(int group, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk, \
                                const CUtensorMap *tmv, int grid);
PKV_PREFIX_DECL(f16)
PKV_PREFIX_DECL(bf16)
PKV_PREFIX_DECL(fp8_f16)
PKV_PREFIX_DECL(fp8_bf16)
PKV_PREFIX_DECL(e5m2_f16)
PKV_PREFIX_DECL(e5m2_bf16)
PKV_PREFIX_DECL(int8_f16)
PKV_PREFIX_DECL(int8_bf16)
PKV_PREFIX_DECL(e4m3i4_f16)
PKV_PREFIX_DECL(e4m3i4_bf16)
#undef PKV_PREFIX_DECL

// Prefix kernel on tcgen05 tensor cores (decode_prefix_umma.cuh): 16-bit caches
// with a query of the same type, head_dim 128.
cudaError_t prefix_umma_call_f16(int group, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                                 const CUtensorMap *tmv, int grid);
cudaError_t prefix_umma_call_bf16(int group, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                                  const CUtensorMap *tmv, int grid);

// The process-wide prefix-kernel choice (pkv_set_prefix_kernel): whether a
// cascade over a cache of this type runs the tcgen05 kernel, and the tiles
// one of its CTAs attends.
bool prefix_uses_umma(pkv_dtype q_dtype, pkv_dtype cache_dtype);
int32_t prefix_umma_chunk_tiles();

// paged_attention_decode (k_new == v_new == NULL) or
// paged_attention_decode_append, with a choice of launch: programmatic ==
// true lets the kernel start while the stream's previous kernel finishes.
// Only for callers that know that kernel writes neither the block tables nor
// the context lengths (the decode kernel reads those before it waits).
// `epoch` >= 0 is one the caller reserved with take_epochs; -1 takes the
// workspace's next one.  `host_lens`: optional host copy of context_lens,
// passed in the launch parameters when the batch is small enough.  `plan`:
// optional cascade (tensor-core path only): the prefix kernel runs first and
// the decode folds its partials in.
// programmatic: 0 ordinary launch; 1 programmatic dependent of the stream's
// previous kernel; 2 the same, and that kernel writes no K/V cache memory.
pkv_status attention_decode(int programmatic, const void *k_new, const void *v_new, void *out, pkv_dtype out_dtype,
                            const void *q, pkv_dtype q_dtype,
                            const void *k_cache, const void *v_cache, pkv_dtype cache_dtype, const float *k_scale,
                            const float *v_scale, const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                            int32_t block_size, float scale, void *workspace, size_t workspace_bytes,
                            int32_t *d_error, pkv_stream_t stream, int64_t epoch = -1,
                            const int32_t *host_lens = nullptr, const CascadePlan *plan = nullptr);

// The calling thread's launch count (pkv_launch_count), adjusted by `delta`:
// a stream capture records launches that run only when the graph is replayed.
void add_launches(int64_t delta);

// Reserve `count` consecutive epochs (counter-bank numbers) of a decode
// workspace for calls the caller issues itself, the first in *first; clear
// the split counters on `stream` first if a call with these shapes would
// (the workspace's first call, or new shapes), so that a stream capture of
// those calls records no clearing.
pkv_status take_epochs(void *workspace, int32_t num_seqs, int32_t num_kv_heads, int32_t count,
                       cudaStream_t stream, uint32_t *first);

}  // namespace pkv
