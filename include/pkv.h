/*
 * pkv.h -- C ABI of the GB300 paged KV cache decode library (libpkv.so).
 *
 * The calls follow the pages' statement of the problem ("KV Cache 与 vLLM"
 * (zwxr.cn) §3.1-§3.4; "KV Cache优化实战" §4.2): the KV cache is cut into
 * fixed physical blocks of 16 tokens, taken on demand; each sequence keeps a
 * block table (logical block -> physical block); sequences with a common
 * prefix share physical blocks and copy a shared block on write; a finished
 * sequence's blocks are freed at once; every decode step appends the new
 * token's K/V and the new query attends over the sequence's cache through
 * its table.  Running out of blocks must not crash a request
 * ("企业官网建设流程全解析" §6.4): the allocator fails the whole request with
 * PKV_ERR_NO_BLOCKS and changes nothing.
 *
 * Conventions shared by every call:
 *  - Every call returns a pkv_status.  Host calls validate their arguments and
 *    leave all state unchanged on error.  pkv_last_error() gives a one-line
 *    reason for the calling thread's last failure.
 *  - Device calls take device pointers owned by the caller (the library never
 *    allocates device memory), enqueue kernels on `stream` and do not
 *    synchronise.  Launch errors are returned at once; errors that depend on
 *    device data (a slot or block id outside the pool, a context length
 *    beyond the table) are OR-ed into the caller's device word `d_error`
 *    (int32, may be NULL) as PKV_DEVERR_* bits and read back with
 *    pkv_read_device_error().  A kernel that finds such an error skips the
 *    offending access; it never traps.
 *  - Device arrays are dense and row-major in the shapes stated, and every
 *    device pointer must be 16-byte aligned.
 *  - Cache layout, per layer: k_cache, v_cache
 *    [num_blocks][num_kv_heads][block_size][head_dim] (the V cache of
 *    FP8_E4M3_INT4 holds head_dim / 2 bytes a row); coded caches
 *    (FP8_E4M3, FP8_E5M2, INT8, FP8_E4M3_INT4) also have one float32 scale
 *    array [num_blocks][num_kv_heads][2][block_size]: a (block, head)'s K
 *    scales, then its V scales.  Calls take it as k_scale (its start) and
 *    v_scale, which must be k_scale + block_size, and fail with
 *    PKV_ERR_INVALID otherwise.  With 16-token blocks the K and V scales of
 *    a block's tokens are then one 128-byte unit, read with one copy.
 *    block_size is 16 or 32.
 *    Token n of a sequence lives at slot
 *    table[n / block_size] * block_size + n % block_size.
 *  - Several layers are several calls with per-layer cache pointers.
 *  - Not thread-safe per block manager handle.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID = -1,      /* bad argument, unknown sequence or block, misaligned pointer */
  PKV_ERR_NO_BLOCKS = -2,    /* the free list cannot cover the request; nothing changed */
  PKV_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
  PKV_ERR_UNSUPPORTED = -4,  /* head_dim / group size / dtype combination not built */
  PKV_ERR_DEVICE_CHECK = -5, /* pkv_read_device_error found a PKV_DEVERR_* bit set */
  PKV_ERR_WORKSPACE = -6     /* workspace smaller than paged_attention_workspace_bytes */
} pkv_status;

/* Element types.  F16 / BF16: queries, new K/V rows, 16-bit caches.  F32:
 * decode output only.  FP8_E4M3, FP8_E5M2, INT8: one-byte cache codes with
 * one fp32 scale per (token, KV head) ("KV Cache优化实战" §3.2-§3.3 names
 * fp8_e4m3, fp8_e5m2 and 8-bit integer caches, and prefers per-token /
 * per-head scales to one scale per tensor).
 *
 * FP8_E4M3_INT4: the mixed scheme of "KV Cache优化实战" §3.2 (8-bit keys,
 * 4-bit values).  The K cache holds E4M3 codes exactly as FP8_E4M3 does.
 * The V cache holds symmetric 4-bit integers, two a byte: a V row is
 * head_dim / 2 bytes, element 2i in the low nibble of byte i, each nibble
 * code + 8 with code = nearest integer (ties to even) of x / scale clamped
 * to [-7, 7], scale = amax / 7 (1 for an all-zero row).  So a V pool is
 * [num_blocks][num_kv_heads][block_size][head_dim / 2] bytes; both halves
 * keep one fp32 scale per (token, KV head). */
typedef enum {
  PKV_F16 = 0,
  PKV_BF16 = 1,
  PKV_FP8_E4M3 = 2,
  PKV_F32 = 3,
  PKV_FP8_E5M2 = 4,
  PKV_INT8 = 5,
  PKV_FP8_E4M3_INT4 = 6
} pkv_dtype;

/* Bits a kernel ORs into *d_error. */
#define PKV_DEVERR_BAD_SLOT 1        /* append: slot >= num_blocks * block_size */
#define PKV_DEVERR_BAD_BLOCK 2       /* copy / decode: block id outside [0, num_blocks) */
#define PKV_DEVERR_BAD_CONTEXT_LEN 4 /* decode: context_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_WAIT_TIMEOUT 8    /* decode: a staging wait ran out its iteration limit */

/* Tokens per physical block ("KV Cache 与 vLLM" §3.1: 16 by default; §4.2
 * and "KV Cache优化实战" §7.5 treat it as a tuning knob).  Pools, tables and
 * the device calls take a block_size of 16 (PKV_BLOCK_SIZE) or 32; the
 * kernels work on 16-token tiles, two per 32-token block. */
#define PKV_BLOCK_SIZE 16
#define PKV_BLOCK_SIZE_32 32
#define PKV_MAX_SEQS_PER_CALL 1024   /* paged_attention_decode batch limit */

/* ------------------------------------------------------------------------ */
/* Host block manager (pages: "KV Cache 与 vLLM" §3.1-§3.4).                  */
/*                                                                          */
/* Free list: FIFO, initialised to alloc_order (NULL = 0..num_blocks-1); a  */
/* block is taken from the head and returned to the tail.  A block is       */
/* shared while its reference count exceeds 1.                              */
/* ------------------------------------------------------------------------ */
typedef struct pkv_bm pkv_bm;

/* num_blocks > 0; block_size 16 or 32; alloc_order (may be NULL) is a
 * permutation of 0..num_blocks-1 copied by the call.  *out owns host memory
 * released by pkv_bm_destroy. */
pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *alloc_order,
                         pkv_bm **out);
void pkv_bm_destroy(pkv_bm *bm);

/* Take one block from the free list (its count becomes 1); with the prefix
 * cache on and the free list empty, evict a cached block (see below). */
pkv_status kv_block_alloc(pkv_bm *bm, int32_t *block_id);
/* Drop one reference; at 0 the block joins the tail of the free list (or,
 * if it is registered in the prefix cache, stays cached). */
pkv_status kv_block_free(pkv_bm *bm, int32_t block_id);

/* New empty sequence; seq_id must not exist. */
pkv_status pkv_seq_create(pkv_bm *bm, int64_t seq_id);
/* child gets a copy of parent's table and length; every block gains one
 * reference (prefix sharing, "KV Cache 与 vLLM" §3.3). */
pkv_status pkv_seq_fork(pkv_bm *bm, int64_t parent, int64_t child);
/* Drop the sequence's references in logical order (freed blocks join the
 * free list in that order) and forget the sequence. */
pkv_status pkv_seq_free(pkv_bm *bm, int64_t seq_id);

/* Append one token to each seq_ids[i], in order (a sequence may repeat).
 * With bs the manager's block size (16 or 32) and n the sequence's length:
 * if n % bs == 0 a block is taken from the free list and added to its table;
 * else if its last block is shared, a new block is taken, the pair
 * (old -> new) is recorded in cow_src/cow_dst and the old block loses one
 * reference (copy-on-write; the last holder writes in place).
 * slot_mapping[i] = table[n / bs] * bs + n % bs, then n becomes n + 1.
 * Arrays: seq_ids[n], slot_mapping[n], cow_src[n], cow_dst[n] (host memory);
 * *num_cow receives the number of pairs.  All-or-nothing: returns
 * PKV_ERR_NO_BLOCKS, with nothing changed, when the free list cannot cover
 * every block the batch needs. The caller must copy each pair (old -> new)
 * with paged_kv_copy_blocks before writing the new tokens. */
pkv_status pkv_seq_append_slots(pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                                int32_t *slot_mapping, int32_t *cow_src, int32_t *cow_dst,
                                int32_t *num_cow);

/* Export block tables: tables[i][j] = physical block of logical block j of
 * seq_ids[i], -1 past the end (host int32 [n][max_blocks]); context_lens[i]
 * = its token count (host int32 [n]).  PKV_ERR_INVALID if a table is longer
 * than max_blocks. */
pkv_status pkv_build_block_tables(const pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                                  int32_t max_blocks, int32_t *tables, int32_t *context_lens);

/* Blocks a request can take: the free list plus cached, unreferenced blocks. */
int32_t pkv_bm_num_free(const pkv_bm *bm);
int32_t pkv_bm_num_blocks(const pkv_bm *bm);
int32_t pkv_bm_block_size(const pkv_bm *bm);
/* The free list in FIFO order: writes min(cap, free) ids to out, *n = free. */
pkv_status pkv_bm_free_list(const pkv_bm *bm, int32_t *out, int32_t cap, int32_t *n);
pkv_status pkv_bm_refcount(const pkv_bm *bm, int32_t block_id, int32_t *count);
pkv_status pkv_seq_len(const pkv_bm *bm, int64_t seq_id, int32_t *len);

/* ------------------------------------------------------------------------ */
/* Automatic prefix caching ("KV Cache优化实战" §5.2: cached blocks keyed by */
/* a content hash, reused block by block when a new request's prefix        */
/* matches token for token; "企业官网建设流程全解析" §6.2: the key covers    */
/* the model, the token ids and the configuration; §6.3: eviction follows   */
/* the hash chain, since a block's later tokens depend on earlier ones).    */
/*                                                                          */
/* Needs a block manager with 16-token blocks.                              */
/* Only full blocks are cached.  Block j of a prompt is keyed by the chain  */
/* h_j = pkv_block_hash(h_{j-1}, tokens[16j .. 16j+16), config_key),        */
/* h_{-1} = 0; a hit also compares the stored token ids.  A registered      */
/* block whose references drop to 0 stays cached and counts as free         */
/* capacity; the free list is used first, then the cached unreferenced      */
/* block with no cached child is evicted (least recently used -- by the     */
/* admit, commit or release call that last touched it --, then the deepest, */
/* then the lowest id), so no cached block loses a block it depends on.     */
/* ------------------------------------------------------------------------ */

/* FNV-1a 64 (offset basis 0xcbf29ce484222325, prime 0x100000001b3) over
 * parent_hash (8 bytes little-endian), tokens[0..16) (4 bytes each,
 * little-endian two's complement) and config_key (8 bytes little-endian). */
uint64_t pkv_block_hash(uint64_t parent_hash, const int32_t *tokens, uint64_t config_key);

/* Turn the prefix cache on (once per block manager); config_key stands for
 * the model and the settings that change the cached K/V. */
pkv_status pkv_bm_enable_prefix_cache(pkv_bm *bm, uint64_t config_key);

/* Create seq_id for a prompt of num_tokens token ids (host int32) and map
 * the longest chain of cached blocks that matches it, at most
 * (num_tokens - 1) / 16 blocks so that at least one prompt token is
 * computed.  Each mapped block gains a reference.  *num_cached = tokens
 * mapped (the sequence's length, a multiple of 16); the caller appends and
 * writes the rest of the prompt. */
pkv_status pkv_seq_admit(pkv_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens,
                         int32_t *num_cached);

/* Register the full blocks among the first num_tokens tokens of seq_id
 * (num_tokens <= its length; tokens are its token ids, host int32) once
 * their K/V are written.  Registration follows the chain from block 0 and
 * stops at the first block whose key is already held by another block (that
 * block and the rest stay private).  *num_registered (may be NULL) = blocks
 * newly registered. */
pkv_status pkv_seq_commit_prefix(pkv_bm *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens,
                                 int32_t *num_registered);

typedef struct {
  int64_t lookups;    /* full prompt blocks looked up by pkv_seq_admit */
  int64_t hits;       /* of those, reused */
  int64_t evictions;  /* cached blocks evicted to serve allocations */
  int64_t registered; /* blocks in the cache now */
  int64_t evictable;  /* of those, unreferenced */
} pkv_prefix_stats;
pkv_status pkv_prefix_cache_stats(const pkv_bm *bm, pkv_prefix_stats *out);

/* ------------------------------------------------------------------------ */
/* Sizing ("KV Cache优化实战" §2.1: bytes = 2 x layers x kv_heads x head_dim */
/* x tokens x bytes per element).  Coded caches add one fp32 scale per      */
/* (token, KV head) for K and for V; FP8_E4M3_INT4 counts one byte per K    */
/* element and half a byte per V element.  Returns -1 on a bad argument.    */
/* ------------------------------------------------------------------------ */
int64_t pkv_kv_bytes(int32_t layers, int32_t kv_heads, int32_t head_dim, int64_t tokens,
                     pkv_dtype cache_dtype);
/* Whole blocks of block_size (16 or 32) tokens a byte budget buys for all
 * layers' K, V (and scales). */
int64_t pkv_pool_blocks(int64_t budget_bytes, int32_t layers, int32_t kv_heads, int32_t head_dim,
                        pkv_dtype cache_dtype, int32_t block_size);

/* ------------------------------------------------------------------------ */
/* Device calls                                                              */
/* ------------------------------------------------------------------------ */

/* Copy-on-write block copy ("KV Cache 与 vLLM" §3.3): for each pair i, copy
 * all block_size slots of physical block src[i] to dst[i] in k_cache and
 * v_cache (and k_scale / v_scale for coded caches; NULL otherwise).
 * src, dst: device int32 [num_pairs]; ids outside [0, num_blocks) set
 * PKV_DEVERR_BAD_BLOCK and that pair is skipped. */
pkv_status paged_kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                                const int32_t *src, const int32_t *dst, int32_t num_pairs,
                                int32_t num_kv_heads, int32_t head_dim, pkv_dtype cache_dtype,
                                int32_t num_blocks, int32_t block_size, int32_t *d_error,
                                pkv_stream_t stream);

/* Reshape-and-cache ("KV Cache 与 vLLM" §1.3 append; "企业官网建设流程全解析"
 * §3.2): token t's rows k[t], v[t] ([num_kv_heads][head_dim], in_dtype
 * F16 or BF16) are written to slot slot_mapping[t] (device int32
 * [num_tokens]; -1 skips the token; >= num_blocks * block_size sets
 * PKV_DEVERR_BAD_SLOT and skips it).
 * 16-bit caches: cache_dtype must equal in_dtype; the copy is exact.
 * One-byte caches ("KV Cache优化实战" §3.2-§3.3, per-token per-head scale):
 * per (token, KV head) amax = max |x| over head_dim, scale = amax / R in
 * IEEE fp32 (1 when amax == 0) and code = Q(x / scale) with an IEEE fp32
 * division, where
 *   FP8_E4M3: R = 448,   Q = nearest E4M3 code, ties to even, saturating;
 *   FP8_E5M2: R = 57344, Q = nearest E5M2 code, ties to even, saturating;
 *   INT8:     R = 127,   Q = nearest integer, ties to even, clamped to
 *             [-127, 127], stored as the byte Q + 128 (zero point 128);
 *   FP8_E4M3_INT4: K rows as FP8_E4M3; V rows R = 7, Q = nearest integer,
 *             ties to even, clamped to [-7, 7], stored two a byte as
 *             code + 8 (even element in the low nibble);
 * the scale of slot (block, offset), head h goes to
 * k_scale[((block * num_kv_heads + h) * 2) * block_size + offset] (K) and
 * to v_scale at the same index (V). */
pkv_status paged_kv_append(const void *k, const void *v, pkv_dtype in_dtype, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t *slot_mapping,
                           void *k_cache, void *v_cache, pkv_dtype cache_dtype, float *k_scale,
                           float *v_scale, int32_t num_blocks, int32_t block_size, int32_t *d_error,
                           pkv_stream_t stream);

/* Which decode kernel runs.  SIMT: CUDA-core dot products (any head_dim).
 * MMA: tensor-core mma.sync m16n8k16 tiles fed by swizzled tensor TMA
 * (head_dim 128; other head_dims use SIMT).  AUTO (default) picks MMA for
 * head_dim 128.  Process-wide; affects calls issued after it. */
typedef enum { PKV_DECODE_AUTO = 0, PKV_DECODE_SIMT = 1, PKV_DECODE_MMA = 2 } pkv_decode_kernel;
pkv_status pkv_set_decode_kernel(pkv_decode_kernel kind);
pkv_decode_kernel pkv_get_decode_kernel(void);

/* Which kernel attends the shared prefixes of the step executor's cascade
 * ("KV Cache 与 vLLM" §3.3, "KV Cache优化实战" §5.2; see pkv_stepper_use_cascade).
 * MMA_SYNC: warp-level mma.sync m16n8k16 over 16-token tiles, any cache
 * type.  TCGEN05: fifth-generation tensor-core MMAs (tcgen05, accumulators
 * in tensor memory) over 64-token sub-chunks, for f16 / bf16 caches with a
 * query of the same type (other caches keep MMA_SYNC).  AUTO (default):
 * MMA_SYNC, the faster of the two on the measured workloads.
 * chunk_tiles: 16-token tiles a tcgen05 CTA attends (the prefix is cut into
 * ceil(tiles / chunk_tiles) chunks, at most 16); 0 keeps the default (16).
 * Process-wide; affects steps issued after it.  PKV_ERR_INVALID for an
 * unknown kind or a chunk_tiles outside [0, 4096]. */
typedef enum { PKV_PREFIX_AUTO = 0, PKV_PREFIX_MMA_SYNC = 1, PKV_PREFIX_TCGEN05 = 2 } pkv_prefix_kernel;
pkv_status pkv_set_prefix_kernel(pkv_prefix_kernel kind, int32_t chunk_tiles);
pkv_prefix_kernel pkv_get_prefix_kernel(void);

/* Device workspace (bytes) paged_attention_decode needs for these shapes on
 * the current device (split-KV partials and per-(sequence, KV head)
 * counters).  Depends on the device's SM count.  Fill a new workspace with
 * zeros once before its first use; after that it can be reused by any
 * number of calls (serialised on the GPU) without clearing, also with other
 * shapes (a call whose shapes differ from the previous call on the same
 * workspace clears the counters itself with one cudaMemsetAsync). */
pkv_status paged_attention_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           pkv_dtype q_dtype, pkv_dtype cache_dtype,
                                           size_t *bytes);

/* PagedAttention decode ("企业官网建设流程全解析" §1.2: softmax(q K^T * scale)
 * V; "KV Cache 与 vLLM" §3.2: through the block table, reading only the
 * sequence's blocks).  For sequence b and query head h, with G =
 * num_q_heads / num_kv_heads and KV head h / G:
 *   out[b][h] = sum_j softmax_j(scale * <q[b][h], K_j>) V_j
 * over tokens j < context_lens[b] (the token appended this step included).
 * q: [num_seqs][num_q_heads][head_dim] in q_dtype (F16 / BF16); out: same
 * shape in out_dtype, either F32 (the fp32 accumulator result) or q_dtype
 * (that result rounded once to nearest even).  Caches F16 or BF16 (q_dtype must match) or
 * coded (FP8_E4M3, FP8_E5M2, INT8, FP8_E4M3_INT4: code value x scale,
 * dequantised in the kernel with k_scale / v_scale).
 * block_tables: device int32 [num_seqs][max_blocks_per_seq]; context_lens:
 * device int32 [num_seqs]; max_context_len bounds every context_len.
 * A context_len of 0 gives a zero output.  Work is split across the GPU
 * in equal shares of (sequence, KV head, 16-token block) tiles; shares that
 * cover part of a sequence leave fp32 partials in `workspace` (at least
 * paged_attention_workspace_bytes, zero-filled before its first use); the
 * warp that stores the last partial of a (sequence, KV head) merges them by
 * log-sum-exp in the same kernel.
 * Supported: head_dim 64 or 128; G in {1, 2, 4, 8}; num_seqs <=
 * PKV_MAX_SEQS_PER_CALL. */
pkv_status paged_attention_decode(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                  const void *k_cache,
                                  const void *v_cache, pkv_dtype cache_dtype, const float *k_scale,
                                  const float *v_scale, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens,
                                  int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                  int32_t block_size, float scale, void *workspace, size_t workspace_bytes,
                                  int32_t *d_error, pkv_stream_t stream);

/* Append and decode in one launch ("KV Cache 与 vLLM" §1.3: every step
 * appends the new token's K/V, then the query attends over the whole
 * cache).  Same arguments and result as paged_attention_decode, plus the new
 * rows: k_new, v_new [num_seqs][num_kv_heads][head_dim] in q_dtype, row b
 * written at position context_lens[b] - 1 of sequence b (the last token
 * the table covers) exactly as paged_kv_append would write it (16-bit copy,
 * or one-byte codes with the scale to k_scale / v_scale), before the
 * attention reads that block.  The caller has already grown the tables
 * (pkv_seq_append_slots) and copied any shared block it writes into
 * (paged_kv_copy_blocks).  The cache pointers are written. */
pkv_status paged_attention_decode_append(void *out, pkv_dtype out_dtype, const void *q, pkv_dtype q_dtype,
                                         const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                                         pkv_dtype cache_dtype, float *k_scale, float *v_scale,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, int32_t block_size, float scale, void *workspace,
                                         size_t workspace_bytes,
                                         int32_t *d_error, pkv_stream_t stream);

/* Decode without a workspace argument, for callers that cannot allocate
 * device memory: a plugin whose host framework owns every device
 * allocation, or a latency-critical loop where an allocation could
 * synchronise the device.  The pages have no counterpart of this call; it
 * is a packaging variant of paged_attention_decode with the same arguments
 * (minus workspace / workspace_bytes) and the same results.
 * Scratch: a PKV_STATIC_SCRATCH_BYTES (16 MiB) __device__ buffer inside the
 * library; every GPU that loads the library holds one until the process
 * exits.  Shapes whose paged_attention_workspace_bytes exceeds it return
 * PKV_ERR_WORKSPACE with the size in pkv_last_error().  The call allocates
 * nothing.  Its first call on a device looks up the buffer's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  The split counters in the buffer are cleared
 * on the caller's stream by the same per-workspace rule as
 * paged_attention_decode (first call on the buffer, or a change of
 * num_seqs / num_kv_heads); nothing else in it needs an initial value.  All
 * calls on a device share the buffer and it keeps the last call's contents;
 * calls whose kernels overlap on the GPU race, so serialise them. */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)
pkv_status paged_attention_decode_static(void *out, pkv_dtype out_dtype, const void *q,
                                         pkv_dtype q_dtype, const void *k_cache, const void *v_cache,
                                         pkv_dtype cache_dtype, const float *k_scale,
                                         const float *v_scale, const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *context_lens,
                                         int32_t max_context_len, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, int32_t block_size, float scale, int32_t *d_error,
                                         pkv_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Decode step executor: one call runs a whole decode step of a batch        */
/* ("KV Cache 与 vLLM" §3.1-§3.4, "企业官网建设流程全解析" §3.2): the block    */
/* manager gives every sequence a slot (taking or copying blocks), the slot   */
/* mapping, copy pairs, lengths and block tables are written to page-locked   */
/* host staging that the first layer's kernels read in place (with more than  */
/* one layer, one small kernel also copies them to device memory for the     */
/* later layers), and for every layer the shared blocks are copied, the new   */
/* K/V rows are written and the new queries attend.  Host work is             */
/* O(batch + table size); all device work is enqueued on `stream`.            */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t num_layers, num_blocks, num_kv_heads, num_q_heads, head_dim;
  pkv_dtype q_dtype, cache_dtype;
  void *k_cache, *v_cache;          /* layer 0; layer l at + l * cache_layer_stride bytes */
  int64_t cache_layer_stride;
  float *k_scale, *v_scale;         /* coded caches only (else NULL): v_scale = k_scale + block_size;
                                       layer l at + l * scale_layer_stride bytes */
  int64_t scale_layer_stride;
  int32_t block_size;               /* 16 or 32: must match the block manager's */
  int64_t v_cache_layer_stride;     /* V layer stride in bytes; 0: the same as cache_layer_stride */
} pkv_pool_desc;

typedef struct pkv_stepper pkv_stepper;

/* Bytes of pinned host staging and of device metadata a stepper needs for
 * batches of up to max_seqs sequences of up to max_blocks_per_seq blocks
 * (both double-buffered). */
size_t pkv_stepper_host_bytes(int32_t max_seqs, int32_t max_blocks_per_seq);
size_t pkv_stepper_device_bytes(int32_t max_seqs, int32_t max_blocks_per_seq);

/* All buffers are caller-owned and must outlive the stepper: host_staging
 * page-locked host memory (cudaHostAlloc / cudaHostRegister, or a pinned
 * tensor) of pkv_stepper_host_bytes, read by kernels in place through its
 * device address; dev_meta device memory of pkv_stepper_device_bytes; both
 * 16-byte aligned; workspace of paged_attention_workspace_bytes(max_seqs, ...)
 * (zero-filled once).  The pool descriptor is copied.  The stepper creates
 * two events and nothing else.  Each step uses one half of the staging and of
 * dev_meta, alternating; a step waits (on the host) until the step two calls
 * earlier, which used the same half, has finished on the device, and (when
 * that step ran on another stream) makes `stream` wait for it too.
 * pkv_stepper_destroy waits for the last steps before it returns. */
pkv_status pkv_stepper_create(const pkv_pool_desc *pool, int32_t max_seqs, int32_t max_blocks_per_seq,
                              int32_t *host_staging, size_t host_staging_bytes, int32_t *dev_meta,
                              size_t dev_meta_bytes, void *workspace, size_t workspace_bytes,
                              pkv_stepper **out);
void pkv_stepper_destroy(pkv_stepper *st);

/* One decode step for seq_ids[0..n) (distinct).  Per layer l (byte strides):
 * k_new, v_new + l * kv_layer_stride: [n][num_kv_heads][head_dim] rows of
 * the new token in q_dtype (stride 0 reuses one tensor for every layer);
 * q + l * q_layer_stride: [n][num_q_heads][head_dim] in q_dtype;
 * out + l * out_layer_stride: same shape in out_dtype (F32 or q_dtype).
 * k_new, v_new and q are device memory (the kernels bulk-copy them); out
 * may also be page-locked host memory, which the kernels store to directly.
 * Validated before anything changes: n <= max_seqs, every table stays within
 * max_blocks_per_seq.  PKV_ERR_NO_BLOCKS leaves the block manager as it was.
 * The copy pairs of the step are written to cow_src / cow_dst (host, [n],
 * may be NULL) and their number to *num_cow (may be NULL).  Every layer's
 * copies and appends are enqueued before the first layer's attention; the
 * optional CUDA events attn_begin / attn_end (cudaEvent_t, may be NULL) are
 * recorded on `stream` just before the first and just after the last
 * attention launch (the metadata copy of a multi-layer step included), so a
 * caller can time the attention alone. */
pkv_status pkv_stepper_step(pkv_stepper *st, pkv_bm *bm, const int64_t *seq_ids, int32_t n,
                            const void *k_new, const void *v_new, int64_t kv_layer_stride,
                            const void *q, int64_t q_layer_stride, void *out, pkv_dtype out_dtype,
                            int64_t out_layer_stride, float scale, int32_t *cow_src, int32_t *cow_dst,
                            int32_t *num_cow, int32_t *d_error, void *attn_begin, void *attn_end,
                            pkv_stream_t stream);

/* CUDA-graph replay of the step's attention launches ("KV Cache 与 vLLM"
 * §4.2: CUDA graphs instead of eager launches).  With enable != 0, a step
 * without copy-on-write copies launches one graph instead of its kernels:
 * the metadata copy (more than one layer) and every layer's fused append +
 * attention.  One graph is kept per metadata half; it is captured on a
 * private stream the first time and captured again when the step's batch
 * size, buffers (k_new, v_new, q, out, d_error), their strides, out_dtype or
 * scale differ from those it was captured with, so replays pay off when the
 * caller reuses its buffers from step to step (the usual pattern around
 * graphs).  While enabled, a step's block tables are as wide as the next
 * power of two of its longest table (at most max_blocks_per_seq), and a
 * graph is also captured again when that width changes.  Results are those
 * of eager steps.  Steps with copy-on-write
 * copies run eagerly.  Disabling frees the graphs.  The capture counts as no
 * launch; each replay adds its kernels to pkv_launch_count. */
pkv_status pkv_stepper_use_graphs(pkv_stepper *st, int32_t enable);
/* Cascade for shared prefixes (on by default; head_dim 128 with the
 * tensor-core decode, eager steps of up to 128 sequences).  Sequences whose
 * block tables start with the same physical blocks (forks, prefix-cache
 * hits) form a group; when their common leading blocks that lie wholly
 * before each member's last token make at least 16 tiles of 16 tokens, a
 * prefix kernel streams those tiles once per KV head and attends them for
 * every member's queries (up to 128 query rows a CTA), leaving fp32
 * partials; the decode then attends each member's remaining tiles and merges
 * the partials in.  The result is the same softmax, summed in another order.
 * pkv_stepper_cascade_count: steps that used it. */
pkv_status pkv_stepper_use_cascade(pkv_stepper *st, int32_t enable);
int64_t pkv_stepper_cascade_count(const pkv_stepper *st);

/* Graphs captured and replayed so far by this stepper. */
pkv_status pkv_stepper_graph_stats(const pkv_stepper *st, int64_t *captures, int64_t *replays);

/* Synchronise `stream`, copy *d_error to *h_error and, if clear != 0, zero
 * it.  Returns PKV_ERR_DEVICE_CHECK when any bit was set. */
pkv_status pkv_read_device_error(int32_t *d_error, int32_t *h_error, int32_t clear,
                                 pkv_stream_t stream);

/* Several copies in one kernel launch, for step inputs and outputs that live
 * in page-locked host memory: the kernel reads and writes them in place over
 * the host link (16-byte vectors), so one launch replaces a memcpy per
 * tensor.  dst and src: device memory or page-locked host memory
 * (cudaHostAlloc / cudaHostRegister, or a pinned tensor), 16-byte aligned;
 * bytes a multiple of 16; segments must not overlap.  At most
 * PKV_MAX_COPY_SEGMENTS segments a call; enqueued on `stream`.  A decode
 * launched after it as a programmatic dependent (the step executor's) may
 * start its prologue during the copy. */
#define PKV_MAX_COPY_SEGMENTS 8
typedef struct {
  void *dst;
  const void *src;
  int64_t bytes;
} pkv_copy_segment;
pkv_status pkv_copy_segments(const pkv_copy_segment *segs, int32_t num_segs, pkv_stream_t stream);

/* Register the next pkv_stepper_step's host-to-device input copies (its
 * k_new, v_new and q rows living in page-locked host memory; the step is
 * given the device copies).  The step launches them as one
 * pkv_copy_segments kernel after its host work (block manager, tables) and
 * right before its first attention launch, so the GPU does not wait for
 * the host between the copy and the attention; the first layer's decode may
 * start its first cache copies while the copy runs (the copy writes no
 * cache).  Same rules as pkv_copy_segments (at most PKV_MAX_COPY_SEGMENTS,
 * 16-byte aligned, sizes multiples of 16; PKV_ERR_INVALID otherwise, nothing
 * registered).  The registration applies to the next step call only, which
 * drops it if it fails before launching; a new call replaces it. */
pkv_status pkv_stepper_copy_inputs(pkv_stepper *st, const pkv_copy_segment *segs, int32_t num_segs);

/* Number of kernel launches the calling thread has made through this
 * library (for launch accounting). */
int64_t pkv_launch_count(void);

const char *pkv_status_string(pkv_status status);
/* One-line reason for the calling thread's last failing call ("" if none). */
const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
