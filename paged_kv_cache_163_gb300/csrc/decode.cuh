// PagedAttention decode: split-KV partial kernel and log-sum-exp reduce.
//
// What is computed ("企业官网建设流程全解析" (KV Cache 原理篇) §1.2, §3.2;
// "KV Cache 与 vLLM" (zwxr.cn) §3.2): for sequence b and query head h
// (KV head h / G), out = softmax(scale * q K^T) V over the sequence's
// context_len cached tokens, reached through its block table.
//
// How (GB300 design, not from the pages):
//  * The work is the list of tiles (sequence, KV head, logical block), each
//    one contiguous [16][head_dim] chunk of K and of V in HBM.  The tiles are
//    flattened (sequence-major, then KV head, then block) and every warp of a
//    persistent grid takes an equal contiguous share, so ragged lengths load
//    balance to one tile.  A share that covers a whole (sequence, KV head)
//    writes the output; one that covers part of it writes an fp32 partial
//    (o, m, l) and counts it in on a per-item counter (one atomic add); the
//    warp that stores the item's last partial merges them by log-sum-exp
//    (flash-decoding style split-KV without a second kernel; nothing waits).
//  * Each warp streams its tiles through a private ring of shared-memory
//    stages filled by bulk asynchronous copies (cp.async.bulk, mbarrier
//    completion), so ~100 KB per SM is in flight with no CTA-wide sync.
//  * The GQA group's G query heads stay in registers (fp32, pre-scaled by
//    scale * log2 e).  Scores: lanes split head_dim, partial dot products are
//    reduced across lanes with a transposing butterfly (G heads reduce in
//    G-1+log2(lanes/G) shuffles), online softmax in base 2.
//  * One-byte tiles are dequantised in registers: the per-token K scale multiplies
//    the score and the per-token V scale folds into the probability.
#pragma once

#include <type_traits>

#include <math.h>

#include "common.cuh"
#include "decode.h"

namespace pkv {

constexpr int round_up_c(int x, int m) { return (x + m - 1) / m * m; }
constexpr int clamp_c(int x, int lo, int hi) { return x < lo ? lo : (x > hi ? hi : x); }

template <int D, int G, int CDT, int QDT>
struct DecodeCfg {
  static constexpr int kWarps = 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int KT = k_part(CDT), VT = v_part(CDT);  // storage types of K and of V
  static constexpr int kEsz = is_code8(KT) ? 1 : 2;         // K bytes per element
  static constexpr int kRow = row_bytes(KT, D);             // bytes of one token's K row
  static constexpr int kVRow = row_bytes(VT, D);            // bytes of one token's V row
  static constexpr int kTile = kBS * kRow;                  // one 16-token (block, head) tile of K
  static constexpr int kVTile = kBS * kVRow;                // ... and of V
  static constexpr int kLPT = (D == 128 && G == 8) ? 16 : 8;  // lanes per token in q.K
  static constexpr int kTPP = 32 / kLPT;                    // tokens per pass
  static constexpr int kPasses = kBS / kTPP;
  static constexpr int kChunk = (kRow / kLPT) < 16 ? (kRow / kLPT) : 16;  // bytes per load
  static constexpr int kNChunk = kRow / (kLPT * kChunk);    // loads per lane per token
  static constexpr int kEPC = kChunk / kEsz;                // elements per load
  static constexpr int kEPT = kEPC * kNChunk;               // q elements per lane
  static constexpr int kDPL = D / 32;                       // output elements per lane
  static constexpr int kVSlice = kVRow / 32;                // V row bytes per lane
  static constexpr int kScale = has_scales(CDT) ? kBS * 4 : 0;
  static constexpr int kQ = G * D * 2;
  static constexpr int kOffV = kTile;
  static constexpr int kOffKS = kTile + kVTile;
  static constexpr int kOffVS = kTile + kVTile + kScale;
  static constexpr int kOffQ = kTile + kVTile + 2 * kScale;
  static constexpr int kNew = 2 * D * 2;                    // fused append: the new token's K and V rows
  static constexpr int kOffNew = kOffQ + kQ;
  static constexpr int kStage = round_up_c(kOffNew + kNew, 128);
  static constexpr int kStages = clamp_c(27900 / kStage, 2, 6);
  static constexpr int kCumBytes = round_up_c((PKV_MAX_SEQS_PER_CALL + 1) * 4, 128);
  static constexpr int kMiscBytes = 128;                    // scan scratch
  static constexpr int kBarBytes = round_up_c(kWarps * kStages * 8, 128);
  static constexpr int kDescBytes = kWarps * 64 * 8;        // two windows of 32 tile descriptors
  static constexpr int kSmem = kCumBytes + kMiscBytes + kBarBytes + kDescBytes + kWarps * kStages * kStage;
  static_assert(G <= kLPT, "group larger than lanes per token");
  static_assert((kBS + 3) * G * 4 <= kTile, "probability buffer must fit in the K tile");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kEPT * kLPT == D, "q.K lane split");
};

// Butterfly over the kLPT lanes of one token: v[G] partial dot products per
// lane in, the full dot product of head (lane % LPT) / (LPT / G) out.
template <int G, int LPT>
__device__ __forceinline__ float reduce_heads(float (&v)[G], int lane) {
  int n = G;
#pragma unroll
  for (int off = LPT / 2; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < n / 2) {
          const float send = up ? v[i] : v[i + n / 2];
          const float keep = up ? v[i + n / 2] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, off);
        }
      }
      n >>= 1;
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], off);
    }
  }
  return v[0];
}

// Context length of sequence b: from the launch parameters when they carry
// the lengths, else from memory.
__device__ __forceinline__ int seq_len(const DecodeParams &p, int b) {
  return p.lens_inline_n ? p.lens_inline[b] : __ldg(p.context_lens + b);
}

// Tile index t -> (sequence, KV head, block) using the exclusive prefix sum
// cum[] of blocks per sequence (in shared memory).
__device__ __forceinline__ int find_seq(const int32_t *cum, int num_seqs, int hkv, int64_t t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(hkv) * cum[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Descriptor of one 16-token tile: x = its row index in the pool divided by
// 16, i.e. ((physical block * Hkv + KV head) * tiles per block + tile within
// the block) (-1 if the block id is invalid); the tile's K rows start at
// k_cache + x * 16 rows, its scales at scale + x * 16.
// y = item << 7 | first << 6 | last << 5 | valid tokens.
__device__ __forceinline__ int2 tile_desc(const DecodeParams &p, const int32_t *cum, int64_t t) {
  const int b = find_seq(cum, p.num_seqs, p.num_kv_heads, t);
  const int nb = cum[b + 1] - cum[b];
  const int64_t r = t - static_cast<int64_t>(p.num_kv_heads) * cum[b];
  const int kvh = static_cast<int>(r / nb);
  const int skip = p.pfx_n ? p.pfx_start[b] : 0;  // tiles the prefix kernel attended
  const int ls = static_cast<int>(r - static_cast<int64_t>(kvh) * nb);
  const int lb = ls + skip;
  const int L = seq_len(p, b);
  const int ntok = min(kBS, L - lb * kBS);
  const int tpb = p.tiles_per_block;
  const int32_t blk = __ldg(p.block_tables + static_cast<int64_t>(b) * p.max_blocks_per_seq + lb / tpb);
  int32_t x = -1;
  if (blk < 0 || blk >= p.num_blocks) {
    report(p.d_error, PKV_DEVERR_BAD_BLOCK);
  } else {
    x = (blk * p.num_kv_heads + kvh) * tpb + lb % tpb;
  }
  const int item = b * p.num_kv_heads + kvh;
  return make_int2(x, (item << 7) | ((ls == 0) << 6) | ((ls == nb - 1) << 5) | ntok);
}

// CTA prologue shared by the decode kernels, reading only the context lengths:
// blocks per sequence (validating every length), their exclusive prefix sum
// cum[0..num_seqs] in shared memory, and each warp's kStages stage barriers.
template <int kWarps, int kStages>
__device__ __forceinline__ void scan_blocks(const DecodeParams &p, int32_t *cum, int32_t *misc, uint64_t *bars_all) {
  constexpr int kThreads = kWarps * 32;
  constexpr int PER = (PKV_MAX_SEQS_PER_CALL + kThreads - 1) / kThreads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int nbk[PER];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int s = tid * PER + i;
    int nb = 0;
    if (s < p.num_seqs) {
      const int L = seq_len(p, s);
      if (L < 0 || L > p.max_context_len ||
          static_cast<int64_t>(L) > static_cast<int64_t>(p.max_blocks_per_seq) * p.block_size) {
        report(p.d_error, PKV_DEVERR_BAD_CONTEXT_LEN);
      } else {
        nb = (L + kBS - 1) / kBS;
        if (p.pfx_n) nb -= p.pfx_start[s];  // the prefix kernel's tiles (fewer than nb)
      }
    }
    nbk[i] = nb;
    sum += nb;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) misc[warp] = incl;
  if (lane < kStages) mbar_init(bars_all + warp * kStages + lane, 1);
  __syncthreads();
  if (warp == 0) {
    int x = lane < kWarps ? misc[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += n;
    }
    if (lane < kWarps) misc[16 + lane] = x;  // inclusive warp totals
  }
  __syncthreads();
  int run = incl - sum + (warp > 0 ? misc[16 + warp - 1] : 0);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int s = tid * PER + i;
    if (s < p.num_seqs) cum[s] = run;
    run += nbk[i];
  }
  if (tid == 0) cum[p.num_seqs] = misc[16 + kWarps - 1];
  fence_barrier_init();
  __syncthreads();
}

// Global writes of the prologue, after griddep_wait(): the next call's
// counter bank starts from zero (all CTAs share the clearing), and CTA 0
// writes zero output for sequences without tokens (or with an invalid
// length), which read nothing.
template <int kThreads>
__device__ __forceinline__ void publish_scan(const DecodeParams &p, const int32_t *cum, int out_row_elems) {
  const int tid = threadIdx.x;
  const int items = p.num_seqs * p.num_kv_heads;
  uint32_t *other = p.ws_ctr + ((p.epoch & 1) ^ 1) * items;
  for (int i = blockIdx.x * kThreads + tid; i < items; i += gridDim.x * kThreads) other[i] = 0u;
  if (blockIdx.x == 0) {
    for (int s = tid; s < p.num_seqs; s += kThreads) {
      if (cum[s + 1] != cum[s]) continue;
      const size_t base = static_cast<size_t>(s) * out_row_elems;
      for (int e = 0; e < out_row_elems; e += 2) {
        if (p.out_f32) *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.out) + base + e) = make_float2(0.f, 0.f);
        else *reinterpret_cast<uint32_t *>(p.out + (base + e) * 2) = 0u;
      }
    }
  }
}

// Programmatic dependent launch: a decode kernel launched as a dependent may
// start while the previous kernel on the stream finishes; it reads only the
// lengths and tables (which that kernel does not write) before waiting here.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Warps in [w_first, w_last] (the warps whose shares meet an item) that own
// at least one tile; with fewer tiles than warps some own none.
__device__ __forceinline__ int owning_warps(int64_t w_first, int64_t w_last, int64_t total, int64_t nwarps) {
  if (total >= nwarps) return static_cast<int>(w_last - w_first + 1);
  int n = 0;
  for (int64_t w = w_first; w <= w_last; ++w) n += (w * total / nwarps) != ((w + 1) * total / nwarps);
  return n;
}

// First and last warp whose shares meet `item` (tiles start .. start + nb - 1).
__device__ __forceinline__ void item_warps(const int32_t *cum, int hkv, int item, int64_t total, int64_t nwarps,
                                           int64_t &w_first, int64_t &w_last) {
  const int b = item / hkv;
  const int kvh = item - b * hkv;
  const int nb = cum[b + 1] - cum[b];
  const int64_t start = static_cast<int64_t>(hkv) * cum[b] + static_cast<int64_t>(kvh) * nb;
  // warp owning tile t: the w with floor(w T / W) <= t < floor((w + 1) T / W)
  w_first = ((start + 1) * nwarps - 1) / total;
  w_last = ((start + nb) * nwarps - 1) / total;
}

// Called by a whole warp after it stored a partial of `item`: counts it in
// with one atomic add and returns (on every lane) whether this warp stored
// the item's last one.  Counters come in two banks used by alternate calls
// (bank = epoch & 1); every call clears the other bank in its prologue, so
// the next call starts from zero even if this one is cut short.
__device__ __forceinline__ bool count_partial(const DecodeParams &p, int item, int expected) {
  __threadfence();
  __syncwarp();
  int last = 0;
  if ((threadIdx.x & 31) == 0) {
    const int items = p.num_seqs * p.num_kv_heads;
    const uint32_t old = atomicAdd(p.ws_ctr + (p.epoch & 1) * items + item, 1u);
    last = static_cast<int>(old) + 1 == expected;
  }
  last = __shfl_sync(kFull, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// One warp merges the partials of `item`:
// out = sum_w 2^(m_w - M) o_w / sum_w 2^(m_w - M) l_w, M = max_w m_w.
// Partials of other CTAs are read through L2 (ld.global.cg).  One pass over
// chunks of 32 partials: each lane takes one partial's (m, l) per head, the
// chunk maximum updates the running maximum M (earlier sums are rescaled by
// 2^(M_old - M_new)), and then every lane accumulates its head_dim slice of
// the chunk's o rows, kBatch partials at a time with all their loads issued
// before the first use (kLoads vector loads a lane, sized to the caller's
// register budget).  A warp that owns no tile (possible when there are fewer
// tiles than warps) has weight 0 and its slot's contents are ignored.
template <int D, int G, int QDT, int kLoads>
__device__ __noinline__ void merge_item(const DecodeParams &p, int item, int64_t w_first, int64_t w_last,
                                        int64_t total, int64_t nwarps) {
  constexpr int DPL = D / 32;
  constexpr int kBatch = kLoads / G > 0 ? kLoads / G : 1;  // partials in flight per batch
  const int lane = threadIdx.x & 31;
  const bool all_own = total >= nwarps;
  auto owns = [&](int64_t w) { return all_own || (w * total / nwarps) != ((w + 1) * total / nwarps); };
  const int nw = static_cast<int>(w_last - w_first + 1);  // warps' partials
  const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + (w_first + item) * G;  // [k][g] = (m, l)
  const float *po = p.ws_o + (w_first + item) * G * D;                                 // [k][g][D]
  // then the prefix kernel's partials of this item, if any (always valid)
  const int bs = item / p.num_kv_heads;
  const int nx = p.pfx_n ? p.pfx_chunks[bs] : 0;
  const int64_t xs = nx ? p.pfx_base[bs] + static_cast<int64_t>(item - bs * p.num_kv_heads) * nx : 0;
  const float2 *xml = reinterpret_cast<const float2 *>(p.pfx_ml) + xs * G;
  const float *xo = p.pfx_o + xs * G * D;
  const int np = nw + nx;
  if (nx) griddep_wait();  // the prefix kernel, running beside this grid, has finished its partials
  float acc[G][DPL], run_m[G], den[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    run_m[g] = -INFINITY;
    den[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[g][e] = 0.f;
  }
  using Vec = typename std::conditional<DPL == 4, float4, float2>::type;
  Vec v[kBatch][G];
  // o rows of partials k0 + j0 .. k0 + j0 + kBatch - 1 (clamped to the chunk's last)
  auto load_batch = [&](int k0, int j0, int nk) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int kk = k0 + min(j0 + b, nk - 1);  // stays inside the item's slots
      const float *src = (kk < nw ? po + static_cast<int64_t>(kk) * G * D : xo + static_cast<int64_t>(kk - nw) * G * D) +
                         lane * DPL;
#pragma unroll
      for (int g = 0; g < G; ++g) v[b][g] = __ldcg(reinterpret_cast<const Vec *>(src + g * D));
    }
  };
  for (int k0 = 0; k0 < np; k0 += 32) {
    const int k = k0 + lane;
    const int nk = min(32, np - k0);
    const bool mine = k < nw ? owns(w_first + k) : k < np;
    const float2 *mk = k < nw ? ml + static_cast<int64_t>(k) * G : xml + static_cast<int64_t>(k - nw) * G;
    float2 mlk[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mlk[g] = mine ? __ldcg(mk + g) : make_float2(-INFINITY, 0.f);
    load_batch(k0, 0, nk);  // in flight while the weights are formed
    float wk[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float cm = mlk[g].x;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(kFull, cm, o));
      const float nm = fmaxf(run_m[g], cm);
      const float rescale = run_m[g] == -INFINITY ? 0.f : exp2f(run_m[g] - nm);
      run_m[g] = nm;
      den[g] *= rescale;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[g][e] *= rescale;
      wk[g] = mlk[g].x == -INFINITY ? 0.f : exp2f(mlk[g].x - nm);
      den[g] = fmaf(wk[g], mlk[g].y, den[g]);
    }
    for (int j0 = 0; j0 < nk; j0 += kBatch) {
      if (j0 > 0) load_batch(k0, j0, nk);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float w = __shfl_sync(kFull, wk[g], (j0 + b) & 31);
          if (j0 + b >= nk) w = 0.f;
          const float *x = reinterpret_cast<const float *>(&v[b][g]);
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[g][e] = fmaf(w, w != 0.f ? x[e] : 0.f, acc[g][e]);
        }
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den[g] += __shfl_xor_sync(kFull, den[g], o);
  const size_t obase = static_cast<size_t>(item) * G * D + lane * DPL;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float inv = den[g] > 0.f ? 1.f / den[g] : 0.f;
    const size_t at = obase + g * D;
    // one vector store a lane (whole sectors, also into page-locked host memory)
    if constexpr (DPL == 4) {
      if (p.out_f32) {
        *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + at) =
            make_float4(acc[g][0] * inv, acc[g][1] * inv, acc[g][2] * inv, acc[g][3] * inv);
      } else {
        *reinterpret_cast<uint2 *>(p.out + at * 2) =
            make_uint2(pack2<QDT>(acc[g][0] * inv, acc[g][1] * inv), pack2<QDT>(acc[g][2] * inv, acc[g][3] * inv));
      }
    } else {
      if (p.out_f32) {
        *reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.out) + at) =
            make_float2(acc[g][0] * inv, acc[g][1] * inv);
      } else {
        *reinterpret_cast<uint32_t *>(p.out + at * 2) = pack2<QDT>(acc[g][0] * inv, acc[g][1] * inv);
      }
    }
  }
}

// After a warp stored its partial of `item`: count it in; the last one merges.
template <int D, int G, int QDT, int kLoads = 16>
__device__ __forceinline__ void finish_partial(const DecodeParams &p, const int32_t *cum, int item, int64_t total,
                                               int64_t nwarps) {
  int64_t w_first, w_last;
  item_warps(cum, p.num_kv_heads, item, total, nwarps, w_first, w_last);
  if (count_partial(p, item, owning_warps(w_first, w_last, total, nwarps)))
    merge_item<D, G, QDT, kLoads>(p, item, w_first, w_last, total, nwarps);
}

template <int D, int G, int CDT, int QDT>
__global__ void __launch_bounds__(DecodeCfg<D, G, CDT, QDT>::kThreads, 1)
    paged_decode_kernel(const __grid_constant__ DecodeParams p) {
  using C = DecodeCfg<D, G, CDT, QDT>;
  extern __shared__ __align__(128) uint8_t smem[];
  int32_t *cum = reinterpret_cast<int32_t *>(smem);
  int32_t *misc = reinterpret_cast<int32_t *>(smem + C::kCumBytes);
  uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + C::kCumBytes + C::kMiscBytes);
  int2 *desc_all = reinterpret_cast<int2 *>(smem + C::kCumBytes + C::kMiscBytes + C::kBarBytes);
  uint8_t *stage_all = smem + C::kCumBytes + C::kMiscBytes + C::kBarBytes + C::kDescBytes;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  scan_blocks<C::kWarps, C::kStages>(p, cum, misc, bars_all);

  // ---- this warp's share of the tiles --------------------------------------
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * C::kWarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * C::kWarps + warp;
  const int64_t total = static_cast<int64_t>(cum[p.num_seqs]) * p.num_kv_heads;
  const int64_t t0 = gw * total / nwarps;
  const int64_t t1 = (gw + 1) * total / nwarps;
  const int count = static_cast<int>(t1 - t0);

  uint64_t *bars = bars_all + warp * C::kStages;
  int2 *desc = desc_all + warp * 64;
  uint8_t *stages = stage_all + warp * C::kStages * C::kStage;
  const uint64_t pol = policy_evict_first();

  auto fill_window = [&](int w) {  // descriptors of warp-local tiles [32 w, 32 w + 32)
    const int64_t t = t0 + 32 * static_cast<int64_t>(w) + lane;
    int2 d = make_int2(-1, 0);
    if (t < t1) d = tile_desc(p, cum, t);
    desc[(w & 1) * 32 + lane] = d;
  };

  auto issue = [&](int m) {  // lane 0 starts the copies of warp-local tile m
    const int2 d = desc[((m >> 5) & 1) * 32 + (m & 31)];
    if (lane == 0) {
      const int st = m % C::kStages;
      uint8_t *sb = stages + st * C::kStage;
      const int item = d.y >> 7;
      const bool need_q = (m == 0) || ((d.y >> 6) & 1);
      const bool need_new = p.k_new && d.x >= 0 && ((d.y >> 5) & 1);  // the item's last tile: its new token
      const uint32_t bytes =
          (d.x >= 0 ? C::kTile + C::kVTile + 2 * C::kScale : 0) + (need_q ? C::kQ : 0) + (need_new ? C::kNew : 0);
      fence_proxy_async_smem();
      if (bytes == 0) {
        mbar_arrive(bars + st);
      } else {
        mbar_arrive_expect_tx(bars + st, bytes);
        if (d.x >= 0) {
          const size_t tile = static_cast<size_t>(d.x);
          bulk_g2s(sb, p.k_cache + tile * C::kTile, C::kTile, bars + st, pol);
          bulk_g2s(sb + C::kOffV, p.v_cache + tile * C::kVTile, C::kVTile, bars + st, pol);
          if constexpr (C::kScale > 0) {  // one 128-byte unit for 16-token blocks
            const int64_t si = scale_index(static_cast<int64_t>(tile), p.tiles_per_block);
            if (p.tiles_per_block == 1) {
              bulk_g2s(sb + C::kOffKS, p.k_scale + si, 2 * C::kScale, bars + st, pol);
            } else {
              bulk_g2s(sb + C::kOffKS, p.k_scale + si, C::kScale, bars + st, pol);
              bulk_g2s(sb + C::kOffVS, p.v_scale + si, C::kScale, bars + st, pol);
            }
          }
        }
        if (need_q) bulk_g2s(sb + C::kOffQ, p.q + static_cast<size_t>(item) * C::kQ, C::kQ, bars + st);
        if (need_new) {
          bulk_g2s(sb + C::kOffNew, p.k_new + static_cast<size_t>(item) * D * 2, D * 2, bars + st);
          bulk_g2s(sb + C::kOffNew + D * 2, p.v_new + static_cast<size_t>(item) * D * 2, D * 2, bars + st);
        }
      }
    }
  };

  if (count > 0) {
    fill_window(0);
    fill_window(1);
  }
  griddep_wait();  // from here the previous kernel's writes are visible
  publish_scan<C::kThreads>(p, cum, G * D * p.num_kv_heads);
  if (count <= 0) {
    griddep_launch_dependents();
    return;
  }
  __syncwarp();
#pragma unroll 1
  for (int i = 0; i < C::kStages && i < count; ++i) issue(i);

  const int jl = lane % C::kLPT;  // lane within its token group
  const int tg = lane / C::kLPT;  // token group
  const int hd = jl / (C::kLPT / G);                  // head this lane's score belongs to
  const bool lead = (jl % (C::kLPT / G)) == 0;        // one writer per (token, head)

  float qreg[G][C::kEPT];
  float o[G][C::kDPL];
  float m[G], l[G];
  float m_mine = -INFINITY;
  int cur_item = -1;
  bool whole_start = false, saw_last = false;

  auto flush = [&](int item, bool whole) {
    if (whole) {
      const size_t base = (static_cast<size_t>(item) * G) * D + lane * C::kDPL;  // element index
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float inv = l[g] > 0.f ? 1.f / l[g] : 0.f;
        float r[C::kDPL];
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) r[e] = o[g][e] * inv;
        if (p.out_f32) {
          float *dst = reinterpret_cast<float *>(p.out) + base + g * D;
          if constexpr (C::kDPL == 4) {
            *reinterpret_cast<float4 *>(dst) = make_float4(r[0], r[1], r[2], r[3]);
          } else {
            *reinterpret_cast<float2 *>(dst) = make_float2(r[0], r[1]);
          }
        } else {
          uint8_t *dst = p.out + (base + g * D) * 2;
          if constexpr (C::kDPL == 4) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pack2<QDT>(r[0], r[1]), pack2<QDT>(r[2], r[3]));
          } else {
            *reinterpret_cast<uint32_t *>(dst) = pack2<QDT>(r[0], r[1]);
          }
        }
      }
    } else {
      const int64_t slot = gw + item;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float *op = p.ws_o + (slot * G + g) * D + lane * C::kDPL;
        if constexpr (C::kDPL == 4) {
          *reinterpret_cast<float4 *>(op) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
        } else {
          *reinterpret_cast<float2 *>(op) = make_float2(o[g][0], o[g][1]);
        }
        if (lane == 0) {
          p.ws_ml[(slot * G + g) * 2] = m[g];
          p.ws_ml[(slot * G + g) * 2 + 1] = l[g];
        }
      }
      finish_partial<D, G, QDT>(p, cum, item, total, nwarps);
    }
  };

#pragma unroll 1
  for (int n = 0; n < count; ++n) {
    if (n > 0 && (n & 31) == 0) {
      __syncwarp();
      fill_window((n >> 5) + 1);
      __syncwarp();
    }
    const int2 d = desc[((n >> 5) & 1) * 32 + (n & 31)];
    const int st = n % C::kStages;
    uint8_t *sb = stages + st * C::kStage;
    const bool ok = __all_sync(kFull, mbar_wait(bars + st, (n / C::kStages) & 1));
    if (!ok) {
      if (lane == 0) report(p.d_error, PKV_DEVERR_WAIT_TIMEOUT);
      // let the copies this warp still has in flight land before leaving
      for (int k = n + 1; k < count && k < n + C::kStages; ++k)
        mbar_wait(bars + k % C::kStages, (k / C::kStages) & 1);
      return;
    }
    const int item = d.y >> 7;
    const int ntok = d.y & 31;
    if (item != cur_item) {
      if (cur_item >= 0) flush(cur_item, whole_start && saw_last);
      cur_item = item;
      whole_start = (d.y >> 6) & 1;
      // this item's G query heads -> registers, pre-scaled by scale * log2(e)
      const uint8_t *qs = sb + C::kOffQ;
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c) {
          const int d0 = (jl + c * C::kLPT) * C::kEPC;
#pragma unroll
          for (int e = 0; e < C::kEPC; e += 2) {
            const float2 f = unpack2<QDT>(*reinterpret_cast<const uint32_t *>(qs + (g * D + d0 + e) * 2));
            qreg[g][c * C::kEPC + e] = f.x * p.scale_log2;
            qreg[g][c * C::kEPC + e + 1] = f.y * p.scale_log2;
          }
        }
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) o[g][e] = 0.f;
        m[g] = -INFINITY;
        l[g] = 0.f;
      }
      m_mine = -INFINITY;
    }
    saw_last = (d.y >> 5) & 1;

    if (p.k_new && d.x >= 0 && saw_last) {
      // Fused append: the item's new token is row r of this tile.  Encode the
      // staged K / V rows as the cache holds them, put them into the staged
      // tile and into the cache for later steps.  No other warp reads this
      // tile, and its copy has landed, so nothing races.
      const int r = (d.y & 31) - 1;
      const int64_t grow = static_cast<int64_t>(d.x) * kBS + r;
      float kscl, vscl;
      const uint2 kb = encode_slice<D, QDT, C::KT>(sb + C::kOffNew, lane, kscl);
      const uint2 vb = encode_slice<D, QDT, C::VT>(sb + C::kOffNew + D * 2, lane, vscl);
      constexpr int BK = slice_bytes<D, C::KT>(), BV = slice_bytes<D, C::VT>();
      store_slice<D, C::KT>(sb + r * C::kRow + lane * BK, kb);
      store_slice<D, C::VT>(sb + C::kOffV + r * C::kVRow + lane * BV, vb);
      // the caches are read-only everywhere else in the kernel
      store_slice<D, C::KT>(const_cast<uint8_t *>(p.k_cache) + grow * C::kRow + lane * BK, kb);
      store_slice<D, C::VT>(const_cast<uint8_t *>(p.v_cache) + grow * C::kVRow + lane * BV, vb);
      if constexpr (C::kScale > 0) {
        if (lane == 0) {
          reinterpret_cast<float *>(sb + C::kOffKS)[r] = kscl;
          reinterpret_cast<float *>(sb + C::kOffVS)[r] = vscl;
          const int64_t gs = scale_index(d.x, p.tiles_per_block) + r;
          const_cast<float *>(p.k_scale)[gs] = kscl;
          const_cast<float *>(p.v_scale)[gs] = vscl;
        }
      }
      __syncwarp();
    }

    if (d.x >= 0) {
      const uint8_t *ks = sb;
      const uint8_t *vs = sb + C::kOffV;
      // -- scores of this tile: s = (q . k) * scale * log2 e, base-2 domain --
      float sc[C::kPasses];
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        const int tok = ps * C::kTPP + tg;
        float part[G];
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = 0.f;
#pragma unroll
        for (int c = 0; c < C::kNChunk; ++c) {
          float x[C::kEPC];
          unpack_row<C::KT, C::kChunk>(ks + tok * C::kRow + (jl + c * C::kLPT) * C::kChunk, x);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::kEPC; ++e) part[g] = fmaf(qreg[g][c * C::kEPC + e], x[e], part[g]);
        }
        float r = reduce_heads<G, C::kLPT>(part, lane);
        if constexpr (is_coded(C::KT)) r *= reinterpret_cast<const float *>(sb + C::kOffKS)[tok];
        sc[ps] = tok < ntok ? r : -INFINITY;
      }
      // -- online softmax over this tile (per head) --
      float mx = sc[0];
#pragma unroll
      for (int ps = 1; ps < C::kPasses; ++ps) mx = fmaxf(mx, sc[ps]);
#pragma unroll
      for (int off = C::kLPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      const float m_new = fmaxf(m_mine, mx);
      const float alpha = exp2f(m_mine - m_new);
      float pr[C::kPasses];
      float psum = 0.f;
#pragma unroll
      for (int ps = 0; ps < C::kPasses; ++ps) {
        pr[ps] = exp2f(sc[ps] - m_new);
        psum += pr[ps];
      }
#pragma unroll
      for (int off = C::kLPT; off < 32; off <<= 1) psum += __shfl_xor_sync(kFull, psum, off);
      m_mine = m_new;
      __syncwarp();  // every lane is done with K: its space now holds probabilities
      float *pbuf = reinterpret_cast<float *>(sb);  // [16][G] probabilities, then alpha, sum, max
      if (lead) {
#pragma unroll
        for (int ps = 0; ps < C::kPasses; ++ps) {
          const int tok = ps * C::kTPP + tg;
          float pv = pr[ps];
          if constexpr (is_coded(C::VT)) pv *= reinterpret_cast<const float *>(sb + C::kOffVS)[tok];
          pbuf[tok * G + hd] = pv;
        }
        if (tg == 0) {
          pbuf[kBS * G + hd] = alpha;
          pbuf[(kBS + 1) * G + hd] = psum;
          pbuf[(kBS + 2) * G + hd] = m_new;
        }
      }
      __syncwarp();
      // -- o = o * alpha + P V --
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float a = pbuf[kBS * G + g];
        l[g] = l[g] * a + pbuf[(kBS + 1) * G + g];
        m[g] = pbuf[(kBS + 2) * G + g];
#pragma unroll
        for (int e = 0; e < C::kDPL; ++e) o[g][e] *= a;
      }
#pragma unroll
      for (int t = 0; t < kBS; ++t) {
        if (t < ntok) {
          float x[C::kDPL];
          if constexpr (C::VT == kInt4) {
            unpack_int4<C::kVSlice>(vs + t * C::kVRow + lane * C::kVSlice, x);
          } else {
            unpack_row<C::VT, C::kVSlice>(vs + t * C::kVRow + lane * C::kVSlice, x);
          }
          float pw[G];
#pragma unroll
          for (int g = 0; g < G; ++g) pw[g] = pbuf[t * G + g];
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < C::kDPL; ++e) o[g][e] = fmaf(pw[g], x[e], o[g][e]);
        }
      }
    }
    __syncwarp();  // the stage is free again
    if (n + C::kStages < count) issue(n + C::kStages);
  }
  griddep_launch_dependents();
  flush(cur_item, whole_start && saw_last);
}

template <int D, int G, int CDT, int QDT>
struct DecodeInstance {
  using C = DecodeCfg<D, G, CDT, QDT>;
  static cudaError_t prepare(DecodeShape *shape) {
    static int cached = -1;
    if (cached < 0) {
      cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<D, G, CDT, QDT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_kernel<D, G, CDT, QDT>,
                                                        C::kThreads, C::kSmem);
      if (e != cudaSuccess) return e;
      cached = n > 0 ? n : 1;
    }
    *shape = DecodeShape{cached, C::kWarps};
    return cudaSuccess;
  }
  static cudaError_t launch(const DecodeParams &p, int grid, int64_t *launches) {
    const cudaError_t e = launch_decode(paged_decode_kernel<D, G, CDT, QDT>, grid, C::kThreads, C::kSmem, p.stream,
                                        p.programmatic, p);
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
};

}  // namespace pkv

namespace pkv {

template <int D, int G, int CDT, int QDT>
cudaError_t decode_op(int op, const DecodeParams *p, int grid, int64_t *launches, DecodeShape *shape) {
  using I = DecodeInstance<D, G, CDT, QDT>;
  if (op == kDecodePrepare) return I::prepare(shape);
  return I::launch(*p, grid, launches);
}

template <int CDT, int QDT>
cudaError_t decode_family(int D, int G, int op, const DecodeParams *p, int grid, int64_t *launches,
                          DecodeShape *shape) {
  if (D == 128) {
    switch (G) {
      case 1: return decode_op<128, 1, CDT, QDT>(op, p, grid, launches, shape);
      case 2: return decode_op<128, 2, CDT, QDT>(op, p, grid, launches, shape);
      case 4: return decode_op<128, 4, CDT, QDT>(op, p, grid, launches, shape);
      case 8: return decode_op<128, 8, CDT, QDT>(op, p, grid, launches, shape);
    }
  } else if (D == 64) {
    switch (G) {
      case 1: return decode_op<64, 1, CDT, QDT>(op, p, grid, launches, shape);
      case 2: return decode_op<64, 2, CDT, QDT>(op, p, grid, launches, shape);
      case 4: return decode_op<64, 4, CDT, QDT>(op, p, grid, launches, shape);
      case 8: return decode_op<64, 8, CDT, QDT>(op, p, grid, launches, shape);
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
