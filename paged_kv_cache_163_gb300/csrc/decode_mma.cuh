// Tensor-core variant of the paged decode partial kernel (head_dim 128).
//
// Same work split, staging ring, partial format and in-kernel merge as
// paged_decode_kernel; the arithmetic of one (block, KV head) tile moves to
// mma.sync m16n8k16 (fp32 accumulate):
//   S^T[16 tokens x 8 heads] = K[16 x 128] . Q^T[128 x 8]      (8 MMAs)
//   O^T[128 x 8]            += V^T[128 x 16] . P^T[16 x 8]     (8 MMAs, 16 for bf16)
// The GQA group (G <= 8 heads, zero-padded to 8) is the MMA's N.  K and V
// tiles arrive by tensor TMA with the 128-byte swizzle; every lane's reads
// are conflict-free because the head_dim order inside the MMAs is permuted
// (a dot product and the output rows do not depend on the order, only on
// using the same order for K and Q, and writing O with the matching d).
// One-byte codes (FP8 E4M3 / E5M2, INT8) and 4-bit V codes become fp16 in
// registers (exact); a bf16 P is split into a high and a low bf16 half so
// the probabilities keep fp16-class precision.
#pragma once

#include <cuda.h>

#include "decode.cuh"

namespace pkv {

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          bool bf16) {
  if (bf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Transpose of an 8x8 16-bit matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Tensor-map bulk load of a 2D box into shared memory (complete_tx on bar).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

template <int G, int CDT, int QDT>
struct MmaCfg {
  static constexpr int kD = 128;
  static constexpr int KT = k_part(CDT), VT = v_part(CDT);  // storage types of K and of V
  static constexpr bool kCode8 = is_code8(KT);  // one-byte K codes (FP8 E4M3 / E5M2, INT8) with scales
  static constexpr bool kVInt4 = VT == kInt4;   // 4-bit V codes: plain 64-byte rows, no swizzle
  // INT8 K codes enter the score MMA biased (1152 + k); the bias comes off
  // the score as 1152 x the query head's sum, once per item.
  static constexpr bool kKBias = KT == PKV_INT8;
  // INT8 / 4-bit V codes enter the output MMA biased; the bias comes off the
  // accumulator in the per-tile rescale (an FFMA instead of an FMUL), with the
  // tile's column sums of P from one more MMA against all-ones A.
  static constexpr bool kVBias = VT == PKV_INT8 || VT == kInt4;
  static constexpr float kBiasLo = VT == kInt4 ? kInt4LoBias : kInt8Bias;  // accumulator rows g
  static constexpr float kBiasHi = VT == kInt4 ? kInt4HiBias : kInt8Bias;  // rows g + 8
  static constexpr float kHiScale = VT == kInt4 ? 0.0625f : 1.f;          // 4-bit high nibbles carry x16
  // The per-tile softmax's exponentials and the V-scale reciprocal by the
  // hardware approximations (fast_exp2, fast_rcp).  Measured per instance
  // (same box, A/B of two builds): 3% faster with 4-bit V codes, 4% slower
  // with E4M3 codes, no change for the others; so 4-bit V only.
  static constexpr bool kFastSoftmax = kVInt4;
  // One-byte tiles are half the bytes, so an SM holds twice the warps (with
  // at most 128 registers a thread).  They form one 16-warp CTA: two 8-warp
  // CTAs on an SM were measured to run unevenly (the CTA launched first
  // streamed ~13% faster), leaving the SM half idle at the end of a call.
  static constexpr int kWarps = kCode8 ? 16 : 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr bool kBf16 = !kCode8 && CDT == PKV_BF16;  // MMA operand type: bf16, else f16
  static constexpr int kEsz = kCode8 ? 1 : 2;
  static constexpr int kTile = kBS * kD * kEsz;  // K tile bytes (1024-aligned in shared memory)
  static constexpr int kVTile = kVInt4 ? kBS * kD / 2 : kTile;
  static constexpr int kKV = kTile + kVTile;
  static constexpr int kScale = has_scales(CDT) ? kBS * 4 : 0;
  static constexpr int kQ = G * kD * 2;
  static constexpr int kNew = 2 * kD * 2;  // fused append: the new token's K and V rows (query dtype)
  static constexpr int kOffNew = 2 * kScale + kQ;
  static constexpr int kAux = round_up_c(2 * kScale + kQ + kNew, 128);  // [k scales][v scales][q rows][new rows]
  // Two stages per warp: measured faster than deeper rings on GB300 (more
  // copies in flight than HBM needs only lengthen the queues).
  static constexpr int kStages = 2;
  static constexpr int kMinBlocks = 1;
  static constexpr int kCumBytes = round_up_c((PKV_MAX_SEQS_PER_CALL + 1) * 4, 128);
  static constexpr int kMiscBytes = 128;
  static constexpr int kBarBytes = round_up_c(kWarps * kStages * 8, 128);
  static constexpr int kDescBytes = kWarps * 64 * 8;
  static constexpr int kHead = kCumBytes + kMiscBytes + kBarBytes + kDescBytes;
  static constexpr int kTilesOff = round_up_c(kHead, 1024);
  static constexpr int kSmem = 1024 + kTilesOff + kWarps * kStages * (kKV + kAux);
  static_assert(G >= 1 && G <= 8, "group size");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kKV % 1024 == 0, "swizzled K tiles stay 1024-aligned");
  static_assert(!kVInt4 || kCode8, "4-bit V only beside one-byte K");
};

// head_dim index of output row m (0..15) of m-tile i for lane group g (see kernel comment).
template <bool CODE8>
__device__ __forceinline__ int out_d(int g, int i, int hrow) {
  return CODE8 ? 16 * g + 2 * i + hrow : 64 * (i >> 2) + 8 * g + 2 * (i & 3) + hrow;
}

template <int G, int CDT, int QDT>
__global__ void __launch_bounds__(MmaCfg<G, CDT, QDT>::kThreads, MmaCfg<G, CDT, QDT>::kMinBlocks)
    paged_decode_mma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
  using C = MmaCfg<G, CDT, QDT>;
  constexpr int D = C::kD;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);  // 1024-aligned base
  int32_t *cum = reinterpret_cast<int32_t *>(smem);
  int32_t *misc = reinterpret_cast<int32_t *>(smem + C::kCumBytes);
  uint64_t *bars_all = reinterpret_cast<uint64_t *>(smem + C::kCumBytes + C::kMiscBytes);
  int2 *desc_all = reinterpret_cast<int2 *>(smem + C::kCumBytes + C::kMiscBytes + C::kBarBytes);
  uint8_t *tiles_all = smem + C::kTilesOff;
  uint8_t *aux_all = tiles_all + C::kWarps * C::kStages * C::kKV;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;   // MMA row group
  const int q4 = lane & 3;   // thread within the group

  scan_blocks<C::kWarps, C::kStages>(p, cum, misc, bars_all);

  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * C::kWarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * C::kWarps + warp;
  const int64_t total = static_cast<int64_t>(cum[p.num_seqs]) * p.num_kv_heads;
  const int64_t t0 = gw * total / nwarps;
  const int64_t t1 = (gw + 1) * total / nwarps;
  const int count = static_cast<int>(t1 - t0);

  uint64_t *bars = bars_all + warp * C::kStages;
  int2 *desc = desc_all + warp * 64;
  uint8_t *tiles = tiles_all + warp * C::kStages * C::kKV;
  uint8_t *aux = aux_all + warp * C::kStages * C::kAux;
  const uint64_t pol = policy_evict_first();

  auto fill_window = [&](int w) {
    const int64_t t = t0 + 32 * static_cast<int64_t>(w) + lane;
    int2 d = make_int2(-1, 0);
    if (t < t1) d = tile_desc(p, cum, t);
    desc[(w & 1) * 32 + lane] = d;
  };

  // Copies of warp-local tile m into its stage.  part 0: all of them; 1: the
  // cache copies only (with the stage's arrival for all its bytes; nothing
  // for a tile without a block); 2: the rest (queries, new rows).
  auto issue = [&](int m, int part) {
    const int2 d = desc[((m >> 5) & 1) * 32 + (m & 31)];
    if (lane == 0) {
      const int st = m % C::kStages;
      uint8_t *tb = tiles + st * C::kKV;
      uint8_t *ab = aux + st * C::kAux;
      const int item = d.y >> 7;
      const bool need_q = (m == 0) || ((d.y >> 6) & 1);
      const bool need_new = p.k_new && d.x >= 0 && ((d.y >> 5) & 1);  // the item's last tile: its new token
      const uint32_t bytes =
          (d.x >= 0 ? C::kKV + 2 * C::kScale : 0) + (need_q ? C::kQ : 0) + (need_new ? C::kNew : 0);
      fence_proxy_async_smem();
      if (part == 0 || (part == 1) == (d.x >= 0)) {  // the part that arrives on the stage's barrier
        if (bytes == 0) {
          mbar_arrive(bars + st);
          return;
        }
        mbar_arrive_expect_tx(bars + st, bytes);
      }
      {
        if (d.x >= 0 && part != 2) {
          const int64_t tile = d.x;
          const int row = static_cast<int>(tile * kBS);
          if constexpr (C::kCode8) {
            tma_load_2d(tb, &tmk, 0, row, bars + st, pol);
            if constexpr (C::kVInt4) {  // a 16-token V tile is one contiguous kilobyte
              bulk_g2s(tb + C::kTile, p.v_cache + tile * C::kVTile, C::kVTile, bars + st, pol);
            } else {
              tma_load_2d(tb + C::kTile, &tmv, 0, row, bars + st, pol);
            }
            const int64_t si = scale_index(tile, p.tiles_per_block);
            if (p.tiles_per_block == 1) {  // K and V scales: one 128-byte unit
              bulk_g2s(ab, p.k_scale + si, 2 * C::kScale, bars + st, pol);
            } else {
              bulk_g2s(ab, p.k_scale + si, C::kScale, bars + st, pol);
              bulk_g2s(ab + C::kScale, p.v_scale + si, C::kScale, bars + st, pol);
            }
          } else {
            tma_load_2d(tb, &tmk, 0, row, bars + st, pol);
            tma_load_2d(tb + 2048, &tmk, 64, row, bars + st, pol);
            tma_load_2d(tb + C::kTile, &tmv, 0, row, bars + st, pol);
            tma_load_2d(tb + C::kTile + 2048, &tmv, 64, row, bars + st, pol);
          }
        }
        if (part != 1) {
          if (need_q) bulk_g2s(ab + 2 * C::kScale, p.q + static_cast<size_t>(item) * C::kQ, C::kQ, bars + st);
          if (need_new) {
            bulk_g2s(ab + C::kOffNew, p.k_new + static_cast<size_t>(item) * D * 2, D * 2, bars + st);
            bulk_g2s(ab + C::kOffNew + D * 2, p.v_new + static_cast<size_t>(item) * D * 2, D * 2, bars + st);
          }
        }
      }
    }
  };

  if (count > 0) {
    fill_window(0);
    fill_window(1);
  }
  // Behind a kernel that writes no K/V cache memory the first tiles' cache
  // copies may start now; their queries and new rows (inputs that kernel
  // may write) follow the wait.
  const bool early = p.early_kv && !p.pfx_n && count > 0;
  if (early) {
    __syncwarp();
#pragma unroll 1
    for (int i = 0; i < C::kStages && i < count; ++i) issue(i, 1);
  }
  // from here the previous kernel's writes are visible.  Behind a prefix
  // kernel (cascade) that kernel's predecessors are done already (it waited
  // for them before it let this grid start), and its own partials are
  // waited for before the first merge that reads them.
  if (!p.pfx_n) griddep_wait();
  publish_scan<C::kThreads>(p, cum, G * D * p.num_kv_heads);
  if (count <= 0) {
    griddep_launch_dependents();
    return;
  }
  __syncwarp();
#pragma unroll 1
  for (int i = 0; i < C::kStages && i < count; ++i) issue(i, early ? 2 : 0);

  uint32_t qb[8][2];   // Q^T B fragments (8 k-steps)
  float oacc[8][4];    // O^T accumulators (8 m-tiles of 16 head_dim rows x 8 heads)
  float m_run[2], l_run[2];  // heads 2 q4 and 2 q4 + 1 (running max: base-2 domain)
  // One-byte caches: oacc holds O / vunit, where vunit is the largest V scale
  // of the latest tile (P carries the tile's scales relative to it, so the
  // fp16 B operand stays in [0, 1] whatever the scales' magnitude).
  float vunit = 1.f;
  float kbias0 = 0.f, kbias1 = 0.f;  // INT8 K: 1152 x sum of the f16 query of heads 2 q4, 2 q4 + 1
  int cur_item = -1;
  bool whole_start = false, saw_last = false;

  auto flush = [&](int item, bool whole) {
    // an item with prefix-kernel partials always merges (its own share is one partial)
    const bool prefixed = p.pfx_n && p.pfx_chunks[item / p.num_kv_heads] > 0;
    const bool direct = whole && !prefixed;
    float lt[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l_run[j];
      v += __shfl_xor_sync(kFull, v, 4);
      v += __shfl_xor_sync(kFull, v, 8);
      v += __shfl_xor_sync(kFull, v, 16);
      lt[j] = v;
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = 2 * q4 + j;
      if (n >= G) continue;
      // m-tiles ib .. ib + 3 hold 8 consecutive head_dim values of this lane
      // (out_d(g, ib + c, 0) = out_d(g, ib, 0) + 2 c): 16-byte stores, which
      // also keep writes to page-locked host memory whole
      if (direct) {
        const float inv = (lt[j] > 0.f ? 1.f / lt[j] : 0.f) * vunit;
        const size_t row = (static_cast<size_t>(item) * G + n) * D;
#pragma unroll
        for (int ib = 0; ib < 8; ib += 4) {
          const int d0 = out_d<C::kCode8>(g, ib, 0);
          float r[8];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            r[2 * c] = oacc[ib + c][j] * inv;
            r[2 * c + 1] = oacc[ib + c][2 + j] * (inv * C::kHiScale);
          }
          if (p.out_f32) {
            float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) + row + d0);
            dst[0] = make_float4(r[0], r[1], r[2], r[3]);
            dst[1] = make_float4(r[4], r[5], r[6], r[7]);
          } else {
            *reinterpret_cast<uint4 *>(p.out + (row + d0) * 2) =
                make_uint4(pack2<QDT>(r[0], r[1]), pack2<QDT>(r[2], r[3]), pack2<QDT>(r[4], r[5]),
                           pack2<QDT>(r[6], r[7]));
          }
        }
      } else {
        const int64_t slot = gw + item;
        float *op = p.ws_o + (slot * G + n) * D;
#pragma unroll
        for (int ib = 0; ib < 8; ib += 4) {
          float4 *dst = reinterpret_cast<float4 *>(op + out_d<C::kCode8>(g, ib, 0));
          const float vh = vunit * C::kHiScale;
          dst[0] = make_float4(oacc[ib][j] * vunit, oacc[ib][2 + j] * vh, oacc[ib + 1][j] * vunit,
                               oacc[ib + 1][2 + j] * vh);
          dst[1] = make_float4(oacc[ib + 2][j] * vunit, oacc[ib + 2][2 + j] * vh, oacc[ib + 3][j] * vunit,
                               oacc[ib + 3][2 + j] * vh);
        }
        if (g == 0) {
          p.ws_ml[(slot * G + n) * 2] = m_run[j];
          p.ws_ml[(slot * G + n) * 2 + 1] = lt[j];
        }
      }
    }
    // merge batches sized to the register budget (one-byte instances: 128 a thread)
    if (!whole) {
      finish_partial<D, G, QDT, C::kCode8 ? 8 : 32>(p, cum, item, total, nwarps);
    } else if (prefixed) {  // the only share of the item: merge with the prefix partials now
      __threadfence_block();
      __syncwarp();
      merge_item<D, G, QDT, C::kCode8 ? 8 : 32>(p, item, gw, gw, total, nwarps);
    }
  };

  // tokens whose V rows this lane reads (B-fragment k rows of P^T)
  const int tk0 = 2 * q4, tk1 = 2 * q4 + 1, tk2 = 2 * q4 + 8, tk3 = 2 * q4 + 9;
  const int tks[4] = {tk0, tk1, tk2, tk3};
  // 4-bit V: byte permutes that put byte b of the pair's first token at
  // byte 0 and of its second token at byte 2 (operands swapped for odd q4)
  uint32_t vsel[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) vsel[b] = (0x4400u + 0x1111u * b) ^ ((q4 & 1) ? 0x4444u : 0u);

#pragma unroll 1
  for (int n = 0; n < count; ++n) {
    if (n > 0 && (n & 31) == 0) {
      __syncwarp();
      fill_window((n >> 5) + 1);
      __syncwarp();
    }
    const int2 d = desc[((n >> 5) & 1) * 32 + (n & 31)];
    const int st = n % C::kStages;
    const uint8_t *kt = tiles + st * C::kKV;
    const uint8_t *vt = kt + C::kTile;
    const uint8_t *ab = aux + st * C::kAux;
    const bool ok = __all_sync(kFull, mbar_wait(bars + st, (n / C::kStages) & 1));
    if (!ok) {
      if (lane == 0) report(p.d_error, PKV_DEVERR_WAIT_TIMEOUT);
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
      const uint8_t *qs = ab + 2 * C::kScale;  // [G][128] rows in the query dtype
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int d0 = C::kCode8 ? 32 * q4 + 4 * s : 64 * (s >> 2) + 16 * q4 + 4 * (s & 3);
        uint2 raw = make_uint2(0u, 0u);
        if (g < G) raw = *reinterpret_cast<const uint2 *>(qs + (g * D + d0) * 2);
        if constexpr (C::kCode8 && QDT == PKV_BF16) {  // f16 MMA operands
          const float2 a = unpack2<QDT>(raw.x), b = unpack2<QDT>(raw.y);
          qb[s][0] = pack2<PKV_F16>(a.x, a.y);
          qb[s][1] = pack2<PKV_F16>(b.x, b.y);
        } else {
          qb[s][0] = raw.x;
          qb[s][1] = raw.y;
        }
      }
      if constexpr (C::kKBias) {
        // head g's query sum: this lane's 32 head_dim values, then the other three lanes of the group
        float qs = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const float2 a = unpack2<PKV_F16>(qb[s][0]), b = unpack2<PKV_F16>(qb[s][1]);
          qs += (a.x + a.y) + (b.x + b.y);
        }
        qs += __shfl_xor_sync(kFull, qs, 1);
        qs += __shfl_xor_sync(kFull, qs, 2);
        kbias0 = kInt8Bias * __shfl_sync(kFull, qs, 8 * q4);      // head 2 q4 (lane group 2 q4)
        kbias1 = kInt8Bias * __shfl_sync(kFull, qs, 8 * q4 + 4);  // head 2 q4 + 1
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) oacc[i][c] = 0.f;
      m_run[0] = m_run[1] = -INFINITY;
      vunit = 1.f;
      l_run[0] = l_run[1] = 0.f;
    }
    saw_last = (d.y >> 5) & 1;

    if (p.k_new && d.x >= 0 && saw_last) {
      // Fused append: the item's new token is row r of this tile.  Encode the
      // staged K / V rows as the cache holds them, put them into the staged
      // tile (swizzled layout) and into the cache for later steps.  No other
      // warp reads this tile, and its copy has landed, so nothing races.
      const int r = (d.y & 31) - 1;
      const int64_t grow = static_cast<int64_t>(d.x) * kBS + r;
      float ks, vs;
      const uint2 kb = encode_slice<D, QDT, C::KT>(ab + C::kOffNew, lane, ks);
      const uint2 vb = encode_slice<D, QDT, C::VT>(ab + C::kOffNew + D * 2, lane, vs);
      const int off = C::kCode8 ? r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + (lane & 3) * 4
                                : (lane >> 4) * 2048 + r * 128 + ((((lane & 15) >> 1) ^ (r & 7)) << 4) + (lane & 1) * 8;
      constexpr int BK = slice_bytes<D, C::KT>(), BV = slice_bytes<D, C::VT>();
      const int voff = C::kVInt4 ? r * (D / 2) + lane * BV : off;
      store_slice<D, C::KT>(tiles + st * C::kKV + off, kb);
      store_slice<D, C::VT>(tiles + st * C::kKV + C::kTile + voff, vb);
      // the caches are read-only everywhere else in the kernel
      store_slice<D, C::KT>(const_cast<uint8_t *>(p.k_cache) + grow * (BK * 32) + lane * BK, kb);
      store_slice<D, C::VT>(const_cast<uint8_t *>(p.v_cache) + grow * (BV * 32) + lane * BV, vb);
      if constexpr (C::kCode8) {
        if (lane == 0) {
          float *sab = reinterpret_cast<float *>(aux + st * C::kAux);
          sab[r] = ks;
          sab[kBS + r] = vs;
          const int64_t gs = scale_index(d.x, p.tiles_per_block) + r;
          const_cast<float *>(p.k_scale)[gs] = ks;
          const_cast<float *>(p.v_scale)[gs] = vs;
        }
      }
      __syncwarp();
    }

    if (d.x >= 0) {
      // ---- S^T = K Q^T: lane rows g and g + 8, head columns 2 q4, 2 q4 + 1 ----
      float sacc4[4][4] = {};  // four independent accumulation chains over the 8 k-steps
      if constexpr (C::kCode8) {
        uint4 kr[2][2];  // [row g, g + 8][chunk 2 q4 + j]
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int row = g + 8 * r, c = 2 * q4 + j;
            kr[r][j] = *reinterpret_cast<const uint4 *>(kt + row * 128 + ((c ^ (row & 7)) << 4));
          }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t a[4];
          if constexpr (C::kKBias) {
            int8x4_to_f16x2_biased(word(kr[0][s >> 2], s & 3), a[0], a[2]);
            int8x4_to_f16x2_biased(word(kr[1][s >> 2], s & 3), a[1], a[3]);
          } else {
            code4_to_f16x2<C::KT>(word(kr[0][s >> 2], s & 3), a[0], a[2]);
            code4_to_f16x2<C::KT>(word(kr[1][s >> 2], s & 3), a[1], a[3]);
          }
          mma_16816(sacc4[s & 3], a, qb[s][0], qb[s][1], false);
        }
      } else {
        uint4 kr[2][2][2];  // [row][half][chunk 2 q4 + j]
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int row = g + 8 * r, c = 2 * q4 + j;
              kr[r][h][j] = *reinterpret_cast<const uint4 *>(kt + h * 2048 + row * 128 + ((c ^ (row & 7)) << 4));
            }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int h = s >> 2, j = (s & 3) >> 1, t = s & 1;
          uint32_t a[4] = {word(kr[0][h][j], 2 * t), word(kr[1][h][j], 2 * t), word(kr[0][h][j], 2 * t + 1),
                           word(kr[1][h][j], 2 * t + 1)};
          mma_16816(sacc4[s & 3], a, qb[s][0], qb[s][1], C::kBf16);
        }
      }
      float sacc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[c] = (sacc4[0][c] + sacc4[1][c]) + (sacc4[2][c] + sacc4[3][c]);
      if constexpr (C::kKBias) {
        sacc[0] -= kbias0;
        sacc[1] -= kbias1;
        sacc[2] -= kbias0;
        sacc[3] -= kbias1;
      }
      // ---- scale, mask, online softmax (base 2) ----
      float sc0 = p.scale_log2, sc1 = p.scale_log2;
      if constexpr (C::kCode8) {
        const float *ksc = reinterpret_cast<const float *>(ab);
        sc0 *= ksc[g];
        sc1 *= ksc[g + 8];
      }
      const bool v0 = g < ntok, v1 = g + 8 < ntok;
      float s00 = v0 ? sacc[0] * sc0 : -INFINITY;  // token g,     head 2 q4
      float s01 = v0 ? sacc[1] * sc0 : -INFINITY;  // token g,     head 2 q4 + 1
      float s10 = v1 ? sacc[2] * sc1 : -INFINITY;  // token g + 8, head 2 q4
      float s11 = v1 ? sacc[3] * sc1 : -INFINITY;  // token g + 8, head 2 q4 + 1
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      auto ex2 = [](float x) { return C::kFastSoftmax ? fast_exp2(x) : exp2f(x); };
      float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);
      m_run[0] = mn0;
      m_run[1] = mn1;
      float p00 = ex2(s00 - mn0), p01 = ex2(s01 - mn1), p10 = ex2(s10 - mn0), p11 = ex2(s11 - mn1);
      l_run[0] = l_run[0] * al0 + (p00 + p10);
      l_run[1] = l_run[1] * al1 + (p01 + p11);
      if constexpr (C::kCode8) {  // per-token V scales, relative to the tile's largest, go into P
        const float *vsc = reinterpret_cast<const float *>(ab + C::kScale);
        const float vs0 = v0 ? vsc[g] : 0.f, vs1 = v1 ? vsc[g + 8] : 0.f;
        float vmax = fmaxf(vs0, vs1);  // over the tile's 16 tokens (lane groups g hold tokens g, g + 8)
        vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 4));
        vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 8));
        vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 16));
        if (!(vmax > 0.f)) vmax = 1.f;  // all scales zero: the tile adds nothing either way
        const float rv = C::kFastSoftmax ? fast_rcp(vmax) : 1.f / vmax;
        const float w0 = vs0 * rv, w1 = vs1 * rv;
        p00 *= w0;
        p01 *= w0;
        p10 *= w1;
        p11 *= w1;
        const float ru = vunit * rv;  // oacc changes units from the old vunit to vmax
        al0 *= ru;
        al1 *= ru;
        vunit = vmax;
      }
      // ---- P^T B fragments (k rows = tokens, n columns = heads) ----
      uint32_t pb[2][2];  // [hi / lo][b0, b1]
      if constexpr (C::kBf16) {
        const uint32_t h0 = pack2<PKV_BF16>(p00, p01), h1 = pack2<PKV_BF16>(p10, p11);
        const float2 r0 = unpack2<PKV_BF16>(h0), r1 = unpack2<PKV_BF16>(h1);
        const uint32_t l0 = pack2<PKV_BF16>(p00 - r0.x, p01 - r0.y), l1 = pack2<PKV_BF16>(p10 - r1.x, p11 - r1.y);
        pb[0][0] = movmatrix_t(h0);
        pb[0][1] = movmatrix_t(h1);
        pb[1][0] = movmatrix_t(l0);
        pb[1][1] = movmatrix_t(l1);
      } else {
        pb[0][0] = movmatrix_t(pack2<PKV_F16>(p00, p01));
        pb[0][1] = movmatrix_t(pack2<PKV_F16>(p10, p11));
      }
      // ---- rescale O to the new maximum (and V scale unit); biased V codes:
      //      also take off the bias the tile's MMAs are about to add ----
      if constexpr (C::kVBias) {
        float ps[4] = {0.f, 0.f, 0.f, 0.f};  // column sums of P^T: heads 2 q4, 2 q4 + 1 (rows g, g + 8 alike)
        const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
        mma_16816(ps, ones, pb[0][0], pb[0][1], false);
        const float b0 = -C::kBiasLo * ps[0], b1 = -C::kBiasLo * ps[1];
        const float b2 = -C::kBiasHi * ps[0], b3 = -C::kBiasHi * ps[1];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          oacc[i][0] = fmaf(oacc[i][0], al0, b0);
          oacc[i][1] = fmaf(oacc[i][1], al1, b1);
          oacc[i][2] = fmaf(oacc[i][2], al0, b2);
          oacc[i][3] = fmaf(oacc[i][3], al1, b3);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          oacc[i][0] *= al0;
          oacc[i][1] *= al1;
          oacc[i][2] *= al0;
          oacc[i][3] *= al1;
        }
      }
      // ---- O^T += V^T P^T ----
      const bool tail = ntok < kBS;
      if constexpr (C::kVInt4) {
        // 4-bit V: lane group g holds bytes 8 g .. 8 g + 7 of a row, i.e.
        // head_dim 16 g .. 16 g + 15, the same rows out_d gives the
        // one-byte layout.  Byte i gives m-tile i: its low nibbles are row
        // g, its high nibbles row g + 8.  Lanes with odd q4 read the two
        // tokens of a pair in the other order (rows of the other parity),
        // so each load spreads over all 32 banks; the byte permute's
        // selector swaps them back.  Masked tokens need no clearing: every
        // nibble decodes to a finite value and their P is 0.
        uint2 vr[4];
        const int flip = q4 & 1;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          vr[k] = *reinterpret_cast<const uint2 *>(vt + (tks[k] ^ flip) * (D / 2) + g * 8);
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const uint32_t x0 = w ? vr[0].y : vr[0].x, y0 = w ? vr[1].y : vr[1].x;
          const uint32_t x1 = w ? vr[2].y : vr[2].x, y1 = w ? vr[3].y : vr[3].x;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t a[4];
            int4_pair_to_f16x2_biased(prmt(x0, y0, vsel[b]), a[0], a[1]);
            int4_pair_to_f16x2_biased(prmt(x1, y1, vsel[b]), a[2], a[3]);
            mma_16816(oacc[4 * w + b], a, pb[0][0], pb[0][1], false);
          }
        }
      } else if constexpr (C::kCode8) {
        uint4 vr[4];  // tokens tk0..tk3, chunk g (head_dim 16 g .. 16 g + 15)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          vr[k] = *reinterpret_cast<const uint4 *>(vt + tks[k] * 128 + ((g ^ (tks[k] & 7)) << 4));
          if (tail && tks[k] >= ntok) vr[k] = make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t x0 = word(vr[0], w), y0 = word(vr[1], w), x1 = word(vr[2], w), y1 = word(vr[3], w);
          uint32_t a[4], b[4];
          if constexpr (C::kVBias) {  // INT8
            int8x4_to_f16x2_biased(prmt(x0, y0, 0x5140), a[0], a[1]);
            int8x4_to_f16x2_biased(prmt(x1, y1, 0x5140), a[2], a[3]);
            int8x4_to_f16x2_biased(prmt(x0, y0, 0x7362), b[0], b[1]);
            int8x4_to_f16x2_biased(prmt(x1, y1, 0x7362), b[2], b[3]);
          } else {
            code4_to_f16x2<C::VT>(prmt(x0, y0, 0x5140), a[0], a[1]);
            code4_to_f16x2<C::VT>(prmt(x1, y1, 0x5140), a[2], a[3]);
            code4_to_f16x2<C::VT>(prmt(x0, y0, 0x7362), b[0], b[1]);
            code4_to_f16x2<C::VT>(prmt(x1, y1, 0x7362), b[2], b[3]);
          }
          mma_16816(oacc[2 * w], a, pb[0][0], pb[0][1], false);
          mma_16816(oacc[2 * w + 1], b, pb[0][0], pb[0][1], false);
        }
      } else {
        uint4 vr[4][2];  // [token][half], chunk g
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            vr[k][h] = *reinterpret_cast<const uint4 *>(vt + h * 2048 + tks[k] * 128 + ((g ^ (tks[k] & 7)) << 4));
            if (tail && tks[k] >= ntok) vr[k][h] = make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int h = i >> 2, w = i & 3;
          const uint32_t x0 = word(vr[0][h], w), y0 = word(vr[1][h], w);
          const uint32_t x1 = word(vr[2][h], w), y1 = word(vr[3][h], w);
          const uint32_t a[4] = {prmt(x0, y0, 0x5410), prmt(x0, y0, 0x7632), prmt(x1, y1, 0x5410),
                                 prmt(x1, y1, 0x7632)};
          mma_16816(oacc[i], a, pb[0][0], pb[0][1], C::kBf16);
          if constexpr (C::kBf16) mma_16816(oacc[i], a, pb[1][0], pb[1][1], true);
        }
      }
    }
    __syncwarp();  // the stage is free again
    if (n + C::kStages < count) issue(n + C::kStages, 0);
  }
  griddep_launch_dependents();
  flush(cur_item, whole_start && saw_last);
}

template <int G, int CDT, int QDT>
struct MmaInstance {
  using C = MmaCfg<G, CDT, QDT>;
  static cudaError_t prepare(DecodeShape *shape) {
    static int cached = -1;
    if (cached < 0) {
      cudaError_t e = cudaFuncSetAttribute(paged_decode_mma_kernel<G, CDT, QDT>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
      if (e != cudaSuccess) return e;
      int n = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_mma_kernel<G, CDT, QDT>, C::kThreads,
                                                        C::kSmem);
      if (e != cudaSuccess) return e;
      cached = n > 0 ? n : 1;
    }
    *shape = DecodeShape{cached, C::kWarps};
    return cudaSuccess;
  }
  static cudaError_t launch(const DecodeParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv, int grid,
                            int64_t *launches) {
    const cudaError_t e = launch_decode(paged_decode_mma_kernel<G, CDT, QDT>, grid, C::kThreads, C::kSmem,
                                        p.stream, p.programmatic, p, tmk, tmv);
    if (e == cudaSuccess) *launches += 1;
    return e;
  }
};

template <int CDT, int QDT>
cudaError_t decode_mma_family(int G, int op, const DecodeParams *p, const CUtensorMap *tmk,
                              const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape) {
  switch (G) {
#define PKV_MMA_CASE(GG)                                                   \
  case GG:                                                                 \
    if (op == kDecodePrepare) return MmaInstance<GG, CDT, QDT>::prepare(shape); \
    return MmaInstance<GG, CDT, QDT>::launch(*p, *tmk, *tmv, grid, launches);
    PKV_MMA_CASE(1)
    PKV_MMA_CASE(2)
    PKV_MMA_CASE(4)
    PKV_MMA_CASE(8)
#undef PKV_MMA_CASE
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
