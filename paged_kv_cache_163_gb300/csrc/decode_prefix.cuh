// Cascade decode for shared prefixes: the prefix kernel.
//
// Sequences forked from one parent, or admitted through the prefix cache,
// hold the same physical blocks for their common prefix ("KV Cache 与
// vLLM" (zwxr.cn) §3.3, "KV Cache优化实战" §5.2).  Attention over those
// tiles is the same K and V against each member's own queries, so one CTA
// streams each shared tile once and attends it for up to 128 query rows
// (the members' GQA groups of one KV head), instead of every member reading
// the tile again.  Its output is an fp32 partial (m, l, o) per row and
// chunk of the prefix, in the decode workspace's partial format; the decode
// kernel then attends each member's own tiles and folds these partials into
// its log-sum-exp merge.  The sum is the same softmax; only the order of the
// fp32 additions changes.
//
// It runs beside the decode: it triggers its programmatic dependents at
// entry, the decode (launched as one, on the SMs this grid leaves free)
// streams the members' own tiles meanwhile, and waits for this grid only
// before its first merge that reads these partials.
//
// A CTA: compute warps of 8 kNT query rows each (kNT MMA n-tiles of 8), and
// one producer warp that streams the chunk's K / V tiles (the tensor-core
// decode's layout and TMA maps) through an 8-stage ring with full / empty
// mbarriers.  Per tile a compute warp does the decode's K Q^T and V^T P^T
// MMAs for its n-tiles, sharing the K and V fragment conversion between
// them.  Prefix tiles are always full (16 tokens).
#pragma once

#include "decode_mma.cuh"

namespace pkv {

template <int G, int CDT, int QDT>
struct PrefixCfg {
  using M = MmaCfg<G, CDT, QDT>;
  static constexpr int kNT = 2;                          // MMA n-tiles (8 query rows each) a warp
  static constexpr int kWarps = kPrefixRows / (8 * kNT);  // compute warps
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kStages = 8;
  static constexpr int kStage = round_up_c(M::kKV + 2 * M::kScale, 1024);  // K, V (swizzled, 1024-aligned), scales
  static constexpr int kSmem = 1024 + kStages * kStage + 128;
  static_assert(kWarps * 8 * kNT == kPrefixRows, "rows per CTA");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int G, int CDT, int QDT>
__global__ void __launch_bounds__(PrefixCfg<G, CDT, QDT>::kThreads, 1)
    paged_prefix_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ PrefixParams pp,
                        const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using PC = PrefixCfg<G, CDT, QDT>;
  using C = typename PC::M;
  constexpr int D = C::kD;
  constexpr int S = PC::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * PC::kStage);
  uint64_t *empty = full + S;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q4 = lane & 3;

  // this CTA's unit: group, KV head, chunk, row block
  int gi = 0;
  while (gi + 1 < pp.num_groups && static_cast<int>(blockIdx.x) >= pp.group[gi + 1].unit0) ++gi;
  const PrefixGroup &grp = pp.group[gi];
  int local = static_cast<int>(blockIdx.x) - grp.unit0;
  const int kvh = local % p.num_kv_heads;
  local /= p.num_kv_heads;
  const int chunk = local % grp.chunks;
  const int rb = local / grp.chunks;
  const int t0 = static_cast<int>(static_cast<int64_t>(chunk) * grp.tiles / grp.chunks);
  const int count = static_cast<int>(static_cast<int64_t>(chunk + 1) * grp.tiles / grp.chunks) - t0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, PC::kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  griddep_wait();              // the caches may come from the kernel before this one
  griddep_launch_dependents();  // the decode may start on the free SMs now

  if (warp == PC::kWarps) {  // ---- producer: the chunk's tiles through the ring ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int tpb = p.tiles_per_block;
      const int32_t *table = p.block_tables + static_cast<int64_t>(grp.lead) * p.max_blocks_per_seq;
      for (int i = 0; i < count; ++i) {
        const int st = i % S;
        if (i >= S && !mbar_wait(empty + st, ((i / S) - 1) & 1)) {
          report(p.d_error, PKV_DEVERR_WAIT_TIMEOUT);
          break;
        }
        uint8_t *tb = smem + st * PC::kStage;
        const int lb = t0 + i;
        const int32_t blk = __ldg(table + lb / tpb);
        fence_proxy_async_smem();
        if (blk < 0 || blk >= p.num_blocks) {
          report(p.d_error, PKV_DEVERR_BAD_BLOCK);
          mbar_arrive(full + st);  // nothing to wait for: the consumers use stale bytes, the flag says so
          continue;
        }
        const int64_t tile = (static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * tpb + lb % tpb;
        const int row = static_cast<int>(tile * kBS);
        mbar_arrive_expect_tx(full + st, C::kKV + 2 * C::kScale);
        if constexpr (C::kCode8) {
          tma_load_2d(tb, &tmk, 0, row, full + st, pol);
          if constexpr (C::kVInt4) {
            bulk_g2s(tb + C::kTile, p.v_cache + tile * C::kVTile, C::kVTile, full + st, pol);
          } else {
            tma_load_2d(tb + C::kTile, &tmv, 0, row, full + st, pol);
          }
          const int64_t si = scale_index(tile, p.tiles_per_block);
          if (p.tiles_per_block == 1) {  // K and V scales: one 128-byte unit
            bulk_g2s(tb + C::kKV, p.k_scale + si, 2 * C::kScale, full + st, pol);
          } else {
            bulk_g2s(tb + C::kKV, p.k_scale + si, C::kScale, full + st, pol);
            bulk_g2s(tb + C::kKV + C::kScale, p.v_scale + si, C::kScale, full + st, pol);
          }
        } else {
          tma_load_2d(tb, &tmk, 0, row, full + st, pol);
          tma_load_2d(tb + 2048, &tmk, 64, row, full + st, pol);
          tma_load_2d(tb + C::kTile, &tmv, 0, row, full + st, pol);
          tma_load_2d(tb + C::kTile + 2048, &tmv, 64, row, full + st, pol);
        }
      }
      // let the copies in flight land before the CTA can retire
      for (int i = count > S ? count - S : 0; i < count; ++i) mbar_wait(full + i % S, (i / S) & 1);
    }
    return;
  }

  // ---- compute warps: rows r0 .. r0 + 8 NT - 1 of the group's (member, head) rows ----
  constexpr int NT = PC::kNT;
  const int r0 = rb * kPrefixRows + warp * 8 * NT;
  const int hq = p.num_kv_heads * G;
  // Q^T B fragments per n-tile (column g = row r0 + 8 nt + g)
  uint32_t qb[NT][8][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int rn = r0 + 8 * nt + g;
    const int mi = rn / G, gr = rn - (rn / G) * G;
    const uint8_t *qrow = nullptr;
    if (mi < grp.members) {
      const int b = pp.member[grp.member0 + mi];
      qrow = p.q + (static_cast<size_t>(b) * hq + kvh * G + gr) * D * 2;
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int d0 = C::kCode8 ? 32 * q4 + 4 * s : 64 * (s >> 2) + 16 * q4 + 4 * (s & 3);
      uint2 raw = make_uint2(0u, 0u);
      if (qrow) raw = *reinterpret_cast<const uint2 *>(qrow + d0 * 2);
      if constexpr (C::kCode8 && QDT == PKV_BF16) {  // f16 MMA operands
        const float2 a = unpack2<QDT>(raw.x), b2 = unpack2<QDT>(raw.y);
        qb[nt][s][0] = pack2<PKV_F16>(a.x, a.y);
        qb[nt][s][1] = pack2<PKV_F16>(b2.x, b2.y);
      } else {
        qb[nt][s][0] = raw.x;
        qb[nt][s][1] = raw.y;
      }
    }
  }
  float oacc[NT][8][4];
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) oacc[nt][i][c] = 0.f;
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }
  float vunit = 1.f;
  const int tks[4] = {2 * q4, 2 * q4 + 1, 2 * q4 + 8, 2 * q4 + 9};
  uint32_t vsel[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) vsel[b] = (0x4400u + 0x1111u * b) ^ ((q4 & 1) ? 0x4444u : 0u);

#pragma unroll 1
  for (int i = 0; i < count; ++i) {
    const int st = i % S;
    if (!__all_sync(kFull, mbar_wait(full + st, (i / S) & 1))) {
      if (lane == 0) report(p.d_error, PKV_DEVERR_WAIT_TIMEOUT);
      return;
    }
    const uint8_t *kt = smem + st * PC::kStage;
    const uint8_t *vt = kt + C::kTile;
    const uint8_t *ab = kt + C::kKV;
    // ---- S^T = K Q^T for both n-tiles ----
    float sacc4[NT][2][4] = {};  // [n-tile][chain][c]
    if constexpr (C::kCode8) {
      uint4 kr[2][2];
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
        code4_to_f16x2<C::KT>(word(kr[0][s >> 2], s & 3), a[0], a[2]);
        code4_to_f16x2<C::KT>(word(kr[1][s >> 2], s & 3), a[1], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(sacc4[nt][s & 1], a, qb[nt][s][0], qb[nt][s][1], false);
      }
    } else {
      uint4 kr[2][2][2];
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
        const uint32_t a[4] = {word(kr[0][h][j], 2 * t), word(kr[1][h][j], 2 * t), word(kr[0][h][j], 2 * t + 1),
                               word(kr[1][h][j], 2 * t + 1)};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(sacc4[nt][s & 1], a, qb[nt][s][0], qb[nt][s][1], C::kBf16);
      }
    }
    // ---- scale, online softmax (base 2); V scales relative to the tile's largest ----
    float sc0 = p.scale_log2, sc1 = p.scale_log2;
    float w0 = 1.f, w1 = 1.f, ru = 1.f;
    if constexpr (C::kCode8) {
      const float *ksc = reinterpret_cast<const float *>(ab);
      sc0 *= ksc[g];
      sc1 *= ksc[g + 8];
      const float *vsc = reinterpret_cast<const float *>(ab + C::kScale);
      const float vs0 = vsc[g], vs1 = vsc[g + 8];
      float vmax = fmaxf(vs0, vs1);
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 4));
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 8));
      vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, 16));
      if (!(vmax > 0.f)) vmax = 1.f;
      const float rv = 1.f / vmax;
      w0 = vs0 * rv;
      w1 = vs1 * rv;
      ru = vunit * rv;
      vunit = vmax;
    }
    uint32_t pb[NT][2][2];  // [n-tile][hi / lo][b0, b1]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float sacc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) sacc[c] = sacc4[nt][0][c] + sacc4[nt][1][c];
      const float s00 = sacc[0] * sc0, s01 = sacc[1] * sc0, s10 = sacc[2] * sc1, s11 = sacc[3] * sc1;
      float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, o));
      }
      const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
      const float e0 = exp2f(m_run[nt][0] - mn0), e1 = exp2f(m_run[nt][1] - mn1);
      m_run[nt][0] = mn0;
      m_run[nt][1] = mn1;
      float p00 = exp2f(s00 - mn0), p01 = exp2f(s01 - mn1), p10 = exp2f(s10 - mn0), p11 = exp2f(s11 - mn1);
      l_run[nt][0] = l_run[nt][0] * e0 + (p00 + p10);
      l_run[nt][1] = l_run[nt][1] * e1 + (p01 + p11);
      const float al0 = e0 * ru, al1 = e1 * ru;  // O also changes units to the tile's V scale
      p00 *= w0;
      p01 *= w0;
      p10 *= w1;
      p11 *= w1;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        oacc[nt][m][0] *= al0;
        oacc[nt][m][1] *= al1;
        oacc[nt][m][2] *= al0;
        oacc[nt][m][3] *= al1;
      }
      if constexpr (C::kBf16) {
        const uint32_t h0 = pack2<PKV_BF16>(p00, p01), h1 = pack2<PKV_BF16>(p10, p11);
        const float2 e0 = unpack2<PKV_BF16>(h0), e1 = unpack2<PKV_BF16>(h1);
        const uint32_t l0 = pack2<PKV_BF16>(p00 - e0.x, p01 - e0.y), l1 = pack2<PKV_BF16>(p10 - e1.x, p11 - e1.y);
        pb[nt][0][0] = movmatrix_t(h0);
        pb[nt][0][1] = movmatrix_t(h1);
        pb[nt][1][0] = movmatrix_t(l0);
        pb[nt][1][1] = movmatrix_t(l1);
      } else {
        pb[nt][0][0] = movmatrix_t(pack2<PKV_F16>(p00, p01));
        pb[nt][0][1] = movmatrix_t(pack2<PKV_F16>(p10, p11));
        pb[nt][1][0] = pb[nt][1][1] = 0u;
      }
    }
    // ---- O^T += V^T P^T for both n-tiles (V fragments converted once) ----
    if constexpr (C::kVInt4) {
      uint2 vr[4];
      const int flip = q4 & 1;
#pragma unroll
      for (int k = 0; k < 4; ++k) vr[k] = *reinterpret_cast<const uint2 *>(vt + (tks[k] ^ flip) * (D / 2) + g * 8);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t x0 = w ? vr[0].y : vr[0].x, y0 = w ? vr[1].y : vr[1].x;
        const uint32_t x1 = w ? vr[2].y : vr[2].x, y1 = w ? vr[3].y : vr[3].x;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t a[4];
          int4_pair_to_f16x2(prmt(x0, y0, vsel[b]), a[0], a[1]);
          int4_pair_to_f16x2(prmt(x1, y1, vsel[b]), a[2], a[3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(oacc[nt][4 * w + b], a, pb[nt][0][0], pb[nt][0][1], false);
        }
      }
    } else if constexpr (C::kCode8) {
      uint4 vr[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) vr[k] = *reinterpret_cast<const uint4 *>(vt + tks[k] * 128 + ((g ^ (tks[k] & 7)) << 4));
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t x0 = word(vr[0], w), y0 = word(vr[1], w), x1 = word(vr[2], w), y1 = word(vr[3], w);
        uint32_t a[4], b[4];
        code4_to_f16x2<C::VT>(prmt(x0, y0, 0x5140), a[0], a[1]);
        code4_to_f16x2<C::VT>(prmt(x1, y1, 0x5140), a[2], a[3]);
        code4_to_f16x2<C::VT>(prmt(x0, y0, 0x7362), b[0], b[1]);
        code4_to_f16x2<C::VT>(prmt(x1, y1, 0x7362), b[2], b[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816(oacc[nt][2 * w], a, pb[nt][0][0], pb[nt][0][1], false);
          mma_16816(oacc[nt][2 * w + 1], b, pb[nt][0][0], pb[nt][0][1], false);
        }
      }
    } else {
      uint4 vr[4][2];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          vr[k][h] = *reinterpret_cast<const uint4 *>(vt + h * 2048 + tks[k] * 128 + ((g ^ (tks[k] & 7)) << 4));
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int h = m >> 2, w = m & 3;
        const uint32_t x0 = word(vr[0][h], w), y0 = word(vr[1][h], w);
        const uint32_t x1 = word(vr[2][h], w), y1 = word(vr[3][h], w);
        const uint32_t a[4] = {prmt(x0, y0, 0x5410), prmt(x0, y0, 0x7632), prmt(x1, y1, 0x5410),
                               prmt(x1, y1, 0x7632)};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma_16816(oacc[nt][m], a, pb[nt][0][0], pb[nt][0][1], C::kBf16);
          if constexpr (C::kBf16) mma_16816(oacc[nt][m], a, pb[nt][1][0], pb[nt][1][1], true);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + st);  // this warp is done with the stage
  }

  // ---- partials: rows r0 + 8 nt + 2 q4 + j ----
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float lt = l_run[nt][j];
      lt += __shfl_xor_sync(kFull, lt, 4);
      lt += __shfl_xor_sync(kFull, lt, 8);
      lt += __shfl_xor_sync(kFull, lt, 16);
      const int rn = r0 + 8 * nt + 2 * q4 + j;
      const int mi = rn / G, gr = rn - (rn / G) * G;
      if (mi >= grp.members) continue;
      const int b = pp.member[grp.member0 + mi];
      const int64_t slot = pp.base[b] + static_cast<int64_t>(kvh) * grp.chunks + chunk;
      float *op = pp.o + (slot * G + gr) * D;
#pragma unroll
      for (int ib = 0; ib < 8; ib += 4) {
        float4 *dst = reinterpret_cast<float4 *>(op + out_d<C::kCode8>(g, ib, 0));
        dst[0] = make_float4(oacc[nt][ib][j] * vunit, oacc[nt][ib][2 + j] * vunit, oacc[nt][ib + 1][j] * vunit,
                             oacc[nt][ib + 1][2 + j] * vunit);
        dst[1] = make_float4(oacc[nt][ib + 2][j] * vunit, oacc[nt][ib + 2][2 + j] * vunit,
                             oacc[nt][ib + 3][j] * vunit, oacc[nt][ib + 3][2 + j] * vunit);
      }
      if (g == 0) {
        pp.ml[(slot * G + gr) * 2] = m_run[nt][j];
        pp.ml[(slot * G + gr) * 2 + 1] = lt;
      }
    }
  }
}

template <int G, int CDT, int QDT>
cudaError_t launch_prefix_instance(const DecodeParams &p, const PrefixParams &pp, const CUtensorMap &tmk,
                                   const CUtensorMap &tmv, int grid) {
  using PC = PrefixCfg<G, CDT, QDT>;
  static bool ready = false;
  if (!ready) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefix_kernel<G, CDT, QDT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PC::kSmem);
    if (e != cudaSuccess) return e;
    ready = true;
  }
  return launch_decode(paged_prefix_kernel<G, CDT, QDT>, grid, PC::kThreads, PC::kSmem, p.stream, 0, p, pp, tmk,
                       tmv);
}

template <int CDT, int QDT>
cudaError_t prefix_family(int G, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                          const CUtensorMap *tmv, int grid) {
  switch (G) {
    case 1: return launch_prefix_instance<1, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 2: return launch_prefix_instance<2, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 4: return launch_prefix_instance<4, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 8: return launch_prefix_instance<8, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
