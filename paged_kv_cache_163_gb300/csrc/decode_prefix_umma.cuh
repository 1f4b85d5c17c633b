// Cascade decode for shared prefixes: the prefix kernel on the fifth-
// generation tensor cores (tcgen05 MMAs with accumulators in tensor memory),
// for 16-bit caches and head_dim 128.
//
// What it computes is the same as paged_prefix_kernel (decode_prefix.cuh):
// for up to 128 query rows (a group's members' GQA heads of one KV head) and
// a chunk of the group's shared 16-token tiles ("KV Cache 与 vLLM" (zwxr.cn)
// §3.3, "KV Cache优化实战" §5.2), the fp32 partial (m, l, o) of
// softmax(scale q K^T) V over the chunk, in the decode workspace's partial
// format, for the decode kernel's log-sum-exp merge.
//
// How:
//  * The chunk is streamed in sub-chunks of up to four tiles (64 tokens).
//    Two producer warps copy each sub-chunk's K tiles and V tiles by tensor
//    TMA (the decode's 128-byte-swizzle maps) into two three-stage rings; a
//    K stage is released as soon as its S MMAs are done, a V stage after
//    its P V MMAs.
//  * One thread issues the MMAs.  S_j = Q K_j^T is one M = 128, N = 16 x
//    tiles, K = 128 product (8 instructions of K = 16), written to one of two
//    tensor-memory S buffers.  O += P_j V_j accumulates in tensor memory
//    across the whole chunk: per 16-token k-step two N = 64 instructions
//    (head_dim 0-63 and 64-127), V read as an MN-major operand straight from
//    the TMA tile; for bf16 a second pair adds the low half of P, so the
//    probabilities keep 16 bits of precision.
//  * Four softmax warps own one query row per thread (its tensor-memory
//    lane).  For sub-chunk j a thread reads its S row and forms P_j against
//    a reference maximum that may lag the row's true maximum by up to 2^8
//    (so P stays <= 256); only when the maximum moves further does the warp
//    rescale its rows of O in tensor memory (after the previous P V MMAs are
//    done).  P_j goes to shared memory in the MMA's layout; the two S and two
//    P buffers let the MMAs of j + 1 and the softmax of j overlap.
//  * tcgen05.ld / st / wait are warp-collective, so every branch that guards
//    one is uniform across the warp.  Every wait is bounded; a wait that runs
//    out reports PKV_DEVERR_WAIT_TIMEOUT and the CTA winds down (the tensor
//    memory is always freed, after every issued MMA has completed).
//
// Operand layouts (shared memory, 128-byte swizzle, 1024-byte atoms of
// 8 rows x 128 bytes):
//  * Q: two halves (head_dim 0-63, 64-127) of 128 rows x 128 bytes, K-major.
//  * K of a sub-chunk: two halves of 64 token rows x 128 bytes, K-major
//    (tile i's TMA boxes at i x 2048 in each half).
//  * V of a sub-chunk: the same layout; as the B operand of O = P V its
//    contiguous dimension is N (head_dim), so it is MN-major.
//  * P: 128 rows x 64 tokens x 2 bytes, K-major.
#pragma once

#include "decode_prefix.cuh"

namespace pkv {

// ---- tcgen05 helpers (inline PTX) --------------------------------------------------

// Instruction descriptor of a kind::f16 MMA: fp32 accumulator, A and B both
// f16 or both bf16, A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n, bool bf16, bool b_mn_major) {
  return (1u << 4)                                      // D format: f32
         | ((bf16 ? 1u : 0u) << 7)                      // A format: f16 / bf16
         | ((bf16 ? 1u : 0u) << 10)                     // B format: f16 / bf16
         | ((b_mn_major ? 1u : 0u) << 16)               // B major-ness (A stays K-major)
         | (static_cast<uint32_t>(n >> 3) << 17)        // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);       // M / 16
}

// Shared-memory matrix descriptor: start address, leading- and stride-dimension
// byte offsets, descriptor version 1, 128-byte swizzle.
__host__ __device__ constexpr uint64_t umma_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Whole warp: allocate `cols` tensor-memory columns; the address lands in *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

// Whole warp: 32 consecutive fp32 columns of this thread's lane (the warp's
// lane quarter is encoded in taddr's lane field).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Tensor-memory stores of 32 consecutive fp32 columns of this thread's lane (whole warp).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- configuration -------------------------------------------------------------------

template <int G, int CDT, int QDT>
struct UmmaPrefixCfg {
  static_assert(CDT == QDT && (CDT == PKV_F16 || CDT == PKV_BF16), "16-bit caches with a query of the same type");
  static constexpr bool kBf16 = CDT == PKV_BF16;
  static constexpr int kD = 128;
  static constexpr int kRows = kPrefixRows;                 // 128: the MMA's M, one per softmax thread
  static constexpr int kSubTiles = 4;                       // tiles per sub-chunk
  static constexpr int kSubTok = kSubTiles * kBS;           // 64 tokens
  static constexpr int kHalfRows = kSubTok * 128;           // one head_dim half of a sub-chunk's K (or V): 8 KB
  static constexpr int kKV = 2 * kHalfRows;                 // K (or V) of a sub-chunk: 16 KB
  static constexpr int kStages = 3;                         // K ring and V ring, each
  static constexpr int kQHalf = kRows * 128;                // one head_dim half of Q: 16 KB
  static constexpr int kP = kRows * 128;                    // P of a sub-chunk: 16 KB
  static constexpr int kPParts = kBf16 ? 2 : 1;             // bf16: high and low halves
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQHalf;
  static constexpr int kOffV = kOffK + kStages * kKV;
  static constexpr int kOffP = kOffV + kStages * kKV;
  static constexpr int kOffBars = kOffP + 2 * kPParts * kP;
  // kfull, kempty, vfull, vempty [kStages] each; sfull, sfree, pfull, odone [2] each; q; done
  static constexpr int kBars = 4 * kStages + 4 * 2 + 2;
  static constexpr int kSmemUsed = kOffBars + kBars * 8 + 16;
  static constexpr int kSmem = 1024 + kSmemUsed;            // + alignment slack
  static constexpr int kKWarp = 4;                          // K copies (and the tensor-memory allocation)
  static constexpr int kVWarp = 5;                          // V copies
  static constexpr int kMmaWarp = 6;
  static constexpr int kThreads = 7 * 32;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kColS = 0;                      // S buffers: columns 0-63, 64-127
  static constexpr uint32_t kColO = 128;                    // O: columns 128-255
  // A row's probabilities are formed against a maximum that may lag the true
  // one by up to 2^kLag (they stay <= 2^kLag); O is rescaled only past that.
  static constexpr float kLag = 8.f;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kKV % 1024 == 0 && kOffP % 1024 == 0,
                "1024-byte swizzle atoms");
};

// ---- the kernel ------------------------------------------------------------------------

template <int G, int CDT, int QDT>
__global__ void __launch_bounds__(UmmaPrefixCfg<G, CDT, QDT>::kThreads, 1)
    paged_prefix_umma_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ PrefixParams pp,
                             const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using C = UmmaPrefixCfg<G, CDT, QDT>;
  constexpr int D = C::kD;
  constexpr int S = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBars);
  uint64_t *kfull = bars;             // [S] a stage's K copies landed (tx count)
  uint64_t *kempty = bars + S;        // [S] S_j, which reads the stage's K, is done (commit)
  uint64_t *vfull = bars + 2 * S;     // [S] V copies landed
  uint64_t *vempty = bars + 3 * S;    // [S] O += P_j V_j is done (commit)
  uint64_t *sfull = bars + 4 * S;     // [2] S_j written (commit)
  uint64_t *sfree = sfull + 2;        // [2] S_j read by the softmax threads (128 arrivals)
  uint64_t *pfull = sfree + 2;        // [2] P_j written and O rescaled if needed (128 arrivals)
  uint64_t *odone = pfull + 2;        // [2] O += P_j V_j done (commit), by j & 1
  uint64_t *qbar = odone + 2;         // Q written (128 arrivals)
  uint64_t *done = qbar + 1;          // every MMA this CTA issued has completed (commit)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::kBars);
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // this CTA's unit: group, KV head, chunk, row block (as paged_prefix_kernel)
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
  const int nsub = (count + C::kSubTiles - 1) / C::kSubTiles;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(kfull + s, 1);
      mbar_init(kempty + s, 1);
      mbar_init(vfull + s, 1);
      mbar_init(vempty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull + b, 1);
      mbar_init(sfree + b, C::kRows);
      mbar_init(pfull + b, C::kRows);
      mbar_init(odone + b, 1);
    }
    mbar_init(qbar, C::kRows);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::kKWarp) tmem_alloc(tmem_slot, C::kTmemCols);
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = *tmem_slot;

  griddep_wait();               // the caches and queries may come from the kernel before this one
  griddep_launch_dependents();  // the decode may start on the free SMs now

  // A bounded wait; once any thread of the CTA gave up, the others stop waiting too.
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort_flag = 1;
    report(p.d_error, PKV_DEVERR_WAIT_TIMEOUT);
    return false;
  };

  if (warp == C::kKWarp || warp == C::kVWarp) {
    // ---- producers: one warp streams the K tiles, one the V tiles, each through its ring ----
    const bool is_k = warp == C::kKWarp;
    uint64_t *fullb = is_k ? kfull : vfull;
    uint64_t *emptyb = is_k ? kempty : vempty;
    const CUtensorMap *map = is_k ? &tmk : &tmv;
    uint8_t *ring = smem + (is_k ? C::kOffK : C::kOffV);
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int tpb = p.tiles_per_block;
      const int32_t *table = p.block_tables + static_cast<int64_t>(grp.lead) * p.max_blocks_per_seq;
      for (int j = 0; j < nsub; ++j) {
        const int st = j % S;
        if (j >= S && !wait(emptyb + st, ((j / S) - 1) & 1)) break;
        uint8_t *dst = ring + st * C::kKV;
        const int nt = min(C::kSubTiles, count - j * C::kSubTiles);
        int64_t tile[C::kSubTiles];
        int valid = 0;
        for (int i = 0; i < nt; ++i) {
          const int lb = t0 + j * C::kSubTiles + i;
          const int32_t blk = __ldg(table + lb / tpb);
          if (blk < 0 || blk >= p.num_blocks) {
            if (is_k) report(p.d_error, PKV_DEVERR_BAD_BLOCK);  // stale bytes are used; the flag says so
            tile[i] = -1;
          } else {
            tile[i] = (static_cast<int64_t>(blk) * p.num_kv_heads + kvh) * tpb + lb % tpb;
            ++valid;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(fullb + st, static_cast<uint32_t>(valid) * 2 * 2048);
        for (int i = 0; i < nt; ++i) {
          if (tile[i] < 0) continue;
          const int row = static_cast<int>(tile[i] * kBS);
          tma_load_2d(dst + i * 2048, map, 0, row, fullb + st, pol);
          tma_load_2d(dst + C::kHalfRows + i * 2048, map, 64, row, fullb + st, pol);
        }
      }
      // the copies of the last stages land before the CTA can retire (bounded)
      for (int j = nsub > S ? nsub - S : 0; j < nsub; ++j) mbar_wait(fullb + j % S, (j / S) & 1);
    }
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    // ---- MMA issuer: S_j = Q K_j^T, then O += P_{j-1} V_{j-1} ----
    if (lane == 0) {
      const uint32_t base = smem_addr(smem);
      const uint32_t q_addr = base + C::kOffQ;
      constexpr uint32_t kIdescPV = umma_idesc_f16(128, 64, C::kBf16, true);
      bool ok = wait(qbar, 0);
      for (int j = 0; ok && j <= nsub; ++j) {
        if (j < nsub) {
          const int st = j % S;
          const int nt = min(C::kSubTiles, count - j * C::kSubTiles);
          ok = wait(kfull + st, (j / S) & 1) && (j < 2 || wait(sfree + (j & 1), ((j - 2) >> 1) & 1));
          if (!ok) break;
          tmem_fence_after();
          const uint32_t k_addr = base + C::kOffK + st * C::kKV;
          const uint32_t idesc = umma_idesc_f16(128, 16 * nt, C::kBf16, false);
          const uint32_t d = tmem + C::kColS + 64 * (j & 1);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::kQHalf + (k & 3) * 32;
            const uint32_t koff = (k >> 2) * C::kHalfRows + (k & 3) * 32;
            umma_f16(d, umma_sdesc(q_addr + off, 1024, 1024), umma_sdesc(k_addr + koff, 1024, 1024), idesc, k > 0);
          }
          umma_commit(sfull + (j & 1));
          umma_commit(kempty + st);
        }
        if (j >= 1) {
          const int jp = j - 1;
          const int st = jp % S;
          const int nt = min(C::kSubTiles, count - jp * C::kSubTiles);
          ok = wait(pfull + (jp & 1), (jp >> 1) & 1) && wait(vfull + st, (jp / S) & 1);
          if (!ok) break;
          tmem_fence_after();
          const uint32_t v_addr = base + C::kOffV + st * C::kKV;
          const uint32_t p_addr = base + C::kOffP + (jp & 1) * C::kPParts * C::kP;
          for (int t = 0; t < nt; ++t) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t bdesc = umma_sdesc(v_addr + h * C::kHalfRows + t * 2048, 1024, 1024);
              umma_f16(tmem + C::kColO + 64 * h, umma_sdesc(p_addr + t * 32, 1024, 1024), bdesc, kIdescPV,
                       jp > 0 || t > 0);
              if constexpr (C::kBf16)
                umma_f16(tmem + C::kColO + 64 * h, umma_sdesc(p_addr + C::kP + t * 32, 1024, 1024), bdesc, kIdescPV,
                         true);
            }
          }
          umma_commit(odone + (jp & 1));
          umma_commit(vempty + st);
        }
      }
      // nothing may still write tensor memory when it is freed (bounded wait)
      umma_commit(done);
      mbar_wait(done, 0);
    }
    __syncwarp();
  } else {
    // ---- softmax warps: thread = query row r (tensor-memory lane r) ----
    const int r = tid;  // warps 0-3
    const int rn = rb * C::kRows + r;
    const int mi = rn / G, gr = rn - (rn / G) * G;
    const bool real = mi < grp.members;
    const int hq = p.num_kv_heads * G;
    int b = 0;
    if (real) b = pp.member[grp.member0 + mi];
    // Q row into the K-major swizzled layout (zeros for rows past the members)
    {
      const uint4 *src = real ? reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(b) * hq + kvh * G + gr) * D * 2)
                              : nullptr;
#pragma unroll
      for (int c = 0; c < 16; ++c) {  // 16-byte chunks of the 256-byte row
        const uint4 v = real ? src[c] : make_uint4(0u, 0u, 0u, 0u);
        const int h = c >> 3, cc = c & 7;
        *reinterpret_cast<uint4 *>(smem + C::kOffQ + h * C::kQHalf + (r >> 3) * 1024 + (r & 7) * 128 +
                                   ((cc ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      mbar_arrive(qbar);
    }
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_row = tmem + lane_base + C::kColO;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;

    // tcgen05.ld / st / wait are warp-collective (.sync.aligned): every
    // decision that guards one is made for the whole warp (uwait: a bounded
    // wait whose result all 32 lanes share).
    auto uwait = [&](uint64_t *bar, uint32_t parity) -> bool { return __all_sync(kFull, wait(bar, parity)); };
    bool ok = true;
    for (int j = 0; ok && j < nsub; ++j) {
      const int nt = min(C::kSubTiles, count - j * C::kSubTiles);
      if (!(ok = uwait(sfull + (j & 1), (j >> 1) & 1))) break;
      tmem_fence_after();
      float s[64];
      {
        float v[32];
        tmem_ld32(tmem + lane_base + C::kColS + 64 * (j & 1), v);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[e] = v[e];
        tmem_ld32(tmem + lane_base + C::kColS + 64 * (j & 1) + 32, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) s[32 + e] = v[e];
        tmem_ld_wait();
      }
      tmem_fence_before();
      mbar_arrive(sfree + (j & 1));
      float mx = -INFINITY;
      if (nt == C::kSubTiles) {
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          s[e] *= sl2;
          mx = fmaxf(mx, s[e]);
        }
      } else {
        const int ncol = 16 * nt;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          s[e] = e < ncol ? s[e] * sl2 : -INFINITY;
          mx = fmaxf(mx, s[e]);
        }
      }
      // A row whose maximum moved past its reference by more than 2^kLag takes
      // a new reference; O (all earlier sub-chunks) and l change units.  The
      // tensor-memory rescale runs for the whole warp (factor 1 on rows that
      // keep their reference).
      const bool mine = mx > m_run + C::kLag;
      if (__any_sync(kFull, mine)) {
        const float m_new = mine ? mx : m_run;
        if (j > 0) {
          if (!(ok = uwait(odone + ((j - 1) & 1), ((j - 1) >> 1) & 1))) break;
          tmem_fence_after();
          const float a = mine ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v[32];
            tmem_ld32(o_row + 32 * q, v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= a;
            tmem_st32(o_row + 32 * q, v);
          }
          tmem_st_wait();
          l_run *= a;
        }
        m_run = m_new;
      }
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        s[e] = fast_exp2(s[e] - m_run);  // 0 past the sub-chunk's tokens; at most 2^kLag
        sum += s[e];
      }
      l_run += sum;
      // P buffer j & 1 was read by O += P_{j-2} V_{j-2}
      if (j >= 2 && !(ok = uwait(odone + (j & 1), ((j - 2) >> 1) & 1))) break;
      uint8_t *pb = smem + C::kOffP + (j & 1) * C::kPParts * C::kP + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // tokens 8c .. 8c + 7
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = s[8 * c + 2 * u], bb = s[8 * c + 2 * u + 1];
          hi[u] = pack2<CDT>(a, bb);
          if constexpr (C::kBf16) {
            const float2 h2 = unpack2<CDT>(hi[u]);
            lo[u] = pack2<CDT>(a - h2.x, bb - h2.y);
          }
        }
        const int off = (c ^ (r & 7)) << 4;
        *reinterpret_cast<uint4 *>(pb + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if constexpr (C::kBf16) *reinterpret_cast<uint4 *>(pb + C::kP + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      tmem_fence_before();
      mbar_arrive(pfull + (j & 1));
    }
    // ---- partial (m, l, o) of this row and chunk, natural head_dim order ----
    if (ok) ok = uwait(odone + ((nsub - 1) & 1), ((nsub - 1) >> 1) & 1);
    if (ok) {
      tmem_fence_after();
      const int64_t slot = real ? pp.base[b] + static_cast<int64_t>(kvh) * grp.chunks + chunk : 0;
      float4 *op = reinterpret_cast<float4 *>(pp.o + (slot * G + gr) * D);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[32];
        tmem_ld32(o_row + 32 * q, v);
        tmem_ld_wait();
        if (real) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) op[(32 * q + e) / 4] = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      if (real) {
        pp.ml[(slot * G + gr) * 2] = m_run;
        pp.ml[(slot * G + gr) * 2 + 1] = l_run;
      }
    }
  }

  tmem_fence_before();
  __syncthreads();
  if (warp == C::kKWarp) {
    tmem_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int G, int CDT, int QDT>
cudaError_t launch_prefix_umma_instance(const DecodeParams &p, const PrefixParams &pp, const CUtensorMap &tmk,
                                        const CUtensorMap &tmv, int grid) {
  using C = UmmaPrefixCfg<G, CDT, QDT>;
  static bool ready = false;
  if (!ready) {
    cudaError_t e = cudaFuncSetAttribute(paged_prefix_umma_kernel<G, CDT, QDT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    ready = true;
  }
  return launch_decode(paged_prefix_umma_kernel<G, CDT, QDT>, grid, C::kThreads, C::kSmem, p.stream, 0, p, pp, tmk,
                       tmv);
}

template <int CDT, int QDT>
cudaError_t prefix_umma_family(int G, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                               const CUtensorMap *tmv, int grid) {
  switch (G) {
    case 1: return launch_prefix_umma_instance<1, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 2: return launch_prefix_umma_instance<2, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 4: return launch_prefix_umma_instance<4, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
    case 8: return launch_prefix_umma_instance<8, CDT, QDT>(*p, *pp, *tmk, *tmv, grid);
  }
  return cudaErrorNotSupported;
}

}  // namespace pkv
