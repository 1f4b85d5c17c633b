// Decode kernel instances: cache BF16, query BF16.
#include "decode.cuh"
#include "decode_mma.cuh"
#include "decode_prefix.cuh"
#include "decode_prefix_umma.cuh"

namespace pkv {

cudaError_t decode_call_bf16(int head_dim, int group, int op, const DecodeParams *p, int grid,
                         int64_t *launches, DecodeShape *shape) {
  return decode_family<PKV_BF16, PKV_BF16>(head_dim, group, op, p, grid, launches, shape);
}

cudaError_t decode_mma_call_bf16(int group, int op, const DecodeParams *p, const CUtensorMap *tmk,
                             const CUtensorMap *tmv, int grid, int64_t *launches, DecodeShape *shape) {
  return decode_mma_family<PKV_BF16, PKV_BF16>(group, op, p, tmk, tmv, grid, launches, shape);
}

cudaError_t prefix_call_bf16(int group, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                             const CUtensorMap *tmv, int grid) {
  return prefix_family<PKV_BF16, PKV_BF16>(group, p, pp, tmk, tmv, grid);
}

cudaError_t prefix_umma_call_bf16(int group, const DecodeParams *p, const PrefixParams *pp, const CUtensorMap *tmk,
                                 const CUtensorMap *tmv, int grid) {
  return prefix_umma_family<PKV_BF16, PKV_BF16>(group, p, pp, tmk, tmv, grid);
}

}  // namespace pkv
