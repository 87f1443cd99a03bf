// Pieces shared by the grouped expert GEMMs (MXFP4 and FP8 weights).
#pragma once
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {

constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;   // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Work item w -> (token tile, weight-row item).  Items are ordered expert by
// expert, and inside an expert weight-row item major, token tile minor, so the
// token tiles of one expert that share a weight item run on neighbouring
// CTAs at about the same time and read those weights through L2 once.  The
// tiles of expert e are [tile_off[e]/BN, tile_off[e+1]/BN) and its items
// [first*MT, (first+count)*MT), so tiles[w / MT] is one of expert e's tiles.
// Split activation layout (see launch_quant_gather): the hi row of padded
// assignment row r; its lo row is BN rows further.
__host__ __device__ __forceinline__ size_t split_row_hi(int r, int BN) {
  return static_cast<size_t>(r / BN) * 2 * BN + r % BN;
}

template <int BN>
__device__ __forceinline__ int4 decode_item(const MoeGemmParams& p, int w, int& mt) {
  const int e = p.tiles[w / p.MT].x;
  const int first = p.tile_off[e] / BN;
  const int count = p.tile_off[e + 1] / BN - first;
  const int local = w - first * p.MT;
  mt = local / count;
  return p.tiles[first + local % count];
}


}  // namespace lmoe
