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

// Dynamic item distribution of the persistent expert GEMMs.  CTA b starts
// with item b; each later item is claimed from a global counter (zeroed by
// the kernel that runs before the GEMM on its stream) while the CTA's
// producer is still loading its current item, so CTAs that start late (their
// SMs held by a concurrent kernel) take fewer items.  The producer thread
// publishes the CTA's item sequence through a ring in shared memory, which
// the MMA thread and the epilogue warps read in the same order; -1 ends it.
constexpr int kRingSlots = 4;
struct ItemRing {
  int item[kRingSlots];
  uint64_t full[kRingSlots], empty[kRingSlots];
};
// One thread.  Consumers of a slot: the MMA thread and one lane of each of
// the epi_warps epilogue warps.
__device__ __forceinline__ void ring_init(ItemRing& r, int epi_warps) {
  for (int i = 0; i < kRingSlots; ++i) {
    mbar_init(&r.full[i], 1);
    mbar_init(&r.empty[i], 1 + epi_warps);
  }
}
// Producer: publish the n-th item (or -1).  False if the wait timed out.
__device__ __forceinline__ bool ring_put(ItemRing& r, uint32_t n, int w, int* err) {
  const uint32_t s = n % kRingSlots;
  if (n >= kRingSlots && !mbar_wait(&r.empty[s], ((n / kRingSlots) - 1) & 1, err, kErrTimeout)) return false;
  r.item[s] = w;
  mbar_arrive(&r.full[s]);
  return true;
}
// Consumer: the n-th item, -1 at the end, -2 if the wait timed out.  The
// slot is released at once (the item number is all a consumer keeps).
__device__ __forceinline__ int ring_take(ItemRing& r, uint32_t n, int* err) {
  const uint32_t s = n % kRingSlots;
  if (!mbar_wait(&r.full[s], (n / kRingSlots) & 1, err, kErrTimeout)) return -2;
  const int w = *reinterpret_cast<volatile int*>(&r.item[s]);
  mbar_arrive(&r.empty[s]);
  return w;
}
// Epilogue warp: lane 0 takes the item, the warp shares it.
__device__ __forceinline__ int ring_take_warp(ItemRing& r, uint32_t n, int* err) {
  int w = 0;
  if ((threadIdx.x & 31) == 0) w = ring_take(r, n, err);
  return __shfl_sync(0xFFFFFFFFu, w, 0);
}
// Producer: claim the next item (an index >= total means none).
__device__ __forceinline__ int claim_item(int* counter) {
  return static_cast<int>(gridDim.x) + atomicAdd(counter, 1);
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
