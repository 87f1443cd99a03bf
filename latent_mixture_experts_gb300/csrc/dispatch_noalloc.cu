// Token -> expert dispatch for callers that cannot allocate device memory.
//
// lmoe_create sizes a workspace with cudaMalloc, which some callers cannot
// do: code running inside a CUDA-graph capture that must not allocate,
// plug-ins of a host framework that owns the device memory budget, or
// allocator-free runtimes.  lmoe_dispatch_noalloc needs no handle: its
// scratch (per-chunk expert histograms, padded rows, the tile list) is the
// file-scope device array below, which every GPU that loads this library
// holds until the process exits (about 2.4 MiB).
#include <mutex>

#include "../../include/lmoe.h"
#include "lmoe_internal.h"

namespace lmoe {
namespace {

constexpr int kNoAllocMaxAssignments = LMOE_NOALLOC_MAX_ASSIGNMENTS;   // T * k
constexpr int kNoAllocMaxExperts = LMOE_NOALLOC_MAX_EXPERTS;
constexpr int kNoAllocChunks = kNoAllocMaxAssignments / kDispatchChunk;
constexpr int kNoAllocBN = 16;
constexpr int kNoAllocMaxTiles = kNoAllocMaxAssignments / kNoAllocBN + kNoAllocMaxExperts + 1;
static_assert(kNoAllocMaxExperts <= kMaxExperts, "dispatch scan limit");
static_assert(kNoAllocMaxAssignments % kDispatchChunk == 0, "whole chunks");

// Byte offsets inside the scratch array (each 256-byte aligned).
constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
constexpr size_t kOffBlockcnt = 0;
constexpr size_t kOffInvPad = align256(kOffBlockcnt + sizeof(int32_t) * kNoAllocChunks * kNoAllocMaxExperts);
constexpr size_t kOffTileOff = align256(kOffInvPad + sizeof(int32_t) * kNoAllocMaxAssignments);
constexpr size_t kOffNtiles = align256(kOffTileOff + sizeof(int32_t) * (kNoAllocMaxExperts + 1));
constexpr size_t kOffTiles = align256(kOffNtiles + sizeof(int32_t) * 4);
constexpr size_t kScratchBytes = align256(kOffTiles + sizeof(int4) * kNoAllocMaxTiles);

static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device, looked up
// once per device.  In host code the symbol is only a host-side stand-in, so
// kernels must be given this address, never the symbol itself.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace lmoe

using namespace lmoe;

extern "C" lmoe_status lmoe_dispatch_noalloc(const int32_t* topk_idx, int T, int k, int n_experts, int32_t* counts,
                                             int32_t* offsets, int32_t* perm, cudaStream_t stream) {
  if (T < 0 || k < 1 || n_experts < 1) return LMOE_ERR_INVALID_ARG;
  if (n_experts > kNoAllocMaxExperts || static_cast<long long>(T) * k > kNoAllocMaxAssignments)
    return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!topk_idx || !counts || !offsets || !perm) return LMOE_ERR_INVALID_ARG;
  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return LMOE_ERR_CUDA;
  unsigned char* s = static_cast<unsigned char*>(base);
  DispatchBufs b;
  b.counts = counts;
  b.offsets = offsets;
  b.perm = perm;
  b.blockcnt = reinterpret_cast<int32_t*>(s + kOffBlockcnt);
  b.inv_pad = reinterpret_cast<int32_t*>(s + kOffInvPad);
  b.tile_off = reinterpret_cast<int32_t*>(s + kOffTileOff);
  b.ntiles = reinterpret_cast<int32_t*>(s + kOffNtiles);
  b.tiles = reinterpret_cast<int4*>(s + kOffTiles);
  b.err = nullptr;   // out-of-range ids are skipped, not reported
  e = launch_dispatch(topk_idx, T, k, n_experts, kNoAllocBN, b, stream);
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}
