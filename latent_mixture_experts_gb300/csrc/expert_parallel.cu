// Expert parallelism: the device work around the two token exchanges of the
// Kimi K2 card's moe_infer when ep_size > 1 (count exchange, token
// all-to-all, local regrouping, expert compute, reverse all-to-all, weighted
// sum), at the latent width for Stable LatentMoE (the walk-through notes
// that both passes then move 3584-wide rows).  Experts are split into
// contiguous ranges, E / ep_size per rank.
//
//   pack     send[pos] = bf16(x^c[token of assignment perm[pos]]): the local
//            dispatch groups the assignments by global expert, so rows bound
//            for each rank are contiguous and in the order of that rank's
//            experts.
//   expand   recv_counts [ep_size][E_loc] (rows from each source rank per
//            local expert, source-major as the exchange delivers them) ->
//            the local expert of every received row.
//   cast     out[row] = bf16(sum of the K-split planes of y[row]): the expert
//            outputs go back in the order the rows arrived.
//   unpack   y[perm[pos]] = G[perm[pos]] * ret[pos]: the returned outputs in
//            assignment order, weighted, for the slot-ordered sum.
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {
namespace {

__global__ void ep_pack_kernel(const float* __restrict__ xc, const __nv_bfloat16* __restrict__ xb, int dx, int k,
                               const int32_t* __restrict__ perm, int P, __nv_bfloat16* __restrict__ send) {
  griddep_launch();
  griddep_wait();
  const int per = dx / 4;   // four values per thread
  const size_t n = static_cast<size_t>(P) * per;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / per), c = static_cast<int>(i % per) * 4;
    const int t = perm[pos] / k;
    uint2 w;
    if (xc) {
      const float4 v = *reinterpret_cast<const float4*>(xc + static_cast<size_t>(t) * dx + c);
      const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
      w.x = *reinterpret_cast<const uint32_t*>(&a);
      w.y = *reinterpret_cast<const uint32_t*>(&b);
    } else {
      w = *reinterpret_cast<const uint2*>(xb + static_cast<size_t>(t) * dx + c);
    }
    *reinterpret_cast<uint2*>(send + static_cast<size_t>(pos) * dx + c) = w;
  }
}

// Every block scans the R x E_loc counts in shared memory (at most
// kMaxExperts of them), then each thread finds its rows' segment by binary
// search.  A count sum different from n is reported in err[1].
__global__ void ep_expand_kernel(const int32_t* __restrict__ counts, int nseg, int E_loc, int n,
                                 int32_t* __restrict__ idx_loc, int* __restrict__ err) {
  griddep_launch();
  griddep_wait();
  __shared__ int off[kMaxExperts + 1];
  if (threadIdx.x == 0) {
    int s = 0;
    off[0] = 0;
    for (int i = 0; i < nseg; ++i) {
      const int c = counts[i];
      s += c < 0 ? 0 : c;
      off[i + 1] = s;
    }
    if (blockIdx.x == 0 && s != n && err) atomicExch(err + 1, 1);
  }
  __syncthreads();
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < n; row += gridDim.x * blockDim.x) {
    int lo = 0, hi = nseg;   // the segment i with off[i] <= row < off[i+1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= row) lo = mid; else hi = mid;
    }
    idx_loc[row] = row < off[nseg] ? lo % E_loc : 0;
  }
}

__global__ void ep_cast_kernel(const float* __restrict__ y, int n, int dx, int ks, size_t plane,
                               __nv_bfloat16* __restrict__ out) {
  griddep_launch();
  griddep_wait();
  const size_t total = static_cast<size_t>(n) * dx / 2;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float a = 0.f, b = 0.f;
    for (int s = 0; s < ks; ++s) {
      const float2 v = *reinterpret_cast<const float2*>(y + s * plane + 2 * i);
      a += v.x;
      b += v.y;
    }
    reinterpret_cast<__nv_bfloat162*>(out)[i] = __floats2bfloat162_rn(a, b);
  }
}

__global__ void ep_unpack_kernel(const __nv_bfloat16* __restrict__ ret, int P, int dx,
                                 const int32_t* __restrict__ perm, const float* __restrict__ G,
                                 float* __restrict__ y) {
  griddep_launch();
  griddep_wait();
  const int per = dx / 2;
  const size_t n = static_cast<size_t>(P) * per;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(i / per), c = static_cast<int>(i % per) * 2;
    const int a = perm[pos];
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(ret + static_cast<size_t>(pos) * dx + c));
    const float g = G[a];
    *reinterpret_cast<float2*>(y + static_cast<size_t>(a) * dx + c) = make_float2(v.x * g, v.y * g);
  }
}

int ep_grid(size_t n) {
  size_t g = (n + 255) / 256;
  return static_cast<int>(g < 152 * 8 ? (g ? g : 1) : 152 * 8);
}

}  // namespace

cudaError_t launch_ep_pack(const float* xc, const void* xb, int dx, int k, const int32_t* perm, int P, void* send,
                           cudaStream_t s) {
  if (P <= 0) return cudaSuccess;
  if (dx % 4) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(ep_pack_kernel, ep_grid(static_cast<size_t>(P) * dx / 4), 256, 0, s, xc,
                                   static_cast<const __nv_bfloat16*>(xb), dx, k, perm, P,
                                   static_cast<__nv_bfloat16*>(send));
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ep_expand(const int32_t* counts, int nseg, int E_loc, int n, int32_t* idx_loc, int* err,
                             cudaStream_t s) {
  if (nseg < 1 || nseg > kMaxExperts) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(ep_expand_kernel, ep_grid(n > 0 ? n : 1), 256, 0, s, counts, nseg, E_loc, n,
                                   idx_loc, err);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ep_cast(const float* y, int n, int dx, int ks, size_t plane, void* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (dx % 2 || plane % 2) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(ep_cast_kernel, ep_grid(static_cast<size_t>(n) * dx / 2), 256, 0, s, y, n, dx, ks,
                                   plane, static_cast<__nv_bfloat16*>(out));
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_ep_unpack(const void* ret, int P, int dx, const int32_t* perm, const float* G, float* y,
                             cudaStream_t s) {
  if (P <= 0) return cudaSuccess;
  if (dx % 2) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(ep_unpack_kernel, ep_grid(static_cast<size_t>(P) * dx / 2), 256, 0, s,
                                   static_cast<const __nv_bfloat16*>(ret), P, dx, perm, G, y);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace lmoe
