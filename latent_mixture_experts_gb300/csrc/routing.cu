// Router tail and token -> expert dispatch.
//
// topk: per token, sum the router GEMM's split-K partial logits in a fixed
// order, s = sigmoid(z), c = s + b, select the k largest c (exact ties to the
// lower expert index), G = scale * s / sum s over the selection (Kimi K3
// card, router steps; Kimi K2 card adds the 2.827 scale; the selection bias
// steers the choice only, the weights use the raw sigmoid).
//
// dispatch: the counting, argsort and grouping of moe_infer as a stable
// counting sort that never leaves the device: per-chunk histograms, a scan
// over chunks and experts, then a per-chunk stable scatter.  It also lays
// out each expert's assignments in BN-row tiles (segments padded to a
// multiple of BN) and writes the tile list the grouped expert GEMMs walk.
#include <algorithm>

#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {

namespace {

constexpr int kTopkMaxThreads = 1024;
constexpr int kTopkPer = kMaxExperts / kTopkMaxThreads;   // experts per thread
constexpr int kTopkMaxK = 32;

// Strict order of the selection: larger biased score first, exact ties to
// the lower expert index (NaN scores rank below every number).
__device__ __forceinline__ bool topk_before(float va, int ea, float vb, int eb) {
  return va > vb || (va == vb && ea < eb);
}

// One block per token, one thread per expert.  Each thread sums its
// expert's split-K partial logits in split order (loads issued eight at a
// time), forms s = sigmoid(z) and c = s + b.  The k-th largest of the
// per-warp maxima is a lower bound of the k-th largest c (k distinct experts
// reach it), so only experts at or above it can be selected; each such
// candidate counts the candidates that precede it in the selection order,
// and that count is its output position.  The selection is the one of
// sorting all experts by (c descending, index ascending) and keeping k.
__global__ void __launch_bounds__(kTopkMaxThreads) topk_kernel(const float* __restrict__ part, int splits, int T,
                                                              int E, const float* __restrict__ bias, int k,
                                                              float scale, int32_t* __restrict__ idx,
                                                              float* __restrict__ G, float* __restrict__ z_out) {
  griddep_launch();
  griddep_wait();
  __shared__ float wmax[32];
  __shared__ float thr;
  __shared__ int ncand;
  __shared__ int sel_e[kTopkMaxK];
  __shared__ float sel_s[kTopkMaxK];
  extern __shared__ float tk_smem[];
  float* cand_c = tk_smem;                                   // [E]
  float* cand_s = tk_smem + E;                               // [E]
  int* cand_e = reinterpret_cast<int*>(tk_smem + 2 * E);     // [E]
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x;
  const size_t plane = static_cast<size_t>(T) * E;
  const float* pt = part + static_cast<size_t>(t) * E;
  if (tid == 0) ncand = 0;

  float cv[kTopkPer], sv[kTopkPer];
  float m = -INFINITY;
#pragma unroll
  for (int q = 0; q < kTopkPer; ++q) {
    const int e = tid + q * nthr;
    cv[q] = -INFINITY;
    sv[q] = 0.f;
    if (e < E) {
      float z = 0.f;
      for (int s0 = 0; s0 < splits; s0 += 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = s0 + i < splits ? __ldg(pt + (s0 + i) * plane + e) : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (s0 + i < splits) z += v[i];
      }
      z_out[static_cast<size_t>(t) * E + e] = z;
      sv[q] = sigmoidf_(z);
      const float c = sv[q] + bias[e];
      cv[q] = c == c ? c : -INFINITY;
    }
    m = fmaxf(m, cv[q]);
  }
  m = warp_max(m);
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr >> 5;
    const float mv = lane < nw ? wmax[lane] : -INFINITY;
    float th = -INFINITY;
    if (nw >= k) {
      int rank = 0;
      for (int j = 0; j < nw; ++j) {
        const float o = __shfl_sync(0xFFFFFFFFu, mv, j);
        rank += topk_before(o, j, mv, lane) ? 1 : 0;
      }
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, lane < nw && rank == k - 1);
      th = __shfl_sync(0xFFFFFFFFu, mv, __ffs(hit) - 1);
    }
    if (lane == 0) thr = th;
  }
  __syncthreads();
  const float th = thr;
#pragma unroll
  for (int q = 0; q < kTopkPer; ++q) {
    const int e = tid + q * nthr;
    const bool is = e < E && cv[q] >= th;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, is);
    int base = 0;
    if (lane == 0 && bal) base = atomicAdd(&ncand, __popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (is) {
      const int slot = base + __popc(bal & ((1u << lane) - 1u));
      cand_c[slot] = cv[q];
      cand_s[slot] = sv[q];
      cand_e[slot] = e;
    }
  }
  __syncthreads();
  const int n = ncand;
  for (int i = tid; i < n; i += nthr) {
    const float v = cand_c[i];
    const int e = cand_e[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += topk_before(cand_c[j], cand_e[j], v, e) ? 1 : 0;
    if (rank < k) {
      sel_e[rank] = e;
      sel_s[rank] = cand_s[i];
    }
  }
  __syncthreads();
  if (warp == 0) {
    float sum = 0.f;
    if (lane == 0)
      for (int j = 0; j < k; ++j) sum += sel_s[j];
    sum = __shfl_sync(0xFFFFFFFFu, sum, 0);
    const float inv = scale / sum;
    if (lane < k) {
      idx[static_cast<size_t>(t) * k + lane] = sel_e[lane];
      G[static_cast<size_t>(t) * k + lane] = sel_s[lane] * inv;
    }
  }
}

// Whole dispatch in one block, for batches of at most kSmallDispatch
// assignments: shared-memory histogram, block scans over the experts, then
// one warp walks the assignments in order for the stable placement.

__global__ void __launch_bounds__(1024) dispatch_small_kernel(const int32_t* __restrict__ idx, int P, int E, int BN,
                                                              int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ perm,
                                                              int32_t* __restrict__ inv_pad,
                                                              int32_t* __restrict__ tile_off,
                                                              int4* __restrict__ tiles, int32_t* __restrict__ ntiles,
                                                              int* err) {
  griddep_launch();
  griddep_wait();
  __shared__ int32_t hist[kMaxExperts];
  __shared__ int32_t s_off[kMaxExperts + 1];
  __shared__ int32_t s_toff[kMaxExperts + 1];
  __shared__ int32_t wsum[3][32];
  extern __shared__ int16_t s_idx[];                     // [P] expert ids, -1 for an invalid id
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (int a = tid; a < P; a += blockDim.x) {
    const int e = idx[a];
    const bool ok = e >= 0 && e < E;
    s_idx[a] = static_cast<int16_t>(ok ? e : -1);
    if (ok) atomicAdd(&hist[e], 1);
    else if (err) atomicExch(err + 1, 1);
  }
  __syncthreads();
  // exclusive scans of (count, padded count, tiles): thread owns experts 2*tid, 2*tid+1
  int v[2][3];
  int loc[3] = {0, 0, 0};
  for (int q = 0; q < 2; ++q) {
    const int e = 2 * tid + q;
    const int c = e < E ? hist[e] : 0;
    const int n = (c + BN - 1) / BN;
    v[q][0] = c;
    v[q][1] = n * BN;
    v[q][2] = n;
    for (int m = 0; m < 3; ++m) loc[m] += v[q][m];
  }
  int incl[3];
  for (int m = 0; m < 3; ++m) {
    int x = loc[m];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    incl[m] = x;
    if (lane == 31) wsum[m][warp] = x;
  }
  __syncthreads();
  if (warp == 0) {
    for (int m = 0; m < 3; ++m) {
      int x = lane < (blockDim.x >> 5) ? wsum[m][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      wsum[m][lane] = x;   // inclusive over warps
    }
  }
  __syncthreads();
  int base[3];
  for (int m = 0; m < 3; ++m) base[m] = (warp ? wsum[m][warp - 1] : 0) + incl[m] - loc[m];
  for (int q = 0; q < 2; ++q) {
    const int e = 2 * tid + q;
    if (e < E) {
      s_off[e] = base[0];
      s_toff[e] = base[1];
      counts[e] = v[q][0];
      offsets[e] = base[0];
      tile_off[e] = base[1];
      for (int i = 0; i < v[q][2]; ++i)
        tiles[base[2] + i] = make_int4(e, base[1] + i * BN, min(BN, v[q][0] - i * BN), base[0] + i * BN);
    }
    for (int m = 0; m < 3; ++m) base[m] += v[q][m];
  }
  if (tid == blockDim.x - 1) {
    offsets[E] = base[0];
    tile_off[E] = base[1];
    *ntiles = base[2];
  }
  __syncthreads();
  // stable placement: warp 0 walks the assignments in order, 32 at a time
  if (warp == 0) {
    for (int a0 = 0; a0 < P; a0 += 32) {
      const int a = a0 + lane;
      const int e = a < P ? s_idx[a] : -1;
      const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int b = e >= 0 ? s_off[e] : 0;
      __syncwarp();
      if (e >= 0) {
        const int pidx = b + rank;
        perm[pidx] = a;
        inv_pad[a] = s_toff[e] + (pidx - offsets[e]);
        if (rank == 0) s_off[e] = b + __popc(peers);
      }
      __syncwarp();
    }
  }
}

// Per-chunk histogram of expert ids.
__global__ void dispatch_count_kernel(const int32_t* __restrict__ idx, int P, int E, int32_t* __restrict__ blockcnt,
                                      int* err) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kDispatchChunk;
  for (int a = a0 + threadIdx.x; a < min(P, a0 + kDispatchChunk); a += blockDim.x) {
    const int e = idx[a];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else if (err) atomicExch(err + 1, 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) blockcnt[static_cast<size_t>(blockIdx.x) * E + e] = hist[e];
}

// One warp per expert: exclusive prefix of the expert's per-chunk counts, in
// place, and the expert's total.  Lane l owns a contiguous run of chunks, so
// the prefix is a warp scan of the 32 run sums plus a sequential pass.
__global__ void __launch_bounds__(256) dispatch_chunkscan_kernel(int32_t* __restrict__ blockcnt, int nchunks, int E,
                                                                 int32_t* __restrict__ counts) {
  griddep_launch();
  griddep_wait();
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (e >= E) return;                                    // whole warp
  const int per = (nchunks + 31) / 32;
  const int b0 = min(nchunks, lane * per), b1 = min(nchunks, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) sum += blockcnt[static_cast<size_t>(b) * E + e];
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  int run = incl - sum;
  for (int b = b0; b < b1; ++b) {
    const int c = blockcnt[static_cast<size_t>(b) * E + e];
    blockcnt[static_cast<size_t>(b) * E + e] = run;
    run += c;
  }
  if (lane == 31) counts[e] = incl;
}

// One block of 1024 threads, two experts per thread: exclusive scans over
// the experts of the counts, the BN-padded counts and the tile counts
// (offsets, tile_off, first tile), then the tile list.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(const int32_t* __restrict__ counts, int E, int BN,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ tile_off, int4* __restrict__ tiles,
                                                             int32_t* __restrict__ ntiles) {
  griddep_launch();
  griddep_wait();
  __shared__ int wsum[3][32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int e0 = 2 * t;
  int c[2], n[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    c[j] = e0 + j < E ? counts[e0 + j] : 0;
    n[j] = (c[j] + BN - 1) / BN;
  }
  const int own[3] = {c[0] + c[1], (n[0] + n[1]) * BN, n[0] + n[1]};
  int inc[3] = {own[0], own[1], own[2]};
#pragma unroll
  for (int off = 1; off < 32; off <<= 1)
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, inc[q], off);
      if (lane >= off) inc[q] += v;
    }
  if (lane == 31)
#pragma unroll
    for (int q = 0; q < 3; ++q) wsum[q][w] = inc[q];
  __syncthreads();
  if (w == 0) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int x = wsum[q][lane];
      int y = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, y, off);
        if (lane >= off) y += v;
      }
      wsum[q][lane] = y - x;                             // exclusive over warps
    }
  }
  __syncthreads();
  int start[3];
#pragma unroll
  for (int q = 0; q < 3; ++q) start[q] = wsum[q][w] + inc[q] - own[q];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int e = e0 + j;
    if (e < E) {
      offsets[e] = start[0];
      tile_off[e] = start[1];
      for (int i = 0; i < n[j]; ++i)
        tiles[start[2] + i] = make_int4(e, start[1] + i * BN, min(BN, c[j] - i * BN), start[0] + i * BN);
    }
    if (e == E - 1) {                                    // totals
      offsets[E] = start[0] + c[j];
      tile_off[E] = start[1] + n[j] * BN;
      *ntiles = start[2] + n[j];
    }
    start[0] += c[j];
    start[1] += n[j] * BN;
    start[2] += n[j];
  }
}

// One warp per chunk: stable ranks inside the chunk, in assignment order.
__global__ void __launch_bounds__(32) dispatch_scatter_kernel(const int32_t* __restrict__ idx, int P, int E,
                                                              const int32_t* __restrict__ blockcnt,
                                                              const int32_t* __restrict__ offsets,
                                                              const int32_t* __restrict__ tile_off,
                                                              int32_t* __restrict__ perm,
                                                              int32_t* __restrict__ inv_pad) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int32_t pos[];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) pos[e] = blockcnt[static_cast<size_t>(blockIdx.x) * E + e] + offsets[e];
  __syncwarp();
  const int a0 = blockIdx.x * kDispatchChunk;
  for (int s = 0; s < kDispatchChunk; s += 32) {
    const int a = a0 + s + lane;
    const bool valid = a < P;
    int e = valid ? idx[a] : -1;
    if (e < 0 || e >= E) e = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int base = e >= 0 ? pos[e] : 0;
    __syncwarp();
    if (e >= 0) {
      const int p = base + rank;
      perm[p] = a;
      inv_pad[a] = tile_off[e] + (p - offsets[e]);
      if (rank == 0) pos[e] = base + __popc(peers);
    }
    __syncwarp();
  }
}

__global__ void shared_tiles_kernel(int T, int BN, int4* __restrict__ tiles, int32_t* __restrict__ tile_off,
                                    int32_t* __restrict__ ntiles) {
  griddep_launch();
  griddep_wait();
  const int nt = (T + BN - 1) / BN;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nt; i += gridDim.x * blockDim.x)
    tiles[i] = make_int4(0, i * BN, min(BN, T - i * BN), i * BN);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    tile_off[0] = 0;
    tile_off[1] = nt * BN;
    *ntiles = nt;
  }
}

__global__ void iota_ones_kernel(int32_t* __restrict__ iota, float* __restrict__ ones, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    iota[i] = i;
    ones[i] = 1.0f;
  }
}

}  // namespace

cudaError_t launch_shared_tiles(int T, int BN, int4* tiles, int32_t* tile_off, int32_t* ntiles, cudaStream_t s) {
  if (T <= 0 || BN <= 0) return cudaErrorInvalidValue;
  const int nt = (T + BN - 1) / BN;
  return launch_pdl(shared_tiles_kernel, (nt + 255) / 256, 256, 0, s, T, BN, tiles, tile_off, ntiles);
}

cudaError_t launch_iota_ones(int32_t* iota, float* ones, int n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  iota_ones_kernel<<<(n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024, 256, 0, s>>>(iota, ones, n);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logit_part, int splits, int T, int E, const float* bias, int k,
                        float routed_scale, int32_t* idx, float* G, float* z_out, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (E > kMaxExperts || k > kTopkMaxK || k > E) return cudaErrorInvalidValue;
  const int threads = std::min(kTopkMaxThreads, (E + 31) / 32 * 32);
  const size_t smem = 3 * static_cast<size_t>(E) * sizeof(float);
  {
    const cudaError_t e_ = launch_pdl(topk_kernel, T, threads, smem, s, logit_part,
                                      splits, T, E, bias, k, routed_scale, idx, G, z_out);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const int32_t* idx, int T, int k, int E, int BN, const DispatchBufs& b,
                            cudaStream_t s) {
  const int P = T * k;
  if (P <= 0) return cudaSuccess;
  if (P <= kSmallDispatch) {
    {
      const size_t smem = static_cast<size_t>(P) * sizeof(int16_t);   // staged expert ids
      const cudaError_t e_ = launch_pdl(dispatch_small_kernel, 1, 1024, smem, s, idx,
                                        P, E, BN, b.counts, b.offsets, b.perm, b.inv_pad, b.tile_off, b.tiles,
                                        b.ntiles, b.err);
      if (e_ != cudaSuccess) return e_;
    }
    return cudaGetLastError();
  }
  const int nchunks = (P + kDispatchChunk - 1) / kDispatchChunk;
  const size_t hsmem = static_cast<size_t>(E) * sizeof(int32_t);
  {
    const cudaError_t e_ = launch_pdl(dispatch_count_kernel, nchunks, 256, hsmem, s, idx,
                                      P, E, b.blockcnt, b.err);
    if (e_ != cudaSuccess) return e_;
  }
  {
    const cudaError_t e_ = launch_pdl(dispatch_chunkscan_kernel, (E + 7) / 8, 256, 0, s, b.blockcnt, nchunks, E,
                                      b.counts);
    if (e_ != cudaSuccess) return e_;
  }
  {
    const cudaError_t e_ = launch_pdl(dispatch_scan_kernel, 1, 1024, 0, s, static_cast<const int32_t*>(b.counts), E,
                                      BN, b.offsets, b.tile_off, b.tiles, b.ntiles);
    if (e_ != cudaSuccess) return e_;
  }
  {
    const cudaError_t e_ = launch_pdl(dispatch_scatter_kernel, nchunks, 32, hsmem, s, idx,
                                      P, E, b.blockcnt, b.offsets, b.tile_off, b.perm, b.inv_pad);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace lmoe
