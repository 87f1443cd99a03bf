// Quantile Balancing: the selection-bias update of Stable LatentMoE
// (tutorial "Stable LatentMoE", section "Quantile Balancing: giving every
// expert a fair shot"; walk-through "Kimi K3 模型结构（5）", section
// "Stable 之三：Quantile Balancing" and its appendix-D histogram estimator).
//
// For a batch routed with biases b, token i's cutoff alpha_i is its
// (k+1)-th largest biased score s_i + b; r_ij = alpha_i - s_ij is the bias
// expert j would need to enter token i's top-k.  The exact update sets b_j
// to the (k/n)-quantile of r_{:,j} ("higher": the sorted value at index
// ceil(k/n (m-1))), the histogram update reads the same quantile from n x B
// integer counts of r over [min b - 1, max b + 1]; both are centred.
//
// Order statistics are found by radix selection on the order-preserving
// integer image of the fp32 keys (four 8-bit digits, most significant
// first, a 256-bin shared-memory histogram per digit), which picks the exact
// element whatever the ties.
#include <algorithm>

#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {
namespace {

constexpr int kQbThreads = 256;

// fp32 -> uint32 with the same order (negative values reversed below positives).
__device__ __forceinline__ uint32_t ordered_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Block-wide: the key of ascending rank `rank` (0-based) among n keys that
// get(i) yields (i < n).  get is called four times per key.  Every thread
// returns the same key.
template <class Get>
__device__ uint32_t block_select(int n, int rank, Get get, uint32_t* hist /*[256]*/, uint32_t* shared_out /*[2]*/) {
  uint32_t prefix = 0, mask = 0;
#pragma unroll 1
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint32_t key = get(i);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 0xFFu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // the digit whose cumulative count first exceeds rank (one warp scans 8 bins per lane)
      const int lane = threadIdx.x;
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[lane * 8 + j];
        tot += c[j];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - tot;
      const uint32_t r = static_cast<uint32_t>(rank);
      if (r >= excl && r < incl) {
        uint32_t acc = excl;
        int d = 0;
        for (int j = 0; j < 8; ++j) {
          if (r < acc + c[j]) {
            d = lane * 8 + j;
            break;
          }
          acc += c[j];
        }
        shared_out[0] = static_cast<uint32_t>(d);
        shared_out[1] = acc;   // keys below the digit
      }
    }
    __syncthreads();
    prefix |= shared_out[0] << shift;
    mask |= 0xFFu << shift;
    rank -= static_cast<int>(shared_out[1]);
    __syncthreads();
  }
  return prefix;
}

// alpha_i: the (k+1)-th largest of c_ij = sigmoid(z_ij) + b_j (ascending rank
// E - 1 - k), one block per token.
__global__ void __launch_bounds__(kQbThreads) qb_cutoff_kernel(const float* __restrict__ z, int E,
                                                              const float* __restrict__ bias, int k,
                                                              float* __restrict__ alpha) {
  __shared__ uint32_t keys[kMaxExperts];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t out[2];
  const int t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    keys[e] = ordered_key(sigmoidf_(z[static_cast<size_t>(t) * E + e]) + bias[e]);
  __syncthreads();
  const uint32_t key = block_select(E, E - 1 - k, [&](int i) { return keys[i]; }, hist, out);
  if (threadIdx.x == 0) alpha[t] = key_value(key);
}

// raw_j = the key of ascending rank `rank` among r_ij = alpha_i - sigmoid(z_ij),
// i < T, one block per expert (the column is read from L2 in each pass).
__global__ void __launch_bounds__(kQbThreads) qb_quantile_kernel(const float* __restrict__ z, int T, int E,
                                                                const float* __restrict__ alpha, int rank,
                                                                float* __restrict__ raw) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t out[2];
  const int j = blockIdx.x;
  auto get = [&](int i) { return ordered_key(alpha[i] - sigmoidf_(z[static_cast<size_t>(i) * E + j])); };
  const uint32_t key = block_select(T, rank, get, hist, out);
  if (threadIdx.x == 0) raw[j] = key_value(key);
}

// lo = min b - 1, hi = max b + 1: the range of every required bias.
__global__ void qb_range_kernel(const float* __restrict__ bias, int E, float* __restrict__ range) {
  __shared__ float mn[32], mx[32];
  float a = INFINITY, b = -INFINITY;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    a = fminf(a, bias[e]);
    b = fmaxf(b, bias[e]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a = fminf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    b = fmaxf(b, __shfl_xor_sync(0xFFFFFFFFu, b, o));
  }
  if ((threadIdx.x & 31) == 0) {
    mn[threadIdx.x >> 5] = a;
    mx[threadIdx.x >> 5] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
      a = fminf(a, mn[w]);
      b = fmaxf(b, mx[w]);
    }
    range[0] = a - 1.0f;
    range[1] = b + 1.0f;
  }
}

// counts[j][bin(r_ij)] += 1 for every (token, expert) of the batch.
__global__ void qb_hist_kernel(const float* __restrict__ z, int T, int E, const float* __restrict__ alpha,
                               const float* __restrict__ range, int bins, int32_t* __restrict__ counts) {
  const float lo = range[0], w = (range[1] - range[0]) / static_cast<float>(bins);
  const size_t n = static_cast<size_t>(T) * E;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / E), e = static_cast<int>(i % E);
    const float r = alpha[t] - sigmoidf_(z[i]);
    int c = static_cast<int>(floorf((r - lo) / w));
    c = c < 0 ? 0 : (c >= bins ? bins - 1 : c);
    atomicAdd(&counts[static_cast<size_t>(e) * bins + c], 1);
  }
}

// One warp per expert: m = its total count, target = ceil(m k / E); the first
// bin whose cumulative count reaches the target, linearly interpolated.
__global__ void qb_hist_quantile_kernel(const int32_t* __restrict__ counts, int E, int bins, int k,
                                        const float* __restrict__ range, float* __restrict__ raw) {
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (j >= E) return;
  const int32_t* cj = counts + static_cast<size_t>(j) * bins;
  long long m = 0;
  for (int c = lane; c < bins; c += 32) m += cj[c];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m += __shfl_xor_sync(0xFFFFFFFFu, m, o);
  const long long target = (m * k + E - 1) / E;
  const float lo = range[0], hi = range[1], w = (hi - lo) / static_cast<float>(bins);
  long long before = 0;
  float val = hi;
  for (int c0 = 0; c0 < bins; c0 += 32) {
    const int c = c0 + lane;
    const long long v = c < bins ? cj[c] : 0;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += u;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, v > 0 && before + incl >= target);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long incl_s = __shfl_sync(0xFFFFFFFFu, incl, src);
      const long long v_s = __shfl_sync(0xFFFFFFFFu, v, src);
      const long long cum = before + incl_s - v_s;
      val = lo + w * (static_cast<float>(c0 + src) +
                      static_cast<float>(target - cum) / static_cast<float>(v_s));
      break;
    }
    before += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) raw[j] = val;
}

// new_b = raw - mean(raw) (the mean summed in a fixed order, in double).
__global__ void qb_center_kernel(const float* __restrict__ raw, int E, float* __restrict__ out) {
  __shared__ double part[32];
  __shared__ double mean;
  double s = 0.0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s += raw[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += part[w];
    mean = t / E;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = static_cast<float>(raw[e] - mean);
}

}  // namespace

cudaError_t launch_qb_update(const float* z, int T, int E, int k, const float* bias, float* alpha, float* raw,
                             float* new_bias, cudaStream_t s) {
  if (T <= 0 || k < 1 || k >= E || E > kMaxExperts) return cudaErrorInvalidValue;
  qb_cutoff_kernel<<<T, kQbThreads, 0, s>>>(z, E, bias, k, alpha);
  // the sorted value at index ceil(k/E (T - 1)), in exact integer arithmetic
  const long long num = static_cast<long long>(k) * (T - 1);
  const int rank = static_cast<int>((num + E - 1) / E);
  qb_quantile_kernel<<<E, kQbThreads, 0, s>>>(z, T, E, alpha, rank, raw);
  qb_center_kernel<<<1, 1024, 0, s>>>(raw, E, new_bias);
  return cudaGetLastError();
}

cudaError_t launch_qb_histogram(const float* z, int T, int E, int k, const float* bias, int bins, float* alpha,
                                float* range, int32_t* counts, cudaStream_t s) {
  if (T <= 0 || k < 1 || k >= E || E > kMaxExperts || bins < 1) return cudaErrorInvalidValue;
  qb_range_kernel<<<1, 1024, 0, s>>>(bias, E, range);
  qb_cutoff_kernel<<<T, kQbThreads, 0, s>>>(z, E, bias, k, alpha);
  const size_t n = static_cast<size_t>(T) * E;
  const int grid = static_cast<int>(std::min<size_t>((n + 255) / 256, 152 * 16));
  qb_hist_kernel<<<grid, 256, 0, s>>>(z, T, E, alpha, range, bins, counts);
  return cudaGetLastError();
}

cudaError_t launch_qb_from_histogram(const int32_t* counts, int E, int bins, int k, const float* bias, float* range,
                                     float* raw, float* new_bias, cudaStream_t s) {
  if (k < 1 || k >= E || E > kMaxExperts || bins < 1) return cudaErrorInvalidValue;
  qb_range_kernel<<<1, 1024, 0, s>>>(bias, E, range);
  qb_hist_quantile_kernel<<<(E + 7) / 8, 256, 0, s>>>(counts, E, bins, k, range, raw);
  qb_center_kernel<<<1, 1024, 0, s>>>(raw, E, new_bias);
  return cudaGetLastError();
}

}  // namespace lmoe
