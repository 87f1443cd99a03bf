// Tensor-pipe throughput of this GPU, measured with the same tcgen05 MMA
// forms the layer's kernels issue.  One CTA per SM keeps one elected thread
// issuing M = 128, N = 256 MMAs back to back on operands that stay in shared
// memory (no loads in the loop), accumulating into one tensor-memory tile;
// the kernel's CUDA-event time gives FLOP/s = 2 M N K x MMAs / time.  These
// are the denominators of the tensor-bound rooflines: nothing in the layer
// can issue faster than this loop.
#include "../../include/lmoe_peak.h"
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {
namespace {

constexpr int kM = 128, kN = 256;
// Loop length cap: at the slowest form (bf16, ~0.6 us per four MMAs) the
// loop stays well inside the 2 s limit of the threads' bounded wait.
constexpr int kMaxIters = 1 << 20;
constexpr int kSmemA = kM * 128, kSmemB = kN * 128;   // one 128-byte (swizzled) K row per operand row
constexpr int kSmemSf = 512 * 3;                       // scale atoms: A (128 rows), B (2 x 128 rows)
constexpr int kSmemBytes = kSmemA + kSmemB + kSmemSf + 1024;

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return x;
}

// MMA forms.  K per instruction: 16 (bf16), 32 (8-bit and padded 4-bit),
// 64 (packed 4-bit).
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb) {
  asm volatile(
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], 1;"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb) {
  asm volatile(
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], 1;"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb)
      : "memory");
}

// Instruction descriptor of the packed-FP4 block-scaled forms: A and B E2M1
// (format code 1), K-major, the scale type (UE8M0 = 1, UE4M3 = 0) and each
// operand's scale-factor id.
constexpr uint32_t idesc_fp4(int M, int N, uint32_t scale_ue8m0) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (scale_ue8m0 << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) tc_peak_kernel(int iters, int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sa = sm;
  uint8_t* sb = sm + kSmemA;
  uint8_t* sf = sm + kSmemA + kSmemB;
  __shared__ uint64_t done;
  __shared__ uint32_t tmem_base;
  const int warp = threadIdx.x >> 5;

  // operands: finite random values of each format (no NaN codes), unit scales
  for (int i = threadIdx.x; i < (kSmemA + kSmemB) / 4; i += blockDim.x) {
    uint32_t h = mix32(static_cast<uint32_t>(i) * 2654435761u + blockIdx.x);
    if (KIND == LMOE_TC_BF16) h = (h & 0x807F807Fu) | 0x3F803F80u;   // +-[1, 2)
    if (KIND == LMOE_TC_E4M3_E4M3 || KIND == LMOE_TC_E2M1_E4M3) h &= 0xFEFEFEFEu;   // mantissa lsb 0: never NaN
    reinterpret_cast<uint32_t*>(sm)[i] = h;
  }
  const uint8_t unit = KIND == LMOE_TC_NVFP4 ? 0x38 : 127;   // 1.0 in UE4M3 / UE8M0
  for (int i = threadIdx.x; i < kSmemSf; i += blockDim.x) sf[i] = unit;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t acc = tmem_base;
  const uint32_t sfa = tmem_base + kN;   // 4 columns of A scales, then 8 of B scales
  const uint32_t sfb = sfa + 4;
  if (threadIdx.x == 0) {
    if (KIND != LMOE_TC_BF16) {
      tmem_cp_32x128b_x4(sfa, sdesc_noswz(smem_u32(sf), 16, 128));
      tmem_cp_32x128b_x4(sfb, sdesc_noswz(smem_u32(sf + 512), 16, 128));
      tmem_cp_32x128b_x4(sfb + 4, sdesc_noswz(smem_u32(sf + 1024), 16, 128));
    }
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    constexpr uint32_t id_bf16 = idesc_bf16(kM, kN);
    constexpr uint32_t id_e4 = idesc_mxf8f6f4(kM, kN, 0, 0, 0, 0);
    constexpr uint32_t id_e2e4 = idesc_mxf8f6f4(kM, kN, 5, 0, 0, 0);
    constexpr uint32_t id_mx4 = idesc_fp4(kM, kN, 1);
    constexpr uint32_t id_nv4 = idesc_fp4(kM, kN, 0);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const uint64_t da = sdesc_sw128(a0 + 32 * kb), db = sdesc_sw128(b0 + 32 * kb);
        const uint32_t accum = (it | kb) != 0;
        if constexpr (KIND == LMOE_TC_BF16) mma_bf16(acc, da, db, id_bf16, accum);
        if constexpr (KIND == LMOE_TC_E4M3_E4M3) mma_mxf8f6f4(acc, da, db, id_e4, sfa, sfb, accum);
        if constexpr (KIND == LMOE_TC_E2M1_E4M3) mma_mxf8f6f4(acc, da, db, id_e2e4, sfa, sfb, accum);
        if constexpr (KIND == LMOE_TC_MXFP4) mma_mxf4(acc, da, db, id_mx4, sfa, sfb);
        if constexpr (KIND == LMOE_TC_NVFP4) mma_nvf4(acc, da, db, id_nv4, sfa, sfb);
      }
    }
    mma_commit(&done);
  }
  __syncwarp();
  mbar_wait(&done, 0, err, kErrTimeout);
  tc_fence_after();
  __syncthreads();
  if (warp == 0) tmem_dealloc(acc, 512);
}

template <int KIND>
cudaError_t launch_tc_peak(int grid, int iters, int* err, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(tc_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  tc_peak_kernel<KIND><<<grid, 128, kSmemBytes, s>>>(iters, err);
  return cudaGetLastError();
}

}  // namespace
}  // namespace lmoe

using namespace lmoe;

extern "C" lmoe_status lmoe_tc_peak(int kind, int iters, float* ms, double* flops, cudaStream_t stream) {
  if (!ms || !flops || iters < 1 || iters > kMaxIters) return LMOE_ERR_INVALID_ARG;
  int k_per_mma = 0;
  switch (kind) {
    case LMOE_TC_BF16: k_per_mma = 16; break;
    case LMOE_TC_E4M3_E4M3:
    case LMOE_TC_E2M1_E4M3: k_per_mma = 32; break;
    case LMOE_TC_MXFP4:
    case LMOE_TC_NVFP4: k_per_mma = 64; break;
    default: return LMOE_ERR_INVALID_ARG;
  }
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return LMOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return LMOE_ERR_UNSUPPORTED;
  const int grid = prop.multiProcessorCount;
  int* err = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  lmoe_status st = LMOE_OK;
  if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return LMOE_ERR_OOM;
  if (cudaMemsetAsync(err, 0, sizeof(int), stream) != cudaSuccess || cudaEventCreate(&e0) != cudaSuccess ||
      cudaEventCreate(&e1) != cudaSuccess || cudaEventRecord(e0, stream) != cudaSuccess) {
    st = LMOE_ERR_CUDA;
  } else {
    cudaError_t le = cudaSuccess;
    switch (kind) {
      case LMOE_TC_BF16: le = launch_tc_peak<LMOE_TC_BF16>(grid, iters, err, stream); break;
      case LMOE_TC_E4M3_E4M3: le = launch_tc_peak<LMOE_TC_E4M3_E4M3>(grid, iters, err, stream); break;
      case LMOE_TC_E2M1_E4M3: le = launch_tc_peak<LMOE_TC_E2M1_E4M3>(grid, iters, err, stream); break;
      case LMOE_TC_MXFP4: le = launch_tc_peak<LMOE_TC_MXFP4>(grid, iters, err, stream); break;
      case LMOE_TC_NVFP4: le = launch_tc_peak<LMOE_TC_NVFP4>(grid, iters, err, stream); break;
    }
    int herr = 0;
    if (le != cudaSuccess || cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(ms, e0, e1) != cudaSuccess ||
        cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
      st = LMOE_ERR_CUDA;
    } else if (herr) {
      st = LMOE_ERR_TIMEOUT;
    }
  }
  *flops = 2.0 * kM * kN * k_per_mma * 4.0 * iters * grid;
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(err);
  return st;
}
