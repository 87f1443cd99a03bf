// Routed experts on block-scaled tcgen05 MMA (kind::mxf8f6f4).
//
// Weights stay in their MXFP4 checkpoint form: E2M1 codes reach shared memory
// through TMA (packed in global memory, one 16-byte slot per 16 codes in
// shared memory, 128-byte swizzle) and their E8M0 scales through bulk
// copies into TMEM.  Activations are encoded as two E4M3 terms per element
// (hi + lo, each with its own E8M0 scale per 32 values): the two terms are
// two columns of the same MMA, so the weights are read from shared memory
// once and the sum of the two columns restores ~16-bit activation precision.
//
// One work item = (expert tile of <= BN assignments, 128 output features).
// A persistent grid walks the device-side tile list written by the dispatch
// step.  Warp roles: 0 = TMA producer, 1 = MMA issuer, 2..5 = epilogue.
//
//   gate/up pass: two accumulators (gate rows, up rows of the same 128
//     features), epilogue h = SiTU(g, u) (or SwiGLU), written back as hi/lo
//     E4M3 for the down pass (Kimi K3 card, routed-expert steps).
//   down pass: one accumulator, epilogue multiplies by the routing weight
//     G_i and stores the expert output of that assignment (moe_infer's
//     weighted sum is finished by the combine kernel in slot order).
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {

namespace {

constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;

template <int BN, bool GU>
struct MoeCfg {
  static constexpr int N = 2 * BN;                   // MMA N: hi/lo columns of BN assignments
  static constexpr int NA = (N + 127) / 128;         // 128-column scale atoms of B
  static constexpr int kA = 16384;                   // 128 rows x 128 FP4 codes, 16-byte slots
  static constexpr int kNA = GU ? 2 : 1;             // A operands per stage
  static constexpr int kB = N * 128;                 // N rows x 128 E4M3 codes
  static constexpr int kSfa = 512;
  static constexpr int kSfb = NA * 512;
  static constexpr int kStage = (kNA * kA + kB + kNA * kSfa + kSfb + 1023) / 1024 * 1024;
  static constexpr int kTx = kNA * 8192 + kB + kNA * kSfa + kSfb;    // bytes each stage's copies deliver
  static constexpr int kStages = GU ? (BN >= 64 ? 4 : 5) : (BN >= 64 ? 6 : 8);
  static constexpr int kSmem = kStages * kStage + 1024;
  static constexpr int kAcc = kNA * N;                 // accumulator columns
  static constexpr int kSfCols = kNA * 4 + NA * 4;     // scale columns per stage
  static constexpr int kTmemUsed = kAcc + kStages * kSfCols;
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(kTmemUsed <= 512, "tensor memory budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

template <int BN, bool GU>
__global__ void __launch_bounds__(kThreads, 1) moe_gemm_kernel(const __grid_constant__ MoeGemmParams p) {
  using C = MoeCfg<BN, GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ uint64_t full[C::kStages], empty[C::kStages], acc_full, acc_empty;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEpiWarps * 32);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  const int ntiles = *p.ntiles;
  const int total = ntiles * p.MT;
  const int KG = p.KG;

  // stage sub-buffers
  auto st_a = [&](int s, int j) { return sm + s * C::kStage + j * C::kA; };
  auto st_b = [&](int s) { return sm + s * C::kStage + C::kNA * C::kA; };
  auto st_sfa = [&](int s, int j) { return sm + s * C::kStage + C::kNA * C::kA + C::kB + j * C::kSfa; };
  auto st_sfb = [&](int s) { return sm + s * C::kStage + C::kNA * C::kA + C::kB + C::kNA * C::kSfa; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.a_gate);
      if (GU) tma_prefetch_desc(&p.a_up);
      tma_prefetch_desc(&p.b);
      uint32_t it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const int4 tile = p.tiles[w / p.MT];
        const int mt = w % p.MT;
        const int e = tile.x, row0 = tile.y;
        const int arow = e * p.N_out + mt * 128;
        const size_t sfa_idx = (static_cast<size_t>(e) * p.MT + mt) * KG;
        const size_t sfb_idx = static_cast<size_t>(row0 / BN) * KG;
        for (int g = 0; g < KG; ++g, ++it) {
          const int s = it % C::kStages;
          if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::kTx);
          tma_load_2d(st_a(s, 0), &p.a_gate, &full[s], g * 128, arow);
          if (GU) tma_load_2d(st_a(s, 1), &p.a_up, &full[s], g * 128, arow);
          tma_load_2d(st_b(s), &p.b, &full[s], g * 128, 2 * row0);
          bulk_g2s(st_sfa(s, 0), p.sfa_gate + (sfa_idx + g) * 512, 512, &full[s]);
          if (GU) bulk_g2s(st_sfa(s, 1), p.sfa_up + (sfa_idx + g) * 512, 512, &full[s]);
          bulk_g2s(st_sfb(s), p.sfb + (sfb_idx + g) * C::kSfb, C::kSfb, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, titer = 0;
      bool ok = true;
      const uint32_t d_gate = tbase, d_up = tbase + C::N;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x, ++titer) {
        if (titer > 0 && !mbar_wait(&acc_empty, (titer - 1) & 1, p.err, kErrTimeout)) break;
        tc_fence_after();
        for (int g = 0; g < KG; ++g, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tbase + C::kAcc + s * C::kSfCols;
          const uint32_t sfa_g = sf, sfa_u = sf + 4, sfb = sf + 4 * C::kNA;
          tmem_cp_32x128b_x4(sfa_g, sdesc_noswz(smem_u32(st_sfa(s, 0)), 16, 128));
          if (GU) tmem_cp_32x128b_x4(sfa_u, sdesc_noswz(smem_u32(st_sfa(s, 1)), 16, 128));
#pragma unroll
          for (int a = 0; a < C::NA; ++a)
            tmem_cp_32x128b_x4(sfb + 4 * a, sdesc_noswz(smem_u32(st_sfb(s)) + 512 * a, 16, 128));
          const uint32_t ag = smem_u32(st_a(s, 0));
          const uint32_t au = smem_u32(st_a(s, 1));
          const uint32_t bb = smem_u32(st_b(s));
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t idesc = idesc_mxf8f6f4(128, C::N, 5, 0, kb, kb);
            const uint32_t acc = (g | kb) != 0;
            mma_mxf8f6f4(d_gate, sdesc_sw128(ag + 32 * kb), sdesc_sw128(bb + 32 * kb), idesc, sfa_g, sfb, acc);
            if (GU) mma_mxf8f6f4(d_up, sdesc_sw128(au + 32 * kb), sdesc_sw128(bb + 32 * kb), idesc, sfa_u, sfb, acc);
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full);
      }
    }
  } else {
    // Epilogue warps: lane quarter q of TMEM = features 32q .. 32q+31 of the tile.
    const int q = warp & 3;
    uint32_t titer = 0;
    for (int w = blockIdx.x; w < total; w += gridDim.x, ++titer) {
      if (!mbar_wait(&acc_full, titer & 1, p.err, kErrTimeout)) break;
      tc_fence_after();
      const int4 tile = p.tiles[w / p.MT];
      const int mt = w % p.MT;
      const int row0 = tile.y, nrows = tile.z, p0 = tile.w;
      const int f = mt * 128 + 32 * q + lane;          // output feature of this lane
      const bool f_ok = f < p.N_out;
      const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
#pragma unroll 1
      for (int j0 = 0; j0 < BN; j0 += 16) {
        if (j0 >= nrows) break;
        uint32_t rg[32];
        tmem_ld16(tbase + lane_base + 2 * j0, *reinterpret_cast<uint32_t(*)[16]>(&rg[0]));
        tmem_ld16(tbase + lane_base + 2 * j0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&rg[16]));
        if constexpr (GU) {
          uint32_t ru[32];
          tmem_ld16(tbase + lane_base + C::N + 2 * j0, *reinterpret_cast<uint32_t(*)[16]>(&ru[0]));
          tmem_ld16(tbase + lane_base + C::N + 2 * j0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&ru[16]));
          tmem_ld_wait();
          const int kblk = f >> 5;                         // 32-feature block = this warp
          const int g = kblk >> 2, kb = kblk & 3;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = j0 + jj;
            if (j >= nrows) continue;                      // warp-uniform
            const float gv = __uint_as_float(rg[2 * jj]) + __uint_as_float(rg[2 * jj + 1]);
            const float uv = __uint_as_float(ru[2 * jj]) + __uint_as_float(ru[2 * jj + 1]);
            const float h = f_ok ? glu_act(gv, uv, p.act, p.b1, p.b2) : 0.0f;
            const HiLo e = quant_hilo_warp(h);
            const size_t r = static_cast<size_t>(row0) + j;
            p.hq[(2 * r) * p.Fp + f] = e.q_hi;
            p.hq[(2 * r + 1) * p.Fp + f] = e.q_lo;
            if (lane == 0) {
              const int n = 2 * j;                         // MMA column of the hi term in the down pass
              uint8_t* atom = p.hsf + ((static_cast<size_t>(row0 / BN) * (p.Fp / 128) + g) * C::NA) * 512;
              atom[(n >> 7) * 512 + sf_atom_offset(n & 127, kb)] = static_cast<uint8_t>(e.s_hi);
              atom[((n + 1) >> 7) * 512 + sf_atom_offset((n + 1) & 127, kb)] = static_cast<uint8_t>(e.s_lo);
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int j = j0 + jj;
            if (j >= nrows) continue;
            const int a = p.perm[p0 + j];
            const float y = (__uint_as_float(rg[2 * jj]) + __uint_as_float(rg[2 * jj + 1])) * p.G[a];
            if (f_ok) p.y[static_cast<size_t>(a) * p.N_out + f] = y;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int BN, bool GU>
cudaError_t launch_moe(const MoeGemmParams& p, int grid, cudaStream_t s) {
  using C = MoeCfg<BN, GU>;
  cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<BN, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  moe_gemm_kernel<BN, GU><<<grid, kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------ activation encode
// One warp per assignment: x^c row of its token -> hi/lo E4M3 rows 2r, 2r+1
// of the padded layout, scales into the staging image of the row's tile.
__global__ void quant_gather_kernel(const float* __restrict__ xc, int T, int k, int din, int Kp,
                                    const int32_t* __restrict__ inv_pad, int BN, uint8_t* __restrict__ xq,
                                    uint8_t* __restrict__ xsf) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int P = T * k;
  if (warp >= P) return;
  const int a = warp;
  const int r = inv_pad[a];
  const int t = a / k;
  const int NA = (2 * BN + 127) / 128;
  const int KG = Kp / 128;
  const float* row = xc + static_cast<size_t>(t) * din;
  const int jt = r % BN;
  uint8_t* atoms = xsf + static_cast<size_t>(r / BN) * KG * NA * 512;
  for (int blk = 0; blk < Kp / 32; ++blk) {
    const int c = blk * 32 + lane;
    const float v = c < din ? row[c] : 0.0f;
    const HiLo e = quant_hilo_warp(v);
    xq[(2 * static_cast<size_t>(r)) * Kp + c] = e.q_hi;
    xq[(2 * static_cast<size_t>(r) + 1) * Kp + c] = e.q_lo;
    if (lane == 0) {
      const int g = blk >> 2, kb = blk & 3;
      const int n = 2 * jt;
      uint8_t* at = atoms + static_cast<size_t>(g) * NA * 512;
      at[(n >> 7) * 512 + sf_atom_offset(n & 127, kb)] = static_cast<uint8_t>(e.s_hi);
      at[((n + 1) >> 7) * 512 + sf_atom_offset((n + 1) & 127, kb)] = static_cast<uint8_t>(e.s_lo);
    }
  }
}

// One block per token: u = sum over the token's k slots in slot order, then
// RMSNorm (Kimi K3 card code: routed_expert_norm between the sum and the
// up-projection).
__global__ void combine_norm_kernel(const float* __restrict__ y, int T, int k, int l,
                                    const __nv_bfloat16* __restrict__ w, int use_norm, float eps,
                                    float* __restrict__ u_out, __nv_bfloat16* __restrict__ u_hat) {
  extern __shared__ float cn_u[];
  __shared__ float red[32];
  const int t = blockIdx.x;
  const float* yt = y + static_cast<size_t>(t) * k * l;
  float ss = 0.f;
  for (int i = threadIdx.x; i < l; i += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j) acc += yt[static_cast<size_t>(j) * l + i];
    cn_u[i] = acc;
    u_out[static_cast<size_t>(t) * l + i] = acc;
    ss += acc * acc;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float rs = use_norm ? rsqrtf(red[0] / static_cast<float>(l) + eps) : 1.0f;
  for (int i = threadIdx.x; i < l; i += blockDim.x) {
    const float wv = use_norm ? __bfloat162float(w[i]) : 1.0f;
    u_hat[static_cast<size_t>(t) * l + i] = __float2bfloat16_rn(wv * cn_u[i] * rs);
  }
}

__global__ void relayout_sfa_kernel(const uint8_t* __restrict__ s, int E, int N, int Kb, int MT, int KG,
                                    uint8_t* __restrict__ atoms) {
  const size_t total = static_cast<size_t>(E) * MT * KG * 512;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i & 511);
    size_t rest = i >> 9;
    const int g = static_cast<int>(rest % KG);
    rest /= KG;
    const int mt = static_cast<int>(rest % MT);
    const int e = static_cast<int>(rest / MT);
    const int r0 = b >> 4, c = (b >> 2) & 3, kb = b & 3;
    const int n = mt * 128 + 32 * c + r0;
    const int kblk = 4 * g + kb;
    atoms[i] = (n < N && kblk < Kb) ? s[(static_cast<size_t>(e) * N + n) * Kb + kblk] : static_cast<uint8_t>(127);
  }
}

__global__ void pad_codes_kernel(const uint8_t* __restrict__ q, int E, int N, int K, int Kp, uint8_t* __restrict__ out) {
  const size_t total = static_cast<size_t>(E) * N * (Kp / 2);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t rowi = i / (Kp / 2);
    const int c = static_cast<int>(i % (Kp / 2));
    out[i] = c < K / 2 ? q[rowi * (K / 2) + c] : static_cast<uint8_t>(0);
  }
}

int ew_grid(size_t n) {
  size_t g = (n + 255) / 256;
  return static_cast<int>(g < 152 * 16 ? (g ? g : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_moe_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_moe<16, true>(p, grid, s);
    case 64: return launch_moe<64, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_moe_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_moe<16, false>(p, grid, s);
    case 64: return launch_moe<64, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quant_gather(const float* xc, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                uint8_t* xq, uint8_t* xsf, cudaStream_t s) {
  const int P = T * k;
  if (P <= 0) return cudaSuccess;
  const int warps_per_block = 8;
  quant_gather_kernel<<<(P + warps_per_block - 1) / warps_per_block, 32 * warps_per_block, 0, s>>>(
      xc, T, k, din, Kp, inv_pad, BN, xq, xsf);
  return cudaGetLastError();
}

cudaError_t launch_combine_norm(const float* y, int T, int k, int l, const void* norm_w, int use_norm, float eps,
                                float* u, void* u_hat, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(l) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(combine_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  combine_norm_kernel<<<T, 256, smem, s>>>(y, T, k, l, static_cast<const __nv_bfloat16*>(norm_w), use_norm, eps, u,
                                          static_cast<__nv_bfloat16*>(u_hat));
  return cudaGetLastError();
}

cudaError_t launch_relayout_sfa(const uint8_t* s, int E, int N, int Kb, int MT, int KG, uint8_t* atoms,
                                cudaStream_t st) {
  const size_t total = static_cast<size_t>(E) * MT * KG * 512;
  relayout_sfa_kernel<<<ew_grid(total), 256, 0, st>>>(s, E, N, Kb, MT, KG, atoms);
  return cudaGetLastError();
}

cudaError_t launch_pad_codes(const uint8_t* q, int E, int N, int K, int Kp, uint8_t* out, cudaStream_t st) {
  const size_t total = static_cast<size_t>(E) * N * (Kp / 2);
  pad_codes_kernel<<<ew_grid(total), 256, 0, st>>>(q, E, N, K, Kp, out);
  return cudaGetLastError();
}

}  // namespace lmoe
