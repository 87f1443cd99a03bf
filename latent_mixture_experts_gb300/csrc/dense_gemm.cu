// Dense bf16 GEMMs of the layer on the 5th-generation tensor cores:
// router logits, latent down-projection, shared-expert gate/up, and the
// K-concatenated [u_hat | h_shared] x [W_up ; W_shared_down] output GEMM.
//
// Weights are the MMA's A operand (M = 128 output features per tile) and
// tokens the B operand (N = BN tokens): at decode the token count is small
// and the weights are streamed once.  Operands arrive by TMA with 128-byte
// swizzle into a multi-stage shared-memory ring; one thread issues
// tcgen05.mma into a TMEM fp32 accumulator; all four warps read it back
// with tcgen05.ld and store fp32 partial sums per K split.
#include "common.cuh"
#include "lmoe_internal.h"

namespace lmoe {

namespace {

// MT: 128-row weight tiles per CTA.  MT = 2 (wide, the prefill tile BN =
// 256): one 256-row A box per stage and two accumulators filling tensor
// memory, which halves the activation bytes each CTA moves per MAC.
template <int BN, int MT>
struct DenseCfg {
  static constexpr int kA = MT * 16384;        // MT x 128 rows x 64 bf16
  static constexpr int kB = BN * 128;          // BN rows x 64 bf16
  static constexpr int kStage = kA + kB;
  static constexpr int kStagesFit = (227 * 1024 - 2048) / (kA + BN * 128);
  // decode tiles (BN <= 64) keep a stage ring of ~100 KB so two CTAs share
  // an SM: twice the weight bytes in flight per SM of one deeper ring
  static constexpr int kStages = MT == 2 ? (kStagesFit < 6 ? kStagesFit : 6)
                                         : (BN >= 256 ? 4 : (BN >= 128 ? 5 : (BN >= 64 ? 4 : 5)));
  static constexpr int kSmem = kStages * kStage + 1024;
  static constexpr int kTmemCols = MT * BN < 32 ? 32 : MT * BN;
  static_assert(kTmemCols <= 512, "tensor memory budget");
};

template <int BN, int MT>
__global__ void __launch_bounds__(128, 1) dense_gemm_kernel(const __grid_constant__ DenseParams p) {
  using C = DenseCfg<BN, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  __shared__ uint64_t full[C::kStages], empty[C::kStages], done;
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x, nt = blockIdx.y, sp = blockIdx.z;
  const int mtw0 = (p.mtiles0 + MT - 1) / MT;           // CTA tiles of the first segment
  const bool pair = MT == 2 && p.epi == 2;               // gate rows + up rows of the same features
  const int seg = (!pair && p.mode == 1 && mt >= mtw0) ? 1 : 0;
  const int m0 = pair ? mt * 128 : (seg ? mt - mtw0 : mt) * 128 * MT;
  const int Mseg = seg ? p.M1 : p.M0;
  const int out_row0 = (seg ? p.M0 : 0) + m0;
  const int n0 = nt * BN;
  const int kb0 = static_cast<int>((static_cast<long long>(sp) * p.nkb) / p.splits);
  const int kb1 = static_cast<int>((static_cast<long long>(sp + 1) * p.nkb) / p.splits);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch();
  const bool producer = warp == 0 && lane == 0;
  if (!producer) griddep_wait();   // the producer waits after requesting its first weight tiles
  const uint32_t tacc = tmem_base;

  if (producer) {
    // TMA producer.  The weights are never written by an earlier kernel, so
    // the first stages' weight tiles are requested before waiting for the
    // preceding kernel; its tokens (the B tiles) only after.
    const CUtensorMap* am = MT == 2 ? (seg ? &p.a1w : &p.a0w) : (seg ? &p.a1 : &p.a0);
    tma_prefetch_desc(am);
    tma_prefetch_desc(&p.b0);
    auto load = [&](int kb, int s, bool a_part) {
      const CUtensorMap* A = am;
      const CUtensorMap* B = &p.b0;
      int kc = kb * 64;
      if (p.mode == 2 && kb >= p.nkb0) {
        A = MT == 2 ? &p.a1w : &p.a1;
        B = &p.b1;
        kc = (kb - p.nkb0) * 64;
      }
      uint8_t* st = sm + s * C::kStage;
      if (!a_part) {
        tma_load_2d(st + C::kA, B, &full[s], kc, n0);
      } else if (pair) {   // gate rows then up rows of features m0.. (one 256-row box of the interleaved copy)
        tma_load_2d(st, &p.a0w, &full[s], kc, 2 * m0);
      } else {
        tma_load_2d(st, A, &full[s], kc, m0);
      }
    };
    const int npre = kb1 - kb0 < C::kStages ? kb1 - kb0 : C::kStages;
    for (int i = 0; i < npre; ++i) {
      mbar_arrive_expect_tx(&full[i], C::kStage);
      load(kb0 + i, i, true);
    }
    griddep_wait();
    for (int i = 0; i < npre; ++i) load(kb0 + i, i, false);
    for (int kb = kb0 + npre, i = npre; kb < kb1; ++kb, ++i) {
      const int s = i % C::kStages;
      if (i >= C::kStages && !mbar_wait(&empty[s], ((i / C::kStages) - 1) & 1, p.err, kErrTimeout)) break;
      mbar_arrive_expect_tx(&full[s], C::kStage);
      load(kb, s, true);
      load(kb, s, false);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    constexpr uint32_t idesc = idesc_bf16(128, BN);
    for (int kb = kb0, i = 0; kb < kb1; ++kb, ++i) {
      const int s = i % C::kStages;
      if (!mbar_wait(&full[s], (i / C::kStages) & 1, p.err, kErrTimeout)) break;
      tc_fence_after();
      const uint32_t a_addr = smem_u32(sm + s * C::kStage);
      const uint32_t b_addr = a_addr + C::kA;
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int t = 0; t < MT; ++t)
          mma_bf16(tacc + t * BN, sdesc_sw128(a_addr + t * 16384 + 32 * k), sdesc_sw128(b_addr + 32 * k), idesc,
                   (i | k) != 0);
      mma_commit(&empty[s]);
    }
    mma_commit(&done);
  }
  __syncwarp();

  // Epilogue: lane = output feature, column = token.
  const bool ok = mbar_wait(&done, 0, p.err, kErrTimeout);
  tc_fence_after();
  const bool have = ok && kb1 > kb0;
  if (pair) {
    // h[t][f] = act(gate, up): gate in the first accumulator, up in the second
    const int f = m0 + 32 * warp + lane;
    __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(p.out16);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      if (n0 + c0 >= p.T) break;
      uint32_t g[16], u[16];
      tmem_ld16(tmem_addr(tacc, 32 * warp, c0), g);
      tmem_ld16(tmem_addr(tacc + BN, 32 * warp, c0), u);
      tmem_ld_wait();
      if (f < p.M0) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = n0 + c0 + j;
          const float h =
              have ? glu_act(__uint_as_float(g[j]), __uint_as_float(u[j]), p.act, p.act_b1, p.act_b2) : 0.0f;
          if (t < p.T) o16[static_cast<size_t>(t) * p.ldo + f] = __float2bfloat16_rn(h);
        }
      }
    }
  }
#pragma unroll 1
  for (int mtl = 0; mtl < (pair ? 0 : MT); ++mtl) {
    const int row = m0 + mtl * 128 + 32 * warp + lane;
    const bool row_ok = row < Mseg;
    float* outp = p.out + static_cast<size_t>(sp) * p.T * p.ldo + out_row0 + mtl * 128 + 32 * warp + lane;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      if (n0 + c0 >= p.T) break;
      uint32_t r[16];
      tmem_ld16(tmem_addr(tacc + mtl * BN, 32 * warp, c0), r);
      tmem_ld_wait();
      if (row_ok && p.epi == 1) {
        // direct bf16 result (one K split), plus the optional fp32 addend
        __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(p.out16) + out_row0 + mtl * 128 + 32 * warp + lane;
        const float* ad = p.add ? p.add + out_row0 + mtl * 128 + 32 * warp + lane : nullptr;
        float* o32 = p.out32 ? p.out32 + out_row0 + mtl * 128 + 32 * warp + lane : nullptr;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = n0 + c0 + j;
          if (t < p.T) {
            float v = have ? __uint_as_float(r[j]) : 0.0f;
            if (ad) v += ad[static_cast<size_t>(t) * p.ld_add];
            o16[static_cast<size_t>(t) * p.ldo] = __float2bfloat16_rn(v);
            if (o32) o32[static_cast<size_t>(t) * p.ldo] = v;
          }
        }
      } else if (row_ok) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = n0 + c0 + j;
          if (t < p.T) outp[static_cast<size_t>(t) * p.ldo] = have ? __uint_as_float(r[j]) : 0.0f;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tacc, C::kTmemCols);
}

template <int BN, int MT>
cudaError_t launch_bn(const DenseParams& p, int mtiles, cudaStream_t s) {
  using C = DenseCfg<BN, MT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(dense_gemm_kernel<BN, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // CTA tiles: MT 128-row tiles each, counted per M segment (a gate/up pair
  // CTA covers one 128-row tile of each segment)
  const int seg0 = p.mode == 1 ? p.mtiles0 : mtiles;
  const int ctas_m = (MT == 2 && p.epi == 2) ? p.mtiles0
                                             : (seg0 + MT - 1) / MT + (mtiles - seg0 + MT - 1) / MT;
  dim3 grid(ctas_m, (p.T + BN - 1) / BN, p.splits);
  {
    const cudaError_t e_ = launch_pdl(dense_gemm_kernel<BN, MT>, grid, 128, C::kSmem, s, p);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------- finalizers
__global__ void finalize_sum_f32_kernel(const float* __restrict__ part, int splits, int T, int M, int ld,
                                        float* __restrict__ out, int ldo) {
  griddep_launch();
  griddep_wait();
  const size_t n = static_cast<size_t>(T) * M;
  const size_t plane = static_cast<size_t>(T) * ld;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / M, m = i % M;
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[s * plane + t * ld + m];
    out[t * ldo + m] = acc;
  }
}

__global__ void finalize_sum_bf16_kernel(const float* __restrict__ part, int splits, int T, int M, int ld,
                                         __nv_bfloat16* __restrict__ out, int ldo, const float* __restrict__ add,
                                         int ld_add, float* __restrict__ out32) {
  griddep_launch();
  griddep_wait();
  const size_t n = static_cast<size_t>(T) * M;
  const size_t plane = static_cast<size_t>(T) * ld;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / M, m = i % M;
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) acc += part[s * plane + t * ld + m];
    if (add) acc += add[t * ld_add + m];
    out[t * ldo + m] = __float2bfloat16_rn(acc);
    if (out32) out32[t * ldo + m] = acc;
  }
}

__global__ void finalize_glu_bf16_kernel(const float* __restrict__ part, int splits, int T, int F, int ld,
                                         __nv_bfloat16* __restrict__ out, int act, float b1, float b2) {
  griddep_launch();
  griddep_wait();
  const size_t n = static_cast<size_t>(T) * F;
  const size_t plane = static_cast<size_t>(T) * ld;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / F, f = i % F;
    float g = 0.f, u = 0.f;
    for (int s = 0; s < splits; ++s) {
      g += part[s * plane + t * ld + f];
      u += part[s * plane + t * ld + F + f];
    }
    out[t * F + f] = __float2bfloat16_rn(glu_act(g, u, act, b1, b2));
  }
}

// Shared gate/up weights with gate and up interleaved every 128 rows:
// row r of the copy = gate row (r/256)*128 + r%256 for r%256 < 128, else up
// row (r/256)*128 + r%256 - 128; rows past Fs are zero.
__global__ void interleave_gate_up_kernel(const __nv_bfloat16* __restrict__ gate, const __nv_bfloat16* __restrict__ up,
                                          int Fs, int K, __nv_bfloat16* __restrict__ out, int rows) {
  const size_t total = static_cast<size_t>(rows) * K;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / K), c = static_cast<int>(i % K);
    const int w = r % 256, f = (r / 256) * 128 + (w % 128);
    const __nv_bfloat16* src = w < 128 ? gate : up;
    out[i] = f < Fs ? src[static_cast<size_t>(f) * K + c] : __float2bfloat16_rn(0.0f);
  }
}

int ew_grid(size_t n) {
  size_t g = (n + 255) / 256;
  return static_cast<int>(g < 152 * 16 ? (g ? g : 1) : 152 * 16);
}

// Elementwise finalizers launch early (programmatic serialization) only with
// a small grid: an early-launched grid waits resident on the SMs until its
// predecessor ends, and a large one holds the thread slots that the other
// stream's kernels need (at 64 tokens the activation encoder stalled behind
// the waiting finalizer of the side stream's shared gate/up GEMM).
constexpr int kEarlyLaunchMaxBlocks = 256;
template <class... KArgs, class... Args>
cudaError_t launch_ew(void (*kernel)(KArgs...), size_t n, cudaStream_t s, Args... args) {
  const int g = ew_grid(n);
  if (g <= kEarlyLaunchMaxBlocks) return launch_pdl(kernel, g, 256, 0, s, args...);
  kernel<<<g, 256, 0, s>>>(static_cast<KArgs>(args)...);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_gemm(const DenseParams& p, int mtiles, int BN, cudaStream_t s) {
  // A wide launch of the M-concatenated gate/up GEMM exists only as the
  // gate/up pair (its weights come from the interleaved copy in a0w); no
  // 256-row maps of the separate gate and up matrices are kept.
  if (p.wide && (BN != 256 || (p.mode == 1 && p.epi != 2))) return cudaErrorInvalidValue;
  switch (BN) {
    case 32: return launch_bn<32, 1>(p, mtiles, s);
    case 64: return launch_bn<64, 1>(p, mtiles, s);
    case 128: return launch_bn<128, 1>(p, mtiles, s);
    case 256: return p.wide ? launch_bn<256, 2>(p, mtiles, s) : launch_bn<256, 1>(p, mtiles, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_interleave_gate_up(const void* gate, const void* up, int Fs, int K, void* out, cudaStream_t s) {
  const int rows = 2 * ((Fs + 127) / 128) * 128;
  interleave_gate_up_kernel<<<ew_grid(static_cast<size_t>(rows) * K), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(gate), static_cast<const __nv_bfloat16*>(up), Fs, K,
      static_cast<__nv_bfloat16*>(out), rows);
  return cudaGetLastError();
}

cudaError_t launch_finalize_sum_f32(const float* part, int splits, int T, int M, int ld, float* out, int ldo,
                                    cudaStream_t s) {
  const size_t n = static_cast<size_t>(T) * M;
  {
    const cudaError_t e_ = launch_ew(finalize_sum_f32_kernel, n, s, part, splits, T, M, ld, out, ldo);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize_sum_bf16(const float* part, int splits, int T, int M, int ld, void* out, int ldo,
                                     const float* add_opt, int ld_add, float* out32_opt, cudaStream_t s) {
  const size_t n = static_cast<size_t>(T) * M;
  {
    const cudaError_t e_ = launch_ew(finalize_sum_bf16_kernel, n, s, part, splits, T, M, ld,
                                     static_cast<__nv_bfloat16*>(out), ldo, add_opt, ld_add, out32_opt);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_finalize_glu_bf16(const float* part, int splits, int T, int F, int ld, void* out, int act,
                                     float b1, float b2, cudaStream_t s) {
  const size_t n = static_cast<size_t>(T) * F;
  {
    const cudaError_t e_ = launch_ew(finalize_glu_bf16_kernel, n, s, part, splits, T, F, ld,
                                     static_cast<__nv_bfloat16*>(out), act, b1, b2);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace lmoe
