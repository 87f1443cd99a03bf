// Routed experts with FP8 E4M3 weights and fp32 scales per 128 x 128 block
// (Kimi K2 card: the K2 checkpoint format; SwiGLU experts on the full width).
//
// Same pipeline as the MXFP4 kernel (TMA producer warp, single-thread MMA
// issuer, four epilogue warps, persistent walk of the device tile list), on
// block-scaled tcgen05 MMA (kind::mxf8f6f4, both operands E4M3).  The weight
// scale is an fp32 number per 128 rows x 128 K, which an E8M0 scale cannot
// carry, so the weights enter the MMA with unit scales and every 128-K group
// is accumulated on its own: the MMA writes the group's partial product into
// one of two TMEM buffers, and the epilogue warps add it, times that block's
// fp32 scale, into register accumulators.  After the last group the item's
// epilogue runs from those registers: SwiGLU (or SiTU) and the hi/lo E4M3
// encoding of h for the gate/up pass, the routing weight for the down pass.
#include "moe_common.cuh"

namespace lmoe {

namespace {

template <int BN, bool GU>
struct Fp8Cfg {
  static constexpr int N = 2 * BN;                   // hi/lo columns of BN assignments
  static constexpr int RB = fp8_rows_per_item(BN);   // weight rows per TMA box
  static constexpr int kTiles = RB / 128;
  static constexpr int kBoxes = 2;                   // gate + up, or two down boxes
  static constexpr int IR = GU ? RB : 2 * RB;        // weight rows of one work item
  static constexpr int kNAcc = kBoxes * kTiles;
  static constexpr int kA = RB * 128;                // RB rows x 128 E4M3 codes
  static constexpr int kB = N * 128;
  static constexpr int kTile = kBoxes * kA + kB;
  static constexpr int kSfb = 512;
  static constexpr int kTx = kBoxes * kA + kB + kSfb;
  static constexpr int kStages = RB == 256 ? 3 : 5;
  static constexpr int kSmem = kStages * (kTile + kSfb) + 1024;
  static constexpr int kPart = kNAcc * N;            // columns of one partial-product buffer
  static constexpr int kSfaCol = 2 * kPart;          // constant unit weight scales (4 columns)
  static constexpr int kSfbCol = kSfaCol + 4;        // activation scales, one slot per stage
  static constexpr int kTmemUsed = kSfbCol + 4 * kStages;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static_assert(N <= 128, "one activation scale atom per stage");
  static_assert(kTile % 1024 == 0, "tiles keep 1024-byte alignment");
  static_assert(kTmemUsed <= 512, "tensor memory budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

template <int BN, bool GU>
__global__ void __launch_bounds__(kThreads, 1) moe_fp8_kernel(const __grid_constant__ MoeGemmParams p) {
  using C = Fp8Cfg<BN, GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sf_region = sm + C::kStages * C::kTile;
  __shared__ uint64_t full[C::kStages], empty[C::kStages], part_full[2], part_empty[2];
  __shared__ uint32_t tmem_base;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&part_full[i], 1);
      mbar_init(&part_empty[i], kEpiWarps * 32);
    }
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
  if (warp >= 2) {
    // unit E8M0 scale (127) in every byte of the weight-scale columns
    const uint32_t one = 0x7F7F7F7Fu;
    tmem_st4(tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + C::kSfaCol, one, one, one, one);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int ntiles = *p.ntiles;
  const int total = ntiles * p.MT;
  const int KG = p.KG;
  auto st_a = [&](int s, int j) { return sm + s * C::kTile + j * C::kA; };
  auto st_b = [&](int s) { return sm + s * C::kTile + C::kBoxes * C::kA; };
  auto st_sfb = [&](int s) { return sf_region + s * C::kSfb; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.a_gate);
      if (GU) tma_prefetch_desc(&p.a_up);
      tma_prefetch_desc(&p.b);
      uint32_t it = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        int mt;
        const int4 tile = decode_item<BN>(p, w, mt);
        const int e = tile.x, row0 = tile.y;
        const int arow = e * p.N_out + mt * C::IR;
        const int arow1 = GU ? arow : arow + C::RB;
        const CUtensorMap* map1 = GU ? &p.a_up : &p.a_gate;
        const size_t sfb_idx = static_cast<size_t>(row0 / BN) * KG;
        for (int g = 0; g < KG; ++g, ++it) {
          const int s = it % C::kStages;
          if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], C::kTx);
          tma_load_2d(st_a(s, 0), &p.a_gate, &full[s], g * 128, arow);
          tma_load_2d(st_a(s, 1), map1, &full[s], g * 128, arow1);
          tma_load_2d(st_b(s), &p.b, &full[s], g * 128, 2 * row0);
          bulk_g2s(st_sfb(s), p.sfb + (sfb_idx + g) * C::kSfb, C::kSfb, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      const uint32_t sfa = tbase + C::kSfaCol;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        for (int g = 0; g < KG; ++g, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          const uint32_t pb = it & 1, use = it >> 1;
          if (use > 0 && !mbar_wait(&part_empty[pb], (use - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb = tbase + C::kSfbCol + 4 * s;
          tmem_cp_32x128b_x4(sfb, sdesc_noswz(smem_u32(st_sfb(s)), 16, 128));
          const uint32_t bb = smem_u32(st_b(s));
          const uint32_t d0 = tbase + pb * C::kPart;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t idesc = idesc_mxf8f6f4(128, C::N, 0, 0, kb, kb);
#pragma unroll
            for (int i = 0; i < C::kNAcc; ++i) {
              const uint32_t a_addr = smem_u32(st_a(s, i / C::kTiles)) + (i % C::kTiles) * 16384 + 32 * kb;
              mma_mxf8f6f4(d0 + i * C::N, sdesc_sw128(a_addr), sdesc_sw128(bb + 32 * kb), idesc, sfa, sfb, kb != 0);
            }
          }
          mma_commit(&empty[s]);
          mma_commit(&part_full[pb]);
        }
      }
    }
  } else {
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      int mt;
      const int4 tile = decode_item<BN>(p, w, mt);
      const int e = tile.x, row0 = tile.y, nrows = tile.z, p0 = tile.w;
      // fp32 block scale rows of the accumulators: box j, tile t -> rows mt*IR + j*RB(down)/0(gate,up) + 128t
      const float* bsc[C::kNAcc];
#pragma unroll
      for (int i = 0; i < C::kNAcc; ++i) {
        const int j = i / C::kTiles, t = i % C::kTiles;
        int rt = (mt * C::IR + (GU ? 0 : j * C::RB) + t * 128) / 128;
        rt = rt < p.NB ? rt : p.NB - 1;
        bsc[i] = ((GU && j == 1) ? p.wsc1 : p.wsc0) + (static_cast<size_t>(e) * p.NB + rt) * p.KB;
      }
      float acc[C::kNAcc][C::N];
#pragma unroll
      for (int i = 0; i < C::kNAcc; ++i)
#pragma unroll
        for (int c = 0; c < C::N; ++c) acc[i][c] = 0.f;
      for (int g = 0; g < KG; ++g, ++it) {
        float sc[C::kNAcc];
#pragma unroll
        for (int i = 0; i < C::kNAcc; ++i) sc[i] = __ldg(bsc[i] + g);
        const uint32_t pb = it & 1;
        if (!mbar_wait(&part_full[pb], (it >> 1) & 1, p.err, kErrTimeout)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < C::kNAcc; ++i) {
#pragma unroll
          for (int c0 = 0; c0 < C::N; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(tbase + lane_off + pb * C::kPart + i * C::N + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[i][c0 + c] = fmaf(sc[i], __uint_as_float(v[c]), acc[i][c0 + c]);
          }
        }
        tc_fence_before();
        mbar_arrive(&part_empty[pb]);
      }
      if (!ok) break;
      if constexpr (GU) {
#pragma unroll
        for (int t = 0; t < C::kTiles; ++t) {
          if (mt * C::RB + t * 128 >= p.Fp) break;
          const int f = mt * C::RB + t * 128 + 32 * q + lane;
          const bool f_ok = f < p.N_out;
          const int kblk = f >> 5;
          const int g = kblk >> 2, kb = kblk & 3;
#pragma unroll
          for (int j = 0; j < BN; ++j) {
            if (j < nrows) {                                   // warp-uniform
              const float gv = acc[t][2 * j] + acc[t][2 * j + 1];
              const float uv = acc[C::kTiles + t][2 * j] + acc[C::kTiles + t][2 * j + 1];
              const float h = f_ok ? glu_act_fast(gv, uv, p.act, p.b1, p.b2) : 0.0f;
              const HiLo hl = quant_hilo_warp(h);
              const size_t r = static_cast<size_t>(row0) + j;
              p.hq[(2 * r) * p.Fp + f] = hl.q_hi;
              p.hq[(2 * r + 1) * p.Fp + f] = hl.q_lo;
              if (lane == 0) {
                const int n = 2 * j;
                uint8_t* atom = p.hsf + (static_cast<size_t>(row0 / BN) * (p.Fp / 128) + g) * 512;
                atom[sf_atom_offset(n, kb)] = static_cast<uint8_t>(hl.s_hi);
                atom[sf_atom_offset(n + 1, kb)] = static_cast<uint8_t>(hl.s_lo);
              }
            }
          }
        }
      } else {
        int a_lo = 0;
        float g_lo = 0.f;
        if (lane < nrows) {
          a_lo = p.perm[p0 + lane];
          g_lo = p.G[a_lo];
        }
#pragma unroll
        for (int i = 0; i < C::kNAcc; ++i) {
          const int f = mt * C::IR + i * 128 + 32 * q + lane;
          const bool f_ok = f < p.N_out;
#pragma unroll
          for (int j = 0; j < BN; ++j) {
            if (j < nrows) {
              const int a = __shfl_sync(0xFFFFFFFFu, a_lo, j);
              const float gw = __shfl_sync(0xFFFFFFFFu, g_lo, j);
              if (f_ok) p.y[static_cast<size_t>(a) * p.N_out + f] = (acc[i][2 * j] + acc[i][2 * j + 1]) * gw;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int BN, bool GU>
cudaError_t launch_fp8(const MoeGemmParams& p, int grid, cudaStream_t s) {
  using C = Fp8Cfg<BN, GU>;
  cudaError_t e = cudaFuncSetAttribute(moe_fp8_kernel<BN, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  moe_fp8_kernel<BN, GU><<<grid, kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

// Block-scaled FP8 [N][K] (fp32 scale per 128 x 128) -> bf16 [N][K].
__global__ void dequant_fp8_block128_kernel(const uint8_t* __restrict__ q, const float* __restrict__ s, int N, int K,
                                            __nv_bfloat16* __restrict__ out) {
  const int KB = (K + 127) / 128;
  const size_t total = static_cast<size_t>(N) * K;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(i / K), k = static_cast<int>(i % K);
    out[i] = __float2bfloat16_rn(e4m3_to_f32(q[i]) * s[(n / 128) * KB + k / 128]);
  }
}

}  // namespace

cudaError_t launch_moe_fp8_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp8<16, true>(p, grid, s);
    case 32: return launch_fp8<32, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_moe_fp8_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp8<16, false>(p, grid, s);
    case 32: return launch_fp8<32, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dequant_fp8_block128(const uint8_t* q, const float* s, int N, int K, void* out, cudaStream_t st) {
  const size_t total = static_cast<size_t>(N) * K;
  size_t g = (total + 255) / 256;
  if (g > 152 * 32) g = 152 * 32;
  dequant_fp8_block128_kernel<<<static_cast<unsigned>(g ? g : 1), 256, 0, st>>>(q, s, N, K,
                                                                             static_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

}  // namespace lmoe
