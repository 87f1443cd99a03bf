// Routed experts with FP8 E4M3 weights and fp32 scales per 128 x 128 block
// (Kimi K2 card: the K2 checkpoint format; SwiGLU experts on the full width).
//
// Persistent grouped GEMM over the device tile list: a TMA producer warp, a
// single-thread tcgen05 MMA issuer (kind::mxf8f6f4, both operands E4M3) and
// eight epilogue warps.  A work item is one 128-row block of gate and of up
// weights (gate/up pass) or two 128-row blocks of down weights (down pass),
// times one tile of up to 96 assignments.
//
// Activations are two E4M3 terms (hi + lo, each with an E8M0 scale per 32)
// stored in the split layout: the tile's hi rows, then its lo rows.  Every
// k-block issues one MMA on the hi rows and one on the lo rows into the SAME
// accumulator columns, so tensor memory holds one column per assignment and
// a 96-assignment tile fits; an expert's weights then pass through the SM
// about once per expert instead of once per 32 assignments.
//
// The weight scale is an fp32 number per 128 rows x 128 K, which an E8M0
// scale cannot carry, so the weights enter the MMA with unit scales and each
// 128-K group is accumulated on its own into one buffer of a ring in tensor
// memory; the epilogue warps add it, times that block's scale, into register
// accumulators (two warps per 32-lane quarter, each owning half of the
// tile's columns).  A work item's 128 rows share one scale per 128-K group,
// so each lane holds the item's scales for groups lane and lane + 32 in
// registers (fetched one item ahead) and a group's scale is a warp shuffle.
// After the last group the item's epilogue runs from the registers: SwiGLU
// (or SiTU) and the split hi/lo E4M3 encoding of h for the gate/up pass, the
// routing weight for the down pass.
#include "moe_common.cuh"

namespace lmoe {

namespace {

constexpr int kFp8EpiWarps = 8;
constexpr int kFp8Threads = 64 + 32 * kFp8EpiWarps;   // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue

template <int BN, bool GU>
struct Fp8Cfg {
  static constexpr int RB = kFp8Rows;                // weight rows per TMA box (one fp32 scale block)
  static constexpr int kBoxes = 2;                   // gate + up, or two down boxes
  static constexpr int IR = GU ? RB : 2 * RB;        // weight rows of one work item
  static constexpr int kNAcc = kBoxes;
  static constexpr int kA = RB * 128;                // RB rows x 128 E4M3 codes
  static constexpr int kB = 2 * BN * 128;            // hi rows then lo rows
  static constexpr int kTile = kBoxes * kA + kB;
  static constexpr int kSfb = 1024;                  // hi and lo activation scale atoms
  static constexpr int kTx = kBoxes * kA + kB + kSfb;
  static constexpr int kStagesFit = (227 * 1024 - 2048) / (kTile + kSfb);
  static constexpr int kStages = kStagesFit < 6 ? kStagesFit : 6;
  static constexpr int kSmem = kStages * (kTile + kSfb) + 1024;
  static constexpr int kPart = kNAcc * BN;           // columns of one partial-product buffer
  static constexpr int kRing = kPart <= 128 ? 3 : 2; // partial-product buffers
  static constexpr int kSfaCol = kRing * kPart;      // constant unit weight scales (4 columns)
  static constexpr int kSfbCol = kSfaCol + 4;        // activation scales, 8 columns per stage
  static constexpr int kTmemUsed = kSfbCol + 8 * kStages;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kHalf = BN / 2;               // columns per epilogue warp
  static constexpr int kLd = kHalf % 16 == 0 ? 16 : 8;
  static_assert(BN % 16 == 0 && BN <= 128, "MMA N and one scale atom per half");
  static_assert(kTile % 1024 == 0, "tiles keep 1024-byte alignment");
  static_assert(kStages >= 2, "pipeline depth");
  static_assert(kTmemUsed <= 512, "tensor memory budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* v) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(v));
  } else {
    tmem_ld8(taddr, *reinterpret_cast<uint32_t(*)[8]>(v));
  }
}

// 320 threads, one CTA per SM.  Registers are allocated per SM
// sub-partition and one of the four holds three of the ten warps, so a
// thread gets at most 168.
template <int BN, bool GU>
__global__ void __launch_bounds__(kFp8Threads, 1) moe_fp8_kernel(const __grid_constant__ MoeGemmParams p) {
  using C = Fp8Cfg<BN, GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sf_region = sm + C::kStages * C::kTile;
  __shared__ uint64_t full[C::kStages], empty[C::kStages], part_full[C::kRing], part_empty[C::kRing];
  __shared__ uint32_t tmem_base;
  __shared__ ItemRing ring;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < C::kRing; ++i) {
      mbar_init(&part_full[i], 1);
      mbar_init(&part_empty[i], kFp8EpiWarps * 32);
    }
    ring_init(ring, kFp8EpiWarps);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch();
  griddep_wait();
  const uint32_t tbase = tmem_base;
  if (warp >= 2 && warp < 6) {
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
      // the next item is claimed four k-groups before the current one's last load
      const int claim_g = KG > 4 ? KG - 4 : 0;
      int w = static_cast<int>(blockIdx.x) < total ? static_cast<int>(blockIdx.x) : -1;
      for (uint32_t n = 0; ok; ++n) {
        if (!ring_put(ring, n, w, p.err) || w < 0) break;
        int nxt = total;
        int mt;
        const int4 tile = decode_item<BN>(p, w, mt);
        const int e = tile.x, row0 = tile.y;
        const int arow = e * p.N_out + mt * C::IR;
        const int arow1 = GU ? arow : arow + C::RB;
        const CUtensorMap* map1 = GU ? &p.a_up : &p.a_gate;
        const size_t sfb_idx = static_cast<size_t>(row0 / BN) * KG;
        for (int g = 0; g < KG; ++g, ++it) {
          if (g == claim_g) nxt = claim_item(p.sched);
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
        w = nxt < total ? nxt : -1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      const uint32_t sfa = tbase + C::kSfaCol;
      for (uint32_t n = 0; ok; ++n) {
        if (ring_take(ring, n, p.err) < 0) break;
        for (int g = 0; g < KG; ++g, ++it) {
          const int s = it % C::kStages;
          if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          const uint32_t pb = it % C::kRing, use = it / C::kRing;
          if (use > 0 && !mbar_wait(&part_empty[pb], (use - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfb_hi = tbase + C::kSfbCol + 8 * s, sfb_lo = sfb_hi + 4;
          tmem_cp_32x128b_x4(sfb_hi, sdesc_noswz(smem_u32(st_sfb(s)), 16, 128));
          tmem_cp_32x128b_x4(sfb_lo, sdesc_noswz(smem_u32(st_sfb(s) + 512), 16, 128));
          const uint32_t b_hi = smem_u32(st_b(s)), b_lo = b_hi + BN * 128;
          const uint32_t d0 = tbase + pb * C::kPart;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t idesc = idesc_mxf8f6f4(128, BN, 0, 0, kb, kb);
#pragma unroll
            for (int i = 0; i < C::kNAcc; ++i) {
              const uint64_t a = sdesc_sw128(smem_u32(st_a(s, i)) + 32 * kb);
              mma_mxf8f6f4(d0 + i * BN, a, sdesc_sw128(b_hi + 32 * kb), idesc, sfa, sfb_hi, kb != 0);
              mma_mxf8f6f4(d0 + i * BN, a, sdesc_sw128(b_lo + 32 * kb), idesc, sfa, sfb_lo, true);
            }
          }
          mma_commit(&empty[s]);
          mma_commit(&part_full[pb]);
        }
      }
    }
  } else {
    const int q = warp & 3;                       // 32-lane quarter of tensor memory
    const int half = (warp - 2) >> 2;             // which half of the tile's columns
    const int c_base = half * C::kHalf;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    // fp32 block scales of item w: accumulator i covers weight rows
    // mt*IR + (down: i*RB), one 128-row block; lane l takes K groups l, l + 32.
    auto item_scales = [&](int w, float (&out)[C::kNAcc][2]) {
      int mt;
      const int e = decode_item<BN>(p, w, mt).x;
#pragma unroll
      for (int i = 0; i < C::kNAcc; ++i) {
        int rt = (mt * C::IR + (GU ? 0 : i * C::RB)) / 128;
        rt = rt < p.NB ? rt : p.NB - 1;
        const float* row = ((GU && i == 1) ? p.wsc1 : p.wsc0) + (static_cast<size_t>(e) * p.NB + rt) * p.KB;
        out[i][0] = lane < KG ? __ldg(row + lane) : 0.f;
        out[i][1] = lane + 32 < KG ? __ldg(row + lane + 32) : 0.f;
      }
    };
    float scl[C::kNAcc][2] = {}, nscl[C::kNAcc][2] = {};
    uint32_t it = 0, n = 0;
    bool ok = true;
    int w = ring_take_warp(ring, 0, p.err);
    if (w >= 0) item_scales(w, scl);
    while (w >= 0) {
      int mt;
      const int4 tile = decode_item<BN>(p, w, mt);
      const int row0 = tile.y, nrows = tile.z, p0 = tile.w;
      float acc[C::kNAcc][C::kHalf];
#pragma unroll
      for (int i = 0; i < C::kNAcc; ++i)
#pragma unroll
        for (int c = 0; c < C::kHalf; ++c) acc[i][c] = 0.f;
      for (int g = 0; g < KG; ++g, ++it) {
        const uint32_t pb = it % C::kRing;
        if (!mbar_wait(&part_full[pb], (it / C::kRing) & 1, p.err, kErrTimeout)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < C::kNAcc; ++i) {
          const float sc = __shfl_sync(0xFFFFFFFFu, g < 32 ? scl[i][0] : scl[i][1], g & 31);
          const uint32_t col = tbase + lane_off + pb * C::kPart + i * BN + c_base;
          // chunks of up to 32 columns: two loads in flight, one wait
#pragma unroll
          for (int c0 = 0; c0 < C::kHalf; c0 += 32) {
            constexpr int kW = 32;
            uint32_t v[kW];
            const int n = C::kHalf - c0 < kW ? C::kHalf - c0 : kW;
#pragma unroll
            for (int c = 0; c < kW; c += C::kLd)
              if (c < n) tmem_ld_cols<C::kLd>(col + c0 + c, v + c);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < kW; ++c)
              if (c < n) acc[i][c0 + c] = fmaf(sc, __uint_as_float(v[c]), acc[i][c0 + c]);
          }
        }
        tc_fence_before();
        mbar_arrive(&part_empty[pb]);
      }
      if (!ok) break;
      // every load of item w has been issued by now, so its successor is
      // published: fetch that item's block scales while w is stored
      const int wn = ring_take_warp(ring, ++n, p.err);
      if (wn >= 0) item_scales(wn, nscl);
      if constexpr (GU) {
        const int f = mt * C::RB + 32 * q + lane;
        const bool f_ok = f < p.N_out;
        const int kblk = f >> 5;
        const int gf = kblk >> 2, kbf = kblk & 3;
        const size_t hi0 = static_cast<size_t>(2) * row0;            // split layout: the tile's first hi row
        uint8_t* atom = p.hsf + (static_cast<size_t>(row0 / BN) * (p.Fp / 128) + gf) * 1024;
        // four tokens at a time: their activations and warp reductions overlap
#pragma unroll
        for (int j0 = 0; j0 < C::kHalf; j0 += 4) {
          if (c_base + j0 >= nrows) break;                             // warp-uniform
          float h[4];
          HiLo hl[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            h[u] = f_ok ? glu_act_fast(acc[0][j0 + u], acc[1][j0 + u], p.act, p.b1, p.b2) : 0.0f;
          quant_hilo_warp_n<4>(h, hl);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int jj = c_base + j0 + u;
            if (jj < nrows) {
              p.hq[(hi0 + jj) * p.Fp + f] = hl[u].q_hi;
              p.hq[(hi0 + BN + jj) * p.Fp + f] = hl[u].q_lo;
              if (lane == 0) {
                atom[sf_atom_offset(jj, kbf)] = static_cast<uint8_t>(hl[u].s_hi);
                atom[512 + sf_atom_offset(jj, kbf)] = static_cast<uint8_t>(hl[u].s_lo);
              }
            }
          }
        }
      } else {
        constexpr int kR = (C::kHalf + 31) / 32;
        int a_l[kR];
        float g_l[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const int jj = c_base + 32 * r + lane;
          a_l[r] = 0;
          g_l[r] = 0.f;
          if (32 * r + lane < C::kHalf && jj < nrows) {
            a_l[r] = p.perm[p0 + jj];
            g_l[r] = p.G[a_l[r]];
          }
        }
#pragma unroll
        for (int i = 0; i < C::kNAcc; ++i) {
          const int f = mt * C::IR + i * C::RB + 32 * q + lane;
          const bool f_ok = f < p.N_out;
#pragma unroll
          for (int j = 0; j < C::kHalf; ++j) {
            if (c_base + j < nrows) {
              const int a = __shfl_sync(0xFFFFFFFFu, a_l[j / 32], j % 32);
              const float gw = __shfl_sync(0xFFFFFFFFu, g_l[j / 32], j % 32);
              if (f_ok) p.y[static_cast<size_t>(a) * p.N_out + f] = acc[i][j] * gw;
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < C::kNAcc; ++i) {
        scl[i][0] = nscl[i][0];
        scl[i][1] = nscl[i][1];
      }
      w = wn;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int BN, bool GU>
cudaError_t launch_fp8(const MoeGemmParams& p, int grid, cudaStream_t s) {
  using C = Fp8Cfg<BN, GU>;
  if (!p.sched || p.KS != 1) return cudaErrorInvalidValue;   // no K split of FP8 items
  cudaError_t e = cudaFuncSetAttribute(moe_fp8_kernel<BN, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  {
    const cudaError_t e_ = launch_pdl(moe_fp8_kernel<BN, GU>, grid, kFp8Threads, C::kSmem, s, p);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_moe_fp8_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp8<16, true>(p, grid, s);
    case 32: return launch_fp8<32, true>(p, grid, s);
    case 64: return launch_fp8<64, true>(p, grid, s);
    case 96: return launch_fp8<96, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_moe_fp8_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp8<16, false>(p, grid, s);
    case 32: return launch_fp8<32, false>(p, grid, s);
    case 64: return launch_fp8<64, false>(p, grid, s);
    case 96: return launch_fp8<96, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lmoe
