// Routed experts with both operands in packed 4-bit form: tcgen05
// kind::mxf4 block-scaled MMAs (scale_vec::2X, one E8M0 scale per 32 values),
// E2M1 x E2M1.
//
// The MXFP4 weights go to shared memory as stored, two codes per byte: a
// 128-byte swizzled row holds 256 K values, half the bytes the E2M1 x E4M3
// form (kind::mxf8f6f4) has to copy, where each code takes a byte.  That form
// needs the activations in 4 bits too: each activation is the sum of `terms`
// MXFP4 terms, every term quantising what the previous ones left, with its
// own E8M0 scale per 32 values (3 terms carry ~1e-3 relative error, the
// precision of two E4M3 terms).  The terms of a tile are separate operands
// accumulated into the same TMEM columns.
//
// The weight scales are the create-time atoms of the other expert kernels
// (per 128 K, the four 32-value scales of each row in one 32-bit TMEM word):
// an MMA of K = 64 reads one half of that word (scale-factor id 0 or 2).
//
// One work item = (expert tile of <= BN assignments, gate + up rows of RB
// features, or 2 x RB down rows), over 256-K stages.  Warp roles: 0 = TMA
// producer, 1 = MMA issuer, 2..5 = epilogue.
#include "common.cuh"
#include "lmoe_internal.h"
#include "moe_common.cuh"

namespace lmoe {
namespace {

template <int BN, bool GU>
struct Fp4Cfg {
  static constexpr int RB = moe_rows_per_item(BN);   // 256 (decode tiles) or 128 (prefill tiles)
  static constexpr int kTiles = RB / 128;
  static constexpr int kBoxes = 2;
  static constexpr int IR = GU ? RB : 2 * RB;
  static constexpr int kNAcc = kBoxes * kTiles;
  static constexpr int N = BN;                        // one accumulator column per assignment
  static constexpr int kA = RB * 128;                 // one weight box: RB rows x 256 packed codes
  static constexpr int kB1 = BN * 128;                // one activation term of the tile
  static constexpr int kSfA = kBoxes * 2 * kTiles * 512;   // weight scale atoms of a 256-K stage
  static constexpr int kAcc = kNAcc * N;
  static_assert(kA % 1024 == 0 && kB1 % 1024 == 0, "swizzle atoms stay aligned");
};

// Per-stage layout for a runtime term count (all multiples of 512 bytes; the
// swizzled tiles of every stage first, 1024-aligned, then the scale atoms).
template <int BN, bool GU>
__host__ __device__ constexpr int fp4_tile_bytes(int terms) {
  return Fp4Cfg<BN, GU>::kBoxes * Fp4Cfg<BN, GU>::kA + terms * Fp4Cfg<BN, GU>::kB1;
}
template <int BN, bool GU>
__host__ __device__ constexpr int fp4_sf_bytes(int terms) {
  return Fp4Cfg<BN, GU>::kSfA + 2 * terms * 512;
}
template <int BN, bool GU>
__host__ __device__ constexpr int fp4_sf_cols(int terms) {
  return Fp4Cfg<BN, GU>::kNAcc * 8 + terms * 8;   // 2 atoms x 4 TMEM columns per accumulator / term
}
constexpr int kFp4MaxStages = 4;
constexpr int kFp4MaxTerms = 4;   // activation terms; the workspace holds up to four per row

// E8M0 scale of an E2M1 block: the smallest power of two 2^p with amax <= 6 x
// 2^p (6 = the largest E2M1 magnitude), as the biased byte p + 127.
__device__ __forceinline__ uint32_t e2m1_block_scale(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int ef = static_cast<int>((bits >> 23) & 0xFF);
  int s = ef - 2 + ((bits & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  s = s < 1 ? 1 : (s > 253 ? 253 : s);
  return static_cast<uint32_t>(s);
}
// Value of an E2M1 code (1 sign, 2 exponent, 1 mantissa bit): 0, 0.5, 1,
// 1.5, 2, 3, 4, 6 and their negatives.
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t m = c & 7u;
  const float mag = m < 2u ? 0.5f * static_cast<float>(m)
                           : __uint_as_float(((m >> 1) + 126u) << 23) * (1.0f + 0.5f * static_cast<float>(m & 1u));
  return (c & 8u) ? -mag : mag;
}
// Two fp32 values -> one byte of two E2M1 codes, `lo` in bits 0-3 and `hi` in
// bits 4-7, rounded to nearest (ties to even) and saturating at +-6: the
// hardware conversion, issued directly (the toolkit's fp4 header emulates it
// in software unless the target is family-specific).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{ .reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tmov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t f32_to_e2m1(float x) { return f32x2_to_e2m1x2(x, 0.0f) & 0xFu; }

// Instruction descriptor of the packed-FP4 forms with E2M1 A and B, UE8M0
// scales (scale_vec::2X), K-major operands, scale-factor ids of A and B.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, uint32_t sf_id) {
  return (sf_id << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) |
         (static_cast<uint32_t>(M >> 4) << 24) | (sf_id << 29);
}
__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Row of term t of padded assignment row r in the packed activation layout:
// per BN-row tile, its terms' BN rows one after the other.
__host__ __device__ __forceinline__ size_t fp4_row(int r, int t, int BN, int terms) {
  return static_cast<size_t>(r / BN) * terms * BN + static_cast<size_t>(t) * BN + r % BN;
}

// Encodes h (one value per lane: the lane's feature f of a 32-feature block
// held by the warp) of N tokens as `terms` MXFP4 terms: packed codes (even
// feature in the low nibble) to rows fp4_row(r_u, t) of hq, scales to the
// atoms of hsf.  The N warp reductions of a term run interleaved.
template <int N>
__device__ __forceinline__ void encode_h_fp4(float (&h)[N], const int (&rr)[N], int nvalid, int terms, int BN, int f,
                                             int Fp, uint8_t* hq, uint8_t* hsf) {
  const int lane = threadIdx.x & 31;
  const int g = f >> 7, kb = (f >> 5) & 3;
  for (int t = 0; t < terms; ++t) {
    float m[N];
#pragma unroll
    for (int u = 0; u < N; ++u) m[u] = fabsf(h[u]);
#pragma unroll
    for (int u = 0; u < N; ++u) m[u] = warp_amax(m[u]);
#pragma unroll
    for (int u = 0; u < N; ++u) {
      const uint32_t s = e2m1_block_scale(m[u]);
      const uint32_t c = f32_to_e2m1(h[u] * e8m0_to_f32(254u - s));
      h[u] -= e2m1_value(c) * e8m0_to_f32(s);
      const uint32_t partner = __shfl_xor_sync(0xFFFFFFFFu, c, 1);
      if (u < nvalid) {
        const int r = rr[u];
        if ((lane & 1) == 0)
          hq[fp4_row(r, t, BN, terms) * (Fp / 2) + (f >> 1)] = static_cast<uint8_t>(c | (partner << 4));
        if (lane == 0)
          hsf[((static_cast<size_t>(r / BN) * (Fp / 128) + g) * terms + t) * 512 + sf_atom_offset(r % BN, kb)] =
              static_cast<uint8_t>(s);
      }
    }
  }
}

// Gate/up epilogue of one K split (16-assignment tile, small batches): the
// partial sums of the warp's rows go to gpart; the split that arrives last at
// these rows adds the KS partials in split order and encodes h.
template <int BN>
__device__ __forceinline__ void fp4_ksplit_gate_up(const MoeGemmParams& p, uint32_t acc_base, int mt, int row0,
                                                   int nrows, int wb, int ks, int q, int lane, const int* a_r,
                                                   uint64_t* acc_empty) {
  using C = Fp4Cfg<BN, true>;
  const size_t plane = static_cast<size_t>(p.P) * p.N_out;
  float* const gp = p.gpart + static_cast<size_t>(ks) * 2 * plane;
#pragma unroll 1
  for (int t = 0; t < C::kTiles; ++t) {
    if (mt * C::RB + t * 128 >= p.Fp) break;
    const int f = mt * C::IR + t * 128 + 32 * q + lane;
    const bool f_ok = f < p.N_out;
    uint32_t rg[16], ru[16];
    tmem_ld16(acc_base + t * C::N, rg);
    tmem_ld16(acc_base + (C::kTiles + t) * C::N, ru);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j >= nrows) break;
      const int a = __shfl_sync(0xFFFFFFFFu, a_r[0], j);
      if (f_ok) {
        gp[static_cast<size_t>(a) * p.N_out + f] = __uint_as_float(rg[j]);
        gp[plane + static_cast<size_t>(a) * p.N_out + f] = __uint_as_float(ru[j]);
      }
    }
  }
  tc_fence_before();
  mbar_arrive(acc_empty);
  __threadfence();
  __syncwarp();
  int* const cnt = p.gcnt + static_cast<size_t>(wb) * 4 + q;
  int old = 0;
  if (lane == 0) old = atomicAdd(cnt, 1);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  if (old != p.KS - 1) return;
  __threadfence();
  if (lane == 0) *cnt = 0;   // counters end every forward at zero
#pragma unroll 1
  for (int t = 0; t < C::kTiles; ++t) {
    if (mt * C::RB + t * 128 >= p.Fp) break;
    const int f = mt * C::IR + t * 128 + 32 * q + lane;
    const bool f_ok = f < p.N_out;
#pragma unroll 1
    for (int j0 = 0; j0 < nrows; j0 += 4) {
      float h[4];
      int rr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        h[u] = 0.f;
        rr[u] = row0 + (j < nrows ? j : 0);
        if (j < nrows && f_ok) {
          const int a = __shfl_sync(0xFFFFFFFFu, a_r[0], j);
          float gv = 0.f, uv = 0.f;
          for (int s = 0; s < p.KS; ++s) {
            const float* src = p.gpart + static_cast<size_t>(s) * 2 * plane + static_cast<size_t>(a) * p.N_out + f;
            gv += __ldcg(src);
            uv += __ldcg(src + plane);
          }
          h[u] = glu_act_fast(gv, uv, p.act, p.b1, p.b2);
        }
      }
      const int nv = nrows - j0 < 4 ? nrows - j0 : 4;
      encode_h_fp4<4>(h, rr, nv, p.terms, BN, f, p.Fp, p.hq, p.hsf);
    }
  }
}

template <int BN, bool GU, bool KSP>
__global__ void __launch_bounds__(kThreads, 1) moe_fp4_kernel(const __grid_constant__ MoeGemmParams p) {
  using C = Fp4Cfg<BN, GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  const int terms = p.terms, nst = p.stages, nbuf = p.accbufs;
  const int tile_bytes = fp4_tile_bytes<BN, GU>(terms);
  const int sf_bytes = fp4_sf_bytes<BN, GU>(terms);
  const int sf_cols = fp4_sf_cols<BN, GU>(terms);
  uint8_t* sf_region = sm + nst * tile_bytes;
  __shared__ uint64_t full[kFp4MaxStages], empty[kFp4MaxStages], acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  __shared__ ItemRing ring;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < nbuf; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps * 32);
    }
    ring_init(ring, kEpiWarps);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch();
  griddep_wait();
  const uint32_t tbase = tmem_base;

  const int ntiles = *p.ntiles;
  const int KS = KSP ? p.KS : 1;
  const int total = ntiles * p.MT * KS;
  const int KG = p.KG;            // 256-K groups
  const int KG128 = 2 * KG;       // the scale atoms run per 128 K
  auto krange = [&](int w, int& g0, int& g1) {
    const int ks = w % KS;
    g0 = ks * KG / KS;
    g1 = (ks + 1) * KG / KS;
  };
  auto st_a = [&](int s, int j) { return sm + s * tile_bytes + j * C::kA; };
  auto st_b = [&](int s, int t) { return sm + s * tile_bytes + C::kBoxes * C::kA + t * C::kB1; };
  // scale atoms of a stage: weights [box][half j][tile], then activations [half j][term]
  auto st_sfa = [&](int s, int box, int j) { return sf_region + s * sf_bytes + (box * 2 + j) * C::kTiles * 512; };
  auto st_sfb = [&](int s, int j) { return sf_region + s * sf_bytes + C::kSfA + j * terms * 512; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.a_gate);
      if (GU) tma_prefetch_desc(&p.a_up);
      tma_prefetch_desc(&p.b);
      uint32_t it = 0;
      bool ok = true;
      const CUtensorMap* map1 = GU ? &p.a_up : &p.a_gate;
      const uint32_t tx = C::kBoxes * C::kA + terms * C::kB1 + C::kSfA + 2 * terms * 512;
      int w = static_cast<int>(blockIdx.x) < total ? static_cast<int>(blockIdx.x) : -1;
      for (uint32_t n = 0; ok; ++n) {
        if (!ring_put(ring, n, w, p.err) || w < 0) break;
        int nxt = total;
        int mt;
        const int4 tile = decode_item<BN>(p, w / KS, mt);
        const int e = tile.x, row0 = tile.y;
        const int arow = e * p.N_out + mt * C::IR;
        const int arow1 = GU ? arow : arow + C::RB;
        int g0, g1;
        krange(w, g0, g1);
        const int claim_g = g1 - g0 > 2 ? g1 - 2 : g0;
        for (int g = g0; g < g1; ++g, ++it) {
          if (g == claim_g) nxt = claim_item(p.sched);
          const int s = it % nst;
          if (it >= static_cast<uint32_t>(nst) &&
              !mbar_wait(&empty[s], ((it / nst) - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], tx);
          tma_load_2d(st_a(s, 0), &p.a_gate, &full[s], g * 128, arow);
          tma_load_2d(st_a(s, 1), map1, &full[s], g * 128, arow1);
          for (int t = 0; t < terms; ++t)
            tma_load_2d(st_b(s, t), &p.b, &full[s], g * 128, row0 * terms + t * BN);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            // atoms [E][KG128][MTa][512]: the item's tiles of one 128-K half are adjacent
            const size_t a_off = ((static_cast<size_t>(e) * KG128 + 2 * g + j) * p.MTa + mt * (C::IR / 128)) * 512;
            bulk_g2s(st_sfa(s, 0, j), p.sfa_gate + a_off, C::kTiles * 512, &full[s]);
            bulk_g2s(st_sfa(s, 1, j), GU ? p.sfa_up + a_off : p.sfa_gate + a_off + C::kTiles * 512, C::kTiles * 512,
                     &full[s]);
            bulk_g2s(st_sfb(s, j), p.sfb + ((static_cast<size_t>(row0 / BN) * KG128 + 2 * g + j) * terms) * 512,
                     terms * 512, &full[s]);
          }
        }
        w = nxt < total ? nxt : -1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, titer = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n, ++titer) {
        const int w = ring_take(ring, n, p.err);
        if (w < 0) break;
        int g0, g1;
        krange(w, g0, g1);
        const int b = titer % nbuf;
        const uint32_t use = titer / nbuf;
        if (use > 0 && !mbar_wait(&acc_empty[b], (use - 1) & 1, p.err, kErrTimeout)) break;
        tc_fence_after();
        const uint32_t d0 = tbase + b * C::kAcc;
        for (int g = g0; g < g1; ++g, ++it) {
          const int s = it % nst;
          if (!mbar_wait(&full[s], (it / nst) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sf = tbase + nbuf * C::kAcc + s * sf_cols;
          const uint32_t sfb = sf + C::kNAcc * 8;
          // scale atoms -> TMEM: accumulator i, half j at columns sf + (2i + j) * 4; term t at sfb + (2t + j) * 4
#pragma unroll
          for (int i = 0; i < C::kNAcc; ++i)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tmem_cp_32x128b_x4(sf + (2 * i + j) * 4,
                                 sdesc_noswz(smem_u32(st_sfa(s, i / C::kTiles, j)) + 512 * (i % C::kTiles), 16, 128));
          for (int t = 0; t < terms; ++t)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tmem_cp_32x128b_x4(sfb + (2 * t + j) * 4, sdesc_noswz(smem_u32(st_sfb(s, j)) + 512 * t, 16, 128));
#pragma unroll
          for (int mk = 0; mk < 4; ++mk) {   // four MMAs of K = 64 per 256-K stage
            const int j = mk >> 1;
            const uint32_t idesc = idesc_mxf4(128, C::N, (mk & 1) * 2);
#pragma unroll
            for (int i = 0; i < C::kNAcc; ++i) {
              const uint32_t a_addr = smem_u32(st_a(s, i / C::kTiles)) + (i % C::kTiles) * 16384 + 32 * mk;
              for (int t = 0; t < terms; ++t) {
                const uint32_t acc = ((g - g0) | mk | t) != 0;
                mma_fp4(d0 + i * C::N, sdesc_sw128(a_addr), sdesc_sw128(smem_u32(st_b(s, t)) + 32 * mk), idesc,
                        sf + (2 * i + j) * 4, sfb + (2 * t + j) * 4, acc);
              }
            }
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[b]);
      }
    }
  } else {
    // Epilogue warps: lane quarter q of TMEM = rows 32q .. 32q+31 of each 128-row tile.
    const int q = warp & 3;
    uint32_t titer = 0;
    for (uint32_t n = 0;; ++n, ++titer) {
      const int w = ring_take_warp(ring, n, p.err);
      if (w < 0) break;
      const int b = titer % nbuf;
      const uint32_t use = titer / nbuf;
      if (!mbar_wait(&acc_full[b], use & 1, p.err, kErrTimeout)) break;
      tc_fence_after();
      const int wb = w / KS, ks = w - wb * KS;
      int mt;
      const int4 tile = decode_item<BN>(p, wb, mt);
      const int row0 = tile.y, nrows = tile.z, p0 = tile.w;
      constexpr int kR = (BN + 31) / 32;
      int a_r[kR];
      float g_r[kR];
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        a_r[r] = 0;
        g_r[r] = 0.f;
        if ((!GU || KSP) && lane + 32 * r < nrows) {
          a_r[r] = p.perm[p0 + lane + 32 * r];
          g_r[r] = p.G[a_r[r]];
        }
      }
      const uint32_t acc_base = tbase + (static_cast<uint32_t>(32 * q) << 16) + b * C::kAcc;
      float* const yk = KSP ? p.y + static_cast<size_t>(ks) * p.y_plane : p.y;
      if constexpr (GU && KSP) {
        fp4_ksplit_gate_up<BN>(p, acc_base, mt, row0, nrows, wb, ks, q, lane, a_r, &acc_empty[b]);
        continue;
      }
#pragma unroll 1
      for (int t = 0; t < (GU ? C::kTiles : C::kNAcc); ++t) {
        if (GU && mt * C::RB + t * 128 >= p.Fp) break;
        const int f = mt * C::IR + t * 128 + 32 * q + lane;
        const bool f_ok = f < p.N_out;
#pragma unroll 1
        for (int j0 = 0; j0 < BN; j0 += 16) {
          if (j0 >= nrows) break;
          uint32_t rg[16];
          const uint32_t a0 = acc_base + t * C::N + j0;
          tmem_ld16(a0, rg);
          if constexpr (GU) {
            uint32_t ru[16];
            tmem_ld16(a0 + C::kTiles * C::N, ru);
            tmem_ld_wait();
#pragma unroll
            for (int jq = 0; jq < 16; jq += 4) {
              if (j0 + jq >= nrows) break;                 // warp-uniform
              float h[4];
              int rr[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                h[u] = f_ok ? glu_act_fast(__uint_as_float(rg[jq + u]), __uint_as_float(ru[jq + u]), p.act, p.b1,
                                           p.b2)
                            : 0.0f;
                rr[u] = row0 + j0 + jq + u;
              }
              const int nv = nrows - (j0 + jq) < 4 ? nrows - (j0 + jq) : 4;
              encode_h_fp4<4>(h, rr, nv, terms, BN, f, p.Fp, p.hq, p.hsf);
            }
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = j0 + jj;
              if (j >= nrows) break;
              const int a = __shfl_sync(0xFFFFFFFFu, a_r[j >> 5], j & 31);
              const float gw = __shfl_sync(0xFFFFFFFFu, g_r[j >> 5], j & 31);
              if (f_ok) yk[static_cast<size_t>(a) * p.N_out + f] = __uint_as_float(rg[jj]) * gw;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int BN, bool GU>
bool fp4_plan(int terms, int& stages, int& bufs, int& smem) {
  using C = Fp4Cfg<BN, GU>;
  const int stage = fp4_tile_bytes<BN, GU>(terms) + fp4_sf_bytes<BN, GU>(terms);
  const int cols = fp4_sf_cols<BN, GU>(terms);
  const int by_smem = (227 * 1024 - 2048) / stage;
  for (bufs = 2; bufs >= 1; --bufs) {
    const int by_tmem = (512 - bufs * C::kAcc) / cols;
    stages = by_smem < by_tmem ? by_smem : by_tmem;
    if (stages > kFp4MaxStages) stages = kFp4MaxStages;
    if (stages >= 2) break;
  }
  smem = stages * stage + 1024;
  return stages >= 2;
}

template <int BN, bool GU, bool KSP>
cudaError_t launch_fp4_k(MoeGemmParams p, int grid, cudaStream_t s) {
  int smem = 0;
  if (!fp4_plan<BN, GU>(p.terms, p.stages, p.accbufs, smem)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(moe_fp4_kernel<BN, GU, KSP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(moe_fp4_kernel<BN, GU, KSP>, grid, kThreads, smem, s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN, bool GU>
cudaError_t launch_fp4(const MoeGemmParams& p, int grid, cudaStream_t s) {
  if (!p.sched || p.KS < 1 || p.KS > p.KG || p.terms < 1 || p.terms > kFp4MaxTerms) return cudaErrorInvalidValue;
  if (p.KS == 1) return launch_fp4_k<BN, GU, false>(p, grid, s);
  if constexpr (BN == 16) {
    if (GU && (!p.gpart || !p.gcnt)) return cudaErrorInvalidValue;
    return launch_fp4_k<16, GU, true>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// One warp per (token, 128-column group) of the expert input: each lane
// holds four consecutive values (a 32-value block is eight lanes) and
// encodes them as `terms` MXFP4 terms, two packed codes per byte, into every
// one of the token's k assignment rows; the E8M0 scales go into the atoms of
// each row's tile, per 128 K and term.
__global__ void quant_gather_fp4_kernel(const float* __restrict__ xc, int T, int k, int din, int Kp,
                                        const int32_t* __restrict__ inv_pad, int BN, int terms,
                                        uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf,
                                        int* __restrict__ sched, int* __restrict__ cnt, int ncnt) {
  griddep_launch();
  griddep_wait();
  if (blockIdx.x == 0) {
    if (sched && threadIdx.x < 2) sched[threadIdx.x] = 0;
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  }
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int KG128 = Kp / 128;
  if (gw >= T * KG128) return;
  const int t = gw / KG128, g = gw % KG128;
  const int c0 = g * 128 + 4 * lane;
  const int kb = lane >> 3;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (c0 < din) {
    const float4 q4 = *reinterpret_cast<const float4*>(xc + static_cast<size_t>(t) * din + c0);
    v[0] = q4.x;
    v[1] = q4.y;
    v[2] = q4.z;
    v[3] = q4.w;
  }
  const int32_t* rows = inv_pad + static_cast<size_t>(t) * k;
  for (int tt = 0; tt < terms; ++tt) {
    float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    const uint32_t s = e2m1_block_scale(m);
    const float inv = e8m0_to_f32(254u - s), sc = e8m0_to_f32(s);
    const uint32_t word = f32x2_to_e2m1x2(v[0] * inv, v[1] * inv) | (f32x2_to_e2m1x2(v[2] * inv, v[3] * inv) << 8);
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] -= e2m1_value((word >> (4 * u)) & 0xFu) * sc;
    for (int j = 0; j < k; ++j) {
      const size_t row = fp4_row(rows[j], tt, BN, terms);
      *reinterpret_cast<uint16_t*>(xq + row * (Kp / 2) + c0 / 2) = static_cast<uint16_t>(word);
    }
    for (int j = lane & 7; j < k; j += 8) {
      const int r = rows[j];
      xsf[((static_cast<size_t>(r / BN) * KG128 + g) * terms + tt) * 512 + sf_atom_offset(r % BN, kb)] =
          static_cast<uint8_t>(s);
    }
  }
}

// Debug read-out of the packed layout: the sum of the terms' values.
__global__ void decode_fp4_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                  const int32_t* __restrict__ inv_pad, int P, int K, int Kp, int BN, int terms,
                                  float* __restrict__ out) {
  const size_t n = static_cast<size_t>(P) * K;
  const int KG128 = Kp / 128;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int a = static_cast<int>(i / K), c = static_cast<int>(i % K);
    const int r = inv_pad[a], g = c >> 7, kb = (c & 127) >> 5;
    float v = 0.f;
    for (int t = 0; t < terms; ++t) {
      const uint8_t byte = q[fp4_row(r, t, BN, terms) * (Kp / 2) + c / 2];
      const uint32_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
      const uint8_t s = sf[((static_cast<size_t>(r / BN) * KG128 + g) * terms + t) * 512 + sf_atom_offset(r % BN, kb)];
      v += e2m1_value(code) * e8m0_to_f32(s);
    }
    out[i] = v;
  }
}

int fp4_ew_grid(size_t n) {
  size_t g = (n + 255) / 256;
  return static_cast<int>(g < 152 * 16 ? (g ? g : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_moe_fp4_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp4<16, true>(p, grid, s);
    case 32: return launch_fp4<32, true>(p, grid, s);
    case 64: return launch_fp4<64, true>(p, grid, s);
    case 96: return launch_fp4<96, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_moe_fp4_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_fp4<16, false>(p, grid, s);
    case 32: return launch_fp4<32, false>(p, grid, s);
    case 64: return launch_fp4<64, false>(p, grid, s);
    case 96: return launch_fp4<96, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quant_gather_fp4(const float* xc, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                    int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                    cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (terms < 1 || terms > kFp4MaxTerms || Kp % 256) return cudaErrorInvalidValue;
  const int warps_per_block = 8;
  const long long warps = static_cast<long long>(T) * (Kp / 128);
  const unsigned blocks = static_cast<unsigned>((warps + warps_per_block - 1) / warps_per_block);
  cudaError_t e = launch_pdl(quant_gather_fp4_kernel, blocks, 32 * warps_per_block, 0, s, xc, T, k, din, Kp, inv_pad,
                             BN, terms, xq, xsf, sched, cnt, ncnt);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode_fp4(const uint8_t* q, const uint8_t* sf, const int32_t* inv_pad, int P, int K, int Kp,
                              int BN, int terms, float* out, cudaStream_t s) {
  if (P <= 0) return cudaSuccess;
  decode_fp4_kernel<<<fp4_ew_grid(static_cast<size_t>(P) * K), 256, 0, s>>>(q, sf, inv_pad, P, K, Kp, BN, terms, out);
  return cudaGetLastError();
}

}  // namespace lmoe
