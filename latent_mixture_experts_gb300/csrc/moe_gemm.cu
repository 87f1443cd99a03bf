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
// One work item = (expert tile of <= BN assignments, 256 weight rows): the
// gate and up rows of 128 features, or 256 consecutive down-projection rows.
// A persistent grid walks the device-side tile list written by the dispatch
// step.  Warp roles: 0 = TMA producer, 1 = MMA issuer, 2..5 = epilogue.
//
//   gate/up pass: two accumulators (gate rows, up rows of the same 128
//     features), epilogue h = SiTU(g, u) (or SwiGLU), written back as hi/lo
//     E4M3 for the down pass (Kimi K3 card, routed-expert steps).
//   down pass: two accumulators (rows 256m.. and 256m+128..), epilogue
//     multiplies by the routing weight
//     G_i and stores the expert output of that assignment (moe_infer's
//     weighted sum is finished by the combine kernel in slot order).
#include <cooperative_groups.h>

#include "common.cuh"
#include "lmoe_internal.h"
#include "moe_common.cuh"

namespace lmoe {

namespace {

template <int BN, bool GU>
struct MoeCfg {
  static constexpr bool SPLIT = moe_split(BN);       // hi and lo as two MMAs into one accumulator
  static constexpr int N = SPLIT ? BN : 2 * BN;      // MMA N (columns per assignment: 1 split, 2 interleaved)
  static constexpr int NA = SPLIT ? 2 : (N + 127) / 128;   // 512-byte scale atoms of B per stage
  static constexpr int RB = moe_rows_per_item(BN);   // weight rows per work item and TMA box
  static constexpr int kTiles = RB / 128;            // 128-row MMA tiles per box
  static constexpr int kBoxes = 2;                   // A boxes per stage: gate + up, or two down boxes
  static constexpr int IR = GU ? RB : 2 * RB;        // weight rows of one work item
  static constexpr int kNAcc = kBoxes * kTiles;      // accumulators per work item
  static constexpr int kA = RB * 128;                // one box: RB rows x 128 FP4 codes in 16-byte slots
  static constexpr int kB = 2 * BN * 128;            // 2*BN rows (hi and lo) x 128 E4M3 codes
  static constexpr int kTile = kBoxes * kA + kB;     // swizzled tiles of one stage (multiple of 1024)
  static constexpr int kSfa = kTiles * 512;          // scale atoms of one box (adjacent in memory)
  static constexpr int kSfb = NA * 512;
  static constexpr int kSf = kBoxes * kSfa + kSfb;   // scale atoms of one stage
  static constexpr int kTx = kBoxes * (kA / 2) + kB + kSf;   // bytes the stage's copies deliver
  static constexpr int kStagesFit = (227 * 1024 - 2048) / (kTile + kSf);
  static constexpr int kStages = RB == 256 ? 3 : (kStagesFit < 4 ? kStagesFit : 4);
  static constexpr int kSmem = kStages * (kTile + kSf) + 1024;
  static constexpr int kAcc = kNAcc * N;             // accumulator columns of one buffer
  static constexpr int kSfCols = kNAcc * 4 + NA * 4; // scale columns per stage
  static constexpr int kAccBufs = (2 * kAcc + kStages * kSfCols <= 512) ? 2 : 1;
  static constexpr int kTmemUsed = kAccBufs * kAcc + kStages * kSfCols;
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kAtoms = kNAcc + NA;           // scale atoms of a stage, in TMEM column order
  static_assert(kSf == kAtoms * 512 && (kAtoms == 4 || kAtoms == 5), "one stage's atoms: 4 TMEM columns each");
  static_assert(kTile % 1024 == 0, "tiles keep 1024-byte alignment");
  static_assert(kTmemUsed <= 512, "tensor memory budget");
  static_assert(kSmem <= 227 * 1024, "shared memory budget");
};

// Gate/up epilogue of one K split of an item (interleaved layout, small
// batches): the warp's rows of the split's partial gate and up sums go to
// gpart, the accumulator buffer is released, and the split that arrives last
// at these rows (counter per item and lane quarter) adds the KS partials in
// split order and finishes them like the unsplit epilogue: h = SiTU(g, u)
// (or SwiGLU) as hi/lo E4M3 codes and block scales for the down pass.
template <int BN>
__device__ __forceinline__ void ksplit_gate_up(const MoeGemmParams& p, uint32_t acc_base, int mt, int row0,
                                               int nrows, int wb, int ks, int q, int lane, const int* a_r,
                                               uint64_t* acc_empty) {
  using C = MoeCfg<BN, true>;
  const size_t plane = static_cast<size_t>(p.P) * p.N_out;
  float* const gp = p.gpart + static_cast<size_t>(ks) * 2 * plane;
#pragma unroll 1
  for (int t = 0; t < C::kTiles; ++t) {
    if (mt * C::RB + t * 128 >= p.Fp) break;
    const int f = mt * C::IR + t * 128 + 32 * q + lane;
    const bool f_ok = f < p.N_out;
#pragma unroll 1
    for (int j0 = 0; j0 < BN; j0 += 16) {
      if (j0 >= nrows) break;
      uint32_t rg[32], ru[32];
      const uint32_t a0 = acc_base + t * C::N + 2 * j0;
      const uint32_t a1 = a0 + C::kTiles * C::N;
      tmem_ld16(a0, *reinterpret_cast<uint32_t(*)[16]>(&rg[0]));
      tmem_ld16(a0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&rg[16]));
      tmem_ld16(a1, *reinterpret_cast<uint32_t(*)[16]>(&ru[0]));
      tmem_ld16(a1 + 16, *reinterpret_cast<uint32_t(*)[16]>(&ru[16]));
      tmem_ld_wait();
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int j = j0 + jj;
        if (j >= nrows) break;   // warp-uniform
        const int a = __shfl_sync(0xFFFFFFFFu, a_r[j >> 5], j & 31);
        if (f_ok) {
          gp[static_cast<size_t>(a) * p.N_out + f] = __uint_as_float(rg[2 * jj]) + __uint_as_float(rg[2 * jj + 1]);
          gp[plane + static_cast<size_t>(a) * p.N_out + f] =
              __uint_as_float(ru[2 * jj]) + __uint_as_float(ru[2 * jj + 1]);
        }
      }
    }
  }
  tc_fence_before();
  mbar_arrive(acc_empty);
  // every lane's partial stores are fenced and the warp has converged before
  // lane 0 announces them with the arrival counter
  __threadfence();
  __syncwarp();
  int* const cnt = p.gcnt + static_cast<size_t>(wb) * 4 + q;
  int old = 0;
  if (lane == 0) old = atomicAdd(cnt, 1);
  old = __shfl_sync(0xFFFFFFFFu, old, 0);
  if (old != p.KS - 1) return;
  __threadfence();
  if (lane == 0) *cnt = 0;   // counters end every forward at zero
  uint8_t* const atom = p.hsf + ((static_cast<size_t>(row0 / BN) * (p.Fp / 128)) * C::NA) * 512;
#pragma unroll 1
  for (int t = 0; t < C::kTiles; ++t) {
    if (mt * C::RB + t * 128 >= p.Fp) break;
    const int f = mt * C::IR + t * 128 + 32 * q + lane;
    const bool f_ok = f < p.N_out;
    const int kblk = f >> 5;   // 32-feature block = this warp
    const int g = kblk >> 2, kb = kblk & 3;
#pragma unroll 1
    for (int j0 = 0; j0 < nrows; j0 += 4) {
      float h[4];
      HiLo e[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        h[u] = 0.f;
        if (j < nrows) {   // warp-uniform
          const int a = __shfl_sync(0xFFFFFFFFu, a_r[j >> 5], j & 31);
          if (f_ok) {
            float gv = 0.f, uv = 0.f;
            for (int s = 0; s < p.KS; ++s) {
              const float* src = p.gpart + static_cast<size_t>(s) * 2 * plane + static_cast<size_t>(a) * p.N_out + f;
              gv += __ldcg(src);
              uv += __ldcg(src + plane);
            }
            h[u] = glu_act_fast(gv, uv, p.act, p.b1, p.b2);
          }
        }
      }
      quant_terms_warp_n<4>(h, e, p.terms);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u;
        if (j >= nrows) break;
        const size_t r = static_cast<size_t>(row0) + j;
        p.hq[(2 * r) * p.Fp + f] = e[u].q_hi;
        p.hq[(2 * r + 1) * p.Fp + f] = e[u].q_lo;
        if (lane == 0) {
          const int n = 2 * j;   // MMA column of the hi term in the down pass
          uint8_t* at = atom + static_cast<size_t>(g) * C::NA * 512;
          at[(n >> 7) * 512 + sf_atom_offset(n & 127, kb)] = static_cast<uint8_t>(e[u].s_hi);
          at[((n + 1) >> 7) * 512 + sf_atom_offset((n + 1) & 127, kb)] = static_cast<uint8_t>(e[u].s_lo);
        }
      }
    }
  }
}

// Scale warps: one per TMEM lane quarter.  Each stage's E8M0 scale atoms go
// from shared memory to the stage's tensor-memory columns by these warps'
// tcgen05.st (every quarter holds the same 32 rows of an atom, as the MMA
// reads them), so the MMA thread's tensor pipe runs MMAs only; a per-stage
// tcgen05.cp ahead of the MMAs held the pipe ~25 ns per atom.
constexpr int kScaleWarps = 4;
constexpr int kMoeThreads = 64 + 32 * (kEpiWarps + kScaleWarps);   // TMA, MMA, epilogue x4, scales x4

// L2 prefetch of the down-pass weights of the experts in the tile list: their
// codes, then their scale atoms, expert by expert (the order in which the
// down pass claims its items), cut into 32 KB chunks and cut off after
// p.pf_budget bytes; this CTA takes chunks blockIdx.x, blockIdx.x + gridDim.x, ...
__device__ __forceinline__ void prefetch_down_weights(const MoeGemmParams& p, int ntiles) {
  constexpr size_t kChunk = 32768;
  const size_t grid = gridDim.x;
  size_t c0 = 0, used = 0;   // chunks and bytes of the ranges before the current one
  for (int i = 0; i < ntiles && used < p.pf_budget; ++i) {
    const int e = p.tiles[i].x;
    if (i > 0 && p.tiles[i - 1].x == e) continue;   // an expert's tiles are adjacent
    for (int r = 0; r < 2 && used < p.pf_budget; ++r) {
      const uint8_t* base = r == 0 ? p.pf_codes + static_cast<size_t>(e) * p.pf_code_bytes
                                   : p.pf_atoms + static_cast<size_t>(e) * p.pf_atom_bytes;
      size_t len = r == 0 ? p.pf_code_bytes : p.pf_atom_bytes;
      if (len > p.pf_budget - used) len = p.pf_budget - used;
      const size_t n = (len + kChunk - 1) / kChunk;
      for (size_t c = (blockIdx.x + grid - c0 % grid) % grid; c < n; c += grid) {
        const size_t off = c * kChunk;
        prefetch_l2_bulk(base + off, static_cast<uint32_t>(len - off < kChunk ? len - off : kChunk));
      }
      c0 += n;
      used += len;
    }
  }
}

// KSP: the K-split form for small batches (p.KS splits per item); without it
// p.KS is taken as 1.
template <int BN, bool GU, bool KSP>
__global__ void __launch_bounds__(kMoeThreads, 1) moe_gemm_kernel(const __grid_constant__ MoeGemmParams p) {
  using C = MoeCfg<BN, GU>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sf_region = sm + C::kStages * C::kTile;
  __shared__ uint64_t full[C::kStages], empty[C::kStages], acc_full[C::kAccBufs], acc_empty[C::kAccBufs];
  __shared__ uint64_t sf_ready[C::kStages];   // the stage's scales are in tensor memory
  __shared__ uint32_t tmem_base;
  __shared__ ItemRing ring;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sf_ready[i], kScaleWarps * 32);
    }
    for (int i = 0; i < C::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps * 32);
    }
    ring_init(ring, kEpiWarps + kScaleWarps);
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

  const int ntiles = *p.ntiles;
  const int KS = KSP ? p.KS : 1;
  // one activation term on a split layout: hi rows only (interleaved layouts
  // keep their zero lo columns)
  const bool one = C::SPLIT && p.terms == 1;
  const int total = ntiles * p.MT * KS;
  const int KG = p.KG;
  // k-groups [g0, g1) of item w (the whole K range unless the batch is K split)
  auto krange = [&](int w, int& g0, int& g1) {
    const int ks = w % KS;
    g0 = ks * KG / KS;
    g1 = (ks + 1) * KG / KS;
  };

  // stage sub-buffers: swizzled tiles first, all scale atoms after them
  auto st_a = [&](int s, int j) { return sm + s * C::kTile + j * C::kA; };
  auto st_b = [&](int s) { return sm + s * C::kTile + C::kBoxes * C::kA; };
  auto st_sfa = [&](int s, int j) { return sf_region + s * C::kSf + j * C::kSfa; };
  auto st_sfb = [&](int s) { return sf_region + s * C::kSf + C::kBoxes * C::kSfa; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&p.a_gate);
      if (GU) tma_prefetch_desc(&p.a_up);
      tma_prefetch_desc(&p.b);
      uint32_t it = 0;
      bool ok = true;
      const CUtensorMap* map1 = GU ? &p.a_up : &p.a_gate;
      // second box: the up rows of the same features, or the next RB down rows
      const uint8_t* sfa1 = GU ? p.sfa_up : p.sfa_gate + C::kSfa;
      int w = static_cast<int>(blockIdx.x) < total ? static_cast<int>(blockIdx.x) : -1;
      for (uint32_t n = 0; ok; ++n) {
        if (!ring_put(ring, n, w, p.err) || w < 0) break;
        int nxt = total;
        int mt;
        const int4 tile = decode_item<BN>(p, w / KS, mt);
        const int e = tile.x, row0 = tile.y;
        const int arow = e * p.N_out + mt * C::IR;
        const int arow1 = GU ? arow : arow + C::RB;
        // atoms [E][KG][MTa][512]: the atoms of an item's tiles are adjacent
        const size_t sfa_row = static_cast<size_t>(e) * KG;
        const size_t sfb_idx = static_cast<size_t>(row0 / BN) * KG;
        int g0, g1;
        krange(w, g0, g1);
        // the next item is claimed four k-groups before this one's last load
        const int claim_g = g1 - g0 > 4 ? g1 - 4 : g0;
        for (int g = g0; g < g1; ++g, ++it) {
          if (g == claim_g) nxt = claim_item(p.sched);
          const int s = it % C::kStages;
          if (it >= C::kStages && !mbar_wait(&empty[s], ((it / C::kStages) - 1) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          const size_t sfa_off = ((sfa_row + g) * p.MTa + mt * (C::IR / 128)) * 512;
          mbar_arrive_expect_tx(&full[s], C::kTx - (one ? C::kB / 2 + 512 : 0));
          tma_load_2d(st_a(s, 0), &p.a_gate, &full[s], g * 128, arow);
          tma_load_2d(st_a(s, 1), map1, &full[s], g * 128, arow1);
          tma_load_2d(st_b(s), &p.b, &full[s], g * 128, 2 * row0);   // one term: the BN hi rows only
          bulk_g2s(st_sfa(s, 0), p.sfa_gate + sfa_off, C::kSfa, &full[s]);
          bulk_g2s(st_sfa(s, 1), sfa1 + sfa_off, C::kSfa, &full[s]);
          bulk_g2s(st_sfb(s), p.sfb + (sfb_idx + g) * C::kSfb, one ? 512 : C::kSfb, &full[s]);
        }
        w = nxt < total ? nxt : -1;
      }
      // the down pass's weights stream into L2 while this pass drains
      if constexpr (GU && KSP)
        if (ok && p.pf_codes) prefetch_down_weights(p, ntiles);
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
        const int b = titer % C::kAccBufs;
        const uint32_t use = titer / C::kAccBufs;
        if (use > 0 && !mbar_wait(&acc_empty[b], (use - 1) & 1, p.err, kErrTimeout)) break;
        tc_fence_after();
        const uint32_t d0 = tbase + b * C::kAcc;
        for (int g = g0; g < g1; ++g, ++it) {
          const int s = it % C::kStages;
          // the stage's operands have landed and the scale warps have put its scales in tensor memory
          if (!mbar_wait(&sf_ready[s], (it / C::kStages) & 1, p.err, kErrTimeout)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // accumulator i = box j, tile t reads scale columns sf + 4i; the activation atoms follow
          const uint32_t sf = tbase + C::kAccBufs * C::kAcc + s * C::kSfCols;
          const uint32_t sfb = sf + 4 * C::kNAcc;
          const uint32_t bb = smem_u32(st_b(s));
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint32_t idesc = idesc_mxf8f6f4(128, C::N, 5, 0, kb, kb);
            const uint32_t acc = ((g - g0) | kb) != 0;
#pragma unroll
            for (int i = 0; i < C::kNAcc; ++i) {
              const uint32_t a_addr = smem_u32(st_a(s, i / C::kTiles)) + (i % C::kTiles) * 16384 + 32 * kb;
              mma_mxf8f6f4(d0 + i * C::N, sdesc_sw128(a_addr), sdesc_sw128(bb + 32 * kb), idesc, sf + 4 * i, sfb, acc);
              if constexpr (C::SPLIT)   // lo rows follow the tile's BN hi rows
                if (!one)
                  mma_mxf8f6f4(d0 + i * C::N, sdesc_sw128(a_addr), sdesc_sw128(bb + BN * 128 + 32 * kb), idesc,
                               sf + 4 * i, sfb + 4, 1u);
            }
          }
          mma_commit(&empty[s]);
        }
        mma_commit(&acc_full[b]);
      }
    }
  } else if (warp >= 2 + kEpiWarps) {
    // Scale warps: lane r of the warp on quarter q writes row r of each of the
    // stage's atoms (16 bytes: the four k-block scales of four row groups) to
    // the four columns of that atom, in the quarter's 32 lanes.
    const uint32_t col0 = tbase + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + C::kAccBufs * C::kAcc;
    uint32_t it = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int w = ring_take_warp(ring, n, p.err);
      if (w < 0) break;
      int g0, g1;
      krange(w, g0, g1);
      for (int g = g0; g < g1; ++g, ++it) {
        const int s = it % C::kStages;
        if (!mbar_wait(&full[s], (it / C::kStages) & 1, p.err, kErrTimeout)) {
          ok = false;
          break;
        }
        const uint4* at = reinterpret_cast<const uint4*>(sf_region + s * C::kSf) + lane;
        uint32_t r[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = at[32 * k];
          r[4 * k] = v.x;
          r[4 * k + 1] = v.y;
          r[4 * k + 2] = v.z;
          r[4 * k + 3] = v.w;
        }
        const uint32_t dst = col0 + s * C::kSfCols;
        tmem_st16(dst, r);
        if constexpr (C::kAtoms == 5) {
          const uint4 v = at[32 * 4];
          tmem_st4(dst + 16, v.x, v.y, v.z, v.w);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sf_ready[s]);
      }
    }
  } else {
    // Epilogue warps: lane quarter q of TMEM = rows 32q .. 32q+31 of each 128-row tile.
    const int q = warp & 3;
    uint32_t titer = 0;
    for (uint32_t n = 0;; ++n, ++titer) {
      const int w = ring_take_warp(ring, n, p.err);
      if (w < 0) break;
      const int b = titer % C::kAccBufs;
      const uint32_t use = titer / C::kAccBufs;
      if (!mbar_wait(&acc_full[b], use & 1, p.err, kErrTimeout)) break;
      tc_fence_after();
      const int wb = w / KS, ks = w - wb * KS;
      int mt;
      const int4 tile = decode_item<BN>(p, wb, mt);
      const int row0 = tile.y, nrows = tile.z, p0 = tile.w;
      // assignment (and, down pass, routing weight) of the tile's rows j = lane + 32r
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
      // down pass: this split's output plane
      float* const yk = KSP ? p.y + static_cast<size_t>(ks) * p.y_plane : p.y;
      if constexpr (GU && KSP) {
        ksplit_gate_up<BN>(p, acc_base, mt, row0, nrows, wb, ks, q, lane, a_r, &acc_empty[b]);
        continue;
      }
#pragma unroll 1
      for (int t = 0; t < (GU ? C::kTiles : C::kNAcc); ++t) {
        // A 256-row item can run past the last 128-row tile of h (whose rows
        // the down pass reads up to Fp): nothing of such a tile is stored.
        if (GU && mt * C::RB + t * 128 >= p.Fp) break;
        const int f = mt * C::IR + t * 128 + 32 * q + lane;   // output feature of this lane
        const bool f_ok = f < p.N_out;
        if constexpr (C::SPLIT) {
          // one column per assignment: gate (or down) at acc_base + t*N + j, up kTiles*N further
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
              const int kblk = f >> 5;
              const int g = kblk >> 2, kb = kblk & 3;
              const size_t hi0 = static_cast<size_t>(2) * row0;      // the tile's first hi row
              uint8_t* atom = p.hsf + (static_cast<size_t>(row0 / BN) * (p.Fp / 128) + g) * 1024;
#pragma unroll
              for (int jq = 0; jq < 16; jq += 4) {
                if (j0 + jq >= nrows) break;                 // warp-uniform
                float h[4];
                HiLo e[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  h[u] = f_ok ? glu_act_fast(__uint_as_float(rg[jq + u]), __uint_as_float(ru[jq + u]), p.act,
                                             p.b1, p.b2)
                              : 0.0f;
                quant_terms_warp_n<4>(h, e, p.terms);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const int j = j0 + jq + u;
                  if (j >= nrows) break;
                  p.hq[(hi0 + j) * p.Fp + f] = e[u].q_hi;
                  if (!one) p.hq[(hi0 + BN + j) * p.Fp + f] = e[u].q_lo;
                  if (lane == 0) {
                    atom[sf_atom_offset(j, kb)] = static_cast<uint8_t>(e[u].s_hi);
                    if (!one) atom[512 + sf_atom_offset(j, kb)] = static_cast<uint8_t>(e[u].s_lo);
                  }
                }
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
        } else {
#pragma unroll 1
        for (int j0 = 0; j0 < BN; j0 += 16) {
          if (j0 >= nrows) break;
          uint32_t rg[32];
          const uint32_t a0 = acc_base + t * C::N + 2 * j0;
          tmem_ld16(a0, *reinterpret_cast<uint32_t(*)[16]>(&rg[0]));
          tmem_ld16(a0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&rg[16]));
          if constexpr (GU) {
            uint32_t ru[32];
            const uint32_t a1 = a0 + C::kTiles * C::N;        // up accumulator of the same tile
            tmem_ld16(a1, *reinterpret_cast<uint32_t(*)[16]>(&ru[0]));
            tmem_ld16(a1 + 16, *reinterpret_cast<uint32_t(*)[16]>(&ru[16]));
            tmem_ld_wait();
            const int kblk = f >> 5;                         // 32-feature block = this warp
            const int g = kblk >> 2, kb = kblk & 3;
            // four tokens at a time: their activations and warp reductions overlap
#pragma unroll
            for (int jq = 0; jq < 16; jq += 4) {
              if (j0 + jq >= nrows) break;                   // warp-uniform
              float h[4];
              HiLo e[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int jj = jq + u;
                const float gv = __uint_as_float(rg[2 * jj]) + __uint_as_float(rg[2 * jj + 1]);
                const float uv = __uint_as_float(ru[2 * jj]) + __uint_as_float(ru[2 * jj + 1]);
                h[u] = f_ok ? glu_act_fast(gv, uv, p.act, p.b1, p.b2) : 0.0f;
              }
              quant_terms_warp_n<4>(h, e, p.terms);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int j = j0 + jq + u;
                if (j >= nrows) break;
                const size_t r = static_cast<size_t>(row0) + j;
                p.hq[(2 * r) * p.Fp + f] = e[u].q_hi;
                p.hq[(2 * r + 1) * p.Fp + f] = e[u].q_lo;
                if (lane == 0) {
                  const int n = 2 * j;                       // MMA column of the hi term in the down pass
                  uint8_t* atom = p.hsf + ((static_cast<size_t>(row0 / BN) * (p.Fp / 128) + g) * C::NA) * 512;
                  atom[(n >> 7) * 512 + sf_atom_offset(n & 127, kb)] = static_cast<uint8_t>(e[u].s_hi);
                  atom[((n + 1) >> 7) * 512 + sf_atom_offset((n + 1) & 127, kb)] =
                      static_cast<uint8_t>(e[u].s_lo);
                }
              }
            }
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              const int j = j0 + jj;
              if (j >= nrows) continue;
              const int a = __shfl_sync(0xFFFFFFFFu, a_r[j >> 5], j & 31);
              const float gw = __shfl_sync(0xFFFFFFFFu, g_r[j >> 5], j & 31);
              const float y = (__uint_as_float(rg[2 * jj]) + __uint_as_float(rg[2 * jj + 1])) * gw;
              if (f_ok) yk[static_cast<size_t>(a) * p.N_out + f] = y;
            }
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
  if (warp == 1) tmem_dealloc(tbase, C::kTmemCols);
}

template <int BN, bool GU, bool KSP>
cudaError_t launch_moe_k(const MoeGemmParams& p, int grid, cudaStream_t s) {
  using C = MoeCfg<BN, GU>;
  cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<BN, GU, KSP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmem);
  if (e != cudaSuccess) return e;
  {
    const cudaError_t e_ = launch_pdl(moe_gemm_kernel<BN, GU, KSP>, grid, kMoeThreads, C::kSmem, s, p);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

// The K-split form exists for the 16-assignment tile, the one small batches use.
template <int BN, bool GU>
cudaError_t launch_moe(const MoeGemmParams& p, int grid, cudaStream_t s) {
  if (!p.sched || p.KS < 1 || p.KS > p.KG || (p.terms != 1 && p.terms != 2)) return cudaErrorInvalidValue;
  if (p.KS == 1) return launch_moe_k<BN, GU, false>(p, grid, s);
  if constexpr (BN == 16) {
    if (GU && (!p.gpart || !p.gcnt)) return cudaErrorInvalidValue;
    return launch_moe_k<16, GU, true>(p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------ activation encode
// One warp per (token, 128-column group) of the expert input: each lane
// encodes four consecutive values, a 32-value block is eight lanes, and the
// hi/lo E4M3 codes are computed once and stored as one 4-byte word per lane
// (a 128-byte row segment per warp) into every one of the token's k
// assignment rows; the block scales go into the staging image of each row's
// tile (launch_quant_gather gives both layouts).
__device__ __forceinline__ float max8(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
  return fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
}
// Four consecutive inputs (din is a multiple of 32, so a lane's four values
// are all inside the row or all past its end).
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  v[0] = q.x;
  v[1] = q.y;
  v[2] = q.z;
  v[3] = q.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(q.x << 16);
  v[1] = __uint_as_float(q.x & 0xFFFF0000u);
  v[2] = __uint_as_float(q.y << 16);
  v[3] = __uint_as_float(q.y & 0xFFFF0000u);
}

template <typename TIn>
__global__ void quant_gather_kernel(const TIn* __restrict__ xc, int T, int k, int din, int Kp,
                                    const int32_t* __restrict__ inv_pad, int BN, int split, int terms,
                                    uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf, int* __restrict__ sched,
                                    int* __restrict__ cnt, int ncnt) {
  griddep_launch();
  griddep_wait();
  // item counters of the two expert GEMMs that follow on this stream, and
  // the K-split arrival counters of the gate/up GEMM
  if (blockIdx.x == 0) {
    if (sched && threadIdx.x < 2) sched[threadIdx.x] = 0;
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0;
  }
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int KG = Kp / 128;
  if (gw >= T * KG) return;
  const int t = gw / KG, g = gw % KG;
  const int c0 = g * 128 + 4 * lane;
  const int kb = lane >> 3;                                  // 32-value block of this lane
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (c0 < din) load4(xc + static_cast<size_t>(t) * din + c0, v);
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  const uint32_t s_hi = e4m3_block_scale(max8(m));
  const float inv_hi = e8m0_to_f32(254u - s_hi), sc_hi = e8m0_to_f32(s_hi);
  uint32_t w_hi = 0;
  float res[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const uint8_t q = f32_to_e4m3(v[u] * inv_hi);
    w_hi |= static_cast<uint32_t>(q) << (8 * u);
    res[u] = v[u] - e4m3_to_f32(q) * sc_hi;
  }
  // second term (the residual), or a zero term with a unit scale in the one-term form
  uint32_t s_lo = 127u, w_lo = 0;
  if (terms == 2) {
    m = fmaxf(fmaxf(fabsf(res[0]), fabsf(res[1])), fmaxf(fabsf(res[2]), fabsf(res[3])));
    s_lo = e4m3_block_scale(max8(m));
    const float inv_lo = e8m0_to_f32(254u - s_lo);
#pragma unroll
    for (int u = 0; u < 4; ++u) w_lo |= static_cast<uint32_t>(f32_to_e4m3(res[u] * inv_lo)) << (8 * u);
  }

  const int32_t* rows = inv_pad + static_cast<size_t>(t) * k;
  if (split) {   // one term: the hi rows and hi atoms only (the GEMMs read nothing else)
    for (int j = 0; j < k; ++j) {
      const size_t row = split_row_hi(rows[j], BN);
      *reinterpret_cast<uint32_t*>(xq + row * Kp + c0) = w_hi;
      if (terms == 2) *reinterpret_cast<uint32_t*>(xq + (row + BN) * Kp + c0) = w_lo;
    }
    for (int j = lane & 7; j < k; j += 8) {
      const int r = rows[j];
      uint8_t* at = xsf + (static_cast<size_t>(r / BN) * KG + g) * 1024 + sf_atom_offset(r % BN, kb);
      at[0] = static_cast<uint8_t>(s_hi);
      if (terms == 2) at[512] = static_cast<uint8_t>(s_lo);
    }
    return;
  }
  const int NA = (2 * BN + 127) / 128;
  for (int j = 0; j < k; ++j) {
    const size_t r = static_cast<size_t>(rows[j]);
    *reinterpret_cast<uint32_t*>(xq + (2 * r) * Kp + c0) = w_hi;
    *reinterpret_cast<uint32_t*>(xq + (2 * r + 1) * Kp + c0) = w_lo;
  }
  for (int j = lane & 7; j < k; j += 8) {
    const int r = rows[j];
    const int n = 2 * (r % BN);
    uint8_t* at = xsf + (static_cast<size_t>(r / BN) * KG + g) * NA * 512;
    at[(n >> 7) * 512 + sf_atom_offset(n & 127, kb)] = static_cast<uint8_t>(s_hi);
    at[((n + 1) >> 7) * 512 + sf_atom_offset((n + 1) & 127, kb)] = static_cast<uint8_t>(s_lo);
  }
}

// One block per token: u = sum over the token's k slots in slot order, then
// RMSNorm (Kimi K3 card code: routed_expert_norm between the sum and the
// up-projection).  float4 loads; the k slot loads of an element are
// independent so they overlap.
__global__ void __launch_bounds__(512) combine_norm_kernel(const float* __restrict__ y, int T, int k, int l,
                                                           int ks, size_t plane,
                                                           const __nv_bfloat16* __restrict__ w, int use_norm,
                                                           float eps, float* __restrict__ u_out,
                                                           __nv_bfloat16* __restrict__ u_hat) {
  griddep_launch();
  griddep_wait();
  extern __shared__ float4 cn_u4[];
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int l4 = l >> 2;
  const float4* yt = reinterpret_cast<const float4*>(y + static_cast<size_t>(t) * k * l);
  float4* ut = reinterpret_cast<float4*>(u_out + static_cast<size_t>(t) * l);
  float ss = 0.f;
  for (int i = threadIdx.x; i < l4; i += blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < ks; ++s) {   // K-split planes of the down pass
      const float4* ys = yt + s * (plane >> 2);
#pragma unroll 8
      for (int j = 0; j < k; ++j) {
        const float4 v = __ldg(ys + static_cast<size_t>(j) * l4 + i);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
    cn_u4[i] = acc;
    ut[i] = acc;
    ss += acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
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
  __nv_bfloat162* ot = reinterpret_cast<__nv_bfloat162*>(u_hat + static_cast<size_t>(t) * l);
  const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(w);
  for (int i = threadIdx.x; i < l4; i += blockDim.x) {
    const float4 a = cn_u4[i];
    float2 w01 = make_float2(1.f, 1.f), w23 = make_float2(1.f, 1.f);
    if (use_norm) {
      w01 = __bfloat1622float2(w2[2 * i]);
      w23 = __bfloat1622float2(w2[2 * i + 1]);
    }
    ot[2 * i] = __floats2bfloat162_rn(w01.x * a.x * rs, w01.y * a.y * rs);
    ot[2 * i + 1] = __floats2bfloat162_rn(w23.x * a.z * rs, w23.y * a.w * rs);
  }
}

// Small batches: the kCombineSlices CTAs of a cluster share one token's
// row.  Inside a CTA, G thread groups (blockDim = 128 G; more groups the
// fewer the tokens, so the CTAs still fill the SMs) each add every G-th of
// the (plane, slot) terms of an element, and the group sums are added in
// group order; the RMSNorm's sum of squares is added across
// the cluster through distributed shared memory (partials of the CTAs in rank
// order).  A token's row is read by several SMs with many loads in flight,
// instead of by one block.
constexpr int kCombineSlices = 8;
constexpr int kCombineClusterMaxT = 256;   // tokens up to which the cluster form is used
constexpr int kCombineLanes = 128;         // float4 columns of a slice handled at once
constexpr int kCombineMaxGroups = 8;

__global__ void __launch_bounds__(kCombineLanes * kCombineMaxGroups) combine_norm_cluster_kernel(
    const float* __restrict__ y, int T, int k, int l, int ks, size_t plane, const __nv_bfloat16* __restrict__ w,
    int use_norm, float eps, float* __restrict__ u_out, __nv_bfloat16* __restrict__ u_hat) {
  namespace cg = cooperative_groups;
  griddep_launch();
  griddep_wait();
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ float4 cc_part[];   // [G][per]; group 0's row then holds u
  __shared__ float red[kCombineLanes / 32];
  __shared__ float part_ss;
  __shared__ float tot_ss;
  const int t = blockIdx.y;
  const int r = static_cast<int>(cl.block_rank());
  const int l4 = l >> 2;
  const int per = (l4 + kCombineSlices - 1) / kCombineSlices;
  const int i0 = r * per;
  const int i1 = min(l4, i0 + per);
  const int lane_c = threadIdx.x % kCombineLanes, grp = threadIdx.x / kCombineLanes;
  const int groups = blockDim.x / kCombineLanes;
  const float4* yt = reinterpret_cast<const float4*>(y + static_cast<size_t>(t) * k * l);
  const size_t plane4 = plane >> 2;
  const int terms = ks * k;
  for (int i = i0 + lane_c; i < i1; i += kCombineLanes) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // term q = s*k + j (plane s, slot j) for q = grp, grp + groups, ...
    int s = grp / k, j = grp - (grp / k) * k;
#pragma unroll 8
    for (int q = grp; q < terms; q += groups) {
      const float4 v = __ldg(yt + s * plane4 + static_cast<size_t>(j) * l4 + i);
      for (j += groups; j >= k; j -= k) ++s;
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    cc_part[grp * per + (i - i0)] = acc;
  }
  __syncthreads();
  float ss = 0.f;
  if (grp == 0) {
    float4* ut = reinterpret_cast<float4*>(u_out + static_cast<size_t>(t) * l);
    for (int i = i0 + lane_c; i < i1; i += kCombineLanes) {
      float4 a = cc_part[i - i0];
#pragma unroll
      for (int g = 1; g < groups; ++g) {
        const float4 v = cc_part[g * per + (i - i0)];
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
      cc_part[i - i0] = a;
      ut[i] = a;
      ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w;
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f;
    for (int i = 0; i < kCombineLanes / 32; ++i) v += red[i];
    part_ss = v;
  }
  cl.sync();   // every CTA's partial is visible cluster-wide
  if (threadIdx.x < 32) {
    float v = threadIdx.x < kCombineSlices ? *cl.map_shared_rank(&part_ss, threadIdx.x) : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) tot_ss = v;
  }
  cl.sync();   // remote reads done before any CTA of the cluster exits; tot_ss visible
  const float rs = use_norm ? rsqrtf(tot_ss / static_cast<float>(l) + eps) : 1.0f;
  __nv_bfloat162* ot = reinterpret_cast<__nv_bfloat162*>(u_hat + static_cast<size_t>(t) * l);
  const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(w);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const float4 a = cc_part[i - i0];
    float2 w01 = make_float2(1.f, 1.f), w23 = make_float2(1.f, 1.f);
    if (use_norm) {
      w01 = __bfloat1622float2(w2[2 * i]);
      w23 = __bfloat1622float2(w2[2 * i + 1]);
    }
    ot[2 * i] = __floats2bfloat162_rn(w01.x * a.x * rs, w01.y * a.y * rs);
    ot[2 * i + 1] = __floats2bfloat162_rn(w23.x * a.z * rs, w23.y * a.w * rs);
  }
}

// Scale atoms [E][KG][MTa][512]: for expert e, k-group g (128 K values) and
// 128-row tile t, line r0 holds for c = 0..3 the four k-block scales of row
// 128t + 32c + r0.  Tiles of one k-group are adjacent, so a 256-row box's
// two atoms arrive in one copy.  Rows past N and k-blocks past Kb read 127.
__global__ void relayout_sfa_kernel(const uint8_t* __restrict__ s, int E, int N, int Kb, int MTa, int KG,
                                    uint8_t* __restrict__ atoms) {
  const size_t total = static_cast<size_t>(E) * KG * MTa * 512;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i & 511);
    size_t rest = i >> 9;
    const int mt = static_cast<int>(rest % MTa);
    rest /= MTa;
    const int g = static_cast<int>(rest % KG);
    const int e = static_cast<int>(rest / KG);
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

// Values the expert GEMMs multiply, back in fp32: for assignment a and
// column c, the sum of its E4M3 terms (hi, and lo for two terms) times their
// E8M0 block scales, read from either activation layout.
__global__ void decode_terms_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                    const int32_t* __restrict__ inv_pad, int P, int K, int Kp, int BN, int split,
                                    int terms, float* __restrict__ out) {
  const size_t n = static_cast<size_t>(P) * K;
  const int KG = Kp / 128;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int a = static_cast<int>(i / K), c = static_cast<int>(i % K);
    const int r = inv_pad[a], g = c >> 7, kb = (c & 127) >> 5;
    uint8_t qh, ql, sh, sl;
    if (split) {
      const size_t row = split_row_hi(r, BN);
      qh = q[row * Kp + c];
      ql = q[(row + BN) * Kp + c];
      const uint8_t* at = sf + (static_cast<size_t>(r / BN) * KG + g) * 1024 + sf_atom_offset(r % BN, kb);
      sh = at[0];
      sl = at[512];
    } else {
      qh = q[static_cast<size_t>(2 * r) * Kp + c];
      ql = q[static_cast<size_t>(2 * r + 1) * Kp + c];
      const int NA = (2 * BN + 127) / 128, nn = 2 * (r % BN);
      const uint8_t* at = sf + (static_cast<size_t>(r / BN) * KG + g) * NA * 512;
      sh = at[(nn >> 7) * 512 + sf_atom_offset(nn & 127, kb)];
      sl = at[((nn + 1) >> 7) * 512 + sf_atom_offset((nn + 1) & 127, kb)];
    }
    float v = e4m3_to_f32(qh) * e8m0_to_f32(sh);
    if (terms == 2) v += e4m3_to_f32(ql) * e8m0_to_f32(sl);
    out[i] = v;
  }
}

}  // namespace

cudaError_t launch_decode_terms(const uint8_t* q, const uint8_t* sf, const int32_t* inv_pad, int P, int K, int Kp,
                                int BN, int split, int terms, float* out, cudaStream_t s) {
  if (P <= 0) return cudaSuccess;
  decode_terms_kernel<<<ew_grid(static_cast<size_t>(P) * K), 256, 0, s>>>(q, sf, inv_pad, P, K, Kp, BN, split, terms,
                                                                          out);
  return cudaGetLastError();
}

cudaError_t launch_moe_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_moe<16, true>(p, grid, s);
    case 32: return launch_moe<32, true>(p, grid, s);
    case 64: return launch_moe<64, true>(p, grid, s);
    case 96: return launch_moe<96, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_moe_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s) {
  switch (BN) {
    case 16: return launch_moe<16, false>(p, grid, s);
    case 32: return launch_moe<32, false>(p, grid, s);
    case 64: return launch_moe<64, false>(p, grid, s);
    case 96: return launch_moe<96, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quant_gather(const float* xc, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                int split, int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (terms != 1 && terms != 2) return cudaErrorInvalidValue;
  const int warps_per_block = 8;
  const long long warps = static_cast<long long>(T) * (Kp / 128);
  {
    const unsigned blocks = static_cast<unsigned>((warps + warps_per_block - 1) / warps_per_block);
    const cudaError_t e_ = launch_pdl(quant_gather_kernel<float>, blocks, 32 * warps_per_block, 0, s, xc, T, k, din,
                                      Kp, inv_pad, BN, split, terms, xq, xsf, sched, cnt, ncnt);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_gather_bf16(const void* x, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                     int split, int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                     cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (terms != 1 && terms != 2) return cudaErrorInvalidValue;
  const int warps_per_block = 8;
  const long long warps = static_cast<long long>(T) * (Kp / 128);
  {
    const unsigned blocks = static_cast<unsigned>((warps + warps_per_block - 1) / warps_per_block);
    const cudaError_t e_ = launch_pdl(quant_gather_kernel<__nv_bfloat16>, blocks, 32 * warps_per_block, 0, s,
                                      static_cast<const __nv_bfloat16*>(x), T, k, din, Kp, inv_pad, BN, split, terms,
                                      xq, xsf, sched, cnt, ncnt);
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_combine_norm(const float* y, int T, int k, int l, int ks, size_t plane, const void* norm_w,
                                int use_norm, float eps, float* u, void* u_hat, int num_sms, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (ks < 1 || plane % 4) return cudaErrorInvalidValue;
  const int per = (l / 4 + kCombineSlices - 1) / kCombineSlices;
  // dynamic shared memory without opting in: 48 KB less the kernel's static arrays
  static size_t dyn_limit = 0;
  if (!dyn_limit) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, combine_norm_cluster_kernel);
    if (e != cudaSuccess) return e;
    dyn_limit = 48 * 1024 - fa.sharedSizeBytes;
  }
  if (T <= kCombineClusterMaxT && static_cast<size_t>(per) * sizeof(float4) <= dyn_limit) {
    int groups = kCombineMaxGroups;   // about one wave of CTAs, within the group-sum budget
    while (groups > 1 && (static_cast<long long>(T) * kCombineSlices * groups > 2LL * num_sms ||
                          static_cast<size_t>(groups) * per * sizeof(float4) > dyn_limit))
      groups >>= 1;
    const size_t smem = static_cast<size_t>(groups) * per * sizeof(float4);
    const cudaError_t e_ = launch_pdl_cluster(combine_norm_cluster_kernel, dim3(kCombineSlices, T), kCombineLanes * groups,
                                              smem, kCombineSlices, s, y, T, k, l, ks, plane,
                                              static_cast<const __nv_bfloat16*>(norm_w), use_norm, eps, u,
                                              static_cast<__nv_bfloat16*>(u_hat));
    if (e_ != cudaSuccess) return e_;
    return cudaGetLastError();
  }
  const size_t smem = static_cast<size_t>(l) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(combine_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t e_ = launch_pdl(combine_norm_kernel, T, 512, smem, s, y,
                                      T, k, l, ks, plane, static_cast<const __nv_bfloat16*>(norm_w), use_norm, eps, u,
                                      static_cast<__nv_bfloat16*>(u_hat));
    if (e_ != cudaSuccess) return e_;
  }
  return cudaGetLastError();
}

cudaError_t launch_relayout_sfa(const uint8_t* s, int E, int N, int Kb, int MTa, int KG, uint8_t* atoms,
                                cudaStream_t st) {
  const size_t total = static_cast<size_t>(E) * MTa * KG * 512;
  relayout_sfa_kernel<<<ew_grid(total), 256, 0, st>>>(s, E, N, Kb, MTa, KG, atoms);
  return cudaGetLastError();
}

cudaError_t launch_pad_codes(const uint8_t* q, int E, int N, int K, int Kp, uint8_t* out, cudaStream_t st) {
  const size_t total = static_cast<size_t>(E) * N * (Kp / 2);
  pad_codes_kernel<<<ew_grid(total), 256, 0, st>>>(q, E, N, K, Kp, out);
  return cudaGetLastError();
}

}  // namespace lmoe
