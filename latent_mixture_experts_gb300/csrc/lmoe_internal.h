// Internal interfaces between the C-ABI layer and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

namespace lmoe {

// Error-flag slots in device memory (int[4]): a bounded wait that expired
// writes kErrTimeout into slot 0; an out-of-range expert index sets slot 1.
constexpr int kErrTimeout = 1;
// Largest expert count the dispatch scan handles in one block.
constexpr int kMaxExperts = 2048;

// ----------------------------------------------------------- dense GEMM
// out[s][t][row] (fp32 partial sums over split s) = sum_k A[row][k] * B[t][k]
// for bf16 A (weights, [M][K]) and B (tokens, [T][K]), K-major both.
//   mode 0: one A, one B.
//   mode 1: rows [0, M0) from a0, rows [M0, M0+M1) from a1 (M concatenation).
//   mode 2: k-blocks [0, nkb0) from (a0, b0), the rest from (a1, b1)
//           (K concatenation, one accumulator).
struct DenseParams {
  CUtensorMap a0, a1, b0, b1;
  CUtensorMap a0w, a1w;   // the same weights with 256-row boxes (used when wide)
  int wide;               // 1: each CTA computes 256 weight rows (two accumulators), BN = 256, splits = 1
  // Epilogue: 0 = fp32 partial sums per K split into `out` (finalized by a
  // separate kernel); 1 = bf16 out16[t][row] (+ add[t][row] when add is set),
  // splits = 1; 2 = gate/up pair (wide, mode 1: the CTA's two tiles are gate
  // rows and up rows of the same 128 features, one 256-row box of the
  // interleaved copy in a0w), bf16 out16[t][f] = act(gate, up), splits = 1.
  int epi;
  void* out16;
  float* out32;           // epilogue 1: when set, also the fp32 value before the bf16 rounding, [t][row]
  const float* add;
  int ld_add;
  int act;
  float act_b1, act_b2;   // SiTU caps (epilogue 2)
  float* out;
  int* err;
  int mode;
  int M0, M1, mtiles0;
  int T;
  int nkb, nkb0;
  int splits;
  int ldo;
};
// BN: token tile (32, 64, 128 or 256).  Grid (mtiles, ceil(T/BN), splits);
// mtiles and mtiles0 count 128-row tiles (a wide launch pairs them).
cudaError_t launch_dense_gemm(const DenseParams& p, int mtiles, int BN, cudaStream_t s);

// bf16 [2*ceil(Fs/128)*128][K] copy of the shared gate [Fs][K] and up [Fs][K]
// weights, interleaved every 128 rows (gate block, up block, ...; zero rows
// past Fs): a 256-row box of it is the gate/up tile pair of 128 features.
cudaError_t launch_interleave_gate_up(const void* gate, const void* up, int Fs, int K, void* out, cudaStream_t s);
// Sum `splits` partial planes [splits][T][ld] and apply an epilogue.
cudaError_t launch_finalize_sum_f32(const float* part, int splits, int T, int M, int ld, float* out, int ldo,
                                    cudaStream_t s);
// out32_opt: when set, also the fp32 sum before the bf16 rounding ([T][ldo]).
cudaError_t launch_finalize_sum_bf16(const float* part, int splits, int T, int M, int ld, void* out, int ldo,
                                     const float* add_opt, int ld_add, float* out32_opt, cudaStream_t s);
// gate at columns [0, F), up at [F, 2F) of each partial row.
cudaError_t launch_finalize_glu_bf16(const float* part, int splits, int T, int F, int ld, void* out, int act,
                                     float b1, float b2, cudaStream_t s);

// ------------------------------------------------------------- routing
// Also writes the summed logits z [T][E] (fp32) to z_out.
cudaError_t launch_topk(const float* logit_part, int splits, int T, int E, const float* bias, int k,
                        float routed_scale, int32_t* idx, float* G, float* z_out, cudaStream_t s);

struct DispatchBufs {
  int32_t* counts;      // [E]
  int32_t* offsets;     // [E+1]
  int32_t* perm;        // [T*k]  assignments grouped by expert
  int32_t* inv_pad;     // [T*k]  padded row of each assignment
  int32_t* tile_off;    // [E+1]  padded offsets (multiples of BN)
  int32_t* blockcnt;    // [nchunks][E]
  int4* tiles;          // [max tiles]  {expert, padded row0, rows, unpadded p0}
  int32_t* ntiles;      // [1]
  int* err;
};
constexpr int kDispatchChunk = 256;
// Batches of at most this many assignments are dispatched by one kernel;
// larger ones by the four-kernel chunked path.
constexpr int kSmallDispatch = 8192;
inline int dispatch_launches(int assignments) { return assignments <= kSmallDispatch ? 1 : 4; }
cudaError_t launch_dispatch(const int32_t* idx, int T, int k, int E, int BN, const DispatchBufs& b,
                            cudaStream_t s);

// ------------------------------------------------------- routed experts
// Activation rows of one assignment as two E4M3 rows (hi, lo) of a
// [2*Ppad][Kp] byte matrix, with their E8M0 scales in the tcgen05 staging
// image (512-byte atoms, one per 128 columns and 128-wide k-group).
//   interleaved (split = 0): padded row r -> rows 2r (hi), 2r+1 (lo); the
//     tile's 2*BN rows are one MMA operand of N = 2*BN columns, scale atoms
//     [Ppad/BN][KG][ceil(2BN/128)].
//   split (split = 1): per BN-row tile b, rows 2*BN*b + j (hi) and
//     2*BN*b + BN + j (lo), j = r - BN*b; hi and lo are two operands of
//     N = BN columns, scale atoms [Ppad/BN][KG][2] (BN <= 128).
// terms = 1: the hi term only (split: lo rows not written; interleaved: lo
// rows zero with unit scales).
cudaError_t launch_quant_gather(const float* xc, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                int split, int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                cudaStream_t s);
// Same from bf16 token rows (layers whose experts take x itself).
cudaError_t launch_quant_gather_bf16(const void* x, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                     int split, int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                     cudaStream_t s);

// Weight rows per work item (and per TMA box) of the grouped expert GEMMs:
// 256-row boxes stream FP4 codes at full HBM rate; the large token tiles of
// prefill keep 128-row items so two accumulators fit tensor memory.
__host__ __device__ constexpr int moe_rows_per_item(int BN) { return BN >= 64 ? 128 : 256; }
// Weight rows per TMA box of the FP8-weight expert GEMMs (one fp32 scale block).
constexpr int kFp8Rows = 128;
// Largest contraction length of the FP8-weight expert GEMMs: the epilogue
// holds an item's per-128-K block scales in two registers per lane.
constexpr int kFp8MaxK = 64 * 128;
// Token tile of the FP8-weight expert GEMMs (hi and lo share accumulator
// columns, so a tile of up to 96 assignments fits tensor memory): the
// smallest of 16, 32, 64, 96 that holds the mean assignments per expert.
inline int fp8_tile_tokens(long long assignments, int n_experts) {
  const long long m = (assignments + n_experts - 1) / n_experts;
  return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 96;
}
constexpr int kFp8MaxTile = 96;
// Token tile of the grouped MXFP4 expert GEMMs from the mean assignments per
// expert: 16 or 32 (decode; interleaved hi/lo columns, 256-row boxes), 64 or
// 96 (prefill; split hi/lo operands, 128-row items).
inline int moe_tile_tokens(long long assignments, int n_experts) {
  return assignments <= 4LL * n_experts ? 16 : assignments <= 16LL * n_experts ? 32
         : assignments <= 64LL * n_experts ? 64 : 96;
}
// Activation layout of the grouped MXFP4 expert GEMMs at a token tile: split
// (hi and lo as two MMAs into the same accumulator columns) for the large
// tiles, interleaved (hi/lo as adjacent columns of one MMA) for the small.
__host__ __device__ constexpr bool moe_split(int BN) { return BN >= 64; }

// Launch `kernel` with programmatic stream serialization (see griddep_wait):
// it may begin while the previous kernel on the stream drains.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl for a kernel whose CTAs form clusters of cluster_x along x.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                                      cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = cluster_x;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct MoeGemmParams {
  CUtensorMap a_gate, a_up, b;   // FP4 weights viewed [E*N][Kp] (boxes of moe_rows_per_item rows);
                                 // activations [2*Ppad][Kp]
  const uint8_t* sfa_gate;       // weight scale atoms [E][KG][MTa][512]
  const uint8_t* sfa_up;
  const uint8_t* sfb;            // activation scale atoms [Ppad/BN][G][NA][512]
  const int4* tiles;
  const int32_t* tile_off;       // [E+1] padded row offsets (multiples of BN)
  const int32_t* ntiles;
  const int32_t* perm;
  const float* G;                // [T*k] routing weights (down pass)
  int* err;
  int* sched;                    // item counter of the dynamic distribution (zeroed before the launch)
  // K split of small batches: weight-row item i becomes items i*KS .. i*KS+KS-1 over consecutive
  // k-group ranges.  Gate/up: partial sums to gpart [KS][2][P][N_out], added by the last split to
  // arrive at a lane quarter's rows (gcnt: [item][4] counters, zeroed before the launch).  Down:
  // split s writes its partial outputs to the y plane at y + s*y_plane.
  int KS;
  float* gpart;
  int* gcnt;
  int P;
  size_t y_plane;
  int stages, accbufs;           // packed-FP4 kernel: stage ring depth and accumulator buffers (set at launch)
  int terms;                     // activation terms: 2 (E4M3 hi + lo) or 1 (MXFP8: hi only; split
                                 // layouts then load and multiply only the hi rows, whose TMA box is BN rows)
  int N_out;                     // output features per expert (F for gate/up, din for down)
  int MT;                        // work-item columns per expert tile: ceil(N_out / rows per item)
  int MTa;                       // 128-row tiles per (expert, k-group) in the scale-atom layout (even)
  int KG;                        // Kp / 128
  // gate/up epilogue: h written as hi/lo E4M3 + scale atoms for the down pass
  uint8_t* hq;                   // [2*Ppad][Fp]
  uint8_t* hsf;                  // [Ppad/BN][Fp/128][NA][512]
  int Fp;
  int act;
  float b1, b2;
  // down epilogue
  float* y;                      // [T*k][dx] fp32, G-scaled expert outputs
  // FP8 weights: fp32 scale per 128 x 128 block, [E][NB][KB]; wsc1 = up scales (gate/up pass)
  const float* wsc0;
  const float* wsc1;
  int NB, KB;
  // K-split gate/up pass (MXFP4 weights): once a CTA has issued its last load
  // it prefetches into L2 its share of the down-pass weights of the batch's
  // experts, in the order the down pass takes them, up to pf_budget bytes
  // (pf_codes null: no prefetch).  Sizes are multiples of 16 bytes.
  const uint8_t* pf_codes;       // down codes, pf_code_bytes per expert
  const uint8_t* pf_atoms;       // down scale atoms, pf_atom_bytes per expert
  size_t pf_code_bytes, pf_atom_bytes, pf_budget;
};
// Down-pass weight bytes the K-split gate/up pass prefetches into L2: about
// half of the 129 MB L2, so the prefetch does not evict its own first lines.
constexpr size_t kDownPrefetchBytes = static_cast<size_t>(64) << 20;
cudaError_t launch_moe_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
cudaError_t launch_moe_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
// FP8 E4M3 weights with 128 x 128 fp32 block scales (BN 16 or 32).
cudaError_t launch_moe_fp8_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
cudaError_t launch_moe_fp8_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
// The shared expert of an FP8 layer runs on the FP8 expert GEMMs as one
// expert that every token uses: its tile list for T tokens in BN-token tiles
// (expert 0, rows i*BN.., assignments i*BN..), tile_off = {0, ntiles*BN}.
cudaError_t launch_shared_tiles(int T, int BN, int4* tiles, int32_t* tile_off, int32_t* ntiles, cudaStream_t s);
// iota[i] = i and ones[i] = 1 for i < n (identity rows and unit weights of the shared expert).
cudaError_t launch_iota_ones(int32_t* iota, float* ones, int n, cudaStream_t s);

// u[t] = sum_j y[t*k + j] (slot order); u_hat = w * u / sqrt(mean(u^2) + eps) -> bf16.
// ks > 1: y holds ks planes (partials of a K-split down pass), plane elements apart, all added.
cudaError_t launch_combine_norm(const float* y, int T, int k, int l, int ks, size_t plane, const void* norm_w,
                                int use_norm, float eps, float* u, void* u_hat, int num_sms, cudaStream_t s);

// ------------------------------------------------------ quantile balancing
// Exact update: alpha [T] (scratch) = each token's (k+1)-th largest biased
// score, raw [E] (scratch) = the (k/E)-quantile of alpha_i - s_ij per expert,
// new_bias = raw - mean(raw).  z: router logits fp32 [T][E].
cudaError_t launch_qb_update(const float* z, int T, int E, int k, const float* bias, float* alpha, float* raw,
                             float* new_bias, cudaStream_t s);
// Adds the batch's required biases to counts [E][bins] (int32) over the range
// [min b - 1, max b + 1] (written to range [2]).
cudaError_t launch_qb_histogram(const float* z, int T, int E, int k, const float* bias, int bins, float* alpha,
                                float* range, int32_t* counts, cudaStream_t s);
// new_bias from the accumulated counts (quantile per expert, centred).
cudaError_t launch_qb_from_histogram(const int32_t* counts, int E, int bins, int k, const float* bias, float* range,
                                     float* raw, float* new_bias, cudaStream_t s);

// ------------------------------------------------------ expert parallelism
// send[pos] = bf16 row of the token of assignment perm[pos]: from x^c (fp32,
// latent layers) or from x (bf16 xb, non-latent layers), P rows of dx.
cudaError_t launch_ep_pack(const float* xc, const void* xb, int dx, int k, const int32_t* perm, int P, void* send,
                           cudaStream_t s);
// idx_loc[row] = local expert of received row `row` (< n), from counts [nseg]
// (source rank major, E_loc experts each); err[1] = 1 when they do not sum to n.
cudaError_t launch_ep_expand(const int32_t* counts, int nseg, int E_loc, int n, int32_t* idx_loc, int* err,
                             cudaStream_t s);
// out[row] = bf16(sum over ks planes of y[row]) for n rows of dx.
cudaError_t launch_ep_cast(const float* y, int n, int dx, int ks, size_t plane, void* out, cudaStream_t s);
// y[perm[pos]] = G[perm[pos]] * ret[pos] (bf16 rows) for P rows of dx.
cudaError_t launch_ep_unpack(const void* ret, int P, int dx, const int32_t* perm, const float* G, float* y,
                             cudaStream_t s);

// One warp waits on an mbarrier nothing arrives at, with the given limit;
// the bounded wait then records kErrTimeout in err[0].
cudaError_t launch_wait_timeout_probe(int* err, unsigned long long limit_ns, cudaStream_t s);

// Routed experts with packed E2M1 operands on both sides (kind::mxf4,
// E8M0 scales per 32): weights as stored, activations p.terms MXFP4 terms in
// the packed layout below; p.KG counts 256-K groups (K padded to 256), the
// scale atoms are those of the other expert kernels (per 128 K).
cudaError_t launch_moe_fp4_gate_up(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
cudaError_t launch_moe_fp4_down(const MoeGemmParams& p, int BN, int grid, cudaStream_t s);
// x^c rows -> `terms` MXFP4 terms per value: packed codes [Ppad/BN][terms][BN][Kp/2] (per tile, its
// terms' rows one after the other), scale atoms [Ppad/BN][Kp/128][terms][512].
cudaError_t launch_quant_gather_fp4(const float* xc, int T, int k, int din, int Kp, const int32_t* inv_pad, int BN,
                                    int terms, uint8_t* xq, uint8_t* xsf, int* sched, int* cnt, int ncnt,
                                    cudaStream_t s);
cudaError_t launch_decode_fp4(const uint8_t* q, const uint8_t* sf, const int32_t* inv_pad, int P, int K, int Kp,
                              int BN, int terms, float* out, cudaStream_t s);

// Debug read-out: the values of the encoded activations (hi + lo terms times
// their block scales) of P assignments, fp32 [P][K], from either layout.
cudaError_t launch_decode_terms(const uint8_t* q, const uint8_t* sf, const int32_t* inv_pad, int P, int K, int Kp,
                                int BN, int split, int terms, float* out, cudaStream_t s);

// Create-time repacking of the expert weights.
cudaError_t launch_relayout_sfa(const uint8_t* s, int E, int N, int Kb, int MTa, int KG, uint8_t* atoms,
                                cudaStream_t st);
cudaError_t launch_pad_codes(const uint8_t* q, int E, int N, int K, int Kp, uint8_t* out, cudaStream_t st);

}  // namespace lmoe
