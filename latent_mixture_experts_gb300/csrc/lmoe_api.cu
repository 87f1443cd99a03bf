// C ABI of the Stable LatentMoE layer: handle, workspace, launch sequence.
//
// lmoe_forward, no host synchronisation.  Caller's stream:
//   1 router GEMM (bf16 tcgen05, fp32 split-K partial logits)
//   2 top-k: sum partials, sigmoid, + bias, select, renormalise
//   3 dispatch: counting sort into BN-row expert tiles (1 or 4 kernels)
//   5 x^c rows -> hi/lo E4M3 activations in expert-tile order (after 4)
//   6 grouped gate/up GEMM with SiTU / SwiGLU epilogue -> hi/lo E4M3 h
//   7 grouped down GEMM, epilogue x G_i -> per-assignment outputs
//   8 slot-ordered sum + RMSNorm -> u_hat (bf16)
//  10 [u_hat | h_shared] x [W_up ; W_shared_down] (K-concatenated) -> Delta
//     (after 9); FP8 layers: Delta = sum + the shared expert's output
// Side stream of the handle, forked at entry and joined before 5 and 10:
//   4 latent down-projection x^c = x W_down^T (+ split-K sum)
//   9 shared gate/up GEMM + SiTU -> h_shared (bf16); FP8 layers: the whole
//     shared expert on the FP8 expert GEMMs
// The grouped expert GEMMs are persistent, hand out their items through a
// counter that step 5 zeroes, and split each item's K range for batches of
// a few tokens.  Every kernel is launched with programmatic serialization.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/lmoe.h"
#include "lmoe_internal.h"
#include "tmap.h"

using namespace lmoe;

struct lmoe_ctx {
  lmoe_config cfg;
  lmoe_weights w;
  int dev = 0, num_sms = 148;
  int d = 0, din = 0, E = 0, k = 0, F = 0, Fs = 0;
  int dx = 0;          // width the routed experts read and write: the latent, or d for non-latent layers
  bool fp8 = false;    // experts in FP8 E4M3 with 128 x 128 fp32 block scales
  int terms = 2;       // activation terms per routed-expert input (E4M3: 2 hi + lo, 1 MXFP8; E2M1: 1..4)
  bool fp4 = false;    // packed E2M1 activations x MXFP4 weights (kind::mxf4); K padded to 256
  // expert parallelism: this handle holds experts [ep_rank * E_loc, (ep_rank + 1) * E_loc)
  int ep = 1, ep_rank = 0, E_loc = 0;
  int Pexp = 0;        // rows the expert GEMMs may see: T*k, or the rows received from all ranks
  int32_t* ep_perm = nullptr;   // assignments grouped by global expert (the send order), kept for the combine
  int32_t* idx_loc = nullptr;   // local expert of each received row
  float* ones = nullptr;        // unit routing weights of the received rows
  int ep_T = 0;                 // tokens of the last lmoe_ep_dispatch
  // FP8 layers run the shared expert on the FP8 expert GEMMs, as one expert
  // that every token uses (exact block-scaled weights): its tile list, identity
  // rows and unit weights, hi/lo activations and its fp32 output.
  int4* sh_tiles = nullptr;
  int32_t *sh_tile_off = nullptr, *sh_ntiles = nullptr, *sh_iota = nullptr;
  float *sh_ones = nullptr, *y_sh = nullptr;
  uint8_t *xq_sh = nullptr, *xsf_sh = nullptr, *hq_sh = nullptr, *hsf_sh = nullptr;
  int Tpad_sh = 0;
  int Kp = 0, Fp = 0, MT_gu = 0, MT_dn = 0, KG_gu = 0, KG_dn = 0, MTa_gu = 0, MTa_dn = 0;
  int Tm = 0, Pm = 0, Ppad = 0, max_tiles = 0, nchunks_max = 0;
  // device memory
  void* pool = nullptr;
  size_t pool_bytes = 0;
  int* err = nullptr;
  int* sched = nullptr;       // item counters: routed gate/up, routed down, shared gate/up, shared down
  float* gpart = nullptr;     // K-split partial gate/up sums of small batches
  int* gcnt = nullptr;        // their arrival counters
  int n_gcnt = 0;
  float* part = nullptr;
  float* part_sh = nullptr;   // split-K partials of the GEMMs on `side` (latent down, shared gate/up)
  float* xc = nullptr;
  float* logits = nullptr;
  int32_t* idx = nullptr;
  float* G = nullptr;
  int32_t *counts = nullptr, *offsets = nullptr, *tile_off = nullptr, *perm = nullptr, *inv_pad = nullptr;
  int32_t *blockcnt = nullptr, *ntiles = nullptr;
  int4* tiles = nullptr;
  uint8_t *xq = nullptr, *xsf = nullptr, *hq = nullptr, *hsf = nullptr;
  float* y = nullptr;           // per-assignment G-scaled expert outputs
  float* u = nullptr;
  void* u_hat = nullptr;
  void* h_s = nullptr;
  void* x_stage = nullptr;
  void* out_stage = nullptr;
  float* delta32 = nullptr;   // Delta before its bf16 rounding, [Tm][d] (allocated by lmoe_keep_f32_output)
  float *qb_alpha = nullptr, *qb_raw = nullptr, *qb_range = nullptr;   // quantile-balancing scratch
  uint8_t *sfa_gate = nullptr, *sfa_up = nullptr, *sfa_down = nullptr;
  const uint8_t *codes_gate = nullptr, *codes_up = nullptr, *codes_down = nullptr;
  uint8_t *pad_gate = nullptr, *pad_up = nullptr, *pad_down = nullptr;
  // static tensor maps
  CUtensorMap m_router, m_wdown, m_wup, m_shg, m_shu, m_shd;
  CUtensorMap m_routerw, m_wdownw, m_wupw, m_shdw;   // 256-row boxes (wide dense tiles)
  // bf16 shared MLP: gate and up weights interleaved every 128 rows, so one
  // 256-row box is the gate/up tile pair of 128 features (handle-owned copy)
  void* sh_gu_il = nullptr;
  CUtensorMap m_shgu_il;
  CUtensorMap m_exg[2], m_exu[2], m_exd[2];   // expert codes, boxes of 128 / 256 rows
  CUtensorMap m_sg, m_su, m_sd;               // FP8 shared-expert codes, 128-row boxes
  // The latent down-projection and the shared-expert gate/up GEMM need only
  // x: they run on a side stream forked from the caller's stream at the start
  // of a forward, overlapping the router and dispatch; the caller's stream
  // waits for x^c before encoding the expert inputs (ev_latent) and for
  // h_shared before the output GEMM (ev_join).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_latent = nullptr, ev_join = nullptr;
  int last_T = 0;
  int last_launches = 0;
  int last_BN = 0, last_split = 0;   // activation layout of the last forward's expert GEMMs
  // per-stage event timing
  bool prof = false;
  uint32_t prof_mask = 0;    // stages timed while profiling
  int prof_every = 1;        // time every prof_every-th call while profiling
  long long prof_calls = 0;  // calls since profiling was enabled
  bool prof_now = false;     // this call records its stage events
  std::vector<cudaEvent_t> ev_free;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev_used[LMOE_NUM_STAGES];
};

namespace {

lmoe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return LMOE_OK;
  if (e == cudaErrorMemoryAllocation) return LMOE_ERR_OOM;
  return LMOE_ERR_CUDA;
}
#define LMOE_TRY(expr)                                   \
  do {                                                   \
    cudaError_t e_ = (expr);                             \
    if (e_ != cudaSuccess) return cuda_status(e_);       \
  } while (0)

#define LMOE_TRY_STATUS(expr)                          \
  do {                                                 \
    const lmoe_status s_ = (expr);                     \
    if (s_ != LMOE_OK) return s_;                      \
  } while (0)

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kRouterMaxSplits = 16;

int dense_bn(int T) { return T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }
// Token tile of the routed expert GEMMs of this handle's weight format for P
// rows over its E_loc experts.
int expert_bn_rows(const lmoe_ctx* h, long long P) {
  return h->fp8 ? fp8_tile_tokens(P, h->E_loc) : moe_tile_tokens(P, h->E_loc);
}
int expert_bn(const lmoe_ctx* h, int T) { return expert_bn_rows(h, static_cast<long long>(T) * h->k); }

// K splits of the routed MXFP4 expert GEMMs (1 = none) for a batch of P
// assignments: when the weight-row items of a pass (an upper bound of its
// tiles times the items per tile) come to fewer than two per SM, each item's
// K range is split (up to 4 ways, to about four items per SM) so that the
// items keep every SM streaming to the end.
constexpr long long kKsplitMaxP = 1024;
int expert_ksplit(const lmoe_ctx* h, long long P, bool gate_up) {
  if (h->fp8 || P > kKsplitMaxP) return 1;
  const int BN = moe_tile_tokens(P, h->E_loc);
  if (BN != 16) return 1;   // the K-split form is built for the 16-assignment tile
  const int RB = moe_rows_per_item(BN);
  const long long MT = gate_up ? ceil_div(h->F, RB) : ceil_div(h->dx, 2 * RB);
  const int KG = (gate_up ? h->KG_gu : h->KG_dn) / (h->fp4 ? 2 : 1);   // K groups of the kernel that runs
  const long long tiles = std::min<long long>(P, P / BN + std::min<long long>(h->E_loc, P));
  const long long items = tiles * MT;
  if (items >= 2LL * h->num_sms) return 1;
  const long long want = 4LL * h->num_sms;
  const long long ks = std::min<long long>({(want + items - 1) / items, 4LL, KG / 2});
  return static_cast<int>(std::max(ks, 1LL));
}

// K splits of a dense GEMM over `tiles` CTA tiles: fill about one wave of
// CTAs, at least two 64-wide k-blocks per split.
int dense_splits(int tiles, int nkb, int num_sms) {
  int s = num_sms / std::max(tiles, 1);
  s = std::min(s, std::max(nkb / 2, 1));
  return std::max(s, 1);
}

// Launch plan of a dense GEMM with mt0 (+ mt1, M-concatenated) 128-row
// weight tiles and nt token tiles of BN: plain (one weight tile per CTA) or
// wide (two per CTA: one 256-row box per stage, a third fewer bytes per
// MAC).  Wide is taken at the prefill tile (BN = 256) when the paired tiles
// fill the SMs without a K split; under a K split it doubled the partial
// planes to sum and measured slower at decode.
struct DensePlan {
  int splits, wide;
};
DensePlan dense_plan(int mt0, int mt1, int nt, int nkb, int BN, int num_sms, bool allow_wide) {
  const int tiles1 = (mt0 + mt1) * nt;
  // decode tiles (BN <= 64) leave room for two CTAs per SM: split K for two per SM
  const int s1 = dense_splits(tiles1, nkb, BN <= 64 ? 2 * num_sms : num_sms);
  const int tiles2 = ((mt0 + 1) / 2 + (mt1 + 1) / 2) * nt;
  if (allow_wide && BN == 256 && s1 == 1 && tiles2 >= num_sms) return {1, 1};
  return {s1, 0};
}

struct Carve {
  size_t off = 0;
  template <class T>
  T* take(size_t count, char* base) {
    off = align_up(off, 1024);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

bool map_bf16(CUtensorMap* m, const void* base, int K, int rows, int box_rows) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, K, rows, static_cast<uint64_t>(K) * 2, 64, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_fp4(CUtensorMap* m, const void* base, int K, long long rows, int box_rows) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, base, K, rows, static_cast<uint64_t>(K) / 2, 128,
                      box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_u8(CUtensorMap* m, const void* base, int K, long long rows, int box_rows) {
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, K, rows, K, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Largest (splits x T) a dense GEMM planned by dense_plan needs for T <= Tm.
long long max_split_rows(int mt0, int mt1, int nkb, int Tm, int num_sms, bool allow_wide) {
  long long best = 0;
  for (int T = 1; T <= Tm;) {
    const int BN = dense_bn(T);
    const int nt = ceil_div(T, BN);
    const DensePlan pl = dense_plan(mt0, mt1, nt, nkb, BN, num_sms, allow_wide);
    const int Tend = std::min(Tm, nt * BN);   // same (BN, ntiles) up to here
    best = std::max(best, static_cast<long long>(pl.splits) * Tend);
    T = Tend + 1;
  }
  return best;
}

cudaEvent_t take_event(lmoe_ctx* h) {
  if (!h->ev_free.empty()) {
    cudaEvent_t e = h->ev_free.back();
    h->ev_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Records a CUDA event pair around one stage's launches while profiling.
struct StageTimer {
  lmoe_ctx* h;
  int stage;
  cudaStream_t st;
  cudaEvent_t b = nullptr;
  StageTimer(lmoe_ctx* h_, int stage_, cudaStream_t st_) : h(h_), stage(stage_), st(st_) {
    if (h->prof_now && (h->prof_mask >> stage & 1u) && (b = take_event(h)) != nullptr) cudaEventRecord(b, st);
  }
  void done() {
    if (!b) return;
    cudaEvent_t e = take_event(h);
    if (e) {
      cudaEventRecord(e, st);
      h->ev_used[stage].emplace_back(b, e);
    } else {
      h->ev_free.push_back(b);
    }
    b = nullptr;
  }
};

// Whether the call starting now records stage events (every prof_every-th).
void begin_call(lmoe_ctx* h) {
  h->prof_now = h->prof && (h->prof_calls++ % h->prof_every) == 0;
}

void release_events(lmoe_ctx* h) {
  for (auto& v : h->ev_used) {
    for (auto& pr : v) {
      h->ev_free.push_back(pr.first);
      h->ev_free.push_back(pr.second);
    }
    v.clear();
  }
}

lmoe_status check_err(lmoe_ctx* h) {
  int e[4] = {0, 0, 0, 0};
  LMOE_TRY(cudaMemcpy(e, h->err, sizeof(e), cudaMemcpyDeviceToHost));
  LMOE_TRY(cudaMemset(h->err, 0, sizeof(e)));
  if (e[0]) return LMOE_ERR_TIMEOUT;
  if (e[1]) return LMOE_ERR_INVALID_ARG;
  return LMOE_OK;
}

lmoe_status run_router(lmoe_ctx* h, const void* x, int T, cudaStream_t st, int& launches) {
  StageTimer tm(h, LMOE_STAGE_ROUTER, st);
  const int BN = dense_bn(T);
  DenseParams p;
  std::memset(&p, 0, sizeof(p));
  p.a0 = h->m_router;
  p.a0w = h->m_routerw;
  if (!map_bf16(&p.b0, x, h->d, T, BN)) return LMOE_ERR_CUDA;
  p.mode = 0;
  p.M0 = h->E;
  p.mtiles0 = ceil_div(h->E, 128);
  p.T = T;
  p.nkb = ceil_div(h->d, 64);
  p.nkb0 = p.nkb;
  // plain tiles: wide ones would split K further and top-k sums every split;
  // at most 16 splits, so top-k reads few partial planes (one to four tokens
  // would otherwise split the 7168-long K ~40 ways)
  const DensePlan pl = dense_plan(p.mtiles0, 0, ceil_div(T, BN), p.nkb, BN, h->num_sms, false);
  p.splits = std::min(pl.splits, kRouterMaxSplits);
  p.wide = pl.wide;
  p.ldo = h->E;
  p.out = h->part;
  p.err = h->err;
  LMOE_TRY(launch_dense_gemm(p, p.mtiles0, BN, st));
  LMOE_TRY(launch_topk(h->part, p.splits, T, h->E, h->w.router_bias, h->k, h->cfg.routed_scale, h->idx, h->G,
                       h->logits, st));
  launches += 2;
  tm.done();
  return LMOE_OK;
}

lmoe_status run_dispatch(lmoe_ctx* h, const int32_t* idx, int T, int BN, int32_t* counts, int32_t* offsets,
                         int32_t* perm, cudaStream_t st, int& launches, int k = 0, int E = 0) {
  k = k ? k : h->k;
  E = E ? E : h->E;
  StageTimer tm(h, LMOE_STAGE_DISPATCH, st);
  DispatchBufs b;
  b.counts = counts;
  b.offsets = offsets;
  b.perm = perm;
  b.inv_pad = h->inv_pad;
  b.tile_off = h->tile_off;
  b.blockcnt = h->blockcnt;
  b.tiles = h->tiles;
  b.ntiles = h->ntiles;
  b.err = h->err;
  LMOE_TRY(launch_dispatch(idx, T, k, E, BN, b, st));
  launches += dispatch_launches(T * k);
  tm.done();
  return LMOE_OK;
}

lmoe_status validate_cfg(const lmoe_config* c) {
  if (c->d_model <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->d_expert_ff <= 0 || c->max_tokens <= 0 ||
      c->d_latent < 0 || c->d_shared_ff < 0 || c->top_k > c->n_experts)
    return LMOE_ERR_INVALID_ARG;
  if (c->act != LMOE_ACT_SITU && c->act != LMOE_ACT_SWIGLU) return LMOE_ERR_INVALID_ARG;
  if (c->expert_wfmt != LMOE_W_MXFP4 && c->expert_wfmt != LMOE_W_FP8_BLOCK128) return LMOE_ERR_INVALID_ARG;
  // MXFP4 experts: latent layers (Kimi K3); FP8 block-128 experts: non-latent layers (Kimi K2)
  if (c->expert_wfmt == LMOE_W_MXFP4 && c->d_latent == 0) return LMOE_ERR_UNSUPPORTED;
  if (c->expert_wfmt == LMOE_W_FP8_BLOCK128 &&
      (c->d_latent != 0 || c->use_latent_norm || c->d_model % 128 || c->d_expert_ff % 128 || c->d_shared_ff % 128 ||
       c->d_model > kFp8MaxK || c->d_expert_ff > kFp8MaxK || c->d_shared_ff > kFp8MaxK))
    return LMOE_ERR_UNSUPPORTED;
  if (c->d_model % 32 || c->d_latent % 32 || c->d_expert_ff % 32 || c->d_shared_ff % 32) return LMOE_ERR_UNSUPPORTED;
  if (c->n_experts > kMaxExperts || c->top_k > 32) return LMOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->max_tokens) * c->top_k > (1LL << 30)) return LMOE_ERR_UNSUPPORTED;
  if (c->use_latent_norm && !(c->norm_eps >= 0.f)) return LMOE_ERR_INVALID_ARG;
  if (c->act_format != LMOE_ACT_FMT_E4M3 && c->act_format != LMOE_ACT_FMT_E2M1) return LMOE_ERR_INVALID_ARG;
  if (c->act_terms < 0 || c->act_terms > (c->act_format == LMOE_ACT_FMT_E2M1 ? 4 : 2)) return LMOE_ERR_INVALID_ARG;
  if (c->act_terms == 1 && c->expert_wfmt != LMOE_W_MXFP4) return LMOE_ERR_UNSUPPORTED;
  if (c->act_format == LMOE_ACT_FMT_E2M1 && c->expert_wfmt != LMOE_W_MXFP4) return LMOE_ERR_UNSUPPORTED;
  if (c->ep_size < 0 || c->ep_rank < 0 || c->max_recv_rows < 0) return LMOE_ERR_INVALID_ARG;
  if (c->ep_size > 1 && (c->ep_rank >= c->ep_size || c->n_experts % c->ep_size)) return LMOE_ERR_INVALID_ARG;
  if (c->ep_size > 1 && c->act_format == LMOE_ACT_FMT_E2M1) return LMOE_ERR_UNSUPPORTED;
  return LMOE_OK;
}

lmoe_status validate_weights(const lmoe_config* c, const lmoe_weights* w) {
  const void* need16[] = {w->router_w, w->router_bias};
  for (const void* p : need16)
    if (!p || !aligned(p, 16)) return LMOE_ERR_INVALID_ARG;
  if (c->d_latent) {
    const void* lat[] = {w->w_down_latent, w->w_up_latent};
    for (const void* p : lat)
      if (!p || !aligned(p, 16)) return LMOE_ERR_INVALID_ARG;
  }
  if (c->use_latent_norm && (!w->norm_w || !aligned(w->norm_w, 16))) return LMOE_ERR_INVALID_ARG;
  const void* need32[] = {w->ex_gate_q, w->ex_up_q, w->ex_down_q, w->ex_gate_s, w->ex_up_s, w->ex_down_s};
  for (const void* p : need32)
    if (!p || !aligned(p, 32)) return LMOE_ERR_INVALID_ARG;
  if (c->d_shared_ff) {
    const void* sh[] = {w->sh_gate, w->sh_up, w->sh_down};
    for (const void* p : sh)
      if (!p || !aligned(p, 16)) return LMOE_ERR_INVALID_ARG;
    if (c->expert_wfmt == LMOE_W_FP8_BLOCK128) {
      const void* shs[] = {w->sh_gate_s, w->sh_up_s, w->sh_down_s};
      for (const void* p : shs)
        if (!p || !aligned(p, 16)) return LMOE_ERR_INVALID_ARG;
    }
  }
  return LMOE_OK;
}

}  // namespace

extern "C" {

const char* lmoe_status_string(lmoe_status s) {
  switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_INVALID_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case LMOE_ERR_CUDA: return "CUDA error";
    case LMOE_ERR_OOM: return "out of device memory";
    case LMOE_ERR_TIMEOUT: return "kernel wait timed out";
  }
  return "unknown status";
}

lmoe_status lmoe_create(const lmoe_config* cfg, const lmoe_weights* w, cudaStream_t stream, lmoe_handle* out) {
  if (!out) return LMOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w) return LMOE_ERR_INVALID_ARG;
  lmoe_status vs = validate_cfg(cfg);
  if (vs != LMOE_OK) return vs;
  vs = validate_weights(cfg, w);
  if (vs != LMOE_OK) return vs;

  int dev = 0;
  LMOE_TRY(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  LMOE_TRY(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return LMOE_ERR_UNSUPPORTED;   // built for sm_103a only
  if (!encode_tiled_fn()) return LMOE_ERR_CUDA;

  lmoe_ctx* h = new (std::nothrow) lmoe_ctx();
  if (!h) return LMOE_ERR_OOM;
  h->cfg = *cfg;
  h->w = *w;
  h->dev = dev;
  h->num_sms = prop.multiProcessorCount;
  h->d = cfg->d_model;
  h->din = cfg->d_latent;
  h->E = cfg->n_experts;
  h->k = cfg->top_k;
  h->F = cfg->d_expert_ff;
  h->Fs = cfg->d_shared_ff;
  h->dx = h->din ? h->din : h->d;
  h->fp8 = cfg->expert_wfmt == LMOE_W_FP8_BLOCK128;
  h->fp4 = cfg->act_format == LMOE_ACT_FMT_E2M1;
  h->terms = h->fp4 ? (cfg->act_terms ? cfg->act_terms : 3) : (cfg->act_terms == 1 ? 1 : 2);
  // contraction lengths of the expert GEMMs, padded to their K group (256 for packed 4-bit rows)
  h->Kp = static_cast<int>(align_up(h->dx, h->fp4 ? 256 : 128));
  h->Fp = static_cast<int>(align_up(h->F, h->fp4 ? 256 : 128));
  h->MT_gu = h->Fp / 128;
  h->MT_dn = ceil_div(h->dx, 128);
  h->MTa_gu = (h->MT_gu + 1) / 2 * 2;
  h->MTa_dn = (h->MT_dn + 3) / 4 * 4;   // the down pass copies the atoms of up to four 128-row tiles per stage
  h->KG_gu = h->Kp / 128;
  h->KG_dn = h->Fp / 128;
  h->Tm = cfg->max_tokens;
  h->Pm = h->Tm * h->k;
  h->ep = cfg->ep_size > 1 ? cfg->ep_size : 1;
  h->ep_rank = h->ep > 1 ? cfg->ep_rank : 0;
  h->E_loc = h->E / h->ep;
  // rows the expert GEMMs may see: the batch's own assignments, or under
  // expert parallelism the rows received from every rank
  h->Pexp = h->ep > 1 ? static_cast<int>(cfg->max_recv_rows ? cfg->max_recv_rows
                                                            : std::min<long long>(1LL << 30, 1LL * h->ep * h->Pm))
                      : h->Pm;
  const int bn_max = expert_bn_rows(h, h->Pexp);
  h->Ppad = h->Pexp + h->E_loc * (bn_max - 1);
  h->max_tiles = std::max(h->Pexp / 16 + h->E_loc, h->Pm / 16 + h->E) + 1;
  h->nchunks_max = ceil_div(std::max(h->Pm, h->Pexp), kDispatchChunk);

  // dense partial buffer: max over the four GEMMs of splits * T * ld
  long long part_elems = 0;
  {
    const int nkb_d = ceil_div(h->d, 64);
    part_elems =
        std::max(part_elems, max_split_rows(ceil_div(h->E, 128), 0, nkb_d, h->Tm, h->num_sms, false) * h->E);
    if (h->Fs)
      part_elems = std::max(part_elems,
                            max_split_rows(ceil_div(h->Fs, 128), ceil_div(h->Fs, 128), nkb_d, h->Tm, h->num_sms,
                                           true) * 2LL * h->Fs);
    const int nkb_o = ceil_div(h->din, 64) + (h->Fs ? ceil_div(h->Fs, 64) : 0);
    part_elems = std::max(part_elems, max_split_rows(ceil_div(h->d, 128), 0, nkb_o, h->Tm, h->num_sms, true) * h->d);
  }
  const long long part_sh_elems = std::max(
      h->Fs ? max_split_rows(ceil_div(h->Fs, 128), ceil_div(h->Fs, 128), ceil_div(h->d, 64), h->Tm, h->num_sms, true) *
                  2LL * h->Fs
            : 0LL,
      h->din ? max_split_rows(ceil_div(h->din, 128), 0, ceil_div(h->d, 64), h->Tm, h->num_sms, true) * h->din : 0LL);
  // activation scale atoms per 16-row tile and 128 K: two E4M3 terms, or up to four E2M1 terms
  const int atoms_per = h->fp4 ? 4 : 2;
  const size_t xsf_bytes = static_cast<size_t>(ceil_div(h->Ppad, 16)) * h->KG_gu * atoms_per * 512;
  const size_t hsf_bytes = static_cast<size_t>(ceil_div(h->Ppad, 16)) * h->KG_dn * atoms_per * 512;
  const bool pad_gu = !h->fp8 && h->Kp != h->dx, pad_dn = !h->fp8 && h->Fp != h->F;
  const size_t sfa_gu_bytes = h->fp8 ? 0 : static_cast<size_t>(h->E_loc) * h->MTa_gu * h->KG_gu * 512;
  const size_t sfa_dn_bytes = h->fp8 ? 0 : static_cast<size_t>(h->E_loc) * h->MTa_dn * h->KG_dn * 512;
  const bool sh8 = h->fp8 && h->Fs;   // shared expert on the FP8 expert GEMMs
  h->Tpad_sh = sh8 ? h->Tm + kFp8MaxTile : 0;
  // K-split scratch: partial gate/up sums, arrival counters (fewer than
  // 4 * SMs items when split), and room for the down pass's partial planes
  long long gpart_elems = 0, y_rows = std::max(h->Pm, h->Pexp);
  for (long long P = 1; P <= std::min<long long>(h->Pexp, kKsplitMaxP); ++P) {
    const int kg = expert_ksplit(h, P, true), kd = expert_ksplit(h, P, false);
    if (kg > 1) gpart_elems = std::max(gpart_elems, 2LL * kg * P * h->F);
    y_rows = std::max(y_rows, static_cast<long long>(kd) * P);
  }
  h->n_gcnt = gpart_elems ? 4 * 4 * h->num_sms : 0;

  auto carve = [&](char* base) {
    Carve c;
    h->err = c.take<int>(4, base);
    h->sched = c.take<int>(4, base);
    h->part = c.take<float>(static_cast<size_t>(part_elems), base);
    h->part_sh = c.take<float>(static_cast<size_t>(part_sh_elems), base);
    h->xc = c.take<float>(static_cast<size_t>(h->Tm) * h->din, base);
    h->logits = c.take<float>(static_cast<size_t>(h->Tm) * h->E, base);
    h->idx = c.take<int32_t>(h->Pm, base);
    h->G = c.take<float>(h->Pm, base);
    h->counts = c.take<int32_t>(h->E, base);
    h->offsets = c.take<int32_t>(h->E + 1, base);
    h->tile_off = c.take<int32_t>(h->E + 1, base);
    h->perm = c.take<int32_t>(std::max(h->Pm, h->Pexp), base);
    h->inv_pad = c.take<int32_t>(std::max(h->Pm, h->Pexp), base);
    h->blockcnt = c.take<int32_t>(static_cast<size_t>(h->nchunks_max) * h->E, base);
    // expert-parallel phases (also on a single rank, where they run every expert locally)
    h->ep_perm = c.take<int32_t>(h->Pm, base);
    h->idx_loc = c.take<int32_t>(h->Pexp, base);
    h->ones = c.take<float>(h->Pexp, base);
    h->ntiles = c.take<int32_t>(1, base);
    h->tiles = c.take<int4>(h->max_tiles, base);
    h->xq = c.take<uint8_t>(2 * static_cast<size_t>(h->Ppad) * h->Kp, base);
    h->xsf = c.take<uint8_t>(xsf_bytes, base);
    h->hq = c.take<uint8_t>(2 * static_cast<size_t>(h->Ppad) * h->Fp, base);
    h->hsf = c.take<uint8_t>(hsf_bytes, base);
    h->y = c.take<float>(static_cast<size_t>(y_rows) * h->dx, base);
    h->u = c.take<float>(static_cast<size_t>(h->Tm) * h->dx, base);
    h->u_hat = c.take<uint16_t>(static_cast<size_t>(h->Tm) * h->dx, base);
    h->h_s = c.take<uint16_t>(static_cast<size_t>(h->Tm) * std::max(h->Fs, 1), base);
    h->x_stage = c.take<uint16_t>(static_cast<size_t>(h->Tm) * h->d, base);
    h->out_stage = c.take<uint16_t>(static_cast<size_t>(h->Tm) * h->d, base);
    h->sfa_gate = c.take<uint8_t>(sfa_gu_bytes, base);
    h->sfa_up = c.take<uint8_t>(sfa_gu_bytes, base);
    h->sfa_down = c.take<uint8_t>(sfa_dn_bytes, base);
    if (h->Fs && !sh8)
      h->sh_gu_il = c.take<uint16_t>(2 * static_cast<size_t>(ceil_div(h->Fs, 128)) * 128 * h->d, base);
    if (sh8) {
      const size_t tiles_max = static_cast<size_t>(h->Tpad_sh / 16 + 1);
      h->sh_tiles = c.take<int4>(tiles_max, base);
      h->sh_tile_off = c.take<int32_t>(2, base);
      h->sh_ntiles = c.take<int32_t>(1, base);
      h->sh_iota = c.take<int32_t>(h->Tm, base);
      h->sh_ones = c.take<float>(h->Tm, base);
      h->xq_sh = c.take<uint8_t>(2 * static_cast<size_t>(h->Tpad_sh) * h->d, base);
      h->xsf_sh = c.take<uint8_t>(tiles_max * (h->d / 128) * 1024, base);
      h->hq_sh = c.take<uint8_t>(2 * static_cast<size_t>(h->Tpad_sh) * h->Fs, base);
      h->hsf_sh = c.take<uint8_t>(tiles_max * (h->Fs / 128) * 1024, base);
      h->y_sh = c.take<float>(static_cast<size_t>(h->Tm) * h->d, base);
    }
    if (pad_gu) {
      h->pad_gate = c.take<uint8_t>(static_cast<size_t>(h->E_loc) * h->F * (h->Kp / 2), base);
      h->pad_up = c.take<uint8_t>(static_cast<size_t>(h->E_loc) * h->F * (h->Kp / 2), base);
    }
    if (pad_dn) h->pad_down = c.take<uint8_t>(static_cast<size_t>(h->E_loc) * h->din * (h->Fp / 2), base);
    h->qb_alpha = c.take<float>(h->Tm, base);
    h->qb_raw = c.take<float>(h->E, base);
    h->qb_range = c.take<float>(2, base);
    h->gpart = c.take<float>(static_cast<size_t>(gpart_elems), base);
    h->gcnt = c.take<int>(static_cast<size_t>(std::max(h->n_gcnt, 1)), base);
    return c.off;
  };
  h->pool_bytes = carve(nullptr);
  cudaError_t ae = cudaMalloc(&h->pool, h->pool_bytes);
  if (ae != cudaSuccess) {
    delete h;
    return ae == cudaErrorMemoryAllocation ? LMOE_ERR_OOM : LMOE_ERR_CUDA;
  }
  carve(static_cast<char*>(h->pool));

  auto fail = [&](lmoe_status s) {
    if (h->side) cudaStreamDestroy(h->side);
    if (h->ev_fork) cudaEventDestroy(h->ev_fork);
    if (h->ev_latent) cudaEventDestroy(h->ev_latent);
    if (h->ev_join) cudaEventDestroy(h->ev_join);
    cudaFree(h->pool);
    delete h;
    return s;
  };
  if (cudaMemsetAsync(h->err, 0, 4 * sizeof(int), stream) != cudaSuccess ||
      cudaMemsetAsync(h->sched, 0, 4 * sizeof(int), stream) != cudaSuccess ||
      cudaMemsetAsync(h->gcnt, 0, std::max(h->n_gcnt, 1) * sizeof(int), stream) != cudaSuccess)
    return fail(LMOE_ERR_CUDA);
  if ((h->Fs || h->din) && (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
                            cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
                            cudaEventCreateWithFlags(&h->ev_latent, cudaEventDisableTiming) != cudaSuccess ||
                            cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess))
    return fail(LMOE_ERR_CUDA);
  // expert weights: scale atoms, K padding when a reduction dim is not a multiple of 128
  const uint8_t* sg = static_cast<const uint8_t*>(w->ex_gate_s);
  const uint8_t* su = static_cast<const uint8_t*>(w->ex_up_s);
  const uint8_t* sd = static_cast<const uint8_t*>(w->ex_down_s);
  if (!h->fp8 &&
      (launch_relayout_sfa(sg, h->E_loc, h->F, h->dx / 32, h->MTa_gu, h->KG_gu, h->sfa_gate, stream) != cudaSuccess ||
       launch_relayout_sfa(su, h->E_loc, h->F, h->dx / 32, h->MTa_gu, h->KG_gu, h->sfa_up, stream) != cudaSuccess ||
       launch_relayout_sfa(sd, h->E_loc, h->dx, h->F / 32, h->MTa_dn, h->KG_dn, h->sfa_down, stream) != cudaSuccess))
    return fail(LMOE_ERR_CUDA);
  if (sh8 && launch_iota_ones(h->sh_iota, h->sh_ones, h->Tm, stream) != cudaSuccess) return fail(LMOE_ERR_CUDA);
  if (h->ones && launch_iota_ones(h->idx_loc, h->ones, h->Pexp, stream) != cudaSuccess) return fail(LMOE_ERR_CUDA);
  if (h->sh_gu_il && launch_interleave_gate_up(w->sh_gate, w->sh_up, h->Fs, h->d, h->sh_gu_il, stream) != cudaSuccess)
    return fail(LMOE_ERR_CUDA);
  h->codes_gate = w->ex_gate_q;
  h->codes_up = w->ex_up_q;
  h->codes_down = w->ex_down_q;
  if (pad_gu) {
    if (launch_pad_codes(w->ex_gate_q, h->E_loc, h->F, h->din, h->Kp, h->pad_gate, stream) != cudaSuccess ||
        launch_pad_codes(w->ex_up_q, h->E_loc, h->F, h->din, h->Kp, h->pad_up, stream) != cudaSuccess)
      return fail(LMOE_ERR_CUDA);
    h->codes_gate = h->pad_gate;
    h->codes_up = h->pad_up;
  }
  if (pad_dn) {
    if (launch_pad_codes(w->ex_down_q, h->E_loc, h->din, h->F, h->Fp, h->pad_down, stream) != cudaSuccess)
      return fail(LMOE_ERR_CUDA);
    h->codes_down = h->pad_down;
  }
  bool ok = true;
  ok &= map_bf16(&h->m_router, w->router_w, h->d, h->E, 128);
  if (h->din) {
    ok &= map_bf16(&h->m_wdown, w->w_down_latent, h->d, h->din, 128);
    ok &= map_bf16(&h->m_wup, w->w_up_latent, h->din, h->d, 128);
  }
  if (h->Fs && !sh8) {
    ok &= map_bf16(&h->m_shg, w->sh_gate, h->d, h->Fs, 128);
    ok &= map_bf16(&h->m_shu, w->sh_up, h->d, h->Fs, 128);
    ok &= map_bf16(&h->m_shd, w->sh_down, h->Fs, h->d, 128);
  }
  if (sh8) {
    ok &= map_u8(&h->m_sg, w->sh_gate, h->d, h->Fs, kFp8Rows);
    ok &= map_u8(&h->m_su, w->sh_up, h->d, h->Fs, kFp8Rows);
    ok &= map_u8(&h->m_sd, w->sh_down, h->Fs, h->d, kFp8Rows);
  }
  ok &= map_bf16(&h->m_routerw, w->router_w, h->d, h->E, 256);
  if (h->din) {
    ok &= map_bf16(&h->m_wdownw, w->w_down_latent, h->d, h->din, 256);
    ok &= map_bf16(&h->m_wupw, w->w_up_latent, h->din, h->d, 256);
  }
  if (h->Fs && !sh8) {
    ok &= map_bf16(&h->m_shgu_il, h->sh_gu_il, h->d, 2 * ceil_div(h->Fs, 128) * 128, 256);
    ok &= map_bf16(&h->m_shdw, w->sh_down, h->Fs, h->d, 256);
  }
  for (int i = 0; i < 2; ++i) {
    const int rows = 128 << i;
    if (h->fp8) {
      ok &= map_u8(&h->m_exg[i], h->codes_gate, h->Kp, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_u8(&h->m_exu[i], h->codes_up, h->Kp, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_u8(&h->m_exd[i], h->codes_down, h->Fp, static_cast<long long>(h->E_loc) * h->dx, rows);
    } else if (h->fp4) {   // packed codes as bytes: a 128-byte box row is 256 K values
      ok &= map_u8(&h->m_exg[i], h->codes_gate, h->Kp / 2, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_u8(&h->m_exu[i], h->codes_up, h->Kp / 2, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_u8(&h->m_exd[i], h->codes_down, h->Fp / 2, static_cast<long long>(h->E_loc) * h->dx, rows);
    } else {
      ok &= map_fp4(&h->m_exg[i], h->codes_gate, h->Kp, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_fp4(&h->m_exu[i], h->codes_up, h->Kp, static_cast<long long>(h->E_loc) * h->F, rows);
      ok &= map_fp4(&h->m_exd[i], h->codes_down, h->Fp, static_cast<long long>(h->E_loc) * h->dx, rows);
    }
  }
  if (!ok) return fail(LMOE_ERR_CUDA);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return fail(LMOE_ERR_CUDA);
  if (cudaGetLastError() != cudaSuccess) return fail(LMOE_ERR_CUDA);
  *out = h;
  return LMOE_OK;
}

lmoe_status lmoe_destroy(lmoe_handle h) {
  if (!h) return LMOE_OK;
  cudaError_t e = cudaDeviceSynchronize();
  release_events(h);
  for (cudaEvent_t ev : h->ev_free) cudaEventDestroy(ev);
  if (h->side) cudaStreamDestroy(h->side);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_latent) cudaEventDestroy(h->ev_latent);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->delta32) cudaFree(h->delta32);
  cudaFree(h->pool);
  delete h;
  return e == cudaSuccess ? LMOE_OK : LMOE_ERR_CUDA;
}

lmoe_status lmoe_keep_f32_output(lmoe_handle h, int enable) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  if (enable && !h->delta32) {
    LMOE_TRY(cudaDeviceSynchronize());
    LMOE_TRY(cudaMalloc(&h->delta32, static_cast<size_t>(h->Tm) * h->d * sizeof(float)));
  } else if (!enable && h->delta32) {
    LMOE_TRY(cudaDeviceSynchronize());
    LMOE_TRY(cudaFree(h->delta32));
    h->delta32 = nullptr;
  }
  return LMOE_OK;
}

// Inputs of a quantile-balancing call: the given logits, or those of the
// handle's last forward (T must then be its token count), and the given
// biases or the handle's router bias.
static lmoe_status qb_inputs(lmoe_ctx* h, const float*& logits, int T, const float*& bias) {
  if (T < 1 || T > h->Tm || h->k >= h->E) return LMOE_ERR_INVALID_ARG;
  if (!logits) {
    if (T != h->last_T) return LMOE_ERR_INVALID_ARG;
    logits = h->logits;
  }
  if (!bias) bias = h->w.router_bias;
  return LMOE_OK;
}

lmoe_status lmoe_qb_update(lmoe_handle h, const float* logits, int T, const float* bias, float* new_bias,
                           cudaStream_t st) {
  if (!h || !new_bias) return LMOE_ERR_INVALID_ARG;
  const lmoe_status s = qb_inputs(h, logits, T, bias);
  if (s != LMOE_OK) return s;
  LMOE_TRY(launch_qb_update(logits, T, h->E, h->k, bias, h->qb_alpha, h->qb_raw, new_bias, st));
  return LMOE_OK;
}

lmoe_status lmoe_qb_histogram(lmoe_handle h, const float* logits, int T, const float* bias, int bins,
                              int32_t* counts, cudaStream_t st) {
  if (!h || !counts || bins < 1 || bins > (1 << 20)) return LMOE_ERR_INVALID_ARG;
  const lmoe_status s = qb_inputs(h, logits, T, bias);
  if (s != LMOE_OK) return s;
  LMOE_TRY(launch_qb_histogram(logits, T, h->E, h->k, bias, bins, h->qb_alpha, h->qb_range, counts, st));
  return LMOE_OK;
}

lmoe_status lmoe_qb_update_from_histogram(lmoe_handle h, const int32_t* counts, int bins, const float* bias,
                                          float* new_bias, cudaStream_t st) {
  if (!h || !counts || !new_bias || bins < 1 || bins > (1 << 20) || h->k >= h->E) return LMOE_ERR_INVALID_ARG;
  if (!bias) bias = h->w.router_bias;
  LMOE_TRY(launch_qb_from_histogram(counts, h->E, bins, h->k, bias, h->qb_range, h->qb_raw, new_bias, st));
  return LMOE_OK;
}

lmoe_status lmoe_selftest_timeout(lmoe_handle h, unsigned long long limit_ns, cudaStream_t st) {
  if (!h || limit_ns < 1000ull || limit_ns > 1000000000ull) return LMOE_ERR_INVALID_ARG;
  LMOE_TRY(launch_wait_timeout_probe(h->err, limit_ns, st));
  return LMOE_OK;
}

lmoe_status lmoe_route(lmoe_handle h, const void* x, int T, int32_t* topk_idx, float* topk_w, cudaStream_t st) {
  if (!h || T < 0 || T > h->Tm) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !aligned(x, 16) || !topk_idx || !topk_w) return LMOE_ERR_INVALID_ARG;
  int launches = 0;
  begin_call(h);
  lmoe_status s = run_router(h, x, T, st, launches);
  if (s != LMOE_OK) return s;
  const size_t n = static_cast<size_t>(T) * h->k;
  LMOE_TRY(cudaMemcpyAsync(topk_idx, h->idx, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
  LMOE_TRY(cudaMemcpyAsync(topk_w, h->G, n * sizeof(float), cudaMemcpyDeviceToDevice, st));
  return LMOE_OK;
}

lmoe_status lmoe_dispatch(lmoe_handle h, const int32_t* topk_idx, int T, int32_t* counts, int32_t* offsets,
                          int32_t* perm, cudaStream_t st) {
  if (!h || T < 0 || T > h->Tm) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!topk_idx || !counts || !offsets || !perm) return LMOE_ERR_INVALID_ARG;
  int launches = 0;
  begin_call(h);
  return run_dispatch(h, topk_idx, T, expert_bn(h, T), counts, offsets, perm, st, launches);
}

// Steps 4 and 9 on the handle's side stream, forked from `st`: the latent
// down-projection (ev_latent) and the shared expert (ev_join), which need
// only x and overlap the router, dispatch and routed experts.
static lmoe_status run_side(lmoe_ctx* h, const void* x, int T, cudaStream_t st, int& launches) {
  const int d = h->d, din = h->din, Fs = h->Fs;
  const int BN = dense_bn(T);
  const int nt = ceil_div(T, BN);
  const int nkb_d = ceil_div(d, 64);
  cudaStream_t ss = h->side;
  if (ss) {
    LMOE_TRY(cudaEventRecord(h->ev_fork, st));
    LMOE_TRY(cudaStreamWaitEvent(ss, h->ev_fork, 0));
  }
  // 4 latent down-projection (latent layers only)
  if (din) {
    StageTimer tm(h, LMOE_STAGE_LATENT_DOWN, ss);
    DenseParams p;
    std::memset(&p, 0, sizeof(p));
    p.a0 = h->m_wdown;
    p.a0w = h->m_wdownw;
    if (!map_bf16(&p.b0, x, d, T, BN)) return LMOE_ERR_CUDA;
    p.mode = 0;
    p.M0 = din;
    p.mtiles0 = ceil_div(din, 128);
    p.T = T;
    p.nkb = nkb_d;
    p.nkb0 = nkb_d;
    const DensePlan pl = dense_plan(p.mtiles0, 0, nt, nkb_d, BN, h->num_sms, true);
    p.splits = pl.splits;
    p.wide = pl.wide;
    p.ldo = din;
    p.out = p.splits == 1 ? h->xc : h->part_sh;
    p.err = h->err;
    LMOE_TRY(launch_dense_gemm(p, p.mtiles0, BN, ss));
    ++launches;
    if (p.splits > 1) {
      LMOE_TRY(launch_finalize_sum_f32(h->part_sh, p.splits, T, din, din, h->xc, din, ss));
      ++launches;
    }
    tm.done();
    LMOE_TRY(cudaEventRecord(h->ev_latent, ss));
  }
  // 9 (FP8 layers) the shared expert on the FP8 expert GEMMs: one expert that
  // every token uses, output y_sh [T][d] fp32
  if (Fs && h->fp8) {
    StageTimer tm(h, LMOE_STAGE_SHARED, ss);
    const int BNs = fp8_tile_tokens(T, 1);
    LMOE_TRY(launch_shared_tiles(T, BNs, h->sh_tiles, h->sh_tile_off, h->sh_ntiles, ss));
    LMOE_TRY(launch_quant_gather_bf16(x, T, 1, d, d, h->sh_iota, BNs, 1, 2, h->xq_sh, h->xsf_sh, h->sched + 2, nullptr,
                                      0, ss));
    MoeGemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.a_gate = h->m_sg;
    p.a_up = h->m_su;
    if (!map_u8(&p.b, h->xq_sh, d, 2LL * h->Tpad_sh, 2 * BNs)) return LMOE_ERR_CUDA;
    p.sfb = h->xsf_sh;
    p.tiles = h->sh_tiles;
    p.tile_off = h->sh_tile_off;
    p.ntiles = h->sh_ntiles;
    p.perm = h->sh_iota;
    p.G = h->sh_ones;
    p.err = h->err;
    p.sched = h->sched + 2;
    p.KS = 1;
    p.terms = 2;
    p.N_out = Fs;
    p.MT = Fs / kFp8Rows;
    p.KG = d / 128;
    p.hq = h->hq_sh;
    p.hsf = h->hsf_sh;
    p.Fp = Fs;
    p.act = h->cfg.act == LMOE_ACT_SWIGLU ? 1 : 0;
    p.b1 = h->cfg.situ_beta;
    p.b2 = h->cfg.situ_linear_beta;
    p.wsc0 = static_cast<const float*>(h->w.sh_gate_s);
    p.wsc1 = static_cast<const float*>(h->w.sh_up_s);
    p.NB = Fs / 128;
    p.KB = d / 128;
    LMOE_TRY(launch_moe_fp8_gate_up(p, BNs, h->num_sms, ss));
    MoeGemmParams q = p;
    q.a_gate = h->m_sd;
    if (!map_u8(&q.b, h->hq_sh, Fs, 2LL * h->Tpad_sh, 2 * BNs)) return LMOE_ERR_CUDA;
    q.sfb = h->hsf_sh;
    q.sched = h->sched + 3;
    q.N_out = d;
    q.MT = ceil_div(d, 2 * kFp8Rows);
    q.KG = Fs / 128;
    q.y = h->y_sh;
    q.wsc0 = static_cast<const float*>(h->w.sh_down_s);
    q.wsc1 = nullptr;
    q.NB = d / 128;
    q.KB = Fs / 128;
    LMOE_TRY(launch_moe_fp8_down(q, BNs, h->num_sms, ss));
    launches += 4;
    tm.done();
    LMOE_TRY(cudaEventRecord(h->ev_join, ss));
  }
  // 9 shared experts gate/up + SiTU (bf16 shared MLP)
  if (Fs && !h->fp8) {
    StageTimer tm(h, LMOE_STAGE_SHARED, ss);
    DenseParams p;
    std::memset(&p, 0, sizeof(p));
    p.a0 = h->m_shg;
    p.a1 = h->m_shu;
    p.a0w = h->m_shgu_il;   // wide: the gate/up tile pair as one 256-row box
    if (!map_bf16(&p.b0, x, d, T, BN)) return LMOE_ERR_CUDA;
    p.mode = 1;
    p.M0 = Fs;
    p.M1 = Fs;
    p.mtiles0 = ceil_div(Fs, 128);
    p.T = T;
    p.nkb = nkb_d;
    p.nkb0 = nkb_d;
    const DensePlan pl = dense_plan(p.mtiles0, p.mtiles0, nt, nkb_d, BN, h->num_sms, true);
    p.splits = pl.splits;
    p.wide = pl.wide;
    p.err = h->err;
    if (p.wide && p.splits == 1) {
      // gate and up tiles of the same features in one CTA: the epilogue writes h_shared
      p.epi = 2;
      p.out16 = h->h_s;
      p.ldo = Fs;
      p.act = h->cfg.act == LMOE_ACT_SWIGLU ? 1 : 0;
      p.act_b1 = h->cfg.situ_beta;
      p.act_b2 = h->cfg.situ_linear_beta;
      LMOE_TRY(launch_dense_gemm(p, 2 * p.mtiles0, BN, ss));
      ++launches;
    } else {
      p.ldo = 2 * Fs;
      p.out = h->part_sh;
      LMOE_TRY(launch_dense_gemm(p, 2 * p.mtiles0, BN, ss));
      LMOE_TRY(launch_finalize_glu_bf16(h->part_sh, p.splits, T, Fs, 2 * Fs, h->h_s,
                                        h->cfg.act == LMOE_ACT_SWIGLU ? 1 : 0, h->cfg.situ_beta,
                                        h->cfg.situ_linear_beta, ss));
      launches += 2;
    }
    tm.done();
    LMOE_TRY(cudaEventRecord(h->ev_join, ss));
  }
  return LMOE_OK;
}

// Steps 6-7: the grouped gate/up and down GEMMs over the tiles of the last
// dispatch (P rows, routing weights G per row); the K splits of the down pass
// (planes of P x dx in y) are returned in KSd.
static lmoe_status run_experts(lmoe_ctx* h, long long P, int BNm, int split, const float* G, cudaStream_t st, int& launches,
                        int& KSd) {
  const int dx = h->dx;
  KSd = expert_ksplit(h, P, false);
  {
    MoeGemmParams p;
    std::memset(&p, 0, sizeof(p));
    const int RB = h->fp8 ? kFp8Rows : moe_rows_per_item(BNm);
    const int mi = RB == 256 ? 1 : 0;
    p.a_gate = h->m_exg[mi];
    p.a_up = h->m_exu[mi];
    // activation rows per tile: hi and lo (2 BN), or the BN hi rows of a split tile in the one-term form;
    // packed 4-bit terms: one box of BN rows per term
    const int b_rows = h->fp4 ? BNm : (split && h->terms == 1) ? BNm : 2 * BNm;
    if (h->fp4) {
      if (!map_u8(&p.b, h->xq, h->Kp / 2, static_cast<long long>(h->terms) * h->Ppad, b_rows)) return LMOE_ERR_CUDA;
    } else if (!map_u8(&p.b, h->xq, h->Kp, 2LL * h->Ppad, b_rows)) {
      return LMOE_ERR_CUDA;
    }
    p.terms = h->terms;
    p.sfa_gate = h->sfa_gate;
    p.sfa_up = h->sfa_up;
    p.sfb = h->xsf;
    p.tiles = h->tiles;
    p.tile_off = h->tile_off;
    p.ntiles = h->ntiles;
    p.perm = h->perm;
    p.G = G;
    p.err = h->err;
    p.sched = h->sched;
    p.KS = expert_ksplit(h, P, true);
    p.gpart = h->gpart;
    p.gcnt = h->gcnt;
    p.P = static_cast<int>(P);
    p.N_out = h->F;
    p.MT = ceil_div(h->F, RB);
    p.MTa = h->MTa_gu;
    p.KG = h->fp4 ? h->Kp / 256 : h->KG_gu;
    p.hq = h->hq;
    p.hsf = h->hsf;
    p.Fp = h->Fp;
    p.act = h->cfg.act == LMOE_ACT_SWIGLU ? 1 : 0;
    p.b1 = h->cfg.situ_beta;
    p.b2 = h->cfg.situ_linear_beta;
    p.y = h->y;
    p.wsc0 = static_cast<const float*>(h->w.ex_gate_s);
    p.wsc1 = static_cast<const float*>(h->w.ex_up_s);
    p.NB = ceil_div(h->F, 128);
    p.KB = ceil_div(dx, 128);
    if (!h->fp8 && !h->fp4 && p.KS > 1) {
      // a few tokens: the down weights of the first experts go to L2 while the gate/up pass drains
      p.pf_codes = h->codes_down;
      p.pf_code_bytes = static_cast<size_t>(dx) * (h->Fp / 2);
      p.pf_atoms = h->sfa_down;
      p.pf_atom_bytes = static_cast<size_t>(h->MTa_dn) * h->KG_dn * 512;
      p.pf_budget = kDownPrefetchBytes;
    }
    StageTimer tgu(h, LMOE_STAGE_EXPERT_GU, st);
    LMOE_TRY(h->fp8   ? launch_moe_fp8_gate_up(p, BNm, h->num_sms, st)
             : h->fp4 ? launch_moe_fp4_gate_up(p, BNm, h->num_sms, st)
                      : launch_moe_gate_up(p, BNm, h->num_sms, st));
    ++launches;
    tgu.done();
    MoeGemmParams q = p;
    q.pf_codes = nullptr;
    q.a_gate = h->m_exd[mi];
    if (h->fp4) {
      if (!map_u8(&q.b, h->hq, h->Fp / 2, static_cast<long long>(h->terms) * h->Ppad, b_rows)) return LMOE_ERR_CUDA;
    } else if (!map_u8(&q.b, h->hq, h->Fp, 2LL * h->Ppad, b_rows)) {
      return LMOE_ERR_CUDA;
    }
    q.sfa_gate = h->sfa_down;
    q.sfa_up = nullptr;
    q.sfb = h->hsf;
    q.sched = h->sched + 1;
    q.KS = KSd;
    q.y_plane = static_cast<size_t>(P) * dx;
    q.N_out = dx;
    q.MT = ceil_div(dx, 2 * RB);
    q.MTa = h->MTa_dn;
    q.KG = h->fp4 ? h->Fp / 256 : h->KG_dn;
    q.wsc0 = static_cast<const float*>(h->w.ex_down_s);
    q.wsc1 = nullptr;
    q.NB = ceil_div(dx, 128);
    q.KB = ceil_div(h->F, 128);
    StageTimer tdn(h, LMOE_STAGE_EXPERT_DOWN, st);
    LMOE_TRY(h->fp8   ? launch_moe_fp8_down(q, BNm, h->num_sms, st)
             : h->fp4 ? launch_moe_fp4_down(q, BNm, h->num_sms, st)
                      : launch_moe_down(q, BNm, h->num_sms, st));
    ++launches;
    tdn.done();
  }
  return LMOE_OK;
}

// Steps 8 and 10: the slot-ordered sum of y (KSd planes) with the latent
// RMSNorm, then Delta = u_hat W_up^T + h_shared W_shared_down^T (latent
// layers) or the routed sum plus the shared expert (non-latent layers).
static lmoe_status run_combine_output(lmoe_ctx* h, int T, long long P, int KSd, void* out, cudaStream_t st, int& launches) {
  const int d = h->d, din = h->din, dx = h->dx, Fs = h->Fs;
  const int BN = dense_bn(T);
  const int nt = ceil_div(T, BN);
  // 8 expert sum in slot order + latent RMSNorm
  {
    StageTimer tm(h, LMOE_STAGE_COMBINE, st);
    LMOE_TRY(launch_combine_norm(h->y, T, h->k, dx, KSd, static_cast<size_t>(P) * dx, h->w.norm_w,
                                 din && h->cfg.use_latent_norm, h->cfg.norm_eps, h->u, h->u_hat, h->num_sms, st));
    ++launches;
    tm.done();
  }
  // join the shared gate/up GEMM of the side stream before the output GEMM reads h_shared
  if (Fs) LMOE_TRY(cudaStreamWaitEvent(st, h->ev_join, 0));
  // 10 Delta = u_hat W_up^T + h_shared W_shared_down^T
  if (din) {
    StageTimer tm(h, LMOE_STAGE_OUTPUT, st);
    DenseParams p;
    std::memset(&p, 0, sizeof(p));
    p.a0 = h->m_wup;
    p.a0w = h->m_wupw;
    if (!map_bf16(&p.b0, h->u_hat, din, T, BN)) return LMOE_ERR_CUDA;
    p.nkb0 = ceil_div(din, 64);
    p.nkb = p.nkb0;
    p.mode = 0;
    if (Fs) {
      p.mode = 2;
      p.a1 = h->m_shd;
      p.a1w = h->m_shdw;
      if (!map_bf16(&p.b1, h->h_s, Fs, T, BN)) return LMOE_ERR_CUDA;
      p.nkb += ceil_div(Fs, 64);
    }
    p.M0 = d;
    p.mtiles0 = ceil_div(d, 128);
    p.T = T;
    const DensePlan pl = dense_plan(p.mtiles0, 0, nt, p.nkb, BN, h->num_sms, true);
    p.splits = pl.splits;
    p.wide = pl.wide;
    p.ldo = d;
    p.out = h->part;
    p.err = h->err;
    if (p.splits == 1) {   // one K split: the epilogue writes Delta in bf16
      p.epi = 1;
      p.out16 = out;
      p.out32 = h->delta32;
      LMOE_TRY(launch_dense_gemm(p, p.mtiles0, BN, st));
      ++launches;
    } else {
      LMOE_TRY(launch_dense_gemm(p, p.mtiles0, BN, st));
      LMOE_TRY(launch_finalize_sum_bf16(h->part, p.splits, T, d, d, out, d, nullptr, 0, h->delta32, st));
      launches += 2;
    }
    tm.done();
  } else {
    // non-latent layer (Kimi K2 card): Delta = sum_i G_i E_i + y_shared
    StageTimer tm(h, LMOE_STAGE_OUTPUT, st);
    int splits = 0;
    if (Fs && h->fp8) {
      LMOE_TRY(launch_finalize_sum_bf16(h->y_sh, 1, T, d, d, out, d, h->u, d, h->delta32, st));
      ++launches;
      splits = -1;
    }
    if (splits >= 0) {
      LMOE_TRY(launch_finalize_sum_bf16(h->part, splits, T, d, d, out, d, h->u, d, h->delta32, st));
      ++launches;
    }
    tm.done();
  }
  return LMOE_OK;
}

lmoe_status lmoe_forward(lmoe_handle h, const void* x, int T, void* out, int32_t* topk_idx_opt, float* topk_w_opt,
                         cudaStream_t st) {
  if (!h || T < 0 || T > h->Tm) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !out || !aligned(x, 16) || !aligned(out, 16) || x == out) return LMOE_ERR_INVALID_ARG;
  if (h->ep > 1) return LMOE_ERR_UNSUPPORTED;   // expert-parallel handles run the lmoe_ep_* phases
  int launches = 0;
  const int d = h->d, din = h->din;
  begin_call(h);

  LMOE_TRY_STATUS(run_side(h, x, T, st, launches));
  // 1-2 router
  lmoe_status s = run_router(h, x, T, st, launches);
  if (s != LMOE_OK) return s;
  // 3 dispatch
  const int BNm = expert_bn(h, T);
  const int split = h->fp8 || moe_split(BNm);   // activation layout the expert GEMMs read
  s = run_dispatch(h, h->idx, T, BNm, h->counts, h->offsets, h->perm, st, launches);
  if (s != LMOE_OK) return s;

  const int KSg = expert_ksplit(h, static_cast<long long>(T) * h->k, true);
  if (din) LMOE_TRY(cudaStreamWaitEvent(st, h->ev_latent, 0));   // x^c from the side stream
  // 5 activations -> hi/lo E4M3 in expert-tile order
  {
    StageTimer tm(h, LMOE_STAGE_ACT_QUANT, st);
    if (h->fp4)
      LMOE_TRY(launch_quant_gather_fp4(h->xc, T, h->k, din, h->Kp, h->inv_pad, BNm, h->terms, h->xq, h->xsf, h->sched,
                                       h->gcnt, KSg > 1 ? h->n_gcnt : 0, st));
    else if (din)
      LMOE_TRY(launch_quant_gather(h->xc, T, h->k, din, h->Kp, h->inv_pad, BNm, split, h->terms, h->xq, h->xsf,
                                   h->sched, h->gcnt, KSg > 1 ? h->n_gcnt : 0, st));
    else
      LMOE_TRY(launch_quant_gather_bf16(x, T, h->k, d, h->Kp, h->inv_pad, BNm, split, h->terms, h->xq, h->xsf,
                                        h->sched, h->gcnt, KSg > 1 ? h->n_gcnt : 0, st));
    ++launches;
    tm.done();
  }
  const long long P = static_cast<long long>(T) * h->k;
  int KSd = 1;
  LMOE_TRY_STATUS(run_experts(h, P, BNm, split, h->G, st, launches, KSd));
  LMOE_TRY_STATUS(run_combine_output(h, T, P, KSd, out, st, launches));
  const size_t n = static_cast<size_t>(T) * h->k;
  if (topk_idx_opt) LMOE_TRY(cudaMemcpyAsync(topk_idx_opt, h->idx, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
  if (topk_w_opt) LMOE_TRY(cudaMemcpyAsync(topk_w_opt, h->G, n * sizeof(float), cudaMemcpyDeviceToDevice, st));
  h->last_T = T;
  h->last_launches = launches;
  h->last_BN = BNm;
  h->last_split = split;
  return LMOE_OK;
}

lmoe_status lmoe_ep_dispatch(lmoe_handle h, const void* x, int T, void* send_bf16, int32_t* expert_counts,
                             int32_t* topk_idx_opt, float* topk_w_opt, cudaStream_t st) {
  if (!h || T < 0 || T > h->Tm) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x || !aligned(x, 16) || !send_bf16 || !aligned(send_bf16, 16) || !expert_counts || !h->ep_perm)
    return LMOE_ERR_INVALID_ARG;
  int launches = 0;
  begin_call(h);
  LMOE_TRY_STATUS(run_side(h, x, T, st, launches));
  LMOE_TRY_STATUS(run_router(h, x, T, st, launches));
  // group the assignments by global expert: the rows for each rank become contiguous
  LMOE_TRY_STATUS(run_dispatch(h, h->idx, T, 16, expert_counts, h->offsets, h->ep_perm, st, launches));
  if (h->din) LMOE_TRY(cudaStreamWaitEvent(st, h->ev_latent, 0));
  LMOE_TRY(launch_ep_pack(h->din ? h->xc : nullptr, h->din ? nullptr : x, h->dx, h->k, h->ep_perm, T * h->k,
                          send_bf16, st));
  ++launches;
  const size_t n = static_cast<size_t>(T) * h->k;
  if (topk_idx_opt) LMOE_TRY(cudaMemcpyAsync(topk_idx_opt, h->idx, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, st));
  if (topk_w_opt) LMOE_TRY(cudaMemcpyAsync(topk_w_opt, h->G, n * sizeof(float), cudaMemcpyDeviceToDevice, st));
  h->ep_T = T;
  h->last_launches = launches;
  return LMOE_OK;
}

lmoe_status lmoe_ep_experts(lmoe_handle h, const void* recv_bf16, const int32_t* recv_counts, int n, void* out_bf16,
                            cudaStream_t st) {
  if (!h || !h->idx_loc || n < 0 || n > h->Pexp) return LMOE_ERR_INVALID_ARG;
  if (!recv_counts) return LMOE_ERR_INVALID_ARG;
  if (n == 0) return LMOE_OK;
  if (!recv_bf16 || !aligned(recv_bf16, 16) || !out_bf16 || !aligned(out_bf16, 16)) return LMOE_ERR_INVALID_ARG;
  int launches = 0;
  begin_call(h);
  // the local expert of each received row, then the same grouping and tiles as a local batch of n rows, k = 1
  LMOE_TRY(launch_ep_expand(recv_counts, h->ep * h->E_loc, h->E_loc, n, h->idx_loc, h->err, st));
  const int BN = expert_bn_rows(h, n);
  const int split = h->fp8 || moe_split(BN);
  LMOE_TRY_STATUS(run_dispatch(h, h->idx_loc, n, BN, h->counts, h->offsets, h->perm, st, launches, 1, h->E_loc));
  const int KSg = expert_ksplit(h, n, true);
  {
    StageTimer tm(h, LMOE_STAGE_ACT_QUANT, st);
    LMOE_TRY(launch_quant_gather_bf16(recv_bf16, n, 1, h->dx, h->Kp, h->inv_pad, BN, split, h->terms, h->xq, h->xsf,
                                      h->sched, h->gcnt, KSg > 1 ? h->n_gcnt : 0, st));
    ++launches;
    tm.done();
  }
  int KSd = 1;
  LMOE_TRY_STATUS(run_experts(h, n, BN, split, h->ones, st, launches, KSd));
  LMOE_TRY(launch_ep_cast(h->y, n, h->dx, KSd, static_cast<size_t>(n) * h->dx, out_bf16, st));
  launches += 2;
  h->last_launches = launches + 1;
  return LMOE_OK;
}

lmoe_status lmoe_ep_combine(lmoe_handle h, const void* ret_bf16, int T, void* out_bf16, cudaStream_t st) {
  if (!h || !h->ep_perm || T < 0 || T != h->ep_T) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!ret_bf16 || !aligned(ret_bf16, 16) || !out_bf16 || !aligned(out_bf16, 16)) return LMOE_ERR_INVALID_ARG;
  int launches = 0;
  begin_call(h);
  const long long P = static_cast<long long>(T) * h->k;
  // returned expert outputs back in assignment order, weighted by G, for the slot-ordered sum
  LMOE_TRY(launch_ep_unpack(ret_bf16, static_cast<int>(P), h->dx, h->ep_perm, h->G, h->y, st));
  ++launches;
  LMOE_TRY_STATUS(run_combine_output(h, T, P, 1, out_bf16, st, launches));
  h->last_T = T;
  h->last_launches = launches;
  return LMOE_OK;
}

lmoe_status lmoe_forward_host(lmoe_handle h, const void* x_host, int T, void* out_host, cudaStream_t st) {
  if (!h || T < 0 || T > h->Tm) return LMOE_ERR_INVALID_ARG;
  if (T == 0) return LMOE_OK;
  if (!x_host || !out_host) return LMOE_ERR_INVALID_ARG;
  const size_t bytes = static_cast<size_t>(T) * h->d * 2;
  LMOE_TRY(cudaMemcpyAsync(h->x_stage, x_host, bytes, cudaMemcpyHostToDevice, st));
  lmoe_status s = lmoe_forward(h, h->x_stage, T, h->out_stage, nullptr, nullptr, st);
  if (s != LMOE_OK) return s;
  LMOE_TRY(cudaMemcpyAsync(out_host, h->out_stage, bytes, cudaMemcpyDeviceToHost, st));
  LMOE_TRY(cudaStreamSynchronize(st));
  return check_err(h);
}

lmoe_status lmoe_debug_tensor(lmoe_handle h, const char* name, void* dst, size_t bytes, cudaStream_t st) {
  if (!h || !name || !dst) return LMOE_ERR_INVALID_ARG;
  const size_t T = static_cast<size_t>(h->last_T);
  const void* src = nullptr;
  size_t want = 0;
  if (!std::strcmp(name, "logits")) {
    src = h->logits;
    want = T * h->E * 4;
  } else if (!std::strcmp(name, "xc")) {
    src = h->xc;
    want = T * h->din * 4;
  } else if (!std::strcmp(name, "u")) {
    src = h->u;
    want = T * h->dx * 4;
  } else if (!std::strcmp(name, "u_hat")) {
    src = h->u_hat;
    want = T * h->dx * 2;
  } else if (!std::strcmp(name, "h_shared")) {
    if (h->fp8) return LMOE_ERR_INVALID_ARG;   // FP8 layers keep h of the shared expert as hi/lo codes
    src = h->h_s;
    want = T * h->Fs * 2;
  } else if (!std::strcmp(name, "y_shared")) {
    if (!h->fp8 || !h->Fs) return LMOE_ERR_INVALID_ARG;
    src = h->y_sh;
    want = T * h->d * 4;
  } else if (!std::strcmp(name, "x_expert") || !std::strcmp(name, "h")) {
    // decoded in place into dst: the routed experts' inputs [T*k][dx] or hidden activations [T*k][F]
    const bool xe = name[0] == 'x';
    const int K = xe ? h->dx : h->F;
    if (bytes != T * h->k * K * 4 || !h->last_BN) return LMOE_ERR_INVALID_ARG;
    if (h->fp4)
      LMOE_TRY(launch_decode_fp4(xe ? h->xq : h->hq, xe ? h->xsf : h->hsf, h->inv_pad, static_cast<int>(T * h->k), K,
                                 xe ? h->Kp : h->Fp, h->last_BN, h->terms, static_cast<float*>(dst), st));
    else
      LMOE_TRY(launch_decode_terms(xe ? h->xq : h->hq, xe ? h->xsf : h->hsf, h->inv_pad, static_cast<int>(T * h->k), K,
                                   xe ? h->Kp : h->Fp, h->last_BN, h->last_split, h->terms, static_cast<float*>(dst),
                                   st));
    return LMOE_OK;
  } else if (!std::strcmp(name, "delta_f32")) {
    if (!h->delta32) return LMOE_ERR_INVALID_ARG;
    src = h->delta32;
    want = T * h->d * 4;
  } else if (!std::strcmp(name, "counts")) {
    src = h->counts;
    want = static_cast<size_t>(h->E) * 4;
  } else if (!std::strcmp(name, "offsets")) {
    src = h->offsets;
    want = static_cast<size_t>(h->E + 1) * 4;
  } else if (!std::strcmp(name, "perm")) {
    src = h->perm;
    want = T * h->k * 4;
  } else {
    return LMOE_ERR_INVALID_ARG;
  }
  if (bytes != want) return LMOE_ERR_INVALID_ARG;
  if (want) LMOE_TRY(cudaMemcpyAsync(dst, src, want, cudaMemcpyDeviceToDevice, st));
  return LMOE_OK;
}

lmoe_status lmoe_sync_status(lmoe_handle h, cudaStream_t st) {
  if (!h) return LMOE_ERR_INVALID_ARG;
  LMOE_TRY(cudaStreamSynchronize(st));
  LMOE_TRY(cudaGetLastError());
  return check_err(h);
}

int lmoe_last_launch_count(lmoe_handle h) { return h ? h->last_launches : 0; }

lmoe_status lmoe_set_profiling(lmoe_handle h, int reserve_forwards, uint32_t stage_mask) {
  if (!h || reserve_forwards < 0) return LMOE_ERR_INVALID_ARG;
  release_events(h);
  h->prof_mask = stage_mask & LMOE_PROFILE_ALL_STAGES;
  h->prof = h->prof_mask != 0;
  h->prof_calls = 0;
  int timed = 0;
  for (int i = 0; i < LMOE_NUM_STAGES; ++i) timed += h->prof_mask >> i & 1u;
  const size_t want = static_cast<size_t>(reserve_forwards) * 2 * timed;
  while (h->prof && h->ev_free.size() < want) {
    cudaEvent_t e = nullptr;
    LMOE_TRY(cudaEventCreate(&e));
    h->ev_free.push_back(e);
  }
  return LMOE_OK;
}

lmoe_status lmoe_set_profiling_period(lmoe_handle h, int every) {
  if (!h || every < 1) return LMOE_ERR_INVALID_ARG;
  h->prof_every = every;
  h->prof_calls = 0;
  return LMOE_OK;
}

lmoe_status lmoe_profile_get(lmoe_handle h, int stage, float* total_ms, int* count) {
  if (!h || stage < 0 || stage >= LMOE_NUM_STAGES || !total_ms || !count) return LMOE_ERR_INVALID_ARG;
  double sum = 0.0;
  for (auto& pr : h->ev_used[stage]) {
    LMOE_TRY(cudaEventSynchronize(pr.second));
    float ms = 0.f;
    LMOE_TRY(cudaEventElapsedTime(&ms, pr.first, pr.second));
    sum += ms;
  }
  *total_ms = static_cast<float>(sum);
  *count = static_cast<int>(h->ev_used[stage].size());
  return LMOE_OK;
}

int lmoe_last_active_experts(lmoe_handle h, cudaStream_t st) {
  if (!h || h->last_T <= 0) return 0;
  std::vector<int32_t> c(h->E);
  if (cudaMemcpyAsync(c.data(), h->counts, c.size() * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return -1;
  if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
  int n = 0;
  for (int32_t v : c) n += v > 0;
  return n;
}

}  // extern "C"
