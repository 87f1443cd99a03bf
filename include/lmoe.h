/*
 * lmoe — forward pass of the Stable LatentMoE feed-forward layer on one
 * GB300 (sm_103a).  C ABI: plain pointers and sizes, no C++ or torch types.
 *
 * What the layer computes (Kimi K3 card "Latent mixture of experts", the
 * equations under "All 23 steps" and the KimiSparseMoeBlock.forward /
 * moe_infer excerpt of modeling_kimi_linear.py; Kimi K2 card "Mixture of
 * experts", "All 19 steps"):
 *
 *   z = x W_r^T,  s = sigmoid(z),  S = top_k(s + b)
 *   G_i = routed_scale * s_i / sum_{j in S} s_j       (raw s, not s + b)
 *   x^c = x W_down^T                                   (latent layers only)
 *   for i in S:  g = x^c W_gate,i^T,  u = x^c W_up,i^T,
 *                h = SiTU(g, u) = b1 tanh(g/b1) sigmoid(g) * b2 tanh(u/b2)
 *                (SwiGLU g sigmoid(g) u for LMOE_ACT_SWIGLU),  E_i = h W_down,i^T
 *   u = sum_i G_i E_i,  u_hat = norm_w * u / sqrt(mean(u^2) + eps)
 *   y_routed = u_hat W_up^T                            (latent layers only)
 *   y_shared = SiTU-GLU of x with the shared weights (full width)
 *   Delta = y_routed + y_shared                        (no residual added)
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers unless the name says host.  All
 *     matrices are row-major in nn.Linear [out][in] storage (the input
 *     dimension is contiguous).  bf16 values are raw IEEE bfloat16.
 *   - Weights are BORROWED: the caller owns them, they must stay valid and
 *     unchanged for the handle's lifetime, and the library never writes them.
 *     The handle owns only its workspace, sized at create for max_tokens.
 *   - Calls are stream-ordered and asynchronous unless stated.  Argument
 *     errors are reported synchronously and nothing is launched.  An
 *     asynchronous CUDA error or a kernel-side timeout surfaces on the next
 *     call that checks (lmoe_sync_status, lmoe_forward_host).
 *   - One handle is used by one stream at a time (the workspace is shared by
 *     its calls).  `out` may not alias `x`.
 *   - No call performs a host synchronisation except lmoe_create,
 *     lmoe_destroy, lmoe_forward_host and lmoe_sync_status.
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#if defined(__GNUC__)
#define LMOE_API __attribute__((visibility("default")))
#else
#define LMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LMOE_OK = 0,
  LMOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size, T > max_tokens */
  LMOE_ERR_UNSUPPORTED = 2,  /* a configuration this build does not implement */
  LMOE_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
  LMOE_ERR_OOM = 4,          /* workspace allocation failed */
  LMOE_ERR_TIMEOUT = 5       /* a kernel's bounded wait expired; results are invalid */
} lmoe_status;

typedef enum { LMOE_ACT_SITU = 0, LMOE_ACT_SWIGLU = 1 } lmoe_act;
/* Number format of the routed experts' activations on the tensor cores. */
typedef enum {
  LMOE_ACT_FMT_E4M3 = 0, /* E4M3 terms x the weights' own codes, kind::mxf8f6f4 (act_terms 1 or 2) */
  LMOE_ACT_FMT_E2M1 = 1  /* packed E2M1 terms, E8M0 per 32, x MXFP4 weights as stored, both operands 4-bit in
                            shared memory, kind::mxf4 (act_terms 1..4, 0 = 3); MXFP4 experts only */
} lmoe_act_fmt;
typedef enum { LMOE_W_MXFP4 = 0, LMOE_W_FP8_BLOCK128 = 1 } lmoe_wfmt;

/* Layer shape and constants; keys mirror the model config (num_experts,
 * num_experts_per_token, routed_expert_hidden_size, moe_intermediate_size,
 * num_shared_experts x moe_intermediate_size, latent_moe_use_norm,
 * rms_norm_eps, activation_situ_beta, activation_situ_linear_beta). */
typedef struct {
  int d_model;          /* d: 7168 for Kimi K3 / K2 */
  int d_latent;         /* l: 3584 for K3; 0 = non-latent block (K2) */
  int n_experts;        /* E: 896 (K3), 384 (K2) */
  int top_k;            /* k: 16 (K3), 8 (K2); 1 <= k <= E */
  int d_expert_ff;      /* routed expert hidden width: 3072 (K3), 2048 (K2) */
  int d_shared_ff;      /* shared MLP hidden width: 6144 (K3, two experts merged); 0 = none */
  int use_latent_norm;  /* 1: RMSNorm between the expert sum and the up-projection */
  float norm_eps;       /* RMSNorm epsilon */
  float routed_scale;   /* 1.0 (K3), 2.827 (K2) */
  float situ_beta;      /* 4: cap of the gate's linear factor */
  float situ_linear_beta; /* 25: cap of the up branch */
  lmoe_act act;
  lmoe_wfmt expert_wfmt;
  int max_tokens;       /* largest T any call on this handle will pass */
  int act_terms;        /* E4M3 terms per routed-expert activation (x^c into the gate/up GEMM, h into
                           the down GEMM), each 32-value block with its own E8M0 scale: 2 (or 0, the
                           default) = hi + lo, the second quantising the first one's residual, about
                           16-bit precision; 1 = MXFP8, the deployment precision of the walk-through's
                           "参数账" section (one term, half the activation bytes and MMAs at large
                           batches; ~2-4% error per expert input).  1 needs MXFP4 experts.  With
                           act_format LMOE_ACT_FMT_E2M1: MXFP4 terms, 1..4 (0 = 3). */
  lmoe_act_fmt act_format;
  int ep_size;          /* expert parallelism over ep_size ranks (0 or 1: none); the experts are split
                           into contiguous ranges of n_experts / ep_size, and this handle's weights
                           hold only its own range (ex_* arrays of n_experts / ep_size experts) */
  int ep_rank;          /* this handle's rank, 0 <= ep_rank < ep_size */
  int max_recv_rows;    /* largest number of rows lmoe_ep_experts will receive
                           (0: ep_size * max_tokens * top_k) */
} lmoe_config;

/* Layer weights (all device pointers, borrowed).
 *   router_w       bf16 [E][d]                  router_bias  fp32 [E]
 *   w_down_latent  bf16 [l][d]                  w_up_latent  bf16 [d][l]
 *   norm_w         bf16 [l]                     (latent layers only)
 *   ex_{gate,up}_q  MXFP4: uint8 [E][F][K/2], K = l (or d for K2): two E2M1
 *                   codes per byte, even K index in the low nibble
 *   ex_down_q       MXFP4: uint8 [E][l][F/2]
 *   ex_*_s          MXFP4: E8M0 uint8 [E][N][K/32], one scale per 32 K values
 *   (LMOE_W_FP8_BLOCK128: ex_*_q E4M3 uint8 [E][N][K], ex_*_s fp32
 *    [E][ceil(N/128)][ceil(K/128)]; sh_* the same without E and sh_*_s set.)
 *   sh_gate, sh_up bf16 [Fs][d]                 sh_down bf16 [d][Fs]
 * Alignment: every pointer 16-byte aligned, code/scale arrays 32-byte. */
typedef struct {
  const void* router_w;
  const float* router_bias;
  const void* w_down_latent;
  const void* w_up_latent;
  const void* norm_w;
  const uint8_t* ex_gate_q;
  const uint8_t* ex_up_q;
  const uint8_t* ex_down_q;
  const void* ex_gate_s;
  const void* ex_up_s;
  const void* ex_down_s;
  const void* sh_gate;
  const void* sh_up;
  const void* sh_down;
  const void* sh_gate_s;
  const void* sh_up_s;
  const void* sh_down_s;
} lmoe_weights;

typedef struct lmoe_ctx* lmoe_handle;

/* Validate the config and weights, allocate the workspace for max_tokens and
 * encode the TMA descriptors of the weights.  Synchronises `stream`.
 * Errors: INVALID_ARG (null pointers, bad shapes), UNSUPPORTED (shapes the
 * kernels do not cover: d, l, F, Fs must be multiples of 32; E <= 2048;
 * k <= 32; MXFP4 experts need a latent layer, FP8 block-128 experts a
 * non-latent one without the norm and with d, F, Fs multiples of 128 and
 * two activation terms; the current device is not an sm_103 GPU), OOM,
 * CUDA.  On error *out is NULL. */
LMOE_API lmoe_status lmoe_create(const lmoe_config* cfg, const lmoe_weights* w, cudaStream_t stream, lmoe_handle* out);

/* Router only (Kimi K3 card, router steps; port notes item 3): topk_idx
 * int32 [T][k], sorted by biased score s + b descending, exact ties to the
 * lower expert index; topk_w fp32 [T][k] = routed_scale * s / sum s over
 * the selection.  x: bf16 [T][d].  T = 0 is a no-op. */
LMOE_API lmoe_status lmoe_route(lmoe_handle h, const void* x_bf16, int T, int32_t* topk_idx, float* topk_w,
                       cudaStream_t stream);

/* Whole layer: out bf16 [T][d] = Delta.  topk_idx_opt / topk_w_opt, when not
 * NULL, receive the routing of lmoe_route.  T = 0 is a no-op. */
LMOE_API lmoe_status lmoe_forward(lmoe_handle h, const void* x_bf16, int T, void* out_bf16, int32_t* topk_idx_opt,
                         float* topk_w_opt, cudaStream_t stream);

/* Expert parallelism (Kimi K2 card, moe_infer under ep_size > 1: count
 * exchange, token all-to-all, local regrouping, experts, reverse all-to-all,
 * weighted sum), at the latent width for latent layers (walk-through: both
 * passes then move 3584-wide rows).  The exchanges are the caller's (one
 * process per GPU; an all-to-all of its collective library); the three calls
 * below are the device work between them, stream-ordered, each on the same
 * handle and stream in this order.  A handle with ep_size > 1 rejects
 * lmoe_forward (UNSUPPORTED); with ep_size <= 1 these calls run all experts
 * locally (the exchanges then pass the buffers through unchanged).
 *
 * lmoe_ep_dispatch: router, top-k and the grouping of the T*k assignments by
 * global expert, plus the side-stream steps (latent down-projection, shared
 * expert).  send_bf16 [T*k][l] (d for non-latent layers) receives each
 * assignment's expert input in bf16, rows grouped by expert, so the rows for
 * rank r are the contiguous block of experts [r E/R, (r+1) E/R); its row
 * count is the sum of expert_counts over that range.  expert_counts int32
 * [E] device.  topk_idx_opt / topk_w_opt as in lmoe_forward. */
LMOE_API lmoe_status lmoe_ep_dispatch(lmoe_handle h, const void* x_bf16, int T, void* send_bf16,
                                      int32_t* expert_counts, int32_t* topk_idx_opt, float* topk_w_opt,
                                      cudaStream_t stream);
/* lmoe_ep_experts: the rows this rank received (recv_bf16 [n][l], in the
 * order the exchange delivers them: source rank by source rank, each
 * source's rows grouped by this rank's experts) and recv_counts int32
 * [ep_size][E/ep_size] (device: the rows each source sent to each local
 * expert, the counts exchange's output) -> out_bf16 [n][l], each row's
 * expert output (unweighted) in the same order, ready for the reverse
 * exchange.  n <= max_recv_rows.  Counts that do not sum to n are reported
 * by lmoe_sync_status (INVALID_ARG). */
LMOE_API lmoe_status lmoe_ep_experts(lmoe_handle h, const void* recv_bf16, const int32_t* recv_counts, int n,
                                     void* out_bf16, cudaStream_t stream);
/* lmoe_ep_combine: ret_bf16 [T*k][l] = the expert outputs returned in the
 * order of lmoe_ep_dispatch's send rows; weights them by G, sums each
 * token's k slots in slot order, applies the latent RMSNorm and the output
 * GEMM with the shared expert: out_bf16 [T][d] = Delta.  T must be the last
 * lmoe_ep_dispatch's. */
LMOE_API lmoe_status lmoe_ep_combine(lmoe_handle h, const void* ret_bf16, int T, void* out_bf16, cudaStream_t stream);

/* lmoe_forward on HOST buffers: copies x (bf16 [T][d], host memory; pinned
 * for asynchronous copies) into the workspace, runs the layer and copies
 * Delta back to out_host.  Synchronises `stream` before returning, so the
 * host buffers may be reused at once.  Returns a deferred error, if any. */
LMOE_API lmoe_status lmoe_forward_host(lmoe_handle h, const void* x_host, int T, void* out_host, cudaStream_t stream);

/* Token -> expert dispatch alone (moe_infer's counting, argsort and
 * grouping written as a counting sort): topk_idx int32 [T][k] in; counts
 * int32 [E]; offsets int32 [E+1] (exclusive prefix sum of counts); perm
 * int32 [T*k] = flattened assignments a = t*k + j grouped by expert, in
 * increasing a inside each expert.  Indices outside [0, E) are an error
 * the kernel reports through lmoe_sync_status (LMOE_ERR_INVALID_ARG). */
LMOE_API lmoe_status lmoe_dispatch(lmoe_handle h, const int32_t* topk_idx, int T, int32_t* counts, int32_t* offsets,
                          int32_t* perm, cudaStream_t stream);

/* lmoe_dispatch for callers that cannot allocate device memory.  The paper
 * has no counterpart of this call: it exists for code that may not call
 * cudaMalloc (and therefore cannot lmoe_create a handle), such as a step
 * being recorded into a CUDA graph that must not allocate, a plug-in whose
 * host framework owns the whole device-memory budget, or an allocator-free
 * runtime.  Same inputs and outputs as lmoe_dispatch (topk_idx int32
 * [T][k] in; counts [E], offsets [E+1], perm [T*k] out, all device memory
 * the caller provides) plus k and n_experts, since there is no handle.
 * Scratch: one static device array of about 2.4 MiB inside the library,
 * which every GPU that loads the library holds until the process exits.
 * Limits: T*k <= LMOE_NOALLOC_MAX_ASSIGNMENTS, n_experts <=
 * LMOE_NOALLOC_MAX_EXPERTS; larger sizes return LMOE_ERR_INVALID_ARG before
 * anything is launched.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.  The first call on each device looks up the array's
 * device address (cudaGetSymbolAddress) and caches it: make that first call
 * outside any stream capture.  The cached address belongs to the device's
 * primary context as it was then: after cudaDeviceReset (or anything else
 * that destroys that context) the array may move, so such a process must
 * not call this function again.  All calls share the one array, so calls that
 * overlap on the GPU (other streams, other threads) race and must be
 * serialised by the caller; no part of the array needs to start at zero
 * (every word a call reads is written earlier in the same call).  Expert ids
 * outside [0, n_experts) are skipped without an error report. */
#define LMOE_NOALLOC_MAX_ASSIGNMENTS 65536
#define LMOE_NOALLOC_MAX_EXPERTS 2048
LMOE_API lmoe_status lmoe_dispatch_noalloc(const int32_t* topk_idx, int T, int k, int n_experts, int32_t* counts,
                                           int32_t* offsets, int32_t* perm, cudaStream_t stream);

/* Quantile Balancing: the selection-bias update of Stable LatentMoE (tutorial
 * "Stable LatentMoE", section "Quantile Balancing: giving every expert a
 * fair shot"; walk-through "Kimi K3 模型结构（5）", section "Stable 之三：
 * Quantile Balancing", appendices C and D).  For a batch of T tokens routed
 * with biases b: alpha_t = token t's (k+1)-th largest biased score
 * sigmoid(z_t) + b; r_tj = alpha_t - sigmoid(z_tj), the bias expert j needs to
 * enter t's top-k.  The new biases are stored for the next batch; the batch
 * itself keeps the biases it was routed with.
 *
 * Inputs of all three calls: logits fp32 [T][E] (the router's z; NULL = those
 * of the handle's last lmoe_forward, whose T must then be passed), bias fp32
 * [E] (the biases the batch was routed with; NULL = the handle's
 * router_bias).  E and k are the handle's; k < E is required.  Stream-ordered,
 * no host synchronisation.  Errors: INVALID_ARG (NULL handle or output, T out
 * of [1, max_tokens], bins out of [1, 2^20], k >= E), CUDA.
 *
 * lmoe_qb_update (exact): new_bias fp32 [E] = q_j - mean(q), q_j = the
 * (k/E)-quantile of r_{:,j} with the "higher" convention (the sorted value at
 * index ceil(k (T-1) / E)). */
LMOE_API lmoe_status lmoe_qb_update(lmoe_handle h, const float* logits, int T, const float* bias, float* new_bias,
                                    cudaStream_t stream);
/* lmoe_qb_histogram (appendix D): adds the batch's T x E required biases to
 * counts int32 [E][bins], bins uniform over [min b - 1, max b + 1] (values
 * outside go to the end bins).  The caller zeroes counts at the start of a
 * step; calls for several micro-batches add up, and counts of several ranks
 * add with one integer all-reduce (the bias, hence the range, must be the
 * same on all of them). */
LMOE_API lmoe_status lmoe_qb_histogram(lmoe_handle h, const float* logits, int T, const float* bias, int bins,
                                       int32_t* counts, cudaStream_t stream);
/* lmoe_qb_update_from_histogram: new_bias fp32 [E] from accumulated counts:
 * per expert, m = its total count, target = ceil(m k / E); the first bin c
 * whose cumulative count reaches the target, value = lo + w (c + (target -
 * count before c) / count of c); then the mean is subtracted.  bias: the
 * biases the counts were taken with (for the range). */
LMOE_API lmoe_status lmoe_qb_update_from_histogram(lmoe_handle h, const int32_t* counts, int bins, const float* bias,
                                                   float* new_bias, cudaStream_t stream);

/* Copy an intermediate of the last lmoe_forward on this handle out of the
 * workspace (stream-ordered): "logits" fp32 [T][E] (router z), "xc" fp32
 * [T][l], "u" fp32 [T][l] (expert sum; [T][d] for non-latent layers, where
 * it is y_routed), "u_hat" bf16 [T][l] (latent layers), "h_shared"
 * bf16 [T][Fs] (layers with a bf16 shared MLP), "y_shared" fp32 [T][d]
 * (FP8 layers, whose shared expert runs on the FP8 expert GEMMs), "counts"
 * int32 [E], "offsets" int32 [E+1], "perm" int32 [T*k], "delta_f32" fp32
 * [T][d] (Delta before its bf16 rounding; only while lmoe_keep_f32_output
 * is on), "x_expert" fp32 [T*k][l] ([T*k][d] for non-latent layers) and "h"
 * fp32 [T*k][F]: the routed experts' inputs and hidden activations per
 * assignment a = t*k + j, as the expert GEMMs multiply them (their E4M3
 * terms times the block scales, decoded by a kernel into dst).  `bytes`
 * must equal the tensor's size for the last T; a name the layer does not
 * have returns INVALID_ARG. */
LMOE_API lmoe_status lmoe_debug_tensor(lmoe_handle h, const char* name, void* dst, size_t bytes, cudaStream_t stream);

/* While enabled (enable != 0), every lmoe_forward also stores Delta as fp32
 * before it is rounded to bf16, readable as the "delta_f32" debug tensor:
 * the same launches, each writing one fp32 value beside each bf16 one.  The
 * K3 card's equations end in Delta itself; the bf16 output holds it to half
 * a bf16 spacing, which this lets a test see past.  Enabling allocates a
 * [max_tokens][d] fp32 buffer (device-synchronising); disabling frees it.
 * Errors: INVALID_ARG (NULL handle), OOM, CUDA. */
LMOE_API lmoe_status lmoe_keep_f32_output(lmoe_handle h, int enable);

/* Test of the deferred-error path: launches one warp that waits on a
 * barrier nothing ever arrives at, through the same bounded wait the layer's
 * kernels use, with a wall-clock limit of limit_ns (1,000 ns .. 1 s).  The
 * wait gives up, records a timeout in the handle's error flag and the kernel
 * returns (it holds no TMA copy, MMA or tensor memory), so the next
 * lmoe_sync_status returns LMOE_ERR_TIMEOUT and clears the flag; the
 * handle stays usable.  The pages have no counterpart: the K3 card's code
 * waits on no device barrier.  Errors: INVALID_ARG (NULL handle, limit out
 * of range), CUDA (launch failure). */
LMOE_API lmoe_status lmoe_selftest_timeout(lmoe_handle h, unsigned long long limit_ns, cudaStream_t stream);

/* Synchronise `stream` and return the first deferred error: a CUDA error, a
 * kernel timeout (TIMEOUT) or an out-of-range expert index (INVALID_ARG).
 * Clears the kernel-side error flag. */
LMOE_API lmoe_status lmoe_sync_status(lmoe_handle h, cudaStream_t stream);

/* Number of kernels the last lmoe_forward launched (for launch accounting). */
LMOE_API int lmoe_last_launch_count(lmoe_handle h);

/* Per-stage timing.  While enabled, lmoe_forward records a CUDA event pair
 * on the stage's stream around each stage whose bit (1 << stage) is set in
 * stage_mask (0 disables timing); lmoe_profile_get synchronises the recorded
 * events and returns the stage's summed device time (ms) and the number of
 * timed launches since profiling was last enabled.  Enabling again resets
 * the sums.  reserve_forwards pre-creates event pairs for that many
 * forwards.  An event between two kernels ends the overlap of the second
 * kernel's start with the first one's drain, so timing every stage slows a
 * small forward measurably; time only the stages of interest.  Stages: */
enum {
  LMOE_STAGE_ROUTER = 0,     /* router GEMM + top-k */
  LMOE_STAGE_DISPATCH = 1,   /* counting-sort dispatch */
  LMOE_STAGE_LATENT_DOWN = 2,/* x^c GEMM (+ split-K sum) */
  LMOE_STAGE_ACT_QUANT = 3,  /* x^c -> hi/lo E4M3 in expert-tile order */
  LMOE_STAGE_EXPERT_GU = 4,  /* grouped expert gate/up GEMM (MXFP4 or FP8) + SiTU / SwiGLU */
  LMOE_STAGE_EXPERT_DOWN = 5,/* grouped expert down GEMM x G */
  LMOE_STAGE_COMBINE = 6,    /* slot-ordered sum + RMSNorm */
  LMOE_STAGE_SHARED = 7,     /* shared gate/up GEMM + SiTU (on the handle's side stream) */
  LMOE_STAGE_OUTPUT = 8,     /* [u_hat | h_shared] output GEMM */
  LMOE_NUM_STAGES = 9
};
#define LMOE_PROFILE_ALL_STAGES 0x1FFu
LMOE_API lmoe_status lmoe_set_profiling(lmoe_handle h, int reserve_forwards, uint32_t stage_mask);
/* Time only every `every`-th call (lmoe_forward, lmoe_route, lmoe_dispatch)
 * while profiling is enabled, counting from the call after this one or after
 * lmoe_set_profiling, starting with that call (default 1: every call); the
 * calls in between run without events, so a long timed loop keeps its launch
 * overlap while the sampled calls give the stage times.  every < 1:
 * LMOE_ERR_INVALID_ARG. */
LMOE_API lmoe_status lmoe_set_profiling_period(lmoe_handle h, int every);
LMOE_API lmoe_status lmoe_profile_get(lmoe_handle h, int stage, float* total_ms, int* count);

/* Number of distinct experts the last lmoe_forward's batch selected
 * (synchronises the stream; reads the dispatch counts). */
LMOE_API int lmoe_last_active_experts(lmoe_handle h, cudaStream_t stream);

/* Release the workspace.  Synchronises the device work of this handle.
 * NULL is accepted. */
LMOE_API lmoe_status lmoe_destroy(lmoe_handle h);

/* Static string for a status code. */
LMOE_API const char* lmoe_status_string(lmoe_status s);

#ifdef __cplusplus
}
#endif
#endif /* LMOE_H */
