/*
 * moe.h -- C ABI of libmoe.so: the forward pass of one sparse top-k
 * Mixture-of-Experts FFN layer on one NVIDIA B300 (sm_103a).
 *
 * What the layer computes (sources: page title, then section):
 *   1. router scores  s = W_r x (+ o)        "Mixture of Experts" (llm-tutorial
 *      ch. 11) § The mathematics; "Mixture of experts" (inside-the-model
 *      guide) § The computation; "Chapter 33 — Mixture of Experts" § The Router.
 *   2. top-k selection and gates: softmax over the k chosen logits
 *      (ch. 11 § Top-k routing), the full-softmax probability of a top-1
 *      choice (ch. 11 § Top-1 vs top-2), or sigmoid affinities renormalised
 *      over the chosen (guide § The computation, § Auxiliary-loss-free
 *      balancing); an optional per-expert bias steers only the choice.
 *   3. expert capacity with overflow dropped to the residual, first come by
 *      token index (ch. 11 § Expert capacity and dropped tokens; guide
 *      § Auxiliary loss).
 *   4. permutation of token copies into expert-contiguous order
 *      ("Chapter 33" § Simple MoE Layer Implementation: per-expert gather).
 *   5. expert MLPs: W2 act(W1 x) with GELU or ReLU, or SwiGLU
 *      W2 (silu(W1 x) * (W3 x)); optional always-on shared SwiGLU expert
 *      (guide § Fine-grained and shared experts).
 *   6. combine y = sum_j g_j Expert_j(x) (+ shared), and the balance
 *      statistics f_i, P_i, L = alpha * E * sum_i f_i P_i (guide § Auxiliary
 *      loss; ch. 11 § The auxiliary loss).
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is DEVICE memory owned by the caller, unless the
 *     entry point says "host".  The library allocates no memory, keeps no
 *     state between calls and never synchronises the stream, except
 *     moe_check_status, which does.
 *   - All calls are asynchronous on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  The return value covers
 *     errors detected before or while enqueueing: argument checks and launch
 *     failures.  Errors found on the device (a bounded wait that ran out) are
 *     recorded in a status word inside the workspace.  moe_check_status
 *     reports them.
 *   - Row-major layouts, no padding:
 *       x      [T, d]       dtype          y      [T, d]   dtype
 *       W_r    [E, d]       dtype          W1, W3 [E, f, d] dtype
 *       W2     [E, d, f]    dtype          Ws1,Ws3[f_s, d] dtype
 *       Ws2    [d, f_s]     dtype
 *       topk_idx [T, k] int32, topk_w [T, k] float32
 *     dtype is float32 (MOE_F32) or bfloat16 (MOE_BF16) for all of x, W_r,
 *     the expert weights and y.  logit_offset and sel_bias are float32 [E].
 *     Router arithmetic, gates and statistics are float32 on both paths.
 *   - Pointers to tensors must be 16-byte aligned.  On the bf16 path d, f
 *     and f_s must be multiples of 8; on the float32 path, multiples of 4.
 *   - The workspace is caller-owned device memory of at least
 *     moe_workspace_size() bytes, 256-byte aligned.  Its first 4096 bytes
 *     hold the device status word and the counters the kernels use to find
 *     the last block of a reduction: zero them once when the workspace is
 *     created; every call leaves them valid for the next.  Concurrent calls
 *     on different streams need separate workspaces.
 *   - Kernels are launched with programmatic dependent launch: each may begin
 *     its prologue while the previous kernel in the stream finishes, and waits
 *     for that kernel's results before reading them.  Stream order is kept.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,          /* NULL where a tensor is required, bad size or mode, misalignment */
  MOE_ERR_UNSUPPORTED = 2,  /* valid layer this build does not run (E > 512, k > 32, ...) */
  MOE_ERR_WORKSPACE = 3,    /* workspace NULL, too small or not 256-byte aligned */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5,      /* a bounded device wait ran out (reported by moe_check_status) */
  MOE_ERR_DEVICE = 6,       /* current device is not a compute-capability 10.3 GPU */
  MOE_ERR_BOUNDS = 7        /* bounds-checked build (libmoe_check.so) only: a routing-derived
                               index (expert, capacity position, buffer row, token) was out
                               of range; the access was skipped (reported by
                               moe_check_status) */
};

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_ACT_GELU = 0, MOE_ACT_RELU = 1, MOE_ACT_SWIGLU = 2 } moe_act;
typedef enum {
  MOE_GATE_SOFTMAX_TOPK = 0,    /* g = softmax of the k chosen logits */
  MOE_GATE_SIGMOID_RENORM = 1,  /* g = sigmoid(s_i) / sum over chosen of sigmoid(s_j) */
  MOE_GATE_SOFTMAX_FULL = 2     /* g = softmax over all E logits, read at the chosen i */
} moe_gate;

/* Layer description.  All fields are read by value during the call. */
typedef struct {
  int32_t T;        /* tokens in the batch, >= 0 */
  int32_t d;        /* model width, >= 1 */
  int32_t E;        /* routed experts, 1..512 */
  int32_t k;        /* experts per token, 1..min(E, 32) */
  int32_t f;        /* routed expert width, >= 1 */
  int32_t n_shared; /* 0 or 1 always-on shared SwiGLU expert (bf16: SwiGLU layers only,
                       else MOE_ERR_UNSUPPORTED) */
  int32_t f_shared; /* width of the shared expert (ignored when n_shared = 0) */
  int32_t dtype;    /* moe_dtype */
  int32_t act;      /* moe_act of the routed experts */
  int32_t gate;     /* moe_gate */
  double capacity_factor; /* rho; <= 0 means no capacity limit.  Otherwise the
                             capacity is C = ceil((double)(k*T) * rho / E),
                             the same C for every expert.  NaN or infinite:
                             MOE_ERR_ARG */
  float alpha;      /* coefficient of the balance loss; NaN or infinite:
                       MOE_ERR_ARG */
  int32_t reserved; /* must be 0 */
} moe_config;

/* Number of bytes of workspace moe_forward needs for this layer. */
int moe_workspace_size(const moe_config* cfg, size_t* bytes);

/*
 * moe_forward -- all six stages, enqueued on `stream`.
 *
 * Inputs (device, read only):
 *   x, W_r, W1, W2            required
 *   W3                        required iff act == MOE_ACT_SWIGLU, else NULL
 *   Ws1, Ws3, Ws2             required iff n_shared == 1, else NULL
 *   logit_offset [E] float32  optional: added to every token's logits; it
 *                             enters the gates and P like the logits do
 *   sel_bias [E] float32      optional: added to the affinity (the logit, or
 *                             its sigmoid) for the choice only; gates and P
 *                             ignore it ("Mixture of experts" guide
 *                             § Auxiliary-loss-free balancing)
 * Outputs (device, written):
 *   y [T, d] (dtype)          MoE branch only; a token whose every slot was
 *                             dropped gets 0 (the caller adds the residual)
 *   topk_idx [T, k] int32     chosen experts, descending selection score,
 *                             ties to the lower index
 *   topk_w [T, k] float32     gates (also reported for dropped slots)
 *   expert_counts [E] int32   assignments kept per expert (after capacity)
 *   aux_loss [1] float32      alpha * E * sum_i f_i P_i
 * Optional outputs (device, may be NULL):
 *   routed_counts [E] int32   assignments per expert before capacity
 *   offsets [E+1] int32       exclusive scan of expert_counts
 *   slot_pos [T, k] int32     offsets[e] + position of the assignment among
 *                             the kept ones of expert e, or -1 if dropped
 *   f_out [E] float32         routed_counts / (T*k)
 *   P_out [E] float32         mean over tokens of the full router
 *                             distribution (softmax of s over all E, or
 *                             sigmoid(s) normalised over all E)
 * Errors: MOE_ERR_ARG / _UNSUPPORTED / _WORKSPACE before anything is
 * enqueued; MOE_ERR_CUDA if a launch fails; MOE_ERR_DEVICE off sm_103.
 * T = 0 is valid: counts, offsets, statistics and the loss are set to 0.
 */
int moe_forward(const moe_config* cfg,
                const void* x, const void* W_r,
                const float* logit_offset, const float* sel_bias,
                const void* W1, const void* W3, const void* W2,
                const void* Ws1, const void* Ws3, const void* Ws2,
                void* y, int32_t* topk_idx, float* topk_w,
                int32_t* expert_counts, float* aux_loss,
                int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                float* f_out, float* P_out,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_route -- stages 1-3 and the balance statistics only (no expert
 * MLPs): the routing half of moe_forward, with the same arguments, meaning
 * and errors.  expert_counts and aux_loss are required; the other outputs
 * are optional.  Needs moe_route_workspace_size() bytes.
 */
int moe_route_workspace_size(const moe_config* cfg, size_t* bytes);
int moe_route(const moe_config* cfg,
              const void* x, const void* W_r,
              const float* logit_offset, const float* sel_bias,
              int32_t* topk_idx, float* topk_w,
              int32_t* expert_counts, float* aux_loss,
              int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
              float* f_out, float* P_out,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_router_scores -- stage 1 alone: scores [T, E] float32 (device) gets the
 * router logits s = x W_r^T (+ logit_offset), from the router kernel
 * moe_forward uses for the same layer (bf16 layers with T >= 256: tensor-core
 * products with the reduction added in 128-wide float32 chunks; otherwise
 * float32 FMA).  Needs moe_route_workspace_size() bytes.  x and W_r must be
 * 16-byte aligned.
 */
int moe_router_scores(const moe_config* cfg, const void* x, const void* W_r,
                      const float* logit_offset, float* scores,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_router_scores_noalloc -- moe_router_scores without a workspace, for
 * callers that cannot allocate device memory per call: a host framework that
 * owns all device memory and hands none out, or a latency-critical path that
 * must not enter the CUDA allocator.  The pages have no counterpart of this
 * entry point; it repackages stage 1 for such callers.
 * Inputs and output ([T, E] float32 logits, offset included) are those of
 * moe_router_scores; the logits come from the float32 FMA router (bit for bit
 * what moe_router_scores gives when moe_set_tuning selects MOE_ROUTER_SIMT,
 * and within 5e-6 of its default tensor-core router for large bf16 batches).
 * The router GEMM's scratch (split partial logits and the counters of their
 * reduction) lives in one 8 MiB array inside the library.  Each device on
 * which the library's router module gets loaded (CUDA loads modules lazily:
 * the first router or no-workspace call on that device loads it) holds those
 * 8 MiB until the process exits.  A layer whose partials do not fit (4 KiB of
 * counters plus S*T*E*4 bytes, S the reduction split) returns
 * MOE_ERR_UNSUPPORTED.  The call allocates nothing.  The first call in a CUDA
 * context looks up the array's device address in that context (and caches it
 * under the context's id, so a device reset or another context gets its own
 * lookup); make that first call before any stream capture.  All calls share
 * the one array and it keeps the last call's contents: calls that overlap on
 * the GPU (other streams, other threads) race, so the caller must serialise
 * them.
 */
int moe_router_scores_noalloc(const moe_config* cfg, const void* x, const void* W_r,
                              const float* logit_offset, float* scores, void* stream);

/*
 * moe_forward_fp8 -- moe_forward for a bf16 SwiGLU layer whose gate and up
 * expert weights are stored as fp8 (e4m3).  The pages use no 8-bit formats;
 * this variant halves the bytes of the weights that dominate a decode step.
 *   W1q, W3q  [E, f, d] uint8: e4m3 codes (sign, 4 exponent bits with bias 7,
 *             3 mantissa bits; the FN encoding, no infinities);
 *   W1s, W3s  [E, f] float32: one scale per output channel, so that
 *             W1[e][n][c] = W1s[e][n] * e4m3(W1q[e][n][c]) (likewise W3);
 *   W2        [E, d, f] bf16, as in moe_forward.
 * Routing reads x as in moe_forward.  Every routed row of x is quantised to
 * e4m3 before the up projection: s_t = 2^q with q the smallest integer (not
 * below -126) such that max_c |x[t][c]| / 2^q <= 448 (s_t = 1 for a zero
 * row), values x[t][c] / s_t rounded to the nearest e4m3 value, ties to even.
 * The up projection multiplies e4m3 operands on the tensor cores
 * (kind::f8f6f4) with float32 accumulation and scales each accumulator by
 * s_t * W1s[e][n] (resp. W3s) before SwiGLU; h, the down projection and the
 * combine are those of moe_forward.  Every other argument, output and
 * convention is moe_forward's.  Requirements: cfg->dtype MOE_BF16, act
 * MOE_ACT_SWIGLU, n_shared 0, d a multiple of 16, f a multiple of 8, else
 * MOE_ERR_UNSUPPORTED; W1q, W3q, W1s, W3s 16-byte aligned, else MOE_ERR_ARG.
 * Needs moe_workspace_size_fp8() bytes of workspace (zeroed header as for
 * moe_forward).  moe_forward_fp8_timed takes the stage events of
 * moe_forward_timed (the row quantisation is timed with the permute stage).
 * moe_launch_count_fp8 gives the kernels one call launches.
 */
int moe_workspace_size_fp8(const moe_config* cfg, size_t* bytes);
int moe_forward_fp8(const moe_config* cfg, const void* x, const void* W_r,
                    const float* logit_offset, const float* sel_bias,
                    const uint8_t* W1q, const float* W1s, const uint8_t* W3q, const float* W3s,
                    const void* W2, void* y, int32_t* topk_idx, float* topk_w,
                    int32_t* expert_counts, float* aux_loss, int32_t* routed_counts,
                    int32_t* offsets, int32_t* slot_pos, float* f_out, float* P_out,
                    void* workspace, size_t workspace_bytes, void* stream);
int moe_forward_fp8_timed(const moe_config* cfg, const void* x, const void* W_r,
                          const float* logit_offset, const float* sel_bias,
                          const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                          const float* W3s, const void* W2, void* y, int32_t* topk_idx,
                          float* topk_w, int32_t* expert_counts, float* aux_loss,
                          int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                          float* f_out, float* P_out, void* workspace, size_t workspace_bytes,
                          void* stream, void* const* events);
int moe_launch_count_fp8(const moe_config* cfg, int32_t* launches);

/*
 * moe_forward_fp8_all -- moe_forward_fp8 with the down expert weights stored
 * as e4m3 as well:
 *   W2q  [E, d, f] uint8: e4m3 codes (the encoding of W1q);
 *   W2s  [E, d] float32: one scale per output channel, so that
 *        W2[e][n][c] = W2s[e][n] * e4m3(W2q[e][n][c]).
 * The down projection reads h in bf16 as moe_forward_fp8 does; the codes are
 * expanded to bf16 on chip (exactly: every e4m3 value is a bf16 value), the
 * products accumulate in float32 and each accumulator is multiplied by its
 * channel's scale before the bf16 rounding of the expert output.  So no
 * rounding decision moves to the activations and the parity bar stays that
 * of moe_forward_fp8; the down weights stream at one byte each.  Every other
 * argument, requirement, workspace size (moe_workspace_size_fp8) and launch
 * count (moe_launch_count_fp8) is moe_forward_fp8's; W2q and W2s 16-byte
 * aligned, else MOE_ERR_ARG; f a multiple of 16 (a row of codes is read by
 * TMA) and no MOE_TUNE_FUSED_COMBINE override of 1, else
 * MOE_ERR_UNSUPPORTED.  NaN codes (0x7F, 0xFF) are not weights: they are
 * read as +-480.  The down projection multiplies the weights as the MMA's N
 * operand (token rows as M), or, where expert segments average at most one
 * row in eight, as its M operand (MOE_TUNE_F8_DOWN_FORM overrides); the
 * results agree within float32 accumulation.  moe_forward_fp8_all_timed takes the stage
 * events of moe_forward_fp8_timed; moe_forward_fp8_all_host_io_batches is
 * moe_forward_fp8_host_io_batches for this layer.  The e4m3 down weights pay
 * on decode-sized batches; on prefill-sized ones the on-chip expansion costs
 * more than the halved weight bytes save.
 */
int moe_forward_fp8_all(const moe_config* cfg, const void* x, const void* W_r,
                        const float* logit_offset, const float* sel_bias,
                        const uint8_t* W1q, const float* W1s, const uint8_t* W3q, const float* W3s,
                        const uint8_t* W2q, const float* W2s, void* y, int32_t* topk_idx,
                        float* topk_w, int32_t* expert_counts, float* aux_loss,
                        int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                        float* f_out, float* P_out, void* workspace, size_t workspace_bytes,
                        void* stream);
int moe_forward_fp8_all_timed(const moe_config* cfg, const void* x, const void* W_r,
                              const float* logit_offset, const float* sel_bias,
                              const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                              const float* W3s, const uint8_t* W2q, const float* W2s, void* y,
                              int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                              float* aux_loss, int32_t* routed_counts, int32_t* offsets,
                              int32_t* slot_pos, float* f_out, float* P_out, void* workspace,
                              size_t workspace_bytes, void* stream, void* const* events);

/*
 * moe_router_z_loss -- the router z-loss of a batch of router logits:
 *     z_loss[0] = (1/T) * sum_t ( log sum_e exp(scores[t, e]) )^2
 * "Mixture of Experts" (llm-tutorial ch. 11) § Why MoE is hard names the
 * ST-MoE router z-loss, which penalises large router logits; the pages give
 * no formula, and this is the ST-MoE form without its coefficient (the caller
 * scales it).  scores: [T, E] float32 row-major device memory, finite values,
 * e.g. from moe_router_scores (offset included).  z_loss: one float32 on the
 * device.  T = 0 writes 0.  The log-partition function of each token is taken
 * in float32 with the running row maximum subtracted; the squares are summed
 * in double in a fixed order, so repeated calls give identical bits.  One
 * launch of a single 8-CTA thread-block cluster; no workspace.
 * Errors: MOE_ERR_ARG for T < 0, E outside 1..512, NULL or unaligned (4-byte)
 * pointers; MOE_ERR_DEVICE, MOE_ERR_CUDA as elsewhere.
 */
int moe_router_z_loss(const float* scores, int32_t T, int32_t E, float* z_loss, void* stream);

/*
 * moe_bias_update -- one step of auxiliary-loss-free balancing ("Mixture of
 * experts" (inside-the-model guide) § Auxiliary-loss-free balancing): the
 * selection bias of every expert (sel_bias [E] float32, device, updated in
 * place; the same array moe_forward takes) moves
 *     down by gamma  when routed_counts[i] * E > T * k   (above the mean load),
 *     up by gamma    when routed_counts[i] * E < T * k   (below it),
 * and stays when the expert carries exactly the mean load.  routed_counts
 * [E] int32 (device) is the pre-drop count per expert that moe_forward or
 * moe_route wrote for the T-token batch with top-k; each change is one
 * float32 add, rounded to nearest.  The comparison is exact integer
 * arithmetic.  Errors: MOE_ERR_ARG for E outside 1..512, T < 0, k outside
 * 1..E, NULL or unaligned pointers, gamma negative or not finite.
 */
int moe_bias_update(const int32_t* routed_counts, int32_t E, int32_t T, int32_t k, float gamma,
                    float* sel_bias, void* stream);

/*
 * moe_forward_host_io -- moe_forward with the activations in HOST memory:
 * x_host [T, d] is copied to the device, the layer runs, and y_host [T, d]
 * and aux_loss_host [1] are copied back, all enqueued on `stream` (pinned
 * host memory makes the copies asynchronous; the caller synchronises before
 * reading y_host).  Weights, logit_offset and sel_bias are device pointers
 * as in moe_forward.  topk_idx / topk_w / counts stay in the workspace.
 * Needs moe_host_io_workspace_size() bytes.
 */
int moe_host_io_workspace_size(const moe_config* cfg, size_t* bytes);
int moe_forward_host_io(const moe_config* cfg,
                        const void* x_host, const void* W_r,
                        const float* logit_offset, const float* sel_bias,
                        const void* W1, const void* W3, const void* W2,
                        const void* Ws1, const void* Ws3, const void* Ws2,
                        void* y_host, float* aux_loss_host,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_forward_fp8_host_io -- moe_forward_fp8 with the activations in HOST
 * memory, as moe_forward_host_io is to moe_forward: x_host [T, d] bf16 is
 * copied to the device, the layer runs with the e4m3 gate/up weights, and
 * y_host [T, d] bf16 and aux_loss_host [1] are copied back, all enqueued on
 * `stream`.  Weights, scales, logit_offset and sel_bias are device pointers
 * as in moe_forward_fp8.  Needs moe_host_io_workspace_size_fp8() bytes.
 */
int moe_host_io_workspace_size_fp8(const moe_config* cfg, size_t* bytes);
int moe_forward_fp8_host_io(const moe_config* cfg, const void* x_host, const void* W_r,
                            const float* logit_offset, const float* sel_bias,
                            const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                            const float* W3s, const void* W2, void* y_host,
                            float* aux_loss_host, void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * moe_forward_host_io_batches / moe_forward_fp8_host_io_batches -- n_batches
 * layer calls on host-memory batches (x_host[i] -> y_host[i], aux_loss_host[i]),
 * with the copies of one batch overlapping the layer of another: batch i+1's
 * x travels to the device while batch i computes, and batch i's y travels back
 * while batch i+1 computes.  The layer runs on `stream`, the copies to the
 * device on `copy_in_stream` and the copies back on `copy_out_stream` (both
 * different from `stream`; they may be the same stream, in which case the two
 * directions take turns).  All three streams are the caller's.  Every other
 * argument is that of moe_forward_host_io (resp. moe_forward_fp8_host_io),
 * with arrays of n_batches host pointers in place of x_host / y_host and
 * n_batches floats at aux_loss_host; pinned host memory makes the copies
 * asynchronous.  The workspace (moe_host_io_workspace_size, resp. _fp8) holds
 * two staging slots.  When the call returns, `stream` waits for every copy:
 * synchronising `stream` makes all y_host and losses valid.
 * Errors: MOE_ERR_ARG for n_batches < 0, NULL arrays or entries, or a copy
 * stream equal to `stream`; otherwise those of moe_forward_host_io.
 */
int moe_forward_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                const void* const* x_host, const void* W_r,
                                const float* logit_offset, const float* sel_bias, const void* W1,
                                const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                                const void* Ws2, void* const* y_host, float* aux_loss_host,
                                void* workspace, size_t workspace_bytes, void* stream,
                                void* copy_in_stream, void* copy_out_stream);
int moe_forward_fp8_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                    const void* const* x_host, const void* W_r,
                                    const float* logit_offset, const float* sel_bias,
                                    const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                                    const float* W3s, const void* W2, void* const* y_host,
                                    float* aux_loss_host, void* workspace,
                                    size_t workspace_bytes, void* stream, void* copy_in_stream,
                                    void* copy_out_stream);
int moe_forward_fp8_all_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                        const void* const* x_host, const void* W_r,
                                        const float* logit_offset, const float* sel_bias,
                                        const uint8_t* W1q, const float* W1s,
                                        const uint8_t* W3q, const float* W3s,
                                        const uint8_t* W2q, const float* W2s,
                                        void* const* y_host, float* aux_loss_host,
                                        void* workspace, size_t workspace_bytes, void* stream,
                                        void* copy_in_stream, void* copy_out_stream);

/*
 * Synchronises `stream`, then reads and clears the device status word in
 * `workspace`.  Returns MOE_OK, MOE_ERR_TIMEOUT when a bounded device wait
 * gave up since the last check, MOE_ERR_BOUNDS when the bounds-checked build
 * (libmoe_check.so, the same ABI compiled with MOE_CHECK=1: every index that
 * routing produces is range-tested before the access it drives, and a failed
 * test skips the access instead of trapping) found an index out of range, or
 * MOE_ERR_CUDA if the synchronisation itself failed.
 */
int moe_check_status(void* workspace, void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* moe_error_string(int code);

/* ---- measurement support ------------------------------------------------ */

/* Stages in the order moe_forward enqueues them. */
enum {
  MOE_STAGE_ROUTER = 0,   /* router logits (float32 GEMM) */
  MOE_STAGE_TOPK = 1,     /* top-k, gates, router distribution, expert counts, and the
                             capacity scan: offsets, tile schedule, f, P, L */
  MOE_STAGE_PERMUTE = 2,  /* slot positions and the copy into expert order */
  MOE_STAGE_UP = 3,       /* expert up projection (+ activation / SwiGLU) */
  MOE_STAGE_DOWN = 4,     /* expert down projection */
  MOE_STAGE_COMBINE = 5,  /* gate-weighted combine (+ shared expert) */
  MOE_NUM_STAGES = 6      /* one kernel per stage */
};

/*
 * Same as moe_forward, and also records events[i] (a cudaEvent_t passed as
 * void*) on `stream` before stage i, and events[MOE_NUM_STAGES] after the
 * last one: MOE_NUM_STAGES + 1 caller-created events.  Used to time each
 * kernel on the stream it runs on.
 */
int moe_forward_timed(const moe_config* cfg,
                      const void* x, const void* W_r,
                      const float* logit_offset, const float* sel_bias,
                      const void* W1, const void* W3, const void* W2,
                      const void* Ws1, const void* Ws3, const void* Ws2,
                      void* y, int32_t* topk_idx, float* topk_w,
                      int32_t* expert_counts, float* aux_loss,
                      int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                      float* f_out, float* P_out,
                      void* workspace, size_t workspace_bytes, void* stream,
                      void* const* events);

/* Number of kernels one moe_forward call launches for this layer. */
int moe_launch_count(const moe_config* cfg, int32_t* launches);

/*
 * The kernel path a moe_forward call takes for this layer (under the current
 * moe_set_tuning overrides), as a set of MOE_PLAN_* bits: routing in one
 * launch (E <= 64), in one launch of thread-block clusters (64 < E <= 256),
 * or by the decode-batch router (T <= 16); the routed token rows gathered by
 * the up projection instead of copied; the combine inside the down
 * projection; the up and down projections in one launch.  Host only: plans,
 * launches nothing.  Errors: those of moe_workspace_size.
 */
enum {
  MOE_PLAN_ROUTE_ONE_LAUNCH = 1,
  MOE_PLAN_ROUTE_CLUSTER = 2,
  MOE_PLAN_ROUTE_DECODE = 4,
  MOE_PLAN_GATHER_ROWS = 8,
  MOE_PLAN_COMBINE_IN_DOWN = 16,
  MOE_PLAN_FUSED_PROJECTIONS = 32
};
int moe_plan_flags(const moe_config* cfg, uint32_t* flags);
/* The same for a moe_forward_fp8 / moe_forward_fp8_all call (errors: those of
 * moe_workspace_size_fp8). */
int moe_plan_flags_fp8(const moe_config* cfg, uint32_t* flags);

/*
 * moe_set_tuning -- process-wide override of a kernel choice, for tests and
 * tile sweeps only; production callers leave every knob at its default.
 * Later calls of every entry point (on every thread and device) plan with
 * the override; the results stay within the layer's parity tolerance whatever
 * the choice, only the kernels and their speed change.  value -1 restores the
 * library's own choice.
 *   MOE_TUNE_ROUTER          MOE_ROUTER_SIMT (split float32 FMA logits),
 *                            MOE_ROUTER_FUSED (fused float32 router),
 *                            MOE_ROUTER_TC (tensor-core logits, bf16 only);
 *   MOE_TUNE_GATHER          0: the up projection reads an expert-ordered copy
 *                            of the rows; 1: it gathers the rows of x itself
 *                            with cp.async; 2: with the TMA row gather;
 *   MOE_TUNE_TILE_N_UP / _DOWN  output columns per tensor-core tile (one of the
 *                            compiled widths, else ignored);
 *   MOE_TUNE_PARTIAL_A_ROWS  tiles with at most this many rows load only them;
 *   MOE_TUNE_MMA_M64         1 (the default): expert tiles of at most 64 rows
 *                            multiply with M = 64, 0: always M = 128;
 *   MOE_TUNE_FUSED_COMBINE   1: bf16 layers with k > 1 or a shared expert
 *                            combine in the down projection's epilogue (the
 *                            last row of each token's column slice sums it, in
 *                            the fixed slot order); 0 (the default): a separate
 *                            combine kernel.  y is the same bit for bit;
 *   MOE_TUNE_CLUSTER         1: the TMA-fed expert projections run as clusters
 *                            of two CTAs on adjacent column tiles sharing one
 *                            multicast A tile; 0 (the default): single CTAs;
 *   MOE_TUNE_FUSED_PROJ      1: the up and down projections run as one
 *                            persistent launch wherever a form is compiled for
 *                            the layer's tiling (down tiles wait, bounded, for
 *                            the up tiles of their rows); 0: always two
 *                            launches; the default takes one launch for the
 *                            form that measured faster (gathered ReLU up
 *                            projection with the combine in the down
 *                            projection);
 *   MOE_TUNE_F8_DOWN_FORM    moe_forward_fp8_all's down projection: 1 the
 *                            weights as the MMA's M operand (128 output
 *                            channels per tile, 32 token rows per pass), 0
 *                            the weights as its N operand (token rows as M);
 *                            the default takes the first where segments
 *                            average at most one row in eight (8*T*k <= E).
 * Errors: MOE_ERR_ARG for an unknown knob or a value out of range.  Not
 * synchronised with calls in flight on other threads.
 */
enum {
  MOE_TUNE_ROUTER = 0,
  MOE_TUNE_GATHER = 1,
  MOE_TUNE_TILE_N_UP = 2,
  MOE_TUNE_TILE_N_DOWN = 3,
  MOE_TUNE_PARTIAL_A_ROWS = 4,
  MOE_TUNE_MMA_M64 = 5,
  MOE_TUNE_FUSED_COMBINE = 6,
  MOE_TUNE_CLUSTER = 7,
  MOE_TUNE_FUSED_PROJ = 8,
  MOE_TUNE_F8_DOWN_FORM = 9,
  MOE_TUNE_COUNT = 10
};
enum { MOE_ROUTER_SIMT = 1, MOE_ROUTER_FUSED = 2, MOE_ROUTER_TC = 3 };
int moe_set_tuning(int32_t knob, int32_t value);

/*
 * Self-test of the bounded device waits: launches one block that waits on
 * a barrier nothing will complete, for at most `wait_ns` nanoseconds, then
 * records a timeout in the workspace status word and returns.  A following
 * moe_check_status returns MOE_ERR_TIMEOUT.
 * The workspace needs at least 256 bytes.
 */
int moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                              uint64_t wait_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
