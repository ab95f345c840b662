// moe_internal.h -- host-side plan of one layer call and the launchers of
// the individual kernels.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kThreads = 256;        // block size of the SIMT kernels
constexpr int kRouteTokensPerPass = 16;   // tokens a top-k block handles at once (one per warp)
constexpr int kRouteMaxBlocks = 128;      // routing blocks are sized to stay near this count
constexpr int kRouteMaxBT = 256;
constexpr int kFusedMinT = 1024;          // smaller batches route through the split path
constexpr int kRouterTcMinT = 256;        // bf16 batches from this size use the tensor-core router
constexpr int kMaxE = 512;
constexpr int kMaxK = 32;
constexpr int kSegAlign = 128;       // expert segments start on multiples of this row
constexpr int kTcBM = 128;           // rows per tensor-core tile
constexpr int kSimtBM = 64;          // rows per SIMT tile (fp32 path)
constexpr int kSimtBN = 64;
// Workspace header (zeroed once by the caller): status word at 0, routing
// block-completion counter at 16, the one-launch routers' grid-wait
// counters (arrivals, passes) at 32 and 48 (and 96 and 112, with the row
// copy's counters at 64 and 80), router split-reduction tile
// counters from kTileCounterOffset on.  Every counter is back at zero when a
// call has finished without a timeout.
constexpr int kWsHeaderBytes = 4096;
constexpr int kRouteDoneOffset = 16;
constexpr int kRouteArriveOffset = 32;
constexpr int kRoutePassedOffset = 48;
// The one-launch router for E <= 256: its row-copy work counter and finished
// count, and the counters of its second grid-wide wait.
constexpr int kRouteCopyNextOffset = 64;
constexpr int kRouteCopyDoneOffset = 80;
constexpr int kRouteArrive2Offset = 96;
constexpr int kRoutePassed2Offset = 112;
// Up and down projections in one launch: the CTAs that have finished, the
// up tiles stored in all; the per-M-tile counts of stored up tiles use the
// tile-counter area (only one of
// the two is in use at a time, and both are zero between launches).
constexpr int kUpDownFinOffset = 128;
constexpr int kUpDownAllOffset = 144;   // up tiles stored in all
constexpr int kRouteTcMaxOwn = 16;        // 128-token tiles per CTA of the one-launch router
// One-launch router for 64 < E <= 256 (route_wide.cu): top-k of at most
// kRouteWideMaxK, at most kRouteWideMaxOwn tiles per cluster, a grid of at
// most kRouteWideMaxCtas CTAs, and clusters sized for one wave of
// kRouteWideSlots SMs.
constexpr int kRouteWideMaxK = 8;
constexpr int kRouteWideMaxOwn = 16;
constexpr int kRouteWideMaxCtas = 160;
constexpr int kRouteWideSlots = 148;
// Layers routed by it whose experts average at most this many rows gather
// their rows in the up projection instead of copying them.
constexpr int kWideGatherRows = 32;
constexpr int kSmallT = 16;               // batches up to this size route in one small launch
constexpr int kSmallMaxE = 256;
constexpr int kTileCounterOffset = 256;
constexpr int kMaxTileCounters = (kWsHeaderBytes - kTileCounterOffset) / 4;

// Workspace regions, all 256-byte aligned.  Offsets in bytes.
struct WsLayout {
  size_t status;      // uint32 status word (+ padding)
  size_t scores;      // float  [T][E]     router logits
  size_t score_parts; // float  [S][T][E]  split partial router logits (S > 1)
  size_t blk_cnt;     // int32  [nblk][Es] per-block expert histogram (Es = E rounded up to 4)
  size_t blk_prob;    // float  [nblk][Es] per-block sums of the router distribution
  size_t meta;        // int32  kept[E] | offsets[E+1] | seg_start[E+1] | mtiles[E+1]
                      //        | tp_up[E+2] | tp_dn[E+2]
  size_t key_row;     // int32  [T*k]      padded row of each assignment, -1 if dropped
  size_t row_token;   // int32  [R_cap]    token of each expert-ordered row
  size_t xp;          // dtype  [R_cap][d] token copies in expert order (absent when the
                      //        tensor-core up projection gathers the rows of x itself)
  size_t xq;          // uint8  [R_cap][d] e4m3 token rows in expert order (fp8 weights only)
  size_t xs;          // float  [R_cap]    their power-of-two scales
  size_t h;           // dtype  [R_cap][f] expert hidden activations
  size_t o;           // dtype  [R_cap][d] expert outputs
  size_t hs;          // dtype  [T_pad][f_s] shared-expert hidden
  size_t os;          // [T_pad][d] shared-expert output: float32 (float32 path), or fp16
                      //        scaled per 32-column chunk (tensor-core path)
  size_t os_exp;      // int8   [T_pad][ceil(d/32)] the chunk exponents (tensor-core path)
  size_t cmb_ctr;     // uint32 [T][N tiles of the down projection]: combine arrival counters
  // host-io staging
  size_t x_dev, y_dev, topk_idx, topk_w, counts, aux;
  size_t x_dev2, y_dev2, aux2;   // second staging slot (pipelined batches)
  size_t total;
};

struct Plan {
  moe_config cfg;
  int elem;           // bytes per element of x / weights / y
  int capacity;       // INT32_MAX when unlimited
  int BT;             // tokens per routing block
  int nblk;           // routing blocks
  bool router_tc;     // router logits on the tensor cores
  bool route_tc;      // stages 1-4 in one tensor-core launch (bf16, E <= 64, k <= 8)
  bool route_small;   // stages 1-4 in one launch for decode batches (T <= kSmallT)
  bool route_wide;    // stages 1-4 and the row copy in one launch (bf16, 64 < E <= 256, k <= 8)
  int rw_ks;          // that router's CTAs per 128-token tile
  int blk_stride;     // row stride of blk_cnt / blk_prob (E rounded up to 4)
  bool router_fused;  // one kernel: logits, top-k, histogram, scan (E <= 256)
  int fu_tm, fu_tn;   // fused router: tokens per thread (1, 2), experts per thread
  int sc_tn;          // router GEMM: experts per thread (2 or 4)
  int sc_mblocks, sc_nblocks, sc_splits, sc_ksplit;   // router GEMM grid and K split
  int bm;             // rows per GEMM tile (128 tensor core, 64 SIMT)
  int R_cap;          // rows reserved for the expert-ordered buffers
  int T_pad;          // T rounded up to kSegAlign
  bool tc;            // tensor-core path (bf16)
  // GEMM tiling
  int up_bn;          // output columns per up-projection tile
  int dn_bn;          // output columns per down-projection tile
  int nt_up, nt_dn;           // N tiles of a routed segment
  int nt_up_sh, nt_dn_sh;     // N tiles of the shared segment
  int mt_sh;                  // M tiles of the shared segment
  int max_tiles_up, max_tiles_dn;  // host upper bounds (grid sizing)
  int partial_rows;           // A tiles with at most this many rows load only those rows
  int partial_rows_up;        // the same for the up projection
  bool combine_in_down;       // top-1, no shared expert, bf16: y written by the down epilogue
  bool combine_k;             // other bf16 layers: the down epilogue's last row per token sums y
  bool gather;                // the up projection gathers token rows with cp.async
  bool gather4;               // the up projection gathers token rows with TMA (tile::gather4)
  bool m64;                   // routed GEMM tiles of <= 64 rows multiply with M = 64
  bool cluster2_up;           // the up projection runs as 2-CTA clusters sharing the A tile
  bool cluster2_dn;           // the same for the down projection
  bool fp8;                   // gate/up weights in e4m3: quantised rows, fp8 up projection
  bool fused;                 // up and down projections in one persistent launch
  bool dn_swap;               // e4m3 down weights: the weights as the MMA's M operand
  int num_sms;
  WsLayout ws;
};

enum class WsKind { Forward, Route, HostIO, ForwardFp8, HostIOFp8 };

int make_plan(const moe_config* cfg, WsKind kind, Plan* p);

// Current override of a moe_set_tuning knob, -1 when none is set.
int tuning(int knob);

// Device pointers of the meta region.
struct Meta {
  int* kept;
  int* offsets;
  int* seg_start;
  int* mtiles;
  int* tp_up;
  int* tp_dn;
};
Meta meta_ptrs(const Plan& p, void* ws);

// ---- launchers (return a cudaError_t of the launch) ----------------------
// Caller-visible outputs of the capacity scan.
struct ScanOutputs {
  int32_t* expert_counts;
  float* aux_loss;
  int32_t* routed_counts;
  int32_t* offsets;
  float* f_out;
  float* P_out;
};

cudaError_t launch_router(const Plan& p, const void* x, const void* W_r, const float* logit_offset,
                          const float* sel_bias, int32_t* topk_idx, float* topk_w, void* ws,
                          const ScanOutputs& so, cudaStream_t st, cudaEvent_t mid_event);
bool route_tc_eligible(const moe_config& c);
cudaError_t launch_route_tc(const Plan& p, const void* x, const void* W_r,
                            const float* logit_offset, const float* sel_bias, int32_t* topk_idx,
                            float* topk_w, int32_t* slot_pos, void* ws, const ScanOutputs& so,
                            cudaStream_t st);
cudaError_t launch_gather_rows(const Plan& p, const void* x, void* ws, cudaStream_t st);
bool route_wide_eligible(const moe_config& c);
int route_wide_ks(const moe_config& c);
bool route_wide_copies_rows(const Plan& p);
// Stages 1-4 and, when `copy`, the expert-ordered row copies (in the same
// launch when a row fits the kernel's staging three times, else by the row
// copy kernel after it).
cudaError_t launch_route_wide(const Plan& p, const void* x, const void* W_r,
                              const float* logit_offset, const float* sel_bias,
                              int32_t* topk_idx, float* topk_w, int32_t* slot_pos, bool copy,
                              void* ws, const ScanOutputs& so, cudaStream_t st);
size_t route_small_smem(int E);
int route_small_splits(int d);
cudaError_t launch_route_small(const Plan& p, const void* x, const void* W_r,
                               const float* logit_offset, const float* sel_bias,
                               int32_t* topk_idx, float* topk_w, int32_t* slot_pos, bool copy_rows,
                               void* ws, const ScanOutputs& so, cudaStream_t st);
cudaError_t launch_router_tc(const Plan& p, const void* x, const void* W_r,
                             const float* logit_offset, float* scores, uint32_t* status,
                             cudaStream_t st);
cudaError_t launch_router_scores(const Plan& p, const void* x, const void* W_r,
                                 const float* logit_offset, float* out, void* ws,
                                 cudaStream_t st);
cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* topk_idx,
                           int32_t* slot_pos, bool copy_rows, void* ws, cudaStream_t st,
                           void* y);
cudaError_t launch_experts_tc(const Plan& p, const void* x, const void* W1, const void* W3,
                              const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                              void* ws, cudaStream_t st, cudaEvent_t mid_event, void* y,
                              const float* topk_w, const float* W1s = nullptr,
                              const float* W3s = nullptr, const float* W2s = nullptr);
cudaError_t launch_quant_rows(const Plan& p, const void* x, void* ws, cudaStream_t st);
// Up and down projections in one launch: compiled for this tiling and the
// counters fit the workspace header.
bool updown_eligible(const Plan& p);
bool updown_default(const Plan& p);   // eligible forms that run as one launch by default
int updown_counters(const Plan& p);
cudaError_t launch_experts_simt(const Plan& p, const void* x, const void* W1, const void* W3,
                                const void* W2, const void* Ws1, const void* Ws3,
                                const void* Ws2, void* ws, cudaStream_t st,
                                cudaEvent_t mid_event);
cudaError_t launch_combine(const Plan& p, const float* topk_w, void* y, void* ws,
                           cudaStream_t st);
cudaError_t launch_router_z_loss(const float* scores, int T, int E, float* z_loss,
                                 cudaStream_t st);
cudaError_t launch_bias_update(const int32_t* routed_counts, int E, int T, int k, float gamma,
                               float* sel_bias, cudaStream_t st);
cudaError_t launch_selftest_wait(uint32_t* status, uint64_t wait_ns, cudaStream_t st);

}  // namespace moe
