// moe_api.cu -- the C ABI declared in include/moe.h: argument checks, the
// per-call plan (workspace layout, routing blocks, GEMM tiling) and the
// enqueueing of the stage kernels on the caller's stream.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Output columns per tile: minimise (waves of tiles over the SMs) x (bytes a
// tile moves per k: B rows = mma_mult * bn weight rows plus the 128-row A
// tile re-read for every N tile); ties go to the wider tile.  Matches tile
// sweeps on B300 (Switch, gpt-oss decode, DeepSeek-V3 shapes).
static int choose_bn(const int* cands, int ncand, int N, long long est_mtiles, long long extra_m,
                     int N_extra, int num_sms, int mma_mult) {
  int best = cands[0];
  long long best_cost = LLONG_MAX;
  for (int i = 0; i < ncand; ++i) {
    const int bn = cands[i];
    const long long tiles = est_mtiles * ceil_div(N, bn) + extra_m * ceil_div(N_extra, bn);
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const long long cost = waves * (mma_mult * bn + kTcBM);
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

int make_plan(const moe_config* cfg, WsKind kind, Plan* p, int num_sms);

// Process-wide overrides set through moe_set_tuning (tests and tile sweeps
// only); -1 = no override.  Production calls never read the environment.
static std::atomic<int> g_tune[MOE_TUNE_COUNT] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1};

int tuning(int knob) {
  return knob >= 0 && knob < MOE_TUNE_COUNT ? g_tune[knob].load(std::memory_order_relaxed) : -1;
}

int make_plan(const moe_config* cfg, WsKind kind, Plan* p) { return make_plan(cfg, kind, p, 0); }

int make_plan(const moe_config* cfg, WsKind kind, Plan* p, int num_sms) {
  if (!cfg || !p) return MOE_ERR_ARG;
  const moe_config& c = *cfg;
  if (c.reserved != 0 || c.T < 0 || c.d < 1 || c.E < 1 || c.k < 1 || c.k > c.E || c.f < 1)
    return MOE_ERR_ARG;
  if (c.n_shared != 0 && c.n_shared != 1) return MOE_ERR_ARG;
  if (c.n_shared == 1 && c.f_shared < 1) return MOE_ERR_ARG;
  if (c.dtype != MOE_F32 && c.dtype != MOE_BF16) return MOE_ERR_ARG;
  if (c.act < MOE_ACT_GELU || c.act > MOE_ACT_SWIGLU) return MOE_ERR_ARG;
  if (c.gate < MOE_GATE_SOFTMAX_TOPK || c.gate > MOE_GATE_SOFTMAX_FULL) return MOE_ERR_ARG;
  if (!std::isfinite(c.capacity_factor) || !std::isfinite(c.alpha)) return MOE_ERR_ARG;
  if (c.E > kMaxE || c.k > kMaxK) return MOE_ERR_UNSUPPORTED;
  const int vec = c.dtype == MOE_BF16 ? 8 : 4;
  if (c.d % vec || c.f % vec || (c.n_shared && c.f_shared % vec)) return MOE_ERR_UNSUPPORTED;
  // the tensor-core kernels run the (SwiGLU) shared expert as one more
  // segment of the routed experts' launches, so they need SwiGLU experts too
  if (c.dtype == MOE_BF16 && c.n_shared && c.act != MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED;
  // fp8 gate/up weights: a bf16 SwiGLU layer without a shared expert; rows of
  // d e4m3 bytes must be 16-byte multiples (TMA) and the column scales are
  // read in pairs
  const bool fp8_kind = kind == WsKind::ForwardFp8 || kind == WsKind::HostIOFp8;
  if (fp8_kind &&
      (c.dtype != MOE_BF16 || c.act != MOE_ACT_SWIGLU || c.n_shared != 0 || c.d % 16 ||
       c.f % 4))
    return MOE_ERR_UNSUPPORTED;
  // every row index and element count of one matrix must fit in int32 / the TMA limits
  const long long Tk = (long long)c.T * c.k;
  if (Tk > (1LL << 30) || (long long)c.T * c.d > (1LL << 40)) return MOE_ERR_UNSUPPORTED;

  Plan& P = *p;
  std::memset(&P, 0, sizeof(P));
  P.cfg = c;
  P.fp8 = fp8_kind;
  P.elem = c.dtype == MOE_BF16 ? 2 : 4;
  if (c.capacity_factor > 0) {
    const double cap = std::ceil(static_cast<double>(Tk) * c.capacity_factor / c.E);
    P.capacity = cap >= (double)INT_MAX ? INT_MAX : static_cast<int>(cap);
  } else {
    P.capacity = INT_MAX;
  }
  // Router path.  Fused (E <= 256, batches of at least kFusedMinT tokens):
  // one kernel per 16*TM tokens computes all logits over the full width, then
  // routes; TN = experts per thread = next_pow2(E)/16.  Otherwise the split
  // path: a split-K logits kernel, then the top-k kernel.
  // A router override (moe_set_tuning) of SIMT forces the split path, FUSED
  // the fused one.
  const int router_tune = tuning(MOE_TUNE_ROUTER);
  {
    const bool force_split = router_tune == MOE_ROUTER_SIMT;
    const bool force_fused = router_tune == MOE_ROUTER_FUSED;
    int ep = 32;
    while (ep < c.E) ep <<= 1;
    P.fu_tn = ep <= 256 ? ep / 16 : 0;
    P.fu_tm = ceil_div(c.T, 32) >= 64 ? 2 : 1;
    P.router_fused = P.fu_tn > 0 && !force_split && force_fused;
  }
  // One-launch tensor-core routing (bf16, E <= 64, k <= 8) unless a router
  // override forces another path; its routing blocks are its 128-token tiles.
  {
    const bool forced = router_tune == MOE_ROUTER_SIMT || router_tune == MOE_ROUTER_FUSED ||
                        router_tune == MOE_ROUTER_TC;
    // decode batches (T <= kSmallT): split-K logits, top-k, scan and
    // positions in one small launch
    P.route_small = !forced && c.T >= 1 && c.T <= kSmallT && c.E <= kSmallMaxE;
    P.route_tc = route_tc_eligible(c) && !forced && !P.route_small;
    // 64 < E <= 256: the one-launch cluster router (route_wide.cu)
    P.route_wide = route_wide_eligible(c) && !forced && !P.route_small && !P.route_tc;
    if (P.route_tc || P.route_small || P.route_wide) P.router_fused = false;
  }
  if (P.route_small) {
    P.BT = c.T;
  } else if (P.route_tc) {
    P.BT = kTcBM;
  } else if (P.route_wide) {
    P.rw_ks = route_wide_ks(c);
    P.BT = kTcBM / P.rw_ks;
  } else if (P.router_fused) {
    P.BT = 16 * P.fu_tm;
  } else {
    // routing blocks: 16 tokens per pass (one per warp), enough passes that
    // the batch needs about kRouteMaxBlocks blocks, at most kRouteMaxBT tokens
    const int passes = ceil_div(c.T, kRouteTokensPerPass * kRouteMaxBlocks);
    const int bt = kRouteTokensPerPass * (passes < 1 ? 1 : passes);
    P.BT = bt > kRouteMaxBT ? kRouteMaxBT : bt;
  }
  P.nblk = P.route_wide ? ceil_div(c.T, kTcBM) * P.rw_ks : ceil_div(c.T, P.BT);
  P.blk_stride = (c.E + 3) / 4 * 4;
  P.num_sms = num_sms > 0 ? num_sms : 148;
  // router GEMM: 128-token x (16*TN)-expert tiles, K split until >= 2 blocks per SM
  P.sc_tn = c.E > 32 ? 4 : 2;
  P.sc_mblocks = ceil_div(c.T, 128);
  P.sc_nblocks = ceil_div(c.E, 16 * P.sc_tn);
  {
    // choose the split with the best wave efficiency over 2 blocks per SM
    // (ties: fewer splits), each split at least 128 wide
    const int tiles = P.sc_mblocks * P.sc_nblocks;
    const int max_split = c.d / 128 > 1 ? c.d / 128 : 1;
    const int slots = 2 * 148;    // fixed, so that the workspace layout never depends on the GPU
    int S = 1;
    double best = -1.0;
    for (int s = 1; s <= max_split && tiles > 0; ++s) {
      const int blocks = tiles * s;
      const int waves = ceil_div(blocks, slots);
      double eff = (double)blocks / ((double)waves * slots);
      if (blocks < slots) eff *= 0.999;   // a partial single wave: prefer more work per block
      if (eff > best + 1e-9) {
        best = eff;
        S = s;
      }
      if (waves > 4) break;
    }
    if (tiles > kMaxTileCounters) S = 1;   // plenty of tiles already; no counters needed
    P.sc_ksplit = ceil_div(ceil_div(c.d, S), 32) * 32;
    P.sc_splits = ceil_div(c.d, P.sc_ksplit);
  }
  // Router logits: bf16 layers with at least kRouterTcMinT tokens use the
  // tensor cores with 128-wide float32 chunks (max error ~2e-6 on a 7168-wide
  // router, measured; float32 FMA: ~8e-7); both stay inside half the 1e-5
  // band in which near-tied experts may swap.  Smaller batches and float32
  // layers use the split float32 FMA kernel.  A router override forces a path.
  {
    const bool force_tc = router_tune == MOE_ROUTER_TC;
    const bool forced_other = router_tune == MOE_ROUTER_SIMT || router_tune == MOE_ROUTER_FUSED;
    P.router_tc = c.dtype == MOE_BF16 && (force_tc || (!forced_other && c.T >= kRouterTcMinT));
    if (P.router_tc) P.router_fused = false;
  }
  P.tc = c.dtype == MOE_BF16;
  P.bm = P.tc ? kTcBM : kSimtBM;
  const long long nonempty = Tk < c.E ? Tk : c.E;
  P.R_cap = static_cast<int>(align_up((size_t)(Tk + nonempty * (P.bm - 1)), (size_t)P.bm));
  P.T_pad = static_cast<int>(align_up((size_t)c.T, (size_t)kSegAlign));
  P.mt_sh = c.n_shared ? ceil_div(c.T, P.bm) : 0;

  if (P.tc) {
    long long est = nonempty + Tk / P.bm;
    if (P.capacity != INT_MAX) {
      const long long capb = (long long)c.E * ceil_div(P.capacity, P.bm);
      if (capb < est) est = capb;
    }
    static const int dual_c[] = {128, 96, 64, 32};
    static const int single_c[] = {256, 128, 96, 64};
    static const int down_c[] = {256, 192, 128, 96, 64};
    if (c.act == MOE_ACT_SWIGLU)
      P.up_bn = choose_bn(dual_c, 4, c.f, est, P.mt_sh, c.f_shared, P.num_sms, 2);
    else
      P.up_bn = choose_bn(single_c, 4, c.f, est, P.mt_sh, c.f_shared, P.num_sms, 1);
    P.dn_bn = choose_bn(down_c, 5, c.d, est, P.mt_sh, c.d, P.num_sms, 1);
    // Tuning override (tile sweeps and tests, moe_set_tuning): one of the
    // compiled tile widths; other values are ignored.
    const int up_env = tuning(MOE_TUNE_TILE_N_UP), dn_env = tuning(MOE_TUNE_TILE_N_DOWN);
    const int* up_list = c.act == MOE_ACT_SWIGLU ? dual_c : single_c;
    for (int i = 0; i < 4; ++i)
      if (up_env == up_list[i]) P.up_bn = up_env;
    for (int i = 0; i < 5; ++i)
      if (dn_env == down_c[i]) P.dn_bn = dn_env;
  } else {
    P.up_bn = kSimtBN;
    P.dn_bn = kSimtBN;
  }
  {
    // Partial A tiles (<= 64 real rows loaded as 32-row boxes) measured
    // faster for the single-operand GEMMs (down projections, plain up
    // projections) and slower for the dual-operand SwiGLU up projection.
    const int v = tuning(MOE_TUNE_PARTIAL_A_ROWS);
    P.partial_rows = v >= 0 ? v : 64;
    P.partial_rows_up = v >= 0 ? P.partial_rows : (c.act == MOE_ACT_SWIGLU ? 0 : 64);
    // routed tiles with at most 64 rows (the last tile of a segment, small
    // segments) issue M = 64 MMAs: half the tensor work of an M = 128 tile
    const int m = tuning(MOE_TUNE_MMA_M64);
    P.m64 = m >= 0 ? m != 0 : true;

  }
  P.combine_in_down = P.tc && c.k == 1 && c.n_shared == 0;
  // Other tensor-core layers can combine in the down projection's epilogue
  // as well (the last row of a token's column slice sums it, in the fixed
  // slot order: y is the separate kernel's bit for bit).  The rows it sums
  // were written long before (a token's k slots lie in k different experts),
  // so the fused form moves the same bytes as the separate combine kernel,
  // inside an HBM-bound projection, and stalls its epilogue on the reads:
  // measured slower on every layer shape (DeepSeek-V3-shaped 5.18 -> 5.37 ms,
  // Mixtral-shaped 4.78 -> 4.81, gpt-oss-shaped T = 16 0.486 -> 0.492), so
  // the separate kernel is the default and an override of 1 selects the fused
  // form.
  {
    const int fc = tuning(MOE_TUNE_FUSED_COMBINE);
    P.combine_k = P.tc && !P.combine_in_down && fc == 1;
  }
  // The up projection gathers the token rows itself (cp.async) for
  // tensor-core layers routed in one launch whose experts average at most
  // one 128-row tile: there the weights dominate and the gather costs
  // nothing (measured: Switch layer).  Wider experts re-read each A tile for
  // every N tile, and a gather per N tile costs more than one copy of the
  // rows into expert order (measured on B300 for both the cp.async gather
  // and the TMA row gather, tile::gather4: DeepSeek-V3-shaped up projection
  // 2.96 -> 6.26 ms with the latter), so they read an expert-ordered copy
  // through TMA.  A gather override forces a source: 0 the expert-ordered
  // copy, 1 cp.async, 2 the TMA row gather.
  {
    const long long per_expert = Tk / (c.E > 0 ? c.E : 1);
    P.gather = P.tc && ((P.route_tc && per_expert <= kTcBM) ||
                        (P.route_wide && per_expert <= kWideGatherRows));
    P.gather4 = false;
    const int gv = tuning(MOE_TUNE_GATHER);
    if (gv >= 0 && P.tc) {
      P.gather = gv == 1;
      P.gather4 = gv == 2;
    }
    if (P.fp8) P.gather = P.gather4 = false;   // fp8: the quantised rows are read by TMA
  }
  // On request, the TMA-fed projections run as clusters of two CTAs on
  // adjacent N tiles, each loading half of the shared A tile and multicasting
  // it (the compiled cluster forms: SwiGLU up projections of 128-column tiles,
  // down projections of 192 or 256 columns).  The A tile then crosses from L2
  // once per pair and the power draw drops (SM clock under the cap 1237 ->
  // 1297 MHz on the DeepSeek-V3-shaped layer), but the pair's stages are
  // refilled only when both CTAs have consumed them, and that coupling costs
  // more (DeepSeek-V3-shaped 5.14 -> 5.23 ms; Mixtral-shaped 4.70 -> 4.66),
  // so single CTAs are the default.
  {
    const int cl = tuning(MOE_TUNE_CLUSTER);
    const bool on = cl == 1;
    P.cluster2_up = on && P.tc && !P.fp8 && !P.gather && !P.gather4 &&
                    c.act == MOE_ACT_SWIGLU && P.up_bn == 128;
    P.cluster2_dn = on && P.tc && !P.combine_k && (P.dn_bn == 256 || P.dn_bn == 192);
  }
  P.nt_up = ceil_div(c.f, P.up_bn);
  P.nt_up_sh = c.n_shared ? ceil_div(c.f_shared, P.up_bn) : 0;
  P.nt_dn = ceil_div(c.d, P.dn_bn);
  P.nt_dn_sh = c.n_shared ? ceil_div(c.d, P.dn_bn) : 0;
  P.max_tiles_up = (P.R_cap / P.bm) * P.nt_up + P.mt_sh * P.nt_up_sh;
  P.max_tiles_dn = (P.R_cap / P.bm) * P.nt_dn + P.mt_sh * P.nt_dn_sh;
  // Up and down projections in one persistent launch (down tiles wait for
  // their M tile's up tiles through counters), where a form is compiled for
  // the tiling and measured faster than two launches; a tuning override of 1
  // takes every compiled form, 0 none.
  {
    const int fp = tuning(MOE_TUNE_FUSED_PROJ);
    P.fused = updown_eligible(P) && (fp == 1 || (fp < 0 && updown_default(P)));
  }
  // e4m3 down weights (moe_forward_fp8_all): the weights as the MMA's M
  // operand where expert segments average at most one row in eight (the
  // smallest decode batches: measured faster there), else as its N operand
  {
    const int sw = tuning(MOE_TUNE_F8_DOWN_FORM);
    P.dn_swap = P.fp8 && (sw == 1 || (sw < 0 && 8 * Tk <= (long long)c.E));
  }

  // ---- workspace layout ----
  WsLayout& L = P.ws;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  const size_t E = c.E;
  L.status = take(kWsHeaderBytes);
  L.scores = take(sizeof(float) * (size_t)c.T * E);
  // split partials only when the split float32 router runs (sc_* keep that
  // kernel's geometry whichever path this layer takes)
  const bool split_router = !P.router_tc && !P.router_fused;
  size_t parts = split_router && P.sc_splits > 1 ? sizeof(float) * (size_t)P.sc_splits * c.T * E : 0;
  if (P.route_small) {
    const size_t small = sizeof(float) * (size_t)route_small_splits(c.d) * c.T * E;
    if (small > parts) parts = small;
  }
  L.score_parts = take(parts);
  L.blk_cnt = take(sizeof(int) * (size_t)P.nblk * P.blk_stride);
  L.blk_prob = take(sizeof(float) * (size_t)P.nblk * P.blk_stride);
  L.meta = take(sizeof(int) * (E + (E + 1) * 3 + (E + 2) * 2));
  L.key_row = take(sizeof(int) * (size_t)Tk);
  L.row_token = take(sizeof(int) * (size_t)P.R_cap);
  if (kind != WsKind::Route) {
    const size_t act_elem = P.elem;   // h is bf16 on the tensor-core path, fp32 otherwise
    L.xp = take(P.gather || P.gather4 || P.fp8 ? 0 : (size_t)P.R_cap * c.d * P.elem);
    L.xq = take(P.fp8 ? (size_t)P.R_cap * c.d : 0);
    L.xs = take(P.fp8 ? (size_t)P.R_cap * sizeof(float) : 0);
    L.h = take((size_t)P.R_cap * c.f * act_elem);
    // expert outputs in the layer dtype: bf16 rounded once from the float32
    // accumulator on the tensor-core path, float32 otherwise
    L.o = take((size_t)P.R_cap * c.d * P.elem);
    if (c.n_shared) {
      L.hs = take((size_t)P.T_pad * c.f_shared * act_elem);
      // the shared expert's output: float32 on the float32 path; fp16 with a
      // power-of-two exponent per 32-column chunk on the tensor-core path
      // (shared_out.cuh)
      L.os = take((size_t)P.T_pad * c.d * (P.tc ? 2 : 4));
      L.os_exp = take(P.tc ? (size_t)P.T_pad * ((c.d + 31) / 32) : 0);
    }
    // sized for the narrowest down tile (64 columns), so that the layout does
    // not depend on the tiling (which follows the GPU's SM count)
    L.cmb_ctr = take(P.combine_k ? sizeof(unsigned) * (size_t)c.T * ceil_div(c.d, 64) : 0);
  }
  if (kind == WsKind::HostIO || kind == WsKind::HostIOFp8) {
    L.x_dev = take((size_t)c.T * c.d * P.elem);
    L.y_dev = take((size_t)c.T * c.d * P.elem);
    L.topk_idx = take(sizeof(int) * (size_t)Tk);
    L.topk_w = take(sizeof(float) * (size_t)Tk);
    L.counts = take(sizeof(int) * E);
    L.aux = take(sizeof(float));
    L.x_dev2 = take((size_t)c.T * c.d * P.elem);
    L.y_dev2 = take((size_t)c.T * c.d * P.elem);
    L.aux2 = take(sizeof(float));
  }
  L.total = off;
  return MOE_OK;
}

// Per-device facts, read once per device (the values never change while the
// process runs).  0 = not read yet, else the SM count or -1 for "not sm_103".
static std::atomic<int> g_dev_sms[64];

static int device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    const int v = g_dev_sms[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *sms = v;
      return MOE_OK;
    }
    if (v < 0) return MOE_ERR_DEVICE;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) g_dev_sms[dev].store(ok ? *sms : -1, std::memory_order_relaxed);
  return ok ? MOE_OK : MOE_ERR_DEVICE;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Tensors {
  const void *x, *W_r;
  const float *logit_offset, *sel_bias;
  const void *W1, *W3, *W2, *Ws1, *Ws3, *Ws2;
  void* y;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* expert_counts;
  float* aux_loss;
  int32_t *routed_counts, *offsets, *slot_pos;
  float *f_out, *P_out;
  const float *W1s = nullptr, *W3s = nullptr;   // fp8 gate/up weights: column scales
  const float* W2s = nullptr;   // fp8 down weights too (W2 holds e4m3 codes): column scales
};

static int check_tensors(const moe_config& c, const Tensors& t, bool route_only) {
  // With T = 0 the per-token tensors are empty and may be NULL.
  const bool empty = c.T == 0;
  if (!t.W_r || !t.expert_counts || !t.aux_loss) return MOE_ERR_ARG;
  if (!empty && (!t.x || !t.topk_idx || !t.topk_w)) return MOE_ERR_ARG;
  if (!aligned16(t.x) || !aligned16(t.W_r) || !aligned4(t.topk_idx) || !aligned4(t.topk_w))
    return MOE_ERR_ARG;
  if (route_only) return MOE_OK;
  if (!t.W1 || !t.W2 || (!empty && !t.y)) return MOE_ERR_ARG;
  if (!aligned16(t.W1) || !aligned16(t.W2) || !aligned16(t.y)) return MOE_ERR_ARG;
  if (c.act == MOE_ACT_SWIGLU ? (!t.W3 || !aligned16(t.W3)) : t.W3 != nullptr) return MOE_ERR_ARG;
  if ((t.W1s != nullptr) != (t.W3s != nullptr)) return MOE_ERR_ARG;
  if (t.W1s && (!aligned16(t.W1s) || !aligned16(t.W3s))) return MOE_ERR_ARG;
  if (t.W2s && (!t.W1s || !aligned16(t.W2s))) return MOE_ERR_ARG;
  if (c.n_shared) {
    if (!t.Ws1 || !t.Ws3 || !t.Ws2) return MOE_ERR_ARG;
    if (!aligned16(t.Ws1) || !aligned16(t.Ws3) || !aligned16(t.Ws2)) return MOE_ERR_ARG;
  } else if (t.Ws1 || t.Ws3 || t.Ws2) {
    return MOE_ERR_ARG;
  }
  return MOE_OK;
}

static int check_workspace(const Plan& p, const void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < p.ws.total)
    return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define MOE_TRY_CUDA(expr)                       \
  do {                                           \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

static int zero_outputs(const moe_config& c, const Tensors& t, cudaStream_t st) {
  const size_t E = c.E;
  MOE_TRY_CUDA(cudaMemsetAsync(t.expert_counts, 0, E * sizeof(int32_t), st));
  MOE_TRY_CUDA(cudaMemsetAsync(t.aux_loss, 0, sizeof(float), st));
  if (t.routed_counts) MOE_TRY_CUDA(cudaMemsetAsync(t.routed_counts, 0, E * sizeof(int32_t), st));
  if (t.offsets) MOE_TRY_CUDA(cudaMemsetAsync(t.offsets, 0, (E + 1) * sizeof(int32_t), st));
  if (t.f_out) MOE_TRY_CUDA(cudaMemsetAsync(t.f_out, 0, E * sizeof(float), st));
  if (t.P_out) MOE_TRY_CUDA(cudaMemsetAsync(t.P_out, 0, E * sizeof(float), st));
  return MOE_OK;
}

static int record(void* const* events, int i, cudaStream_t st) {
  if (events && events[i])
    MOE_TRY_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(events[i]), st));
  return MOE_OK;
}

static int forward_impl(const moe_config* cfg, const Tensors& t, void* ws, size_t ws_bytes,
                        cudaStream_t st, void* const* events, bool route_only, WsKind kind) {
  if (!cfg) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, kind, &p, 0);
  if (rc != MOE_OK) return rc;
  rc = check_tensors(*cfg, t, route_only);
  if (rc != MOE_OK) return rc;
  if (p.fp8 != (t.W1s != nullptr)) return MOE_ERR_ARG;   // fp8 weights come with their scales
  rc = check_workspace(p, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  int sms = 0;
  rc = device_sms(&sms);
  if (rc != MOE_OK) return rc;
  if (sms != p.num_sms) {        // tiling depends on the SM count; the layout does not
    rc = make_plan(cfg, kind, &p, sms);
    if (rc != MOE_OK) return rc;
  }
  const moe_config& c = *cfg;
  // e4m3 down weights: rows of f code bytes are TMA rows (16-byte multiples);
  // the down kernel writes the expert outputs or combines a top-1 layer in
  // its epilogue, so the k-slot combine override has no form with them
  if (t.W2s && (c.f % 16 || p.combine_k || p.fused)) return MOE_ERR_UNSUPPORTED;
  if (c.T == 0) return zero_outputs(c, t, st);

  if ((rc = record(events, MOE_STAGE_ROUTER, st)) != MOE_OK) return rc;
  const ScanOutputs so{t.expert_counts, t.aux_loss, t.routed_counts, t.offsets, t.f_out, t.P_out};
  // expert-ordered bf16 copies of the rows, unless the up projection gathers
  // them or reads their e4m3 form
  const bool copy = !route_only && !p.gather && !p.gather4 && !p.fp8;
  if (p.route_small) {
    // stages 1-4 in one launch for a decode batch; top-k and permute are empty
    MOE_TRY_CUDA(launch_route_small(p, t.x, t.W_r, t.logit_offset, t.sel_bias, t.topk_idx,
                                    t.topk_w, t.slot_pos, copy, ws, so, st));
    if ((rc = record(events, MOE_STAGE_TOPK, st)) != MOE_OK) return rc;
    if ((rc = record(events, MOE_STAGE_PERMUTE, st)) != MOE_OK) return rc;
  } else if (p.route_tc) {
    // stages 1-4 in one launch; the top-k and permute stages are empty
    MOE_TRY_CUDA(launch_route_tc(p, t.x, t.W_r, t.logit_offset, t.sel_bias, t.topk_idx, t.topk_w,
                                 t.slot_pos, ws, so, st));
    if ((rc = record(events, MOE_STAGE_TOPK, st)) != MOE_OK) return rc;
    if ((rc = record(events, MOE_STAGE_PERMUTE, st)) != MOE_OK) return rc;
    if (copy) MOE_TRY_CUDA(launch_gather_rows(p, t.x, ws, st));
  } else if (p.route_wide) {
    // stages 1-4 and the row copy in one launch; top-k and permute are empty
    MOE_TRY_CUDA(launch_route_wide(p, t.x, t.W_r, t.logit_offset, t.sel_bias, t.topk_idx,
                                   t.topk_w, t.slot_pos, copy, ws, so, st));
    if ((rc = record(events, MOE_STAGE_TOPK, st)) != MOE_OK) return rc;
    if ((rc = record(events, MOE_STAGE_PERMUTE, st)) != MOE_OK) return rc;
  } else {
    cudaEvent_t topk_ev = events ? static_cast<cudaEvent_t>(events[MOE_STAGE_TOPK]) : nullptr;
    MOE_TRY_CUDA(launch_router(p, t.x, t.W_r, t.logit_offset, t.sel_bias, t.topk_idx, t.topk_w,
                               ws, so, st, topk_ev));
    if ((rc = record(events, MOE_STAGE_PERMUTE, st)) != MOE_OK) return rc;
    // the expert-ordered copies (unless the up projection gathers rows)
    MOE_TRY_CUDA(launch_permute(p, t.x, t.topk_idx, t.slot_pos, copy, ws, st, t.y));
  }
  if (route_only) return MOE_OK;
  if (p.fp8) MOE_TRY_CUDA(launch_quant_rows(p, t.x, ws, st));
  if ((rc = record(events, MOE_STAGE_UP, st)) != MOE_OK) return rc;
  cudaEvent_t mid = events ? static_cast<cudaEvent_t>(events[MOE_STAGE_DOWN]) : nullptr;
  if (p.tc)
    MOE_TRY_CUDA(launch_experts_tc(p, t.x, t.W1, t.W3, t.W2, t.Ws1, t.Ws3, t.Ws2, ws, st, mid,
                                   t.y, t.topk_w, t.W1s, t.W3s, t.W2s));
  else
    MOE_TRY_CUDA(launch_experts_simt(p, t.x, t.W1, t.W3, t.W2, t.Ws1, t.Ws3, t.Ws2, ws, st, mid));
  if ((rc = record(events, MOE_STAGE_COMBINE, st)) != MOE_OK) return rc;
  if (!p.combine_in_down && !p.combine_k)
    MOE_TRY_CUDA(launch_combine(p, t.topk_w, t.y, ws, st));
  if ((rc = record(events, MOE_NUM_STAGES, st)) != MOE_OK) return rc;
  return MOE_OK;
}

// A sequence of batches from and to host memory, with the copies of one batch
// overlapping the layer of another.  The workspace holds two staging slots for
// x, y and the loss.  `ci` carries the copies in (H2D 0, H2D 1, then H2D i+2
// into the slot batch i used, once batch i's layer has read it), `co` the
// copies back (D2H i after batch i's layer); `st` runs the layers, batch i
// after H2D i and after D2H i-2 has read the slot's y.  With ci == co the
// copies share one stream in the order H2D 0, H2D 1, D2H 0, H2D 2, D2H 1, ...
// At the end `st` waits for both copy streams, so that synchronising `st`
// covers every copy.
static int host_io_batches(const moe_config* cfg, int n, const void* const* x_host,
                           void* const* y_host, float* aux_host, Tensors t, WsKind kind,
                           void* workspace, size_t workspace_bytes, cudaStream_t st,
                           cudaStream_t ci, cudaStream_t co) {
  if (!cfg || n < 0) return MOE_ERR_ARG;
  if (n > 0 && (!x_host || !y_host || !aux_host)) return MOE_ERR_ARG;
  if (ci == st || co == st) return MOE_ERR_ARG;   // the copies need streams of their own
  for (int i = 0; i < n; ++i)
    if (!x_host[i] || !y_host[i]) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, kind, &p);
  if (rc != MOE_OK) return rc;
  rc = check_workspace(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  char* w = static_cast<char*>(workspace);
  void* xd[2] = {w + p.ws.x_dev, w + p.ws.x_dev2};
  void* yd[2] = {w + p.ws.y_dev, w + p.ws.y_dev2};
  float* ad[2] = {reinterpret_cast<float*>(w + p.ws.aux), reinterpret_cast<float*>(w + p.ws.aux2)};
  t.x = xd[0];
  t.y = yd[0];
  t.topk_idx = reinterpret_cast<int32_t*>(w + p.ws.topk_idx);
  t.topk_w = reinterpret_cast<float*>(w + p.ws.topk_w);
  t.expert_counts = reinterpret_cast<int32_t*>(w + p.ws.counts);
  t.aux_loss = ad[0];
  rc = check_tensors(*cfg, t, false);
  if (rc != MOE_OK) return rc;
  if (n == 0) return MOE_OK;
  const size_t io = (size_t)cfg->T * cfg->d * p.elem;
  // in[2], layer[2], out[2], joins of ci and co
  cudaEvent_t ev[8] = {};
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      for (auto& f : ev)
        if (f) cudaEventDestroy(f);
      return MOE_ERR_CUDA;
    }
  cudaEvent_t* ev_in = ev;
  cudaEvent_t* ev_layer = ev + 2;
  cudaEvent_t* ev_out = ev + 4;
  auto run = [&]() -> int {
    auto h2d = [&](int i) -> int {
      const int s = i & 1;
      if (i >= 2) MOE_TRY_CUDA(cudaStreamWaitEvent(ci, ev_layer[s], 0));
      if (io) MOE_TRY_CUDA(cudaMemcpyAsync(xd[s], x_host[i], io, cudaMemcpyHostToDevice, ci));
      MOE_TRY_CUDA(cudaEventRecord(ev_in[s], ci));
      return MOE_OK;
    };
    int r = h2d(0);
    if (r == MOE_OK && n > 1) r = h2d(1);
    for (int i = 0; i < n && r == MOE_OK; ++i) {
      const int s = i & 1;
      MOE_TRY_CUDA(cudaStreamWaitEvent(st, ev_in[s], 0));
      if (i >= 2) MOE_TRY_CUDA(cudaStreamWaitEvent(st, ev_out[s], 0));
      Tensors ti = t;
      ti.x = xd[s];
      ti.y = yd[s];
      ti.aux_loss = ad[s];
      r = forward_impl(cfg, ti, workspace, workspace_bytes, st, nullptr, false, kind);
      if (r != MOE_OK) break;
      MOE_TRY_CUDA(cudaEventRecord(ev_layer[s], st));
      MOE_TRY_CUDA(cudaStreamWaitEvent(co, ev_layer[s], 0));
      if (io) MOE_TRY_CUDA(cudaMemcpyAsync(y_host[i], yd[s], io, cudaMemcpyDeviceToHost, co));
      MOE_TRY_CUDA(cudaMemcpyAsync(aux_host + i, ad[s], sizeof(float), cudaMemcpyDeviceToHost, co));
      MOE_TRY_CUDA(cudaEventRecord(ev_out[s], co));
      if (i + 2 < n) r = h2d(i + 2);
    }
    if (r != MOE_OK) return r;
    MOE_TRY_CUDA(cudaEventRecord(ev[6], ci));
    MOE_TRY_CUDA(cudaEventRecord(ev[7], co));
    MOE_TRY_CUDA(cudaStreamWaitEvent(st, ev[6], 0));
    MOE_TRY_CUDA(cudaStreamWaitEvent(st, ev[7], 0));
    return MOE_OK;
  };
  rc = run();
  for (auto& e : ev) cudaEventDestroy(e);   // released once their work completes
  return rc;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::Forward, &p);
  if (rc == MOE_OK) *bytes = p.ws.total;
  return rc;
}

int moe_route_workspace_size(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::Route, &p);
  if (rc == MOE_OK) *bytes = p.ws.total;
  return rc;
}

int moe_host_io_workspace_size(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::HostIO, &p);
  if (rc == MOE_OK) *bytes = p.ws.total;
  return rc;
}

int moe_forward_timed(const moe_config* cfg, const void* x, const void* W_r,
                      const float* logit_offset, const float* sel_bias, const void* W1,
                      const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                      const void* Ws2, void* y, int32_t* topk_idx, float* topk_w,
                      int32_t* expert_counts, float* aux_loss, int32_t* routed_counts,
                      int32_t* offsets, int32_t* slot_pos, float* f_out, float* P_out,
                      void* workspace, size_t workspace_bytes, void* stream,
                      void* const* events) {
  Tensors t{x,  W_r, logit_offset, sel_bias, W1,       W3,      W2,      Ws1,      Ws3,  Ws2,
            y,  topk_idx, topk_w, expert_counts, aux_loss, routed_counts, offsets, slot_pos,
            f_out, P_out};
  return forward_impl(cfg, t, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      events, false, WsKind::Forward);
}

int moe_forward(const moe_config* cfg, const void* x, const void* W_r, const float* logit_offset,
                const float* sel_bias, const void* W1, const void* W3, const void* W2,
                const void* Ws1, const void* Ws3, const void* Ws2, void* y, int32_t* topk_idx,
                float* topk_w, int32_t* expert_counts, float* aux_loss, int32_t* routed_counts,
                int32_t* offsets, int32_t* slot_pos, float* f_out, float* P_out,
                void* workspace, size_t workspace_bytes, void* stream) {
  return moe_forward_timed(cfg, x, W_r, logit_offset, sel_bias, W1, W3, W2, Ws1, Ws3, Ws2, y,
                           topk_idx, topk_w, expert_counts, aux_loss, routed_counts, offsets,
                           slot_pos, f_out, P_out, workspace, workspace_bytes, stream, nullptr);
}

int moe_workspace_size_fp8(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::ForwardFp8, &p);
  if (rc == MOE_OK) *bytes = p.ws.total;
  return rc;
}

int moe_forward_fp8_timed(const moe_config* cfg, const void* x, const void* W_r,
                          const float* logit_offset, const float* sel_bias, const uint8_t* W1q,
                          const float* W1s, const uint8_t* W3q, const float* W3s, const void* W2,
                          void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                          float* aux_loss, int32_t* routed_counts, int32_t* offsets,
                          int32_t* slot_pos, float* f_out, float* P_out, void* workspace,
                          size_t workspace_bytes, void* stream, void* const* events) {
  if (!W1s || !W3s) return MOE_ERR_ARG;
  Tensors t{x,  W_r, logit_offset, sel_bias, W1q,     W3q,     W2,      nullptr,  nullptr, nullptr,
            y,  topk_idx, topk_w, expert_counts, aux_loss, routed_counts, offsets, slot_pos,
            f_out, P_out, W1s, W3s};
  return forward_impl(cfg, t, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      events, false, WsKind::ForwardFp8);
}

int moe_forward_fp8(const moe_config* cfg, const void* x, const void* W_r,
                    const float* logit_offset, const float* sel_bias, const uint8_t* W1q,
                    const float* W1s, const uint8_t* W3q, const float* W3s, const void* W2,
                    void* y, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                    float* aux_loss, int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                    float* f_out, float* P_out, void* workspace, size_t workspace_bytes,
                    void* stream) {
  return moe_forward_fp8_timed(cfg, x, W_r, logit_offset, sel_bias, W1q, W1s, W3q, W3s, W2, y,
                               topk_idx, topk_w, expert_counts, aux_loss, routed_counts, offsets,
                               slot_pos, f_out, P_out, workspace, workspace_bytes, stream,
                               nullptr);
}

int moe_forward_fp8_all_timed(const moe_config* cfg, const void* x, const void* W_r,
                              const float* logit_offset, const float* sel_bias,
                              const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                              const float* W3s, const uint8_t* W2q, const float* W2s, void* y,
                              int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                              float* aux_loss, int32_t* routed_counts, int32_t* offsets,
                              int32_t* slot_pos, float* f_out, float* P_out, void* workspace,
                              size_t workspace_bytes, void* stream, void* const* events) {
  if (!W1s || !W3s || !W2s) return MOE_ERR_ARG;
  Tensors t{x,  W_r, logit_offset, sel_bias, W1q,     W3q,     W2q,     nullptr,  nullptr, nullptr,
            y,  topk_idx, topk_w, expert_counts, aux_loss, routed_counts, offsets, slot_pos,
            f_out, P_out, W1s, W3s, W2s};
  return forward_impl(cfg, t, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      events, false, WsKind::ForwardFp8);
}

int moe_forward_fp8_all(const moe_config* cfg, const void* x, const void* W_r,
                        const float* logit_offset, const float* sel_bias, const uint8_t* W1q,
                        const float* W1s, const uint8_t* W3q, const float* W3s,
                        const uint8_t* W2q, const float* W2s, void* y, int32_t* topk_idx,
                        float* topk_w, int32_t* expert_counts, float* aux_loss,
                        int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
                        float* f_out, float* P_out, void* workspace, size_t workspace_bytes,
                        void* stream) {
  return moe_forward_fp8_all_timed(cfg, x, W_r, logit_offset, sel_bias, W1q, W1s, W3q, W3s, W2q,
                                   W2s, y, topk_idx, topk_w, expert_counts, aux_loss,
                                   routed_counts, offsets, slot_pos, f_out, P_out, workspace,
                                   workspace_bytes, stream, nullptr);
}

int moe_route(const moe_config* cfg, const void* x, const void* W_r, const float* logit_offset,
              const float* sel_bias, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
              float* aux_loss, int32_t* routed_counts, int32_t* offsets, int32_t* slot_pos,
              float* f_out, float* P_out, void* workspace, size_t workspace_bytes,
              void* stream) {
  Tensors t{x,       W_r,     logit_offset, sel_bias, nullptr, nullptr,       nullptr,
            nullptr, nullptr, nullptr,      nullptr,  topk_idx, topk_w,       expert_counts,
            aux_loss, routed_counts, offsets, slot_pos, f_out,  P_out};
  return forward_impl(cfg, t, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                      nullptr, true, WsKind::Route);
}

int moe_router_scores(const moe_config* cfg, const void* x, const void* W_r,
                      const float* logit_offset, float* scores, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!cfg) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, WsKind::Route, &p);
  if (rc != MOE_OK) return rc;
  if (cfg->T > 0 && (!x || !W_r || !scores || !aligned16(x) || !aligned16(W_r)))
    return MOE_ERR_ARG;
  rc = check_workspace(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  int sms = 0;
  rc = device_sms(&sms);
  if (rc != MOE_OK) return rc;
  if (sms != p.num_sms && (rc = make_plan(cfg, WsKind::Route, &p, sms)) != MOE_OK) return rc;
  if (cfg->T == 0) return MOE_OK;
  MOE_TRY_CUDA(launch_router_scores(p, x, W_r, logit_offset, scores, workspace,
                                    static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_forward_host_io(const moe_config* cfg, const void* x_host, const void* W_r,
                        const float* logit_offset, const float* sel_bias, const void* W1,
                        const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                        const void* Ws2, void* y_host, float* aux_loss_host, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!cfg || !x_host || !y_host || !aux_loss_host) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, WsKind::HostIO, &p);
  if (rc != MOE_OK) return rc;
  rc = check_workspace(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  char* w = static_cast<char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t io_bytes = (size_t)cfg->T * cfg->d * p.elem;
  void* x_dev = w + p.ws.x_dev;
  void* y_dev = w + p.ws.y_dev;
  float* aux_dev = reinterpret_cast<float*>(w + p.ws.aux);
  Tensors t{x_dev, W_r, logit_offset, sel_bias, W1, W3, W2, Ws1, Ws3, Ws2, y_dev,
            reinterpret_cast<int32_t*>(w + p.ws.topk_idx), reinterpret_cast<float*>(w + p.ws.topk_w),
            reinterpret_cast<int32_t*>(w + p.ws.counts), aux_dev, nullptr, nullptr, nullptr,
            nullptr, nullptr};
  rc = check_tensors(*cfg, t, false);
  if (rc != MOE_OK) return rc;
  if (io_bytes) MOE_TRY_CUDA(cudaMemcpyAsync(x_dev, x_host, io_bytes, cudaMemcpyHostToDevice, st));
  rc = forward_impl(cfg, t, workspace, workspace_bytes, st, nullptr, false, WsKind::HostIO);
  if (rc != MOE_OK) return rc;
  if (io_bytes) MOE_TRY_CUDA(cudaMemcpyAsync(y_host, y_dev, io_bytes, cudaMemcpyDeviceToHost, st));
  MOE_TRY_CUDA(cudaMemcpyAsync(aux_loss_host, aux_dev, sizeof(float), cudaMemcpyDeviceToHost, st));
  return MOE_OK;
}

int moe_host_io_workspace_size_fp8(const moe_config* cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::HostIOFp8, &p);
  if (rc == MOE_OK) *bytes = p.ws.total;
  return rc;
}

int moe_forward_fp8_host_io(const moe_config* cfg, const void* x_host, const void* W_r,
                            const float* logit_offset, const float* sel_bias,
                            const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                            const float* W3s, const void* W2, void* y_host,
                            float* aux_loss_host, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!cfg || !x_host || !y_host || !aux_loss_host || !W1s || !W3s) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, WsKind::HostIOFp8, &p);
  if (rc != MOE_OK) return rc;
  rc = check_workspace(p, workspace, workspace_bytes);
  if (rc != MOE_OK) return rc;
  char* w = static_cast<char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t io_bytes = (size_t)cfg->T * cfg->d * p.elem;
  void* x_dev = w + p.ws.x_dev;
  void* y_dev = w + p.ws.y_dev;
  float* aux_dev = reinterpret_cast<float*>(w + p.ws.aux);
  Tensors t{x_dev, W_r, logit_offset, sel_bias, W1q, W3q, W2, nullptr, nullptr, nullptr, y_dev,
            reinterpret_cast<int32_t*>(w + p.ws.topk_idx), reinterpret_cast<float*>(w + p.ws.topk_w),
            reinterpret_cast<int32_t*>(w + p.ws.counts), aux_dev, nullptr, nullptr, nullptr,
            nullptr, nullptr, W1s, W3s};
  rc = check_tensors(*cfg, t, false);
  if (rc != MOE_OK) return rc;
  if (io_bytes) MOE_TRY_CUDA(cudaMemcpyAsync(x_dev, x_host, io_bytes, cudaMemcpyHostToDevice, st));
  rc = forward_impl(cfg, t, workspace, workspace_bytes, st, nullptr, false, WsKind::HostIOFp8);
  if (rc != MOE_OK) return rc;
  if (io_bytes) MOE_TRY_CUDA(cudaMemcpyAsync(y_host, y_dev, io_bytes, cudaMemcpyDeviceToHost, st));
  MOE_TRY_CUDA(cudaMemcpyAsync(aux_loss_host, aux_dev, sizeof(float), cudaMemcpyDeviceToHost, st));
  return MOE_OK;
}

int moe_forward_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                const void* const* x_host, const void* W_r,
                                const float* logit_offset, const float* sel_bias, const void* W1,
                                const void* W3, const void* W2, const void* Ws1, const void* Ws3,
                                const void* Ws2, void* const* y_host, float* aux_loss_host,
                                void* workspace, size_t workspace_bytes, void* stream,
                                void* copy_in_stream, void* copy_out_stream) {
  Tensors t{nullptr, W_r, logit_offset, sel_bias, W1, W3, W2, Ws1, Ws3, Ws2, nullptr,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return host_io_batches(cfg, n_batches, x_host, y_host, aux_loss_host, t, WsKind::HostIO,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         static_cast<cudaStream_t>(copy_in_stream),
                         static_cast<cudaStream_t>(copy_out_stream));
}

int moe_forward_fp8_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                    const void* const* x_host, const void* W_r,
                                    const float* logit_offset, const float* sel_bias,
                                    const uint8_t* W1q, const float* W1s, const uint8_t* W3q,
                                    const float* W3s, const void* W2, void* const* y_host,
                                    float* aux_loss_host, void* workspace,
                                    size_t workspace_bytes, void* stream, void* copy_in_stream,
                                    void* copy_out_stream) {
  if (!W1s || !W3s) return MOE_ERR_ARG;
  Tensors t{nullptr, W_r, logit_offset, sel_bias, W1q, W3q, W2, nullptr, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr, W1s, W3s};
  return host_io_batches(cfg, n_batches, x_host, y_host, aux_loss_host, t, WsKind::HostIOFp8,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         static_cast<cudaStream_t>(copy_in_stream),
                         static_cast<cudaStream_t>(copy_out_stream));
}

int moe_forward_fp8_all_host_io_batches(const moe_config* cfg, int32_t n_batches,
                                        const void* const* x_host, const void* W_r,
                                        const float* logit_offset, const float* sel_bias,
                                        const uint8_t* W1q, const float* W1s,
                                        const uint8_t* W3q, const float* W3s,
                                        const uint8_t* W2q, const float* W2s,
                                        void* const* y_host, float* aux_loss_host,
                                        void* workspace, size_t workspace_bytes, void* stream,
                                        void* copy_in_stream, void* copy_out_stream) {
  if (!W1s || !W3s || !W2s) return MOE_ERR_ARG;
  Tensors t{nullptr, W_r, logit_offset, sel_bias, W1q, W3q, W2q, nullptr, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr, W1s, W3s, W2s};
  return host_io_batches(cfg, n_batches, x_host, y_host, aux_loss_host, t, WsKind::HostIOFp8,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         static_cast<cudaStream_t>(copy_in_stream),
                         static_cast<cudaStream_t>(copy_out_stream));
}

int moe_check_status(void* workspace, void* stream) {
  if (!workspace) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t status = 0;
  if (cudaMemcpyAsync(&status, workspace, sizeof(status), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(status), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (status & STATUS_BOUNDS) return MOE_ERR_BOUNDS;
  return status ? MOE_ERR_TIMEOUT : MOE_OK;
}

const char* moe_error_string(int code) {
  switch (code) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_ARG: return "MOE_ERR_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: layer shape not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, small or misaligned";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: needs a compute capability 10.3 GPU";
    case MOE_ERR_BOUNDS:
      return "MOE_ERR_BOUNDS: a routing-derived index was out of range (bounds-checked build)";
  }
  return "MOE_ERR_UNKNOWN";
}

int moe_launch_count(const moe_config* cfg, int32_t* launches) {
  if (!launches) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::Forward, &p);
  if (rc != MOE_OK) return rc;
  // routing: one launch (decode batches; tensor-core routing, plus a row
  // copy unless the up projection gathers rows), two (fused float32 router +
  // permute) or three (logits, top-k, permute); then the two projections and
  // the combine, which top-1 bf16 layers without a shared expert fold into
  // the down projection
  const bool copy = !p.gather && !p.gather4;   // the tensor-core router's row copy
  const int routing = p.route_small ? 1
                      : p.route_tc  ? (copy ? 2 : 1)
                      : p.route_wide ? (copy && !route_wide_copies_rows(p) ? 2 : 1)
                                    : (p.router_fused ? 2 : 3);
  *launches = cfg->T == 0 ? 0
                          : routing + (p.fused ? 1 : 2) + (p.combine_in_down || p.combine_k ? 0 : 1);
  return MOE_OK;
}

static int plan_flags(const moe_config* cfg, WsKind kind, uint32_t* flags) {
  if (!flags) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, kind, &p);
  if (rc != MOE_OK) return rc;
  uint32_t f = 0;
  if (p.route_tc) f |= MOE_PLAN_ROUTE_ONE_LAUNCH;
  if (p.route_wide) f |= MOE_PLAN_ROUTE_CLUSTER;
  if (p.route_small) f |= MOE_PLAN_ROUTE_DECODE;
  if (p.gather || p.gather4) f |= MOE_PLAN_GATHER_ROWS;
  if (p.combine_in_down || p.combine_k) f |= MOE_PLAN_COMBINE_IN_DOWN;
  if (p.fused) f |= MOE_PLAN_FUSED_PROJECTIONS;
  *flags = f;
  return MOE_OK;
}

int moe_plan_flags(const moe_config* cfg, uint32_t* flags) {
  return plan_flags(cfg, WsKind::Forward, flags);
}

int moe_plan_flags_fp8(const moe_config* cfg, uint32_t* flags) {
  return plan_flags(cfg, WsKind::ForwardFp8, flags);
}

int moe_launch_count_fp8(const moe_config* cfg, int32_t* launches) {
  if (!launches) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(cfg, WsKind::ForwardFp8, &p);
  if (rc != MOE_OK) return rc;
  // routing without a row copy, the row quantisation, the two projections
  // and the combine (folded into the down projection for top-1 layers)
  const int routing = p.route_small || p.route_tc || p.route_wide ? 1 : (p.router_fused ? 2 : 3);
  *launches = cfg->T == 0 ? 0 : routing + 1 + 2 + (p.combine_in_down || p.combine_k ? 0 : 1);
  return MOE_OK;
}

int moe_set_tuning(int32_t knob, int32_t value) {
  if (knob < 0 || knob >= MOE_TUNE_COUNT || value < -1) return MOE_ERR_ARG;
  if (knob == MOE_TUNE_ROUTER && value > MOE_ROUTER_TC) return MOE_ERR_ARG;
  if (knob == MOE_TUNE_GATHER && value > 2) return MOE_ERR_ARG;
  if ((knob == MOE_TUNE_MMA_M64 || knob == MOE_TUNE_FUSED_COMBINE ||
       knob == MOE_TUNE_CLUSTER || knob == MOE_TUNE_FUSED_PROJ ||
       knob == MOE_TUNE_F8_DOWN_FORM) && value > 1)
    return MOE_ERR_ARG;
  g_tune[knob].store(value, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t wait_ns,
                              void* stream) {
  if (!workspace || workspace_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_WORKSPACE;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != MOE_OK) return rc;
  MOE_TRY_CUDA(launch_selftest_wait(static_cast<uint32_t*>(workspace), wait_ns,
                                    static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_router_z_loss(const float* scores, int32_t T, int32_t E, float* z_loss, void* stream) {
  if (T < 0 || E < 1 || E > kMaxE || !z_loss || !aligned4(z_loss)) return MOE_ERR_ARG;
  if (T > 0 && (!scores || !aligned4(scores))) return MOE_ERR_ARG;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != MOE_OK) return rc;
  MOE_TRY_CUDA(launch_router_z_loss(scores, T, E, z_loss, static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_bias_update(const int32_t* routed_counts, int32_t E, int32_t T, int32_t k, float gamma,
                    float* sel_bias, void* stream) {
  if (E < 1 || E > kMaxE || T < 0 || k < 1 || k > E) return MOE_ERR_ARG;
  if (!routed_counts || !sel_bias || !aligned4(routed_counts) || !aligned4(sel_bias))
    return MOE_ERR_ARG;
  if (!(gamma >= 0.f) || !std::isfinite(gamma)) return MOE_ERR_ARG;
  int sms = 0;
  const int rc = device_sms(&sms);
  if (rc != MOE_OK) return rc;
  MOE_TRY_CUDA(launch_bias_update(routed_counts, E, T, k, gamma, sel_bias,
                                  static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

}  // extern "C"
