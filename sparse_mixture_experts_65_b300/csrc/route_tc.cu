// route_tc.cu -- stages 1 to 4 in one launch, for bf16 layers with at most 64
// experts and k <= 8: router logits on the tensor cores, selection, top-k and
// gates, the router distribution, the capacity scan, and the positions of the
// kept assignments in expert order.
//
// What is computed is the same as the split path (router.cu, route_scan.cuh,
// route.cu): "Mixture of Experts" (llm-tutorial ch. 11) § The mathematics and
// § Top-k routing (s = W_r x, the k largest, gates from the chosen logits),
// "Mixture of experts" (inside-the-model guide) § The computation and
// § Auxiliary-loss-free balancing (sigmoid affinities, a bias that only
// selects), ch. 11 § Expert capacity and dropped tokens (first come by the
// token-major key t*k + j), and the guide's § Auxiliary loss (f_i, P_i, L).
//
// Launch: one CTA of 192 threads per 128-token tile, persistent over tiles
// (grid <= SM count), cooperative so that every CTA is resident at once:
//   warp 0     TMA: the x tile (128 tokens x 64 k) and W_r (EP experts x 64 k),
//              128-byte swizzle, completion on a transaction barrier;
//   warp 1     tcgen05.mma (M=128, N=EP, K=16) into one of two TMEM
//              accumulators, one per 128-wide chunk of the model width;
//   warps 2-5  one token per thread: the chunk results are added in float32
//              in chunk order (the arithmetic of the tensor-core router, max
//              error ~2e-6 on a 7168-wide router), then selection, top-k,
//              gates and the router distribution; one warp ranks the tile's
//              keys among the earlier keys of the tile; the tile's histogram
//              and probability sums are published.
// Then a grid-wide wait (bounded) until every tile is published, after which
// every CTA reads all tiles' histograms, derives the routed totals, the
// exclusive prefix of its own tiles and the expert segments itself (CTA 0
// also writes the layer's meta data and the balance statistics) and turns its
// tiles' ranks into positions and rows.  No token row is copied: the up
// projection gathers the rows of x through the row -> token map.
//
// Determinism: counts are integers; every float sum has a fixed association
// (chunk order, a fixed butterfly per warp, warps and tiles in order).
#include <atomic>
#include <climits>
#include <cstring>

#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "route_scan.cuh"
#include "tma_host.cuh"

namespace moe {

constexpr int kRtThreads = 192;
constexpr int kRtBK = 64;          // k per stage (128 bytes of bf16: one swizzle row)
// Stages per TMEM accumulator: 128-wide chunks of the model width, whose
// float32 sums the epilogue adds in chunk order (the tensor cores' own
// accumulation then spans at most 8 MMA steps: ~2e-6 on a 7168-wide router).
// Narrow routers (d <= 768) take two chunks of at most 384: at most 24 steps
// each, ~2e-6 on a 768-wide router as well, with a third of the epilogue's
// chunk passes on the latency-bound path of the routing kernel.
constexpr int kRtChunkKB = 2;
__host__ __device__ inline int rt_chunk_kb(int nk) {
  return nk <= 12 ? ((nk + 1) / 2 > kRtChunkKB ? (nk + 1) / 2 : kRtChunkKB) : kRtChunkKB;
}
constexpr int kRtMaxK = 8;
constexpr int kRtLds = kTcBM + 1;  // row stride of the logit columns (odd: no bank conflicts)
constexpr uint64_t kRtTimeoutNs = 2000000000ull;   // 2 s

struct RouteTcArgs {
  const float* logit_offset;   // [E] or null
  const float* sel_bias;       // [E] or null
  int32_t* topk_idx;           // [T*k]
  float* topk_w;               // [T*k]
  int32_t* slot_pos;           // [T*k] or null
  int* key_row;                // [T*k]: rank inside the tile, then the padded row
  int* row_token;              // [R_cap]
  int T, d, E, k, gate, capacity, ntiles, R_cap;
  unsigned* arrive;            // CTAs whose tiles are published
  unsigned* passed;            // CTAs through the wait (the last one re-arms both)
  uint32_t* status;
  uint64_t timeout_ns;
  ScanArgs scan;
};

// Shared memory of the per-CTA capacity scan (route_scan_cta).  E <= 64; the
// 192 threads form 3 groups of 64, one thread per expert in each group.
struct RtScanSmem {
  int seg[3][kRouteTcMaxOwn + 1][64];   // per group: histogram sums between owned tiles
  float psum3[3][64];                   // CTA 0: per-group sums of the router distribution
  int pre[kRouteTcMaxOwn][64];          // exclusive prefix of every owned tile
  int routed[64];
  int segst[64];                        // first row of each expert's segment
  int off[64];                          // first slot of each expert
};

template <int EP>
struct RtCfg {
  static_assert(EP == 32 || EP == 64, "experts per tile");
  static constexpr int A_BYTES = kTcBM * kRtBK * 2;
  static constexpr int B_BYTES = EP * kRtBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int TMEM_COLS = 2 * EP;               // 64 or 128: a power of two >= 32
  static constexpr uint32_t IDESC = idesc_bf16_f32(kTcBM, EP);
  // shared memory after the stages; every region a multiple of 16 bytes
  static constexpr int al16(int b) { return (b + 15) / 16 * 16; }
  static constexpr int BAR_BYTES = al16(8 * (2 * STAGES + 5));
  static constexpr int KEYS_BYTES = 4 * kTcBM * kRtMaxK;  // keys of a tile, then its rows
  static constexpr int CA_BYTES = 4 * kTcBM * kRtMaxK;    // affinities of the chosen experts
  static constexpr int LG_BYTES = al16(4 * EP * kRtLds);  // one column per token: p
  static constexpr int PH_BYTES = 4 * 2 * EP;             // half-tile probability sums
  static constexpr int CNT_BYTES = 4 * EP;
  static constexpr int SCAN_BYTES = al16((int)sizeof(RtScanSmem));
  static constexpr int VEC_BYTES = 4 * 2 * EP;            // selection bias and logit offset
  static constexpr int MISC_BYTES = 64;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + KEYS_BYTES + CA_BYTES +
                              LG_BYTES + PH_BYTES + CNT_BYTES + SCAN_BYTES + VEC_BYTES +
                              MISC_BYTES;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Tree reductions over a register array (the association is fixed, so the
// results are deterministic; max and min are exact in any order anyway).
template <int N>
__device__ __forceinline__ float tree_max(const float (&x)[N]) {
  float t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = x[i];
#pragma unroll
  for (int w = N / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  return t[0];
}

// Routing of one token by one thread.  v[] holds the token's logits (offset
// included; -inf past E) in registers.  Every loop over experts is unrolled
// over the padded width EP and free of branches (selects and reduction
// trees), so the steps of one token overlap.  Writes the k chosen experts and
// their gates (when `valid`), the chosen experts to keys[] and their
// affinities to ca[], and the router distribution p to the token's column
// col[e * kRtLds] (zero for invalid tokens).  The exponentials use the
// hardware exp2 (relative error ~1e-6 over the logit range, inside the 1e-5
// tolerance of gates and P).
template <int EP>
__device__ __forceinline__ void route_token(float (&v)[EP], int E, int k, int gate,
                                            const float* bias_s, bool valid, int32_t* idx_out,
                                            float* w_out, int* keys, float* ca, float* col) {
  const bool sigm = gate == MOE_GATE_SIGMOID_RENORM;
  // affinity: the logit, or its sigmoid (0 past E); hardware exp2 and
  // reciprocal (relative error ~2e-7, far inside the near-tie band)
  if (sigm) {
#pragma unroll
    for (int e = 0; e < EP; ++e) v[e] = __fdividef(1.0f, 1.0f + __expf(-v[e]));
  }
  // selection scores: affinity + bias, -inf past E and for NaN
  float sel[EP];
#pragma unroll
  for (int e0 = 0; e0 < EP; e0 += 4) {
    const float4 b = *reinterpret_cast<const float4*>(bias_s + e0);
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float x = v[e0 + u] + bb[u];
      sel[e0 + u] = (e0 + u < E && x == x) ? x : -INFINITY;
    }
  }
  // k rounds: the largest score, then the lowest index holding it (ties go
  // to the lower index); the chosen expert leaves the race
  for (int r = 0; r < k; ++r) {
    const float best = tree_max<EP>(sel);
    float idx[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) idx[e] = sel[e] == best ? (float)e : (float)EP;
    float mi = idx[0];
#pragma unroll
    for (int w = EP / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) idx[i] = fminf(idx[i], idx[i + w]);
    mi = idx[0];
    const int bix = best == -INFINITY ? -1 : (int)mi;
    float pick[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      pick[e] = e == bix ? v[e] : -INFINITY;
      sel[e] = e == bix ? -INFINITY : sel[e];
    }
    keys[r] = bix >= 0 ? bix : 0;
    ca[r] = bix >= 0 ? tree_max<EP>(pick) : -INFINITY;
  }
  // router distribution over all E: softmax(s), or the sigmoids normalised
  float m_all = -INFINITY;
  if (!sigm) {
    m_all = tree_max<EP>(v);
#pragma unroll
    for (int e = 0; e < EP; ++e) v[e] = __expf(v[e] - m_all);
  }
  float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int e = 0; e < EP; ++e) z[e & 7] += v[e];
  const float z_all = ((z[0] + z[1]) + (z[2] + z[3])) + ((z[4] + z[5]) + (z[6] + z[7]));
  // gates of the chosen experts
  float m_k = -INFINITY, zk = 0.f;
  if (gate == MOE_GATE_SOFTMAX_TOPK) {
    for (int r = 0; r < k; ++r) m_k = fmaxf(m_k, ca[r]);
    for (int r = 0; r < k; ++r) zk += __expf(ca[r] - m_k);
  } else if (sigm) {
    for (int r = 0; r < k; ++r) zk += ca[r];
  }
  const float inv_z = 1.0f / z_all;
  if (valid) {
    const float inv_zk = 1.0f / zk;
    for (int r = 0; r < k; ++r) {
      const float g = gate == MOE_GATE_SOFTMAX_TOPK ? __expf(ca[r] - m_k) * inv_zk
                      : sigm                        ? ca[r] * inv_zk
                                                    : __expf(ca[r] - m_all) * inv_z;
      idx_out[r] = keys[r];
      w_out[r] = g;
    }
  }
  const float scale = valid ? inv_z : 0.f;
#pragma unroll
  for (int e = 0; e < EP; ++e) col[e * kRtLds] = v[e] * scale;
}

// Per-CTA view of the capacity scan, computed by every CTA once all tiles
// are published: routed totals per expert, the exclusive prefix of each tile
// this CTA owns, and the expert segments.  One round of histogram loads (the
// three thread groups take every third tile), one warp for the scans over
// experts.  CTA 0 also writes the layer's meta data and the balance
// statistics.
__device__ void route_scan_cta(const RouteTcArgs& a, RtScanSmem& sm) {
  const ScanArgs& sa = a.scan;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool writer = blockIdx.x == 0;
  const int grid = gridDim.x, me = blockIdx.x;
  const int nown = (a.ntiles - me + grid - 1) / grid;   // owned tiles: me, me + grid, ...
  {
    const int g = tid >> 6, e = tid & 63;
    if (e < a.E) {
      // segment s covers the tiles [me + (s-1)*grid, me + s*grid)
      int s_idx = 0, bound = me, acc = 0;
      float pacc = 0.f;
      constexpr int U = 8;   // loads in flight per thread
      for (int b0 = g; b0 < a.ntiles; b0 += 3 * U) {
        int cv[U];
        float pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = b0 + 3 * u;
          const bool ok = b < a.ntiles;
          cv[u] = ok ? __ldcg(sa.blk_cnt + (size_t)b * a.E + e) : 0;
          pv[u] = (ok && writer) ? __ldcg(sa.blk_prob + (size_t)b * a.E + e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = b0 + 3 * u;
          if (b < a.ntiles) {
            while (b >= bound) {
              sm.seg[g][s_idx][e] = acc;
              acc = 0;
              ++s_idx;
              bound += grid;
            }
            acc += cv[u];
            pacc += pv[u];
          }
        }
      }
      for (; s_idx <= nown; ++s_idx) {
        sm.seg[g][s_idx][e] = acc;
        acc = 0;
      }
      if (writer) sm.psum3[g][e] = pacc;
    }
  }
  __syncthreads();
  if (tid < a.E) {
    int run = 0;
    for (int s = 0; s <= nown; ++s) {
      run += sm.seg[0][s][tid] + sm.seg[1][s][tid] + sm.seg[2][s][tid];
      if (s < nown) sm.pre[s][tid] = run;
    }
    sm.routed[tid] = run;
  }
  __syncthreads();
  if (warp == 0) {
    // experts 2*lane and 2*lane + 1: kept counts, M tiles and tile counts,
    // scanned over the warp
    const int e0 = 2 * lane, e1 = e0 + 1;
    const int r0 = e0 < a.E ? sm.routed[e0] : 0, r1 = e1 < a.E ? sm.routed[e1] : 0;
    const int k0 = r0 < a.capacity ? r0 : a.capacity, k1 = r1 < a.capacity ? r1 : a.capacity;
    const int m0 = (k0 + sa.bm - 1) / sa.bm, m1 = (k1 + sa.bm - 1) / sa.bm;
    int ik = k0 + k1, im = m0 + m1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nk = __shfl_up_sync(0xffffffffu, ik, o);
      const int nm = __shfl_up_sync(0xffffffffu, im, o);
      if (lane >= o) {
        ik += nk;
        im += nm;
      }
    }
    const int xk0 = ik - k0 - k1, xm0 = im - m0 - m1;   // exclusive, expert e0
    const int xk1 = xk0 + k0, xm1 = xm0 + m0;           // exclusive, expert e1
    if (e0 < a.E) {
      sm.segst[e0] = xm0 * sa.bm;
      sm.off[e0] = xk0;
    }
    if (e1 < a.E) {
      sm.segst[e1] = xm1 * sa.bm;
      sm.off[e1] = xk1;
    }
    if (writer) {
      const float P0 = ((sm.psum3[0][e0 & 63] + sm.psum3[1][e0 & 63]) + sm.psum3[2][e0 & 63]) /
                       (float)a.T;
      const float P1 = ((sm.psum3[0][e1 & 63] + sm.psum3[1][e1 & 63]) + sm.psum3[2][e1 & 63]) /
                       (float)a.T;
      const float f0 = (float)r0 / (float)(a.T * a.k), f1 = (float)r1 / (float)(a.T * a.k);
      // tile counts of the two projections are M tiles times N tiles per segment
      if (e0 < a.E) {
        sa.m.kept[e0] = k0;
        sa.m.offsets[e0] = xk0;
        sa.m.seg_start[e0] = xm0 * sa.bm;
        sa.m.mtiles[e0] = m0;
        sa.m.tp_up[e0] = xm0 * sa.nt_up;
        sa.m.tp_dn[e0] = xm0 * sa.nt_dn;
        sa.expert_counts[e0] = k0;
        if (sa.routed_counts) sa.routed_counts[e0] = r0;
        if (sa.offsets_out) sa.offsets_out[e0] = xk0;
        if (sa.f_out) sa.f_out[e0] = f0;
        if (sa.P_out) sa.P_out[e0] = P0;
      }
      if (e1 < a.E) {
        sa.m.kept[e1] = k1;
        sa.m.offsets[e1] = xk1;
        sa.m.seg_start[e1] = xm1 * sa.bm;
        sa.m.mtiles[e1] = m1;
        sa.m.tp_up[e1] = xm1 * sa.nt_up;
        sa.m.tp_dn[e1] = xm1 * sa.nt_dn;
        sa.expert_counts[e1] = k1;
        if (sa.routed_counts) sa.routed_counts[e1] = r1;
        if (sa.offsets_out) sa.offsets_out[e1] = xk1;
        if (sa.f_out) sa.f_out[e1] = f1;
        if (sa.P_out) sa.P_out[e1] = P1;
      }
      if (lane == 31) {   // totals: the inclusive scan at the last lane
        const int sh_up = sa.has_shared ? sa.mt_sh * sa.nt_up_sh : 0;
        const int sh_dn = sa.has_shared ? sa.mt_sh * sa.nt_dn_sh : 0;
        sa.m.offsets[a.E] = ik;
        sa.m.seg_start[a.E] = im * sa.bm;
        sa.m.mtiles[a.E] = sa.has_shared ? sa.mt_sh : 0;
        sa.m.tp_up[a.E] = im * sa.nt_up;
        sa.m.tp_up[a.E + 1] = im * sa.nt_up + sh_up;
        sa.m.tp_dn[a.E] = im * sa.nt_dn;
        sa.m.tp_dn[a.E + 1] = im * sa.nt_dn + sh_dn;
        if (sa.offsets_out) sa.offsets_out[a.E] = ik;
      }
      // L = alpha * E * sum_i f_i P_i in double, a fixed butterfly over the warp
      double l = (e0 < a.E ? (double)f0 * (double)P0 : 0.0) +
                 (e1 < a.E ? (double)f1 * (double)P1 : 0.0);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) sa.aux_loss[0] = (float)((double)sa.alpha * (double)a.E * l);
    }
  }
  __syncthreads();
}

template <int EP>
__global__ void __launch_bounds__(kRtThreads, 1)
    route_tc_kernel(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mW,
                    const RouteTcArgs a) {
  using C = RtCfg<EP>;
  extern __shared__ uint8_t rt_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(rt_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  uint8_t* p = smem + C::STAGES * C::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  p += C::BAR_BYTES;
  int* keys_s = reinterpret_cast<int*>(p);
  p += C::KEYS_BYTES;
  float* ca_s = reinterpret_cast<float*>(p);
  p += C::CA_BYTES;
  float* lg = reinterpret_cast<float*>(p);      // [EP][kRtLds]
  p += C::LG_BYTES;
  float* ph = reinterpret_cast<float*>(p);      // [2][EP]
  p += C::PH_BYTES;
  int* cnt = reinterpret_cast<int*>(p);
  p += C::CNT_BYTES;
  RtScanSmem& scan_sm = *reinterpret_cast<RtScanSmem*>(p);
  p += C::SCAN_BYTES;
  float* bias_s = reinterpret_cast<float*>(p);
  float* offs_s = bias_s + EP;
  p += C::VEC_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(p + 4);
  int* s_fail = reinterpret_cast<int*>(p + 12);
  volatile int* s_stop = reinterpret_cast<volatile int*>(p + 16);

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::STAGES + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *s_fail = 0;
    fence_mbar_init();
  }
  if (tid < EP) cnt[tid] = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mX);
    tma_prefetch_desc(&mW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  // the selection bias and the logit offset are read by the epilogue warps
  // only (after their first named barrier), so the producer and the MMA
  // issuer start streaming without waiting for these loads
  if (tid >= 64 && tid - 64 < EP) {
    bias_s[tid - 64] = (a.sel_bias && tid - 64 < a.E) ? a.sel_bias[tid - 64] : 0.f;
    offs_s[tid - 64] = (a.logit_offset && tid - 64 < a.E) ? a.logit_offset[tid - 64] : 0.f;
  }

  const int nk = (a.d + kRtBK - 1) / kRtBK;
  const int ckb = rt_chunk_kb(nk);
  auto give_up = [&]() {
    atomicOr(a.status, STATUS_TIMEOUT_ROUTE);
    *abort_flag = 1;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.ntiles && ok; tile += gridDim.x) {
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % C::STAGES;
          const uint32_t ph = (g / C::STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          tma_load_2d(sa, &mX, full_bar(s), kb * kRtBK, tile * kTcBM);
          tma_load_2d(sa + C::A_BYTES, &mW, full_bar(s), kb * kRtBK, 0);
        }
      }
      // nothing asynchronous may still target shared memory at exit
      for (int s = 0; s < C::STAGES; ++s) {
        if (g > static_cast<uint32_t>(s)) {
          const uint32_t issues = (g - 1 - s) / C::STAGES + 1;
          if (ok)
            mbar_wait_bounded(empty_bar(s), (issues - 1) & 1u, a.timeout_ns, abort_flag);
          else
            mbar_wait_bounded(full_bar(s), (issues - 1) & 1u, a.timeout_ns, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < a.ntiles && ok; tile += gridDim.x) {
        for (int kb0 = 0; kb0 < nk && ok; kb0 += ckb, ++it) {
          const int ab = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait_bounded(tempty_bar(ab), aph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * EP;
          const int kb1 = kb0 + ckb < nk ? kb0 + ckb : nk;
          for (int kb = kb0; kb < kb1; ++kb, ++g) {
            const int s = g % C::STAGES;
            const uint32_t ph = (g / C::STAGES) & 1u;
            if (!mbar_wait_bounded(full_bar(s), ph, a.timeout_ns, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_base + s * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < kRtBK / 16; ++kk)
              tc_mma_bf16(d_tmem, smem_desc_k128(sa + kk * 32), smem_desc_k128(sb + kk * 32),
                          C::IDESC, (kb != kb0 || kk != 0) ? 1u : 0u);
            tc_commit(empty_bar(s));
          }
          if (!ok) break;
          tc_commit(tfull_bar(ab));
        }
      }
      if (!ok) {
        // let every issued MMA finish before tensor memory is freed
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, a.timeout_ns, nullptr);
      }
    }
  } else {
    // ---------------- routing epilogue (warps 2..5) ----------------
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int tl = q * 32 + lane;            // token inside the tile
    const int ep_tid = tid - 64;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < a.ntiles && ok; tile += gridDim.x) {
      float s[EP];
#pragma unroll
      for (int e = 0; e < EP; ++e) s[e] = 0.f;
      for (int kb0 = 0; kb0 < nk; kb0 += ckb, ++it) {
        const int ab = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_bounded(tfull_bar(ab), aph, a.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * EP;
#pragma unroll
        for (int c = 0; c < EP; c += 32) {
          uint32_t r[32];
          tmem_ld32(t_row + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c + i] += __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(ab));
      }
      // one snapshot of the abort flag, so that all epilogue threads take the
      // same branch (the named barriers below need all 128)
      epi_bar();
      if (ep_tid == 0) *s_stop = *abort_flag;
      epi_bar();
      if (*s_stop) break;
      const int t0 = tile * kTcBM;
      const int t = t0 + tl;
      const bool valid = t < a.T;
      // logits (the tensor-core router's arithmetic: chunk sums in order,
      // then the offset); -inf past E
#pragma unroll
      for (int e = 0; e < EP; ++e) s[e] = e < a.E ? s[e] + offs_s[e] : -INFINITY;
      route_token<EP>(s, a.E, a.k, a.gate, bias_s, valid, a.topk_idx + (size_t)t * a.k,
                      a.topk_w + (size_t)t * a.k, keys_s + tl * a.k, ca_s + tl * a.k, lg + tl);
      epi_bar();
      // probability sums of the tile: two halves of 64 tokens, each as eight
      // interleaved partial sums added in a fixed tree (independent loads)
      if (ep_tid < 2 * a.E) {
        const int e = ep_tid >> 1, half = ep_tid & 1;
        const float* row = lg + e * kRtLds + half * (kTcBM / 2);
        float acc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = row[u];
#pragma unroll
        for (int i = 8; i < kTcBM / 2; i += 8)
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] += row[i + u];
        ph[half * EP + e] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) +
                            ((acc[4] + acc[5]) + (acc[6] + acc[7]));
      }
      const int ntok = a.T - t0 < kTcBM ? a.T - t0 : kTcBM;
      const int nkeys = ntok * a.k;
      const size_t key0 = (size_t)t0 * a.k;
      if (warp == 2) {
        // rank of every key among the earlier keys of the tile with the same
        // expert: keys in order, 32 at a time, equal experts grouped by
        // __match_any_sync, a per-expert count carried across the groups
        for (int c = 0; c < nkeys; c += 32) {
          const int kq = c + lane;
          const bool kv = kq < nkeys;
          const int e = kv ? keys_s[kq] : -1 - lane;   // invalid lanes never match
          const unsigned peers = __match_any_sync(0xffffffffu, e);
          const int before = __popc(peers & ((1u << lane) - 1u));
          const int prior = kv ? cnt[e] : 0;
          __syncwarp();
          if (kv) {
            a.key_row[key0 + kq] = prior + before;
            if (before == 0) cnt[e] = prior + __popc(peers);
          }
          __syncwarp();
        }
      }
      epi_bar();
      if (ep_tid < a.E) {
        const int e = ep_tid;
        a.scan.blk_cnt[(size_t)tile * a.E + e] = cnt[e];
        a.scan.blk_prob[(size_t)tile * a.E + e] = ph[e] + ph[EP + e];
        cnt[e] = 0;
      }
      epi_bar();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  // grid barrier: every CTA has published its tiles (all CTAs are resident:
  // cooperative launch).  The last CTA through re-arms the counters.
  if (tid == 0) {
    bool seen = false;
    if (*abort_flag == 0) {
      __threadfence();
      atomicAdd(a.arrive, 1u);
      const uint64_t t_start = globaltimer_ns();
      for (uint32_t i = 0;; ++i) {
        if (ld_acquire_gpu(a.arrive) >= gridDim.x) {
          seen = true;
          break;
        }
        if ((i & 63u) == 63u && globaltimer_ns() - t_start > a.timeout_ns) break;
      }
    }
    if (!seen) atomicOr(a.status, STATUS_TIMEOUT_ROUTE);
    *s_fail = seen ? 0 : 1;
    if (atomicAdd(a.passed, 1u) == gridDim.x - 1u) {
      *a.arrive = 0u;
      *a.passed = 0u;
    }
  }
  __syncthreads();
  if (*s_fail) return;
  route_scan_cta(a, scan_sm);
  // positions and rows of this CTA's tiles (the up projection gathers the
  // token rows itself)
  for (int tile = blockIdx.x, j = 0; tile < a.ntiles; tile += gridDim.x, ++j) {
    const int t0 = tile * kTcBM;
    const int ntok = a.T - t0 < kTcBM ? a.T - t0 : kTcBM;
    const int nkeys = ntok * a.k;
    const size_t key0 = (size_t)t0 * a.k;
    for (int kq = tid; kq < nkeys; kq += kRtThreads) {
      const int e = __ldcg(a.topk_idx + key0 + kq);
      if (!in_bounds(e >= 0 && e < a.E, a.status)) {
        a.key_row[key0 + kq] = -1;
        if (a.slot_pos) a.slot_pos[key0 + kq] = -1;
        continue;
      }
      const int pos = scan_sm.pre[j][e] + __ldcg(a.key_row + key0 + kq);
      bool keep = pos < a.capacity;
      int row = keep ? scan_sm.segst[e] + pos : -1;
      if (keep && !in_bounds(pos >= 0 && row < a.R_cap, a.status)) {
        keep = false;
        row = -1;
      }
      a.key_row[key0 + kq] = row;
      if (a.slot_pos) a.slot_pos[key0 + kq] = keep ? scan_sm.off[e] + pos : -1;
      if (keep) a.row_token[row] = t0 + kq / a.k;
    }
  }
}

// ---------------------------------------------------------------- host side
// Every CTA owns at most kRouteTcMaxOwn tiles on a GPU with at least 32 SMs.
bool route_tc_eligible(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.E <= 64 && c.k <= kRtMaxK &&
         (long long)c.T <= (long long)kRouteTcMaxOwn * kTcBM * 32;
}

// Launch modes that the runtime accepted: bit 0 = cooperative with
// programmatic dependent launch, bit 1 = that combination was refused and
// the plain cooperative launch is used.
static std::atomic<int> g_rt_launch_mode{0};

template <int EP>
static cudaError_t launch_route_tc_t(const CUtensorMap& mX, const CUtensorMap& mW,
                                     const RouteTcArgs& a, int grid, cudaStream_t st) {
  using C = RtCfg<EP>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = route_tc_kernel<EP>;
  cudaError_t e = smem_attr_once(kern, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if ((g_rt_launch_mode.load(std::memory_order_relaxed) & 2) == 0) {
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, mX, mW, a);
    if (e == cudaSuccess) {
      g_rt_launch_mode.fetch_or(1, std::memory_order_relaxed);
      return e;
    }
    if (g_rt_launch_mode.load(std::memory_order_relaxed) & 1) return e;   // worked before
    (void)cudaGetLastError();   // a refused attribute combination is not sticky
    g_rt_launch_mode.fetch_or(2, std::memory_order_relaxed);
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mX, mW, a);
}

cudaError_t launch_route_tc(const Plan& p, const void* x, const void* W_r,
                            const float* logit_offset, const float* sel_bias, int32_t* topk_idx,
                            float* topk_w, int32_t* slot_pos, void* ws, const ScanOutputs& so,
                            cudaStream_t st) {
  const moe_config& c = p.cfg;
  const int EP = c.E <= 32 ? 32 : 64;
  CUtensorMap mX, mW;
  if (!encode_2d(&mX, x, c.T, c.d, kTcBM) || !encode_2d(&mW, W_r, c.E, c.d, EP))
    return cudaErrorInvalidValue;
  char* w = static_cast<char*>(ws);
  RouteTcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.logit_offset = logit_offset;
  a.sel_bias = sel_bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.slot_pos = slot_pos;
  a.key_row = reinterpret_cast<int*>(w + p.ws.key_row);
  a.row_token = reinterpret_cast<int*>(w + p.ws.row_token);
  a.T = c.T;
  a.d = c.d;
  a.E = c.E;
  a.k = c.k;
  a.gate = c.gate;
  a.capacity = p.capacity;
  a.ntiles = p.nblk;
  a.R_cap = p.R_cap;
  a.arrive = reinterpret_cast<unsigned*>(w + p.ws.status + kRouteArriveOffset);
  a.passed = reinterpret_cast<unsigned*>(w + p.ws.status + kRoutePassedOffset);
  a.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  a.timeout_ns = kRtTimeoutNs;
  a.scan = scan_args(p, ws, so);
  const int grid = p.nblk < p.num_sms ? p.nblk : p.num_sms;
  if ((p.nblk + grid - 1) / grid > kRouteTcMaxOwn) return cudaErrorInvalidValue;
  return EP == 32 ? launch_route_tc_t<32>(mX, mW, a, grid, st)
                  : launch_route_tc_t<64>(mX, mW, a, grid, st);
}

}  // namespace moe
