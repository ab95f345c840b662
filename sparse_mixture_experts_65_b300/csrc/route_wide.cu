// route_wide.cu -- stages 1 to 4, and the copy of the kept token rows into
// expert order, in one launch for bf16 layers with 64 < E <= 256 experts and
// k <= 8 (DeepSeek-V3-shaped routers: 256 experts, top-8).
//
// What is computed is that of the split path (router.cu, route_scan.cuh,
// route.cu): "Mixture of Experts" (llm-tutorial ch. 11) § The mathematics and
// § Top-k routing (s = W_r x, the k largest, gates from the chosen logits),
// "Mixture of experts" (inside-the-model guide) § The computation and
// § Auxiliary-loss-free balancing (sigmoid affinities, a bias that only
// selects), ch. 11 § Expert capacity and dropped tokens (first come by the
// token-major key t*k + j), and the guide's § Auxiliary loss (f_i, P_i, L).
//
// Launch: clusters of KS CTAs (KS in 1, 2, 4, 8), one cluster per 128-token
// tile, persistent over tiles; CTA c of a cluster takes the c-th share of the
// model width's 128-wide chunks, so that each CTA streams 128 x d/KS of x and
// all experts' E x d/KS of W_r (half the bytes of a split over experts, which
// re-reads the whole x tile in every CTA).  320 threads:
//   warp 0     TMA: the x tile (128 tokens x 64 k) and W_r (EPN experts x
//              64 k, rows past E read as zeros), 128-byte swizzle;
//   warp 1     tcgen05.mma (M = 128, N = EPN, K = 16) into one of two TMEM
//              accumulators, one per 128-wide chunk;
//   warps 2-9  two per TMEM lane quarter, each on half of the EPN columns:
//              the chunk results are added in float32 in chunk order (the
//              tensor-core router's arithmetic, ~2e-6 on a 7168-wide router).
// At the end of a tile every CTA writes its partial logits to a scratch
// buffer in global memory and signals the cluster's CTAs (remote mbarrier
// arrivals, release at cluster scope).  CTA c then routes the tile's c-th
// block of 128/KS tokens, one token per warp: the KS partials added in CTA
// order plus the logit offset, selection, top-k, gates, the router
// distribution, and the rank of every key among the earlier keys of the
// block with the same expert; the block's histogram and probability sums are
// published.  A grid-wide wait (bounded; the grid is sized to the clusters
// the GPU holds at once, so every CTA is resident) follows,
// after which every CTA derives the routed totals, the exclusive prefix of
// its own blocks and the expert segments (CTA 0 also writes the meta data
// and the balance statistics), turns its keys' ranks into positions and
// rows, and copies its tokens' rows into their segments (each row read once).
//
// Determinism: counts are integers; every float sum has a fixed association
// (chunk order, CTA order, a fixed butterfly per warp, warps and blocks in
// order), so repeated calls agree bitwise.
#include <atomic>
#include <climits>
#include <cstring>

#include "bulk_rows.cuh"
#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "route_scan.cuh"
#include "tma_host.cuh"

namespace moe {

constexpr int kRwThreads = 320;
constexpr int kRwEpiThreads = 256;        // warps 2..9
constexpr int kRwEpiWarps = kRwEpiThreads / 32;
constexpr int kRwBK = 64;                 // k per stage (128 bytes of bf16)
constexpr int kRwChunkKB = 2;             // stages per accumulator: 128-wide chunks
constexpr int kRwGroups = 5;              // scan: 5 groups of 64 threads, 4 experts each
constexpr uint64_t kRwTimeoutNs = 2000000000ull;   // 2 s

template <int EPN>
struct RwCfg {
  static_assert(EPN == 128 || EPN == 256, "experts per MMA");
  static constexpr int A_BYTES = kTcBM * kRwBK * 2;
  static constexpr int B_BYTES = EPN * kRwBK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = EPN == 256 ? 4 : 6;
  static constexpr int STAGE_AREA = STAGES * STAGE_BYTES;   // also the scan's and copy's space
  static constexpr int TMEM_COLS = 2 * EPN;
  static constexpr int HALF = EPN / 2;                      // columns per epilogue thread
  static constexpr int NPL = EPN / 32;                      // experts per lane when routing
  static constexpr uint32_t IDESC = idesc_bf16_f32(kTcBM, EPN);
  static constexpr int al16(int b) { return (b + 15) / 16 * 16; }
  static constexpr int NBARS = 2 * STAGES + 8;   // + tfull 2, tempty 2, ready 2, drain, released
  // the tile's partial logits, row-major with a padded pitch, over the stages
  static constexpr int PITCH = EPN + 4;
  static_assert(kTcBM * PITCH * 4 <= STAGE_AREA, "partial logits fit the stage area");
  static constexpr int BAR_BYTES = al16(8 * NBARS);
  static constexpr int FAN_BAR_BYTES = 8 * kFanMaxSlots;
  static constexpr int KEYS_BYTES = 4 * kTcBM * kRouteWideMaxK;   // keys of a block, then ranks
  static constexpr int PW_BYTES = 4 * kRwEpiWarps * EPN;
  static constexpr int CNT_BYTES = 4 * EPN;
  static constexpr int VEC_BYTES = 4 * 2 * EPN;             // selection bias and logit offset
  static constexpr int MISC_BYTES = 64;
  static constexpr int SMEM = 1024 + STAGE_AREA + BAR_BYTES + FAN_BAR_BYTES + 2 * KEYS_BYTES +
                              PW_BYTES + CNT_BYTES + VEC_BYTES + MISC_BYTES;
};

// The per-CTA capacity scan's shared memory, laid over the stage area once the
// main loop is done.
struct RwScanSmem {
  int seg[kRwGroups][kRouteWideMaxOwn + 1][256];   // per group: histogram sums between own blocks
  float psum[kRwGroups][256];                      // CTA 0: per-group probability sums
  int pre[kRouteWideMaxOwn][256];                  // exclusive prefix of every own block
  int segst[256];                                  // first row of each expert's segment
  int off[256];                                    // first slot of each expert
  int wk[kRwEpiWarps], wm[kRwEpiWarps];            // warp totals of the expert scans
  double red[kRwEpiWarps];
};
static_assert(sizeof(RwScanSmem) <= RwCfg<128>::STAGE_AREA, "scan scratch fits the stages");
static_assert(sizeof(RwScanSmem) <= RwCfg<256>::STAGE_AREA, "scan scratch fits the stages");

struct RouteWideArgs {
  const float* logit_offset;   // [E] or null
  const float* sel_bias;       // [E] or null
  int32_t* topk_idx;           // [T*k]
  float* topk_w;               // [T*k]
  int32_t* slot_pos;           // [T*k] or null
  int* key_row;                // [T*k]: rank inside the block, then the padded row
  int* row_token;              // [R_cap]
  const char* x_rows;          // x, when the kernel copies the kept rows (else null)
  char* xp;                    // [R_cap][d] expert-ordered copies
  uint32_t row_bytes;
  int T, d, E, Es, k, gate, capacity, ntiles, ks, ncl, R_cap;
  unsigned* arrive;            // CTAs whose blocks are published
  unsigned* passed;            // CTAs through the wait (the last one re-arms both)
  unsigned* arrive2;           // the second wait: CTAs whose positions are written
  unsigned* passed2;
  int* copy_next;              // next token row of the copy to hand out
  unsigned* copy_done;         // CTAs done copying (the last one re-arms both)
  uint32_t* status;
  uint64_t timeout_ns;
  ScanArgs scan;               // blk_cnt / blk_prob rows have stride Es
};

__device__ __forceinline__ void rw_epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ unsigned rw_ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Experts of lane l when routing: four consecutive experts per 128-wide
// group, e = 4 l + 128 (i / 4) + i % 4 (i < NPL), the order in which the
// partial logits are stored (float4 groups, coalesced over token rows).
__device__ __forceinline__ int rw_expert(int lane, int i) {
  return 4 * lane + 128 * (i >> 2) + (i & 3);
}
// Lane and slot holding expert e.
__device__ __forceinline__ int rw_owner_lane(int e) { return (e & 127) >> 2; }
__device__ __forceinline__ int rw_owner_slot(int e) { return ((e >> 7) << 2) | (e & 3); }

// Order-preserving map of a float (not NaN) to an unsigned integer; 0 lies
// below every float.
__device__ __forceinline__ unsigned rw_ord(float v) {
  const unsigned u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One compare-exchange of a descending sort of (hi, lo) keys.
__device__ __forceinline__ void rw_cas(unsigned& ha, unsigned& la, unsigned& hb, unsigned& lb) {
  const bool swap = hb > ha || (hb == ha && lb > la);
  const unsigned th = swap ? hb : ha, tl = swap ? lb : la;
  hb = swap ? ha : hb;
  lb = swap ? la : lb;
  ha = th;
  la = tl;
}

// Descending sort of N = 4 or 8 keys (Batcher's odd-even merge sort: 5 or 19
// compare-exchanges).
template <int N>
__device__ __forceinline__ void rw_sort(unsigned (&h)[N], unsigned (&l)[N]) {
  static_assert(N == 4 || N == 8, "sort width");
#define RW_CAS(i, j) rw_cas(h[i], l[i], h[j], l[j])
  RW_CAS(0, 1); RW_CAS(2, 3); RW_CAS(0, 2); RW_CAS(1, 3); RW_CAS(1, 2);
  if constexpr (N == 8) {
    RW_CAS(4, 5); RW_CAS(6, 7); RW_CAS(4, 6); RW_CAS(5, 7); RW_CAS(5, 6);
    RW_CAS(0, 4); RW_CAS(1, 5); RW_CAS(2, 6); RW_CAS(3, 7);
    RW_CAS(2, 4); RW_CAS(3, 5);
    RW_CAS(1, 2); RW_CAS(3, 4); RW_CAS(5, 6);
  }
#undef RW_CAS
}

// Routing of NT tokens by one warp, interleaved so that their dependent
// chains overlap; lane l holds the logits of experts rw_expert(l, i)
// (offset included, -inf past E).  For each valid token: the k choices and
// gates (lanes < k), the chosen experts to keys[0..k), and the token's router
// distribution added to psum.
//
// Selection: each lane sorts its experts by the key (selection score, then
// the lower index first) once; a round then takes the largest head key of
// the warp (two warp maxima: the score's order-preserving integer form, then
// the inverted index among the lanes holding that score) and the winning
// lane drops its head.  Ties go to the lower index, as in the pages' top-k.
// The sigmoid uses the hardware exponential and an approximate reciprocal
// (~1e-7 relative, far inside the near-tie band and the gate tolerance).
template <int NPL, int NT>
__device__ __forceinline__ void rw_route_tokens(const float (&sv)[NT][NPL], const bool (&valid)[NT],
                                                int E, int k, int gate, const float* bias_s,
                                                int32_t* const (&idx_out)[NT],
                                                float* const (&w_out)[NT], int* const (&keys)[NT],
                                                float (&psum)[NPL]) {
  const int lane = threadIdx.x & 31;
  const bool sigm = gate == MOE_GATE_SIGMOID_RENORM;
  float aff[NT][NPL];
  unsigned kh[NT][NPL], kl[NT][NPL];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = rw_expert(lane, i);
      aff[t][i] = sigm ? __fdividef(1.0f, 1.0f + __expf(-sv[t][i])) : sv[t][i];
      float v = aff[t][i] + bias_s[e];
      if (v != v) v = -INFINITY;
      kh[t][i] = e < E ? rw_ord(v) : 0u;     // experts past E never win a round
      kl[t][i] = ~static_cast<unsigned>(e);
    }
#pragma unroll
  for (int t = 0; t < NT; ++t) rw_sort<NPL>(kh[t], kl[t]);
  int my_idx[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) my_idx[t] = 0;
  for (int r = 0; r < k; ++r) {
    unsigned mh[NT], ml[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) mh[t] = __reduce_max_sync(0xffffffffu, kh[t][0]);
#pragma unroll
    for (int t = 0; t < NT; ++t) ml[t] = __reduce_max_sync(0xffffffffu, kh[t][0] == mh[t] ? kl[t][0] : 0u);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int w = static_cast<int>(~ml[t]);
      if (lane == r) my_idx[t] = w;
      if (kh[t][0] == mh[t] && kl[t][0] == ml[t]) {   // this lane's head won: drop it
#pragma unroll
        for (int i = 0; i + 1 < NPL; ++i) {
          kh[t][i] = kh[t][i + 1];
          kl[t][i] = kl[t][i + 1];
        }
        kh[t][NPL - 1] = 0u;
        kl[t][NPL - 1] = 0u;
      }
    }
  }
  const bool mine = lane < k;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    // the chosen expert's logit, from the lane and slot that hold it
    const int src = rw_owner_lane(my_idx[t]), slot = rw_owner_slot(my_idx[t]);
    float my_s = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const float v = __shfl_sync(0xffffffffu, sv[t][i], src);
      if (slot == i) my_s = v;
    }
    const float s_me = mine ? my_s : -INFINITY;
    float m_all = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPL; ++i) m_all = fmaxf(m_all, sv[t][i]);
    m_all = warp_max(m_all);
    float ex[NPL];
    float z_all = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      ex[i] = sigm ? aff[t][i] : expf(sv[t][i] - m_all);
      if (rw_expert(lane, i) < E) z_all += ex[i];
    }
    z_all = warp_sum(z_all);
    float g;
    if (gate == MOE_GATE_SOFTMAX_TOPK) {
      const float m_k = warp_max(s_me);
      const float ek = mine ? expf(s_me - m_k) : 0.f;
      g = ek / warp_sum(ek);
    } else if (sigm) {
      const float ak = mine ? __fdividef(1.0f, 1.0f + __expf(-s_me)) : 0.f;
      g = ak / warp_sum(ak);
    } else {
      g = expf(s_me - m_all) / z_all;
    }
    if (valid[t]) {
      if (mine) {
        idx_out[t][lane] = my_idx[t];
        w_out[t][lane] = g;
        keys[t][lane] = my_idx[t];
      }
      const float inv_z = 1.0f / z_all;
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (rw_expert(lane, i) < E) psum[i] += ex[i] * inv_z;
    }
  }
}

// Grid-wide wait (bounded; every CTA of the grid is resident): each thread's
// global writes are made visible, thread 0 counts this CTA in and spins until
// every CTA has arrived; the last CTA through re-arms both counters.  A CTA
// whose roles gave up (abort set) does not arrive, so the others time out.
// Returns false (for every thread of the CTA) when the wait ran out.
__device__ bool rw_grid_wait(unsigned* arrive, unsigned* passed, uint32_t* status,
                             uint64_t timeout_ns, const volatile int* abort_flag, int* s_fail) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    bool seen = false;
    if (*abort_flag == 0) {
      atomicAdd(arrive, 1u);
      const uint64_t t_start = globaltimer_ns();
      for (uint32_t i = 0;; ++i) {
        if (rw_ld_acquire_gpu(arrive) >= gridDim.x) {
          seen = true;
          break;
        }
        if ((i & 63u) == 63u && globaltimer_ns() - t_start > timeout_ns) break;
      }
    }
    if (!seen) atomicOr(status, STATUS_TIMEOUT_ROUTE);
    *s_fail = seen ? 0 : 1;
    if (atomicAdd(passed, 1u) == gridDim.x - 1u) {
      *arrive = 0u;
      *passed = 0u;
    }
  }
  __syncthreads();
  return *s_fail == 0;
}

// Per-CTA view of the capacity scan, run by every CTA once all blocks are
// published: routed totals per expert, the exclusive prefix of each block
// this CTA owns (blocks (cl + j*ncl)*KS + c, j < nown) and the expert
// segments.  One round of histogram loads: five groups of 64 threads, each
// thread four experts (16-byte loads), group g taking blocks g, g + 5, ...;
// then one thread per expert.  CTA 0 also writes the layer's meta data and
// the balance statistics.
__device__ void rw_scan_cta(const RouteWideArgs& a, RwScanSmem& sm, int cl, int c, int nown) {
  const ScanArgs& sa = a.scan;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool writer = blockIdx.x == 0;
  const int nblk = a.ntiles * a.ks;
  auto own_block = [&](int j) { return (cl + j * a.ncl) * a.ks + c; };
  {
    const int g = tid >> 6, e0 = 4 * (tid & 63);
    if (e0 < a.E) {
      int s_idx = 0, bound = nown > 0 ? own_block(0) : INT_MAX;
      int4 acc = make_int4(0, 0, 0, 0);
      constexpr int U = 16;   // loads in flight per thread
      for (int b0 = g; b0 < nblk; b0 += kRwGroups * U) {
        int4 cv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = b0 + kRwGroups * u;
          cv[u] = b < nblk
                      ? __ldcg(reinterpret_cast<const int4*>(sa.blk_cnt + (size_t)b * a.Es + e0))
                      : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int b = b0 + kRwGroups * u;
          if (b < nblk) {
            while (b >= bound) {
              *reinterpret_cast<int4*>(&sm.seg[g][s_idx][e0]) = acc;
              acc = make_int4(0, 0, 0, 0);
              ++s_idx;
              bound = s_idx < nown ? own_block(s_idx) : INT_MAX;
            }
            acc.x += cv[u].x;
            acc.y += cv[u].y;
            acc.z += cv[u].z;
            acc.w += cv[u].w;
          }
        }
      }
      for (; s_idx <= nown; ++s_idx) {
        *reinterpret_cast<int4*>(&sm.seg[g][s_idx][e0]) = acc;
        acc = make_int4(0, 0, 0, 0);
      }
      if (writer) {
        // the router distribution's sums over the blocks of group g, in order
        float4 pacc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int b0 = g; b0 < nblk; b0 += kRwGroups * U) {
          float4 pv[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int b = b0 + kRwGroups * u;
            pv[u] = b < nblk ? __ldcg(reinterpret_cast<const float4*>(sa.blk_prob +
                                                                      (size_t)b * a.Es + e0))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (b0 + kRwGroups * u < nblk) {
              pacc.x += pv[u].x;
              pacc.y += pv[u].y;
              pacc.z += pv[u].z;
              pacc.w += pv[u].w;
            }
          }
        }
        *reinterpret_cast<float4*>(&sm.psum[g][e0]) = pacc;
      }
    }
  }
  __syncthreads();
  // one thread per expert: prefixes of the own blocks and the routed total
  const int e = tid;
  const bool ev = e < a.E;
  int routed = 0;
  if (ev) {
    int run = 0;
    for (int s = 0; s <= nown; ++s) {
      int v = 0;
#pragma unroll
      for (int g = 0; g < kRwGroups; ++g) v += sm.seg[g][s][e];
      run += v;
      if (s < nown) sm.pre[s][e] = run;
    }
    routed = run;
  }
  // kept counts and M tiles, exclusive scans over the experts (warps 0..7)
  const int kept = ev ? (routed < a.capacity ? routed : a.capacity) : 0;
  const int mt = ev ? (kept + sa.bm - 1) / sa.bm : 0;
  int ik = kept, im = mt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nk = __shfl_up_sync(0xffffffffu, ik, o);
    const int nm = __shfl_up_sync(0xffffffffu, im, o);
    if (lane >= o) {
      ik += nk;
      im += nm;
    }
  }
  if (lane == 31 && warp < kRwEpiWarps) {
    sm.wk[warp] = ik;
    sm.wm[warp] = im;
  }
  __syncthreads();
  int xk = ik - kept, xm = im - mt, tk = 0, tm = 0;
#pragma unroll
  for (int w = 0; w < kRwEpiWarps; ++w) {
    if (w < warp) {
      xk += sm.wk[w];
      xm += sm.wm[w];
    }
    tk += sm.wk[w];
    tm += sm.wm[w];
  }
  double l = 0.0;
  if (ev) {
    sm.segst[e] = xm * sa.bm;
    sm.off[e] = xk;
    if (writer) {
      float ps = 0.f;
#pragma unroll
      for (int g = 0; g < kRwGroups; ++g) ps += sm.psum[g][e];
      const float P = ps / (float)a.T;
      const float f = (float)routed / (float)(a.T * a.k);
      sa.m.kept[e] = kept;
      sa.m.offsets[e] = xk;
      sa.m.seg_start[e] = xm * sa.bm;
      sa.m.mtiles[e] = mt;
      sa.m.tp_up[e] = xm * sa.nt_up;
      sa.m.tp_dn[e] = xm * sa.nt_dn;
      sa.expert_counts[e] = kept;
      if (sa.routed_counts) sa.routed_counts[e] = routed;
      if (sa.offsets_out) sa.offsets_out[e] = xk;
      if (sa.f_out) sa.f_out[e] = f;
      if (sa.P_out) sa.P_out[e] = P;
      l = (double)f * (double)P;
    }
  }
  if (writer && e == 0) {
    const int sh_up = sa.has_shared ? sa.mt_sh * sa.nt_up_sh : 0;
    const int sh_dn = sa.has_shared ? sa.mt_sh * sa.nt_dn_sh : 0;
    sa.m.offsets[a.E] = tk;
    sa.m.seg_start[a.E] = tm * sa.bm;
    sa.m.mtiles[a.E] = sa.has_shared ? sa.mt_sh : 0;
    sa.m.tp_up[a.E] = tm * sa.nt_up;
    sa.m.tp_up[a.E + 1] = tm * sa.nt_up + sh_up;
    sa.m.tp_dn[a.E] = tm * sa.nt_dn;
    sa.m.tp_dn[a.E + 1] = tm * sa.nt_dn + sh_dn;
    if (sa.offsets_out) sa.offsets_out[a.E] = tk;
  }
  // L = alpha * E * sum_i f_i P_i in double: a fixed butterfly per warp, then
  // the warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0 && warp < kRwEpiWarps) sm.red[warp] = l;
  __syncthreads();
  if (writer && tid == 0) {
    double s = 0.0;
    for (int w = 0; w < kRwEpiWarps; ++w) s += sm.red[w];
    sa.aux_loss[0] = (float)((double)sa.alpha * (double)a.E * s);
  }
}


template <int EPN>
__global__ void __launch_bounds__(kRwThreads, 1)
    route_wide_kernel(const __grid_constant__ CUtensorMap mX,
                      const __grid_constant__ CUtensorMap mW, const RouteWideArgs a) {
  using C = RwCfg<EPN>;
  extern __shared__ uint8_t rw_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(rw_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  uint8_t* p = smem + C::STAGE_AREA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  p += C::BAR_BYTES;
  uint64_t* fan_bars = reinterpret_cast<uint64_t*>(p);
  p += C::FAN_BAR_BYTES;
  int* keys_s = reinterpret_cast<int*>(p);     // [BT][k] experts of the routed block's keys
  p += C::KEYS_BYTES;
  int* rank_s = reinterpret_cast<int*>(p);     // [BT][k] their ranks inside the block
  p += C::KEYS_BYTES;
  float* Pw = reinterpret_cast<float*>(p);     // [8][EPN] per-warp probability sums
  p += C::PW_BYTES;
  int* cnt = reinterpret_cast<int*>(p);
  p += C::CNT_BYTES;
  float* bias_s = reinterpret_cast<float*>(p);
  float* offs_s = bias_s + EPN;
  p += C::VEC_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(p);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(p + 4);
  int* s_fail = reinterpret_cast<int*>(p + 8);
  volatile int* s_stop = reinterpret_cast<volatile int*>(p + 12);

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::STAGES + s); };
  auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + 2 + b); };
  auto ready_bar = [&](int b) { return smem_u32(bars + 2 * C::STAGES + 4 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::STAGES + 6);
  const uint32_t released_bar = smem_u32(bars + 2 * C::STAGES + 7);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KS = a.ks;
  const int c = static_cast<int>(cluster_ctarank());   // share of the width, block of the tile
  const int cl = blockIdx.x / KS;                       // cluster: tiles cl, cl + ncl, ...
  const int BT = kTcBM / KS;                            // tokens per routing block
  const int nk = (a.d + kRwBK - 1) / kRwBK;
  const int nch = (nk + kRwChunkKB - 1) / kRwChunkKB;
  const int ch0 = c * nch / KS, ch1 = (c + 1) * nch / KS;
  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kRwEpiThreads);
      mbar_init(ready_bar(b), KS);   // one arrival per CTA of the cluster
    }
    mbar_init(drain_bar, 1);
    mbar_init(released_bar, KS);   // every CTA of the cluster has read this one's partials
    *abort_flag = 0;
    *s_fail = 0;
    *s_stop = 0;
    fence_mbar_init();
  }
  if (tid < EPN) cnt[tid] = 0;
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
  cluster_sync();   // every CTA's barriers exist before a peer signals them
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  // selection bias and logit offset: read by the epilogue warps only
  if (tid >= 64 && tid - 64 < EPN) {
    const int e = tid - 64;
    bias_s[e] = (a.sel_bias && e < a.E) ? a.sel_bias[e] : 0.f;
    offs_s[e] = (a.logit_offset && e < a.E) ? a.logit_offset[e] : 0.f;
  }
  auto give_up = [&]() {
    atomicOr(a.status, STATUS_TIMEOUT_ROUTE);
    *abort_flag = 1;
  };
  const int kb_lo = ch0 * kRwChunkKB;
  const int kb_hi = ch1 * kRwChunkKB < nk ? ch1 * kRwChunkKB : nk;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t g = 0;
      bool ok = true;
      int n = 0;
      for (int tile = cl; tile < a.ntiles && ok; tile += a.ncl, ++n) {
        // the stage area holds the previous tile's partial logits until every
        // CTA of the cluster has read them
        if (n > 0) {
          if (!mbar_wait_cluster_bounded(released_bar, (n - 1) & 1, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          fence_proxy_async_smem();
        }
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          const int s = g % C::STAGES;
          const uint32_t ph = (g / C::STAGES) & 1u;
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(full_bar(s), C::STAGE_BYTES);
          tma_load_2d(sa, &mX, full_bar(s), kb * kRwBK, tile * kTcBM);
          tma_load_2d(sa + C::A_BYTES, &mW, full_bar(s), kb * kRwBK, 0);
        }
      }
      // nothing asynchronous may still target shared memory afterwards
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
      for (int tile = cl; tile < a.ntiles && ok; tile += a.ncl) {
        for (int ch = ch0; ch < ch1 && ok; ++ch, ++it) {
          const int ab = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait_bounded(tempty_bar(ab), aph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * EPN;
          const int kb0 = ch * kRwChunkKB;
          const int kb1 = kb0 + kRwChunkKB < nk ? kb0 + kRwChunkKB : nk;
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
            for (int kk = 0; kk < kRwBK / 16; ++kk)
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
    // ---------------- epilogue and routing (warps 2..9) ----------------
    const int ew = warp - 2;                 // 0..7
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int h = ew >> 2;                   // half of the columns
    const int row = q * 32 + lane;           // token row of the tile
    const int ep_tid = tid - 64;
    int it = 0, itile = 0;
    for (int tile = cl; tile < a.ntiles; tile += a.ncl, ++itile) {
      float acc[C::HALF];
#pragma unroll
      for (int i = 0; i < C::HALF; ++i) acc[i] = 0.f;
      bool ok = true;
      for (int ch = ch0; ch < ch1; ++ch, ++it) {
        const int ab = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_bounded(tfull_bar(ab), aph, a.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_col =
            tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * EPN + h * C::HALF;
#pragma unroll
        for (int cc = 0; cc < C::HALF; cc += 32) {
          uint32_t r[32];
          tmem_ld32(t_col + cc, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[cc + i] += __uint_as_float(r[i]);
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(ab));
      }
      (void)ok;
      // one snapshot of the abort flag, so that all epilogue threads take the
      // same branch (the named barriers below need all 256)
      rw_epi_bar();
      if (ep_tid == 0) *s_stop = *abort_flag;
      rw_epi_bar();
      if (*s_stop) break;
      // this CTA's partial logits of the tile into its stage area (every MMA
      // of the tile has completed), then the cluster's signal
      const int slot = itile & 1;
      const uint32_t rph = (itile >> 1) & 1;
      float* pbs = reinterpret_cast<float*>(smem);
      {
        float4* dst = reinterpret_cast<float4*>(pbs + row * C::PITCH + h * C::HALF);
#pragma unroll
        for (int i = 0; i < C::HALF / 4; ++i)
          dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
      }
      rw_epi_bar();
      if (ep_tid == 0) {
        for (int r = 0; r < KS; ++r) mbar_arrive_cluster(mapa_shared(ready_bar(slot), r));
        if (!mbar_wait_cluster_bounded(ready_bar(slot), rph, a.timeout_ns, abort_flag)) {
          give_up();
          *s_stop = 1;
        }
      }
      rw_epi_bar();
      if (*s_stop) break;
      (void)mbar_try_wait_cluster(ready_bar(slot), rph);   // acquire for every reader
      // ---- routing of block c of the tile: one token per warp ----
      const int t_base = tile * kTcBM + c * BT;
      int ntok = a.T - t_base;
      ntok = ntok < 0 ? 0 : (ntok > BT ? BT : ntok);
      float psum[C::NPL];
#pragma unroll
      for (int j = 0; j < C::NPL; ++j) psum[j] = 0.f;
      // two tokens per warp at a time; the partials of both are requested
      // together, up to four CTAs' shares per round (KS = 8: two rounds)
      constexpr int NG = C::NPL / 4;   // float4 groups per lane
      constexpr int RQ = 4;            // CTA shares per load round
      for (int i0 = 2 * ew; i0 < ntok; i0 += 2 * kRwEpiWarps) {
        float4 v4[2][NG];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int j = 0; j < NG; ++j) v4[t][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r0 = 0; r0 < KS; r0 += RQ) {
          float4 ld[2][RQ][NG];
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int rr = c * BT + (i0 + t < ntok ? i0 + t : i0);
#pragma unroll
            for (int r = 0; r < RQ; ++r)
#pragma unroll
              for (int j = 0; j < NG; ++j)
                ld[t][r][j] = r0 + r < KS
                                  ? ld_dsmem_f4(mapa_shared(
                                        smem_u32(pbs + rr * C::PITCH + 4 * lane + 128 * j),
                                        r0 + r))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int r = 0; r < RQ; ++r)
#pragma unroll
              for (int j = 0; j < NG; ++j)
                if (r0 + r < KS) {                 // the CTAs' shares in order
                  v4[t][j].x += ld[t][r][j].x;
                  v4[t][j].y += ld[t][r][j].y;
                  v4[t][j].z += ld[t][r][j].z;
                  v4[t][j].w += ld[t][r][j].w;
                }
        }
        float sv[2][C::NPL];
        bool valid[2];
        int32_t* io[2];
        float* wo[2];
        int* ko[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
          for (int j = 0; j < NG; ++j) {
            const float vv[4] = {v4[t][j].x, v4[t][j].y, v4[t][j].z, v4[t][j].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int e = rw_expert(lane, 4 * j + u);
              sv[t][4 * j + u] = e < a.E ? vv[u] + offs_s[e] : -INFINITY;
            }
          }
          const int i = i0 + t < ntok ? i0 + t : i0;
          valid[t] = i0 + t < ntok;
          const size_t tok = (size_t)(t_base + i);
          io[t] = a.topk_idx + tok * a.k;
          wo[t] = a.topk_w + tok * a.k;
          ko[t] = keys_s + i * a.k;
        }
        rw_route_tokens<C::NPL, 2>(sv, valid, a.E, a.k, a.gate, bias_s, io, wo, ko, psum);
      }
#pragma unroll
      for (int j = 0; j < C::NPL; ++j) Pw[ew * EPN + rw_expert(lane, j)] = psum[j];
      rw_epi_bar();
      // every partial this CTA needed is read: the cluster's stage areas may
      // take the next tile
      if (ep_tid == 0)
        for (int r = 0; r < KS; ++r) mbar_arrive_cluster(mapa_shared(released_bar, r));
      const int b = tile * KS + c;
      if (ep_tid < a.Es) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kRwEpiWarps; ++w) s += Pw[w * EPN + ep_tid];
        a.scan.blk_prob[(size_t)b * a.Es + ep_tid] = s;
      }
      const int nkeys = ntok * a.k;
      const size_t key0 = (size_t)t_base * a.k;
      if (ew == 0) {
        // rank of every key among the earlier keys of the block with the
        // same expert: keys in order, 32 at a time, equal experts grouped by
        // __match_any_sync, a per-expert count carried across the groups
        for (int c0 = 0; c0 < nkeys; c0 += 32) {
          const int kq = c0 + lane;
          const bool kv = kq < nkeys;
          const int e = kv ? keys_s[kq] : -1 - lane;   // invalid lanes never match
          const unsigned peers = __match_any_sync(0xffffffffu, e);
          const int before = __popc(peers & ((1u << lane) - 1u));
          const int prior = kv ? cnt[e] : 0;
          __syncwarp();
          if (kv) {
            a.key_row[key0 + kq] = prior + before;
            rank_s[kq] = prior + before;
            if (before == 0) cnt[e] = prior + __popc(peers);
          }
          __syncwarp();
        }
      }
      rw_epi_bar();
      if (ep_tid < a.Es) {
        a.scan.blk_cnt[(size_t)b * a.Es + ep_tid] = cnt[ep_tid];
        cnt[ep_tid] = 0;
      }
      rw_epi_bar();
    }
  }

  tc_fence_before();
  __threadfence();
  __syncthreads();
  // no CTA leaves, or reuses its barriers, while a peer may still signal it
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  // every CTA has published its blocks
  if (!rw_grid_wait(a.arrive, a.passed, a.status, a.timeout_ns, abort_flag, s_fail)) return;
  const int nown = (a.ntiles - cl + a.ncl - 1) / a.ncl;
  RwScanSmem& ssm = *reinterpret_cast<RwScanSmem*>(smem);
  rw_scan_cta(a, ssm, cl, c, nown);
  // positions and rows of this CTA's blocks
  for (int j = 0; j < nown; ++j) {
    const int tile = cl + j * a.ncl;
    const int t_base = tile * kTcBM + c * BT;
    int ntok = a.T - t_base;
    ntok = ntok < 0 ? 0 : (ntok > BT ? BT : ntok);
    const int nkeys = ntok * a.k;
    const size_t key0 = (size_t)t_base * a.k;
    // the last tile's keys and ranks are still in shared memory
    const bool last = j == nown - 1;
    for (int kq = tid; kq < nkeys; kq += kRwThreads) {
      const int e = last ? keys_s[kq] : __ldcg(a.topk_idx + key0 + kq);
      if (!in_bounds(e >= 0 && e < a.E, a.status)) {
        a.key_row[key0 + kq] = -1;
        if (a.slot_pos) a.slot_pos[key0 + kq] = -1;
        continue;
      }
      const int pos = ssm.pre[j][e] + (last ? rank_s[kq] : __ldcg(a.key_row + key0 + kq));
      bool keep = pos < a.capacity;
      int rw = keep ? ssm.segst[e] + pos : -1;
      if (keep && !in_bounds(pos >= 0 && rw < a.R_cap, a.status)) {
        keep = false;
        rw = -1;
      }
      a.key_row[key0 + kq] = rw;
      if (a.slot_pos) a.slot_pos[key0 + kq] = keep ? ssm.off[e] + pos : -1;
      if (keep) a.row_token[rw] = t_base + kq / a.k;
    }
  }
  if (a.x_rows == nullptr) return;
  // the kept rows into their segments, once every CTA's positions are
  // written: token rows handed out two at a time from a shared counter,
  // each read once into shared memory (the stage area) and stored to the
  // rows of its kept slots
  fence_proxy_async_smem();   // the scan's generic accesses before the copies' writes
  if (!rw_grid_wait(a.arrive2, a.passed2, a.status, a.timeout_ns, abort_flag, s_fail)) return;
  constexpr int kBatch = 2;
  bulk_fanout_claimed(
      [&]() { return atomicAdd(a.copy_next, kBatch); }, kBatch, a.T, a.k, a.row_bytes,
      [&](int t) { return static_cast<const void*>(a.x_rows + (size_t)t * a.row_bytes); },
      [&](int t, int jj) {
        const int r = __ldcg(a.key_row + (size_t)t * a.k + jj);
        return r >= 0 && in_bounds(r < a.R_cap, a.status)
                   ? static_cast<void*>(a.xp + (size_t)r * a.row_bytes)
                   : nullptr;
      },
      smem, C::STAGE_AREA, fan_bars, a.status, STATUS_TIMEOUT_ROUTE, a.timeout_ns);
  __syncthreads();
  if (tid == 0 && atomicAdd(a.copy_done, 1u) == gridDim.x - 1u) {
    *a.copy_next = 0;    // every CTA has stopped claiming
    *a.copy_done = 0u;
  }
}

// ---------------------------------------------------------------- host side
static int rw_epn(int E) { return E <= 128 ? 128 : 256; }
static int rw_ceil(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

bool route_wide_eligible(const moe_config& c) {
  return c.dtype == MOE_BF16 && c.E > 64 && c.E <= 256 && c.k <= kRouteWideMaxK &&
         (long long)c.T <= (long long)kRouteWideMaxOwn * kTcBM * 64;
}

// CTAs per 128-token tile: the largest of 8, 4, 2, 1 that keeps the grid
// within one wave of a 148-SM GPU and gives every CTA at least one chunk.
int route_wide_ks(const moe_config& c) {
  const int ntiles = rw_ceil(c.T, kTcBM);
  const int nch = rw_ceil(rw_ceil(c.d, kRwBK), kRwChunkKB);
  int ks = 8;
  while (ks > 1 && ((long long)ntiles * ks > kRouteWideSlots || ks > nch)) ks >>= 1;
  return ks;
}

bool route_wide_copies_rows(const Plan& p) {
  const uint32_t row_bytes = (uint32_t)p.cfg.d * (uint32_t)p.elem;
  const int area = p.cfg.E <= 128 ? RwCfg<128>::STAGE_AREA : RwCfg<256>::STAGE_AREA;
  return row_bytes * 3u <= (uint32_t)area;
}

// Clusters of each size that fit on the GPU at once, per device.
static std::atomic<int> g_rw_max_clusters[2][4][64];

template <int EPN>
static cudaError_t rw_max_clusters(int ks, int* out) {
  using C = RwCfg<EPN>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int ki = ks == 1 ? 0 : ks == 2 ? 1 : ks == 4 ? 2 : 3;
  std::atomic<int>& slot = g_rw_max_clusters[EPN == 256][ki][dev & 63];
  int v = slot.load(std::memory_order_relaxed);
  if (v > 0) {
    *out = v;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks);
  cfg.blockDim = dim3(kRwThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaOccupancyMaxActiveClusters(&v, route_wide_kernel<EPN>, &cfg);
  if (e != cudaSuccess) return e;
  if (v < 1) return cudaErrorInvalidConfiguration;
  slot.store(v, std::memory_order_relaxed);
  *out = v;
  return cudaSuccess;
}

template <int EPN>
static cudaError_t launch_route_wide_t(const CUtensorMap& mX, const CUtensorMap& mW,
                                       RouteWideArgs a, cudaStream_t st) {
  using C = RwCfg<EPN>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = route_wide_kernel<EPN>;
  cudaError_t e = smem_attr_once(kern, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  int maxcl = 0;
  if ((e = rw_max_clusters<EPN>(a.ks, &maxcl)) != cudaSuccess) return e;
  int ncl = a.ntiles;
  if (ncl > maxcl) ncl = maxcl;
  if (ncl > kRouteWideMaxCtas / a.ks) ncl = kRouteWideMaxCtas / a.ks;
  if (ncl < 1 || rw_ceil(a.ntiles, ncl) > kRouteWideMaxOwn) return cudaErrorInvalidValue;
  a.ncl = ncl;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ncl * a.ks);
  cfg.blockDim = dim3(kRwThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  // a cluster launch (no cooperative attribute): the grid holds at most the
  // clusters the GPU keeps resident at once, so every CTA reaches the
  // grid-wide waits (which are bounded in any case)
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mX, mW, a);
}

cudaError_t launch_route_wide(const Plan& p, const void* x, const void* W_r,
                              const float* logit_offset, const float* sel_bias,
                              int32_t* topk_idx, float* topk_w, int32_t* slot_pos, bool copy,
                              void* ws, const ScanOutputs& so, cudaStream_t st) {
  const moe_config& c = p.cfg;
  const int EPN = rw_epn(c.E);
  CUtensorMap mX, mW;
  if (!encode_2d(&mX, x, c.T, c.d, kTcBM) || !encode_2d(&mW, W_r, c.E, c.d, EPN))
    return cudaErrorInvalidValue;
  char* w = static_cast<char*>(ws);
  RouteWideArgs a;
  std::memset(&a, 0, sizeof(a));
  a.logit_offset = logit_offset;
  a.sel_bias = sel_bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.slot_pos = slot_pos;
  a.key_row = reinterpret_cast<int*>(w + p.ws.key_row);
  a.row_token = reinterpret_cast<int*>(w + p.ws.row_token);
  const bool in_kernel = copy && route_wide_copies_rows(p);
  a.x_rows = in_kernel ? static_cast<const char*>(x) : nullptr;
  a.xp = w + p.ws.xp;
  a.row_bytes = (uint32_t)c.d * (uint32_t)p.elem;
  a.T = c.T;
  a.d = c.d;
  a.E = c.E;
  a.Es = p.blk_stride;
  a.k = c.k;
  a.gate = c.gate;
  a.capacity = p.capacity;
  a.ntiles = rw_ceil(c.T, kTcBM);
  a.ks = p.rw_ks;
  a.R_cap = p.R_cap;
  a.arrive = reinterpret_cast<unsigned*>(w + p.ws.status + kRouteArriveOffset);
  a.passed = reinterpret_cast<unsigned*>(w + p.ws.status + kRoutePassedOffset);
  a.arrive2 = reinterpret_cast<unsigned*>(w + p.ws.status + kRouteArrive2Offset);
  a.passed2 = reinterpret_cast<unsigned*>(w + p.ws.status + kRoutePassed2Offset);
  a.copy_next = reinterpret_cast<int*>(w + p.ws.status + kRouteCopyNextOffset);
  a.copy_done = reinterpret_cast<unsigned*>(w + p.ws.status + kRouteCopyDoneOffset);
  a.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  a.timeout_ns = kRwTimeoutNs;
  a.scan = scan_args(p, ws, so);
  if (a.ks < 1 || kTcBM % a.ks != 0 || a.ntiles * a.ks != p.nblk) return cudaErrorInvalidValue;
  cudaError_t e = EPN == 128 ? launch_route_wide_t<128>(mX, mW, a, st)
                             : launch_route_wide_t<256>(mX, mW, a, st);
  if (e != cudaSuccess) return e;
  if (copy && !in_kernel) return launch_gather_rows(p, x, ws, st);
  return cudaSuccess;
}

}  // namespace moe
