// router.cu -- stages 1 and 2 of the layer: router scores s = W_r x (+ o) in
// float32, then top-k selection with the selection bias, gate normalisation,
// the full router distribution for P_i and per-block expert histograms.
//
// "Mixture of Experts" (llm-tutorial ch. 11) § Top-k routing: softmax over the
// k chosen logits; § Top-1 vs top-2: the full-softmax probability of a top-1
// choice; § Why MoE is hard: the router runs in float32 even when the model
// is bf16.  "Mixture of experts" (inside-the-model guide) § The computation
// and § Auxiliary-loss-free balancing: renormalised sigmoid gates and a bias
// that steers only the choice.
//
// Kernel 1 (scores) is a float32 FMA GEMM over [T x d] x [d x E]: 128-token x
// BN-expert tiles, 8 x TN outputs per thread, register-prefetched double
// buffering, and a split of the reduction over blockIdx.z so that small
// batches still fill the GPU.  bf16 x bf16 products are exact in float32;
// each thread adds its products in 128-wide chunks before folding them into
// the running sum, which keeps the rounding error of a 7168-long dot product
// near 1e-7 relative.  Partial sums go to [S][T][E].
//
// Kernel 2 (top-k) gives each warp whole tokens: lanes hold E/32 scores (the
// split partials summed in a fixed order), k rounds of warp arg-max pick the
// experts (larger score first, equal scores to the lower index), then gates,
// the router distribution and the block's expert histogram.
#include <atomic>
#include <cfloat>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>

#include "bulk_rows.cuh"
#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"
#include "route_scan.cuh"

namespace moe {

// ---------------------------------------------------------------- scores
struct ScoresArgs {
  const void* x;       // [T][d]
  const void* W_r;     // [E][d]
  const float* logit_offset;   // [E] or null
  float* part;         // [S][T][E] split partials (S > 1)
  float* scores;       // [T][E] final logits
  unsigned int* tile_counter;  // [mblocks * nblocks] split blocks done per tile
  int T, d, E, k_split, S;
};

constexpr int kScBM = 128, kScBK = 32, kScTM = 8, kScStages = 4;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, bool ok) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  const int n = ok ? 16 : 0;     // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void to_float8(const uint4& u, const __nv_bfloat16*, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void to_float8(const uint4& u, const float*, float (&v)[8]) {
  v[0] = __uint_as_float(u.x);
  v[1] = __uint_as_float(u.y);
  v[2] = __uint_as_float(u.z);
  v[3] = __uint_as_float(u.w);
}

// Raw input tiles stream through a kScStages-deep cp.async pipeline in their
// stored precision.  Each stage is converted once to float32 and transposed
// into a k-major tile; the inner loop then reads 8 token values and TN expert
// values with vector loads and forms products in increasing k order.
// Thread (ty, tx) of 16 x 16 owns tokens ty*8 .. ty*8+7 and experts
// tx*TN .. tx*TN+TN-1.
template <typename TIn, int TN>
__global__ void __launch_bounds__(kThreads) router_scores_kernel(const ScoresArgs a) {
  constexpr int BM = kScBM, BK = kScBK, TM = kScTM, BN = 16 * TN;
  constexpr int EPC = 16 / sizeof(TIn);          // elements per 16-byte chunk
  constexpr int LD = BK + EPC;                   // raw smem row stride (elements)
  constexpr int A_EL = BM * LD, B_EL = BN * LD;
  constexpr int CPR = BK / EPC;                  // 16-byte chunks per tile row
  extern __shared__ __align__(16) uint8_t sc_smem[];
  float* Af = reinterpret_cast<float*>(sc_smem);             // [BK][BM + 4]
  float* Bf = Af + BK * (BM + 4);                            // [BK][BN + 4]
  TIn* As = reinterpret_cast<TIn*>(Bf + BK * (BN + 4));      // [stages][BM][LD]
  TIn* Bs = As + kScStages * A_EL;                           // [stages][BN][LD]
  __shared__ int am_last;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  const int k_beg = blockIdx.z * a.k_split;
  const int k_end = min(a.d, k_beg + a.k_split);
  const TIn* X = static_cast<const TIn*>(a.x);
  const TIn* Wr = static_cast<const TIn*>(a.W_r);
  pdl_wait();
  pdl_trigger();

  auto issue = [&](int stage, int k0) {
    TIn* as = As + stage * A_EL;
    TIn* bs = Bs + stage * B_EL;
    for (int c = tid; c < BM * CPR; c += kThreads) {
      const int r = c % BM, kc = (c / BM) * EPC;
      const int gm = m0 + r, gk = k0 + kc;
      const bool ok = gm < a.T && gk < k_end;
      cp_async16(as + r * LD + kc, X + (ok ? (size_t)gm * a.d + gk : 0), ok);
    }
    for (int c = tid; c < BN * CPR; c += kThreads) {
      const int r = c % BN, kc = (c / BN) * EPC;
      const int gn = n0 + r, gk = k0 + kc;
      const bool ok = gn < a.E && gk < k_end;
      cp_async16(bs + r * LD + kc, Wr + (ok ? (size_t)gn * a.d + gk : 0), ok);
    }
  };
  // raw stage -> float32, transposed to [k][row]; consecutive threads take
  // consecutive rows, so both the 16-byte reads and the scalar writes are
  // free of bank conflicts
  auto convert = [&](int stage) {
    const TIn* as = As + stage * A_EL;
    const TIn* bs = Bs + stage * B_EL;
    for (int c = tid; c < BM * CPR; c += kThreads) {
      const int r = c % BM, kc = (c / BM) * EPC;
      float v[8];
      to_float8(*reinterpret_cast<const uint4*>(as + r * LD + kc), as, v);
#pragma unroll
      for (int i = 0; i < EPC; ++i) Af[(kc + i) * (BM + 4) + r] = v[i];
    }
    for (int c = tid; c < BN * CPR; c += kThreads) {
      const int r = c % BN, kc = (c / BN) * EPC;
      float v[8];
      to_float8(*reinterpret_cast<const uint4*>(bs + r * LD + kc), bs, v);
#pragma unroll
      for (int i = 0; i < EPC; ++i) Bf[(kc + i) * (BN + 4) + r] = v[i];
    }
  };

  float acc[TM][TN], part[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = part[i][j] = 0.f;

  const int nk = (k_end - k_beg + BK - 1) / BK;
#pragma unroll
  for (int s = 0; s < kScStages - 1; ++s) {
    if (s < nk) issue(s, k_beg + s * BK);
    cp_async_commit();
  }
  for (int it = 0; it < nk; ++it) {
    cp_async_wait<kScStages - 2>();
    __syncthreads();                      // stage `it` landed; the float tile is free
    convert(it % kScStages);
    {
      const int nxt = it + kScStages - 1;
      if (nxt < nk) issue(nxt % kScStages, k_beg + nxt * BK);
      cp_async_commit();
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(Af + kk * (BM + 4) + ty * TM);
      const float4 a1 = *reinterpret_cast<const float4*>(Af + kk * (BM + 4) + ty * TM + 4);
      const float av[TM] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float bv[TN];
      if (TN == 4) {
        const float4 b4 = *reinterpret_cast<const float4*>(Bf + kk * (BN + 4) + tx * TN);
        bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
      } else {
        const float2 b2 = *reinterpret_cast<const float2*>(Bf + kk * (BN + 4) + tx * TN);
        bv[0] = b2.x; bv[1] = b2.y;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
    }
    if ((it & 3) == 3 || it + 1 == nk) {   // fold every 128 k into the running sum
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          acc[i][j] += part[i][j];
          part[i][j] = 0.f;
        }
    }
  }
  cp_async_wait<0>();

  if (a.S == 1) {
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int m = m0 + ty * TM + i;
      if (m >= a.T) continue;
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const int n = n0 + tx * TN + j;
        if (n < a.E)
          a.scores[(size_t)m * a.E + n] = acc[i][j] + (a.logit_offset ? a.logit_offset[n] : 0.f);
      }
    }
    return;
  }
  // Split reduction: every split block publishes its partial; the last one
  // to finish for this tile adds the S partials in split order.
  float* out = a.part + (size_t)blockIdx.z * a.T * a.E;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int m = m0 + ty * TM + i;
    if (m >= a.T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int n = n0 + tx * TN + j;
      if (n < a.E) out[(size_t)m * a.E + n] = acc[i][j];
    }
  }
  __threadfence();
  __syncthreads();
  unsigned int* ctr = a.tile_counter + blockIdx.x * gridDim.y + blockIdx.y;
  if (tid == 0) am_last = atomicAdd(ctr, 1u) == (unsigned)(a.S - 1);
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  // all TM x TN partials of one split are loaded before any of them is added
  const size_t TE = (size_t)a.T * a.E;
  float sum[TM][TN];
  for (int z = 0; z < a.S; ++z) {
    float v[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int m = m0 + ty * TM + i;
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const int n = n0 + tx * TN + j;
        v[i][j] = (m < a.T && n < a.E) ? __ldcg(a.part + z * TE + (size_t)m * a.E + n) : 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) sum[i][j] = z == 0 ? v[i][j] : sum[i][j] + v[i][j];
  }
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int m = m0 + ty * TM + i;
    if (m >= a.T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int n = n0 + tx * TN + j;
      if (n < a.E)
        a.scores[(size_t)m * a.E + n] = sum[i][j] + (a.logit_offset ? a.logit_offset[n] : 0.f);
    }
  }
  if (tid == 0) *ctr = 0;
}

// ---------------------------------------------------------------- top-k
// One warp routes one token.  sv[i] holds the logit of expert lane + 32 i
// (logit offset included, -inf past E).  Selection: k rounds of warp arg-max
// over sel = affinity + bias (larger first, equal to the lower index; NaN never
// outranks a number).  Gates from the unbiased logits; the full router
// distribution (softmax, or sigmoid normalised over all E) is added to psum;
// the chosen experts are counted into the block histogram `cnt`.
template <int NPL_MAX>
__device__ __forceinline__ void route_one_token(const float (&sv)[NPL_MAX], int E, int k, int gate,
                                                const float* sel_bias, int32_t* idx_out,
                                                float* w_out, int* cnt,
                                                float (&psum)[NPL_MAX]) {
  const int lane = threadIdx.x & 31;
  const bool sigm = gate == MOE_GATE_SIGMOID_RENORM;
  // affinities, once per score: the logit, or its sigmoid with the hardware
  // exponential and an approximate reciprocal (relative error ~1e-7, far
  // inside the 1e-5 near-tie band and the gate tolerance)
  float aff[NPL_MAX], sel[NPL_MAX];
#pragma unroll
  for (int i = 0; i < NPL_MAX; ++i) {
    const int e = lane + 32 * i;
    aff[i] = sigm ? __fdividef(1.0f, 1.0f + __expf(-sv[i])) : sv[i];
    sel[i] = -INFINITY;
    if (e < E) {
      float v = aff[i];
      if (sel_bias) v += sel_bias[e];
      sel[i] = (v != v) ? -INFINITY : v;
    }
  }
  uint32_t taken = 0;
  int my_idx = 0;
  float my_s = -INFINITY;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY, bs = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < NPL_MAX; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        if (sel[i] > bv || (sel[i] == bv && e < bi)) {
          bv = sel[i];
          bi = e;
          bs = sv[i];
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
        bs = os;
      }
    }
    if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_idx = bi < E ? bi : 0;
      my_s = bs;
    }
  }
  const bool mine = lane < k;
  const float s_me = mine ? my_s : -INFINITY;
  float m_all = -INFINITY;
#pragma unroll
  for (int i = 0; i < NPL_MAX; ++i) m_all = fmaxf(m_all, sv[i]);
  m_all = warp_max(m_all);
  float z_all = 0.f;
#pragma unroll
  for (int i = 0; i < NPL_MAX; ++i)
    if (lane + 32 * i < E) z_all += sigm ? aff[i] : expf(sv[i] - m_all);
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
  if (mine) {
    idx_out[lane] = my_idx;
    w_out[lane] = g;
    atomicAdd(&cnt[my_idx], 1);
  }
#pragma unroll
  for (int i = 0; i < NPL_MAX; ++i)
    if (lane + 32 * i < E)
      psum[i] += sigm ? aff[i] / z_all : expf(sv[i] - m_all) / z_all;
}

// Block epilogue of a routing block: the per-warp probability sums (fixed
// warp order) and the histogram go to the block's row; the last block to
// finish runs the capacity scan for the whole batch.
template <int NT, int NPL_MAX>
__device__ __forceinline__ void publish_and_scan(const ScanArgs& a, const float (&psum)[NPL_MAX],
                                                 float (*Pw)[kMaxE], const int* cnt,
                                                 ScanSmem<NT>& scan_sm, int* am_last) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
#pragma unroll
  for (int i = 0; i < NPL_MAX; ++i)
    if (lane + 32 * i < a.E) Pw[warp][lane + 32 * i] = psum[i];
  __syncthreads();
  for (int e = tid; e < a.E; e += NT) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += Pw[w][e];
    a.blk_prob[(size_t)blockIdx.x * a.E + e] = s;
    a.blk_cnt[(size_t)blockIdx.x * a.E + e] = cnt[e];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *am_last = atomicAdd(a.done_counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!*am_last) return;
  __threadfence();
  scan_block<NT>(a, scan_sm);
  if (tid == 0) *a.done_counter = 0;
}

struct TopkArgs {
  const float* scores;       // [T][E] logits, offset included
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  int T, E, k, BT, gate;
  ScanArgs scan;             // blk_cnt / blk_prob / counter and the scan outputs
};

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;

union TopkSmem {
  struct {
    float Pw[kTopkWarps][kMaxE];
    int cnt[kMaxE];
  } t;
  ScanSmem<kTopkThreads> scan;
};

// Split path: one routing block of BT tokens, warp w takes tokens w, w + 16, ...
// NPL = logits per lane (E <= 32 NPL).
template <int NPL>
__global__ void __launch_bounds__(kTopkThreads) router_topk_kernel(const TopkArgs a) {
  __shared__ TopkSmem sm;
  __shared__ int am_last;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int E = a.E;
  for (int e = tid; e < E; e += kTopkThreads) sm.t.cnt[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;
  const int t0 = blockIdx.x * a.BT;
  for (int tl = warp; tl < a.BT; tl += kTopkWarps) {
    const int t = t0 + tl;
    if (t >= a.T) break;
    float sv[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      sv[i] = e < E ? a.scores[(size_t)t * E + e] : -INFINITY;
    }
    route_one_token<NPL>(sv, E, a.k, a.gate, a.sel_bias, a.topk_idx + (size_t)t * a.k,
                         a.topk_w + (size_t)t * a.k, sm.t.cnt, psum);
  }
  publish_and_scan<kTopkThreads, NPL>(a.scan, psum, sm.t.Pw, sm.t.cnt, sm.scan, &am_last);
}

// ---------------------------------------------------------------- small batches
// Decode-sized batches (T <= kSmallT): stages 1-4 in one launch.  Block s takes
// the 128-wide slice s of the model width and writes float32 partial logits
// for every token and expert (x and W_r staged in shared memory as float32,
// 128 sequential FMAs per output); the last block to finish adds the partials
// in slice order (plus the offset), routes one token per warp, runs the
// capacity scan of the single routing block, ranks the keys in key order and
// writes positions, rows, the row -> token map and the expert-ordered copies.
constexpr int kSmallThreads = 512;
constexpr int kSmallKs = 128;
constexpr uint32_t kSmallStage = 96u << 10;   // bulk-copy staging of the last block

struct SmallArgs {
  const void* x;
  const void* W_r;
  const float* logit_offset;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* slot_pos;
  float* part;      // [S][T][E]
  int* key_row;     // [T*k]
  int* row_token;   // [R_cap]
  void* xp;         // [R_cap][d] or null (no copy)
  int T, d, E, k, gate, capacity, S, nvec, elem, R_cap;
  uint32_t* status;
  ScanArgs scan;
};

template <typename TIn>
__device__ __forceinline__ void load_row_f32(const TIn* src, int n, float* dst) {
  for (int i = 0; i < n; ++i) dst[i] = to_float(src[i]);
}

template <typename TIn, int NPL>
__global__ void __launch_bounds__(kSmallThreads) route_small_kernel(const SmallArgs a) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  __shared__ int am_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, T = a.T;
  const int Ep = E + 1;   // padded row of the transposed weight slice
  pdl_wait();
  pdl_trigger();
  {
    // ---- partial logits of slice s ----
    float* xs = reinterpret_cast<float*>(sm_raw);        // [T][Ks]
    float* ws = xs + kSmallT * kSmallKs;                 // [Ks][Ep]
    const int s = blockIdx.x;
    const int k0 = s * kSmallKs, kn = min(kSmallKs, a.d - k0);
    const TIn* X = static_cast<const TIn*>(a.x);
    const TIn* Wr = static_cast<const TIn*>(a.W_r);
    // 16-byte loads (the slice width and d are multiples of the vector)
    constexpr int V = 16 / (int)sizeof(TIn);
    constexpr int NV = kSmallKs / V;
    for (int i = tid; i < T * NV; i += kSmallThreads) {
      const int t = i / NV, kk = (i - t * NV) * V;
      float v[8];
      if (kk < kn) {
        to_float8(*reinterpret_cast<const uint4*>(X + (size_t)t * a.d + k0 + kk), X, v);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < V; ++j) xs[t * kSmallKs + kk + j] = v[j];
    }
    for (int i = tid; i < E * NV; i += kSmallThreads) {
      const int e = i / NV, kk = (i - e * NV) * V;
      float v[8];
      if (kk < kn) {
        to_float8(*reinterpret_cast<const uint4*>(Wr + (size_t)e * a.d + k0 + kk), Wr, v);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < V; ++j) ws[(kk + j) * Ep + e] = v[j];
    }
    __syncthreads();
    // thread (expert e, group of 4 tokens, part kq of the slice): a weight
    // value is loaded once for the 4 tokens, the x values 4 k at a time
    // (16-byte loads).  Where expert x token-group items leave threads idle
    // (small T), the slice's 128 k are split into KQ parts summed in k order
    // by different threads, then added in part order; otherwise every output
    // sums its 128 products in k order.
    const int ngrp = (T + 3) / 4;
    int KQ = 1;
    while (KQ < 4 && E * ngrp * KQ * 2 <= kSmallThreads) KQ *= 2;
    const int kw = kSmallKs / KQ;
    float* red = ws + kSmallKs * Ep;                     // [KQ][T][E] part sums
    for (int i = tid; i < E * ngrp * KQ; i += kSmallThreads) {
      const int e = i % E, rest = i / E;
      const int t0 = (rest % ngrp) * 4, kq = rest / ngrp;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kk = kq * kw; kk < (kq + 1) * kw; kk += 4) {
        const float w0 = ws[kk * Ep + e], w1 = ws[(kk + 1) * Ep + e];
        const float w2 = ws[(kk + 2) * Ep + e], w3 = ws[(kk + 3) * Ep + e];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (t0 + j < T) {
            const float4 x4 = *reinterpret_cast<const float4*>(xs + (t0 + j) * kSmallKs + kk);
            acc[j] = fmaf(x4.x, w0, acc[j]);
            acc[j] = fmaf(x4.y, w1, acc[j]);
            acc[j] = fmaf(x4.z, w2, acc[j]);
            acc[j] = fmaf(x4.w, w3, acc[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (t0 + j >= T) continue;
        if (KQ == 1)
          a.part[((size_t)s * T + t0 + j) * E + e] = acc[j];
        else
          red[((size_t)kq * T + t0 + j) * E + e] = acc[j];
      }
    }
    if (KQ > 1) {
      __syncthreads();
      for (int i = tid; i < T * E; i += kSmallThreads) {
        float v = red[i];
        for (int kq = 1; kq < KQ; ++kq) v += red[(size_t)kq * T * E + i];
        a.part[(size_t)s * T * E + i] = v;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) am_last = atomicAdd(a.scan.done_counter, 1u) == (unsigned)a.S - 1u;
  __syncthreads();
  if (!am_last) return;
  __threadfence();
  // ---- the last block: logits, routing, scan, positions, copies ----
  float* lg = reinterpret_cast<float*>(sm_raw);                       // [T][E]
  float* Pw = lg + kSmallT * kMaxE;                                   // [16 warps][E]
  int* cnt = reinterpret_cast<int*>(Pw + (kSmallThreads / 32) * kMaxE);   // [E]
  int* row_s = cnt + kMaxE;                                           // [T*k]
  ScanSmem<kSmallThreads>& scan_sm =
      *reinterpret_cast<ScanSmem<kSmallThreads>*>(row_s + kSmallT * kMaxK);
  uint8_t* stage = reinterpret_cast<uint8_t*>(&scan_sm + 1);
  stage = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(stage) + 127) & ~uintptr_t(127));
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + kSmallStage);
  const uint32_t row_bytes = (uint32_t)a.nvec * 16u;
  // When all T token rows fit the stage, they are loaded now, while the
  // logits, routing and scan run, and later stored straight to their rows.
  const bool stage_x = a.xp != nullptr && (size_t)T * row_bytes <= kSmallStage;
  uint64_t* xbar = bars + kBulkIssuers;
  if (stage_x && tid == 0) {
    mbar_init(smem_u32(xbar), 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(smem_u32(xbar), (uint32_t)T * row_bytes);
    for (int t = 0; t < T; ++t)
      bulk_load(smem_u32(stage) + t * row_bytes, static_cast<const char*>(a.x) + (size_t)t * row_bytes,
                row_bytes, smem_u32(xbar));
  }
  const int TE = T * E;
  if (TE <= kSmallThreads || (TE & 3)) {
    for (int i = tid; i < TE; i += kSmallThreads) {
      const int t = i / E, e = i - t * E;
      const float* pp = a.part + (size_t)t * E + e;
      const size_t ss = (size_t)TE;   // slice stride
      float l = 0.f;
      // up to 32 loads in flight, added in slice order
      for (int s0 = 0; s0 < a.S; s0 += 32) {
        float v[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = s0 + u < a.S ? __ldcg(pp + (size_t)(s0 + u) * ss) : 0.f;
#pragma unroll
        for (int u = 0; u < 32; ++u)
          if (s0 + u < a.S) l += v[u];
      }
      lg[t * E + e] = l + (a.logit_offset ? a.logit_offset[e] : 0.f);
    }
  } else {
    // more outputs than threads: four consecutive outputs per thread
    // (16-byte loads), 16 slices in flight, the same additions in slice order
    const float4* p4 = reinterpret_cast<const float4*>(a.part);
    const int n4 = TE / 4;
    for (int i4 = tid; i4 < n4; i4 += kSmallThreads) {
      float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s0 = 0; s0 < a.S; s0 += 16) {
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          v[u] = s0 + u < a.S ? __ldcg(p4 + (size_t)(s0 + u) * n4 + i4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          if (s0 + u < a.S) {
            l.x += v[u].x;
            l.y += v[u].y;
            l.z += v[u].z;
            l.w += v[u].w;
          }
        }
      }
      const int i = 4 * i4;
      const float* off = a.logit_offset;
      lg[i] = l.x + (off ? off[i % E] : 0.f);
      lg[i + 1] = l.y + (off ? off[(i + 1) % E] : 0.f);
      lg[i + 2] = l.z + (off ? off[(i + 2) % E] : 0.f);
      lg[i + 3] = l.w + (off ? off[(i + 3) % E] : 0.f);
    }
  }
  for (int e = tid; e < E; e += kSmallThreads) cnt[e] = 0;
  __syncthreads();
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;
  for (int t = warp; t < T; t += kSmallThreads / 32) {
    float sv[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      sv[i] = e < E ? lg[t * E + e] : -INFINITY;
    }
    route_one_token<NPL>(sv, E, a.k, a.gate, a.sel_bias, a.topk_idx + (size_t)t * a.k,
                         a.topk_w + (size_t)t * a.k, cnt, psum);
  }
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < E) Pw[warp * E + lane + 32 * i] = psum[i];
  __syncthreads();
  // capacity scan of the single routing block: its histogram is the total
  {
    const ScanArgs& sa = a.scan;
    int* seg_s = scan_sm.routed_s;      // first row of each expert's segment
    int* off_s = reinterpret_cast<int*>(scan_sm.psum_s);   // first slot of each expert
    const int e = tid;
    int routed = 0, kept = 0, mt = 0;
    float P = 0.f, fr = 0.f;
    if (e < E) {
      float pe = 0.f;
      for (int w = 0; w < kSmallThreads / 32; ++w) pe += Pw[w * E + e];
      routed = cnt[e];
      kept = routed < a.capacity ? routed : a.capacity;
      mt = (kept + sa.bm - 1) / sa.bm;
      P = pe / (float)T;
      fr = (float)routed / (float)(T * a.k);
    }
    int4 tot;
    const int4 ex = block_exscan4<kSmallThreads>(
        make_int4(kept, mt, mt * sa.nt_up, mt * sa.nt_dn), scan_sm.scratch, &tot);
    if (e < E) {
      seg_s[e] = ex.y * sa.bm;
      off_s[e] = ex.x;
      cnt[e] = 0;
      sa.m.kept[e] = kept;
      sa.m.offsets[e] = ex.x;
      sa.m.seg_start[e] = ex.y * sa.bm;
      sa.m.mtiles[e] = mt;
      sa.m.tp_up[e] = ex.z;
      sa.m.tp_dn[e] = ex.w;
      sa.expert_counts[e] = kept;
      if (sa.routed_counts) sa.routed_counts[e] = routed;
      if (sa.offsets_out) sa.offsets_out[e] = ex.x;
      if (sa.f_out) sa.f_out[e] = fr;
      if (sa.P_out) sa.P_out[e] = P;
    }
    if (tid == 0) {
      const int sh_up = sa.has_shared ? sa.mt_sh * sa.nt_up_sh : 0;
      const int sh_dn = sa.has_shared ? sa.mt_sh * sa.nt_dn_sh : 0;
      sa.m.offsets[E] = tot.x;
      sa.m.seg_start[E] = tot.y * sa.bm;
      sa.m.mtiles[E] = sa.has_shared ? sa.mt_sh : 0;
      sa.m.tp_up[E] = tot.z;
      sa.m.tp_up[E + 1] = tot.z + sh_up;
      sa.m.tp_dn[E] = tot.w;
      sa.m.tp_dn[E + 1] = tot.w + sh_dn;
      if (sa.offsets_out) sa.offsets_out[E] = tot.x;
    }
    // L = alpha * E * sum_i f_i P_i in double: a fixed butterfly inside each
    // warp, then the warp sums in warp order
    double l = e < E ? (double)fr * (double)P : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) scan_sm.red[warp] = l;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < kSmallThreads / 32; ++w) t += scan_sm.red[w];
      sa.aux_loss[0] = (float)((double)sa.alpha * (double)E * t);
    }
  }
  __syncthreads();
  if (warp == 0) {
    // ranks in key order (one routing block: no base), then rows
    const int nk = T * a.k;
    for (int c = 0; c < nk; c += 32) {
      const int q = c + lane;
      bool valid = q < nk;
      int e = valid ? a.topk_idx[q] : -1 - lane;
      if (valid && !in_bounds(e >= 0 && e < E, a.status)) {
        valid = false;
        e = -1 - lane;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int before = __popc(peers & ((1u << lane) - 1u));
      const int prior = valid ? cnt[e] : 0;
      __syncwarp();
      if (valid) {
        const int pos = prior + before;
        bool keep = pos < a.capacity;
        int row = keep ? scan_sm.routed_s[e] + pos : -1;
        if (keep && !in_bounds(row >= 0 && row < a.R_cap, a.status)) {
          keep = false;
          row = -1;
        }
        a.key_row[q] = row;
        if (a.slot_pos)
          a.slot_pos[q] = keep ? reinterpret_cast<const int*>(scan_sm.psum_s)[e] + pos : -1;
        if (keep) a.row_token[row] = q / a.k;
        row_s[q] = row;
        if (before == 0) cnt[e] = prior + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (tid == 0) *a.scan.done_counter = 0;
  if (stage_x) {
    // every kept key's token row from the staged copy of x, four issuers
    if (warp < kBulkIssuers && lane == 0) {
      if (!mbar_wait_bounded(smem_u32(xbar), 0, 2000000000ull, nullptr)) {
        atomicOr(a.status, STATUS_TIMEOUT_ROUTE);
      } else {
        char* xp = static_cast<char*>(a.xp);
        for (int q = warp; q < T * a.k; q += kBulkIssuers) {
          const int row = row_s[q];
          if (row >= 0)
            bulk_store(xp + (size_t)row * row_bytes, smem_u32(stage) + (q / a.k) * row_bytes,
                       row_bytes);
        }
        bulk_commit();
        bulk_wait_all();
      }
    }
  } else if (a.xp) {
    // the kept rows into expert order: bulk copies through shared memory
    const char* xs = static_cast<const char*>(a.x);
    char* xp = static_cast<char*>(a.xp);
    bulk_copy_rows(
        T * a.k, row_bytes,
        [&](int q) { return static_cast<const void*>(xs + (size_t)(q / a.k) * row_bytes); },
        [&](int q) {
          const int row = row_s[q];
          return row >= 0 ? static_cast<void*>(xp + (size_t)row * row_bytes) : nullptr;
        },
        stage, kSmallStage, bars, a.status, STATUS_TIMEOUT_ROUTE, 2000000000ull);
  }
}

size_t route_small_smem(int E) {
  // x and weight slices, then the part sums of the split dot products (at
  // most 4 parts x 4 token groups' worth of outputs per thread: 4 x 512 x 4)
  const size_t p1 = sizeof(float) * ((size_t)kSmallT * kSmallKs + (size_t)kSmallKs * (E + 1) +
                                     (size_t)4 * kSmallThreads * 4);
  const size_t p2 = sizeof(float) * ((size_t)kSmallT * kMaxE + (kSmallThreads / 32) * kMaxE) +
                    sizeof(int) * ((size_t)kMaxE + kSmallT * kMaxK) +
                    sizeof(ScanSmem<kSmallThreads>) + 128 + kSmallStage + 8 * (kBulkIssuers + 1);
  return p1 > p2 ? p1 : p2;
}

int route_small_splits(int d) { return (d + kSmallKs - 1) / kSmallKs; }

template <typename TIn, int NPL>
static cudaError_t launch_small_t(const SmallArgs& a, size_t smem, cudaStream_t st) {
  static std::atomic<uint64_t> attr_done{0};
  auto kern = route_small_kernel<TIn, NPL>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  return launch_pdl(kern, dim3(a.S), dim3(kSmallThreads), smem, st, a);
}

template <typename TIn>
static cudaError_t launch_small_npl(const SmallArgs& a, size_t smem, cudaStream_t st) {
  const int npl = (a.E + 31) / 32;
  if (npl <= 1) return launch_small_t<TIn, 1>(a, smem, st);
  if (npl <= 2) return launch_small_t<TIn, 2>(a, smem, st);
  if (npl <= 4) return launch_small_t<TIn, 4>(a, smem, st);
  return launch_small_t<TIn, 8>(a, smem, st);
}

cudaError_t launch_route_small(const Plan& p, const void* x, const void* W_r,
                               const float* logit_offset, const float* sel_bias,
                               int32_t* topk_idx, float* topk_w, int32_t* slot_pos, bool copy_rows,
                               void* ws, const ScanOutputs& so, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  SmallArgs a;
  a.x = x;
  a.W_r = W_r;
  a.logit_offset = logit_offset;
  a.sel_bias = sel_bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.slot_pos = slot_pos;
  a.part = reinterpret_cast<float*>(w + p.ws.score_parts);
  a.key_row = reinterpret_cast<int*>(w + p.ws.key_row);
  a.row_token = reinterpret_cast<int*>(w + p.ws.row_token);
  a.xp = copy_rows ? static_cast<void*>(w + p.ws.xp) : nullptr;
  a.T = p.cfg.T;
  a.d = p.cfg.d;
  a.E = p.cfg.E;
  a.k = p.cfg.k;
  a.gate = p.cfg.gate;
  a.capacity = p.capacity;
  a.S = route_small_splits(p.cfg.d);
  a.elem = p.elem;
  a.nvec = p.cfg.d * p.elem / 16;
  a.R_cap = p.R_cap;
  a.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  a.scan = scan_args(p, ws, so);
  const size_t smem = route_small_smem(p.cfg.E);
  if (p.cfg.dtype == MOE_BF16) return launch_small_npl<__nv_bfloat16>(a, smem, st);
  return launch_small_npl<float>(a, smem, st);
}

// ---------------------------------------------------------------- fused router
// Fused path (E <= 256): one block computes the float32 logits of BM = 16 TM
// tokens for all experts over the full model width, keeps them in shared
// memory, routes its tokens (one warp per token) and publishes its histogram;
// the last block runs the capacity scan.  Thread (ty, tx) of 16 x 16 owns
// tokens ty*TM .. +TM-1 and experts tx*TN .. +TN-1 (E padded to 16 TN).
struct FusedArgs {
  const void* x;
  const void* W_r;
  const float* logit_offset;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  float* scores_out;         // logits-only mode: write [T][E] and stop
  int T, d, E, k, gate;
  ScanArgs scan;
};

constexpr int kFuBK = 32, kFuStages = 3;

template <typename TIn, int TM, int TN>
struct FusedCfg {
  static constexpr int BM = 16 * TM, EP = 16 * TN;
  static constexpr int EPC = 16 / sizeof(TIn), LD = kFuBK + EPC, CPR = kFuBK / EPC;
  static constexpr size_t A_RAW = (size_t)BM * LD * sizeof(TIn);
  static constexpr size_t B_RAW = (size_t)EP * LD * sizeof(TIn);
  static constexpr size_t AF = (size_t)kFuBK * (BM + 4) * sizeof(float);
  static constexpr size_t BF = (size_t)kFuBK * (EP + 4) * sizeof(float);
  static constexpr size_t PIPE = AF + BF + kFuStages * (A_RAW + B_RAW);
  static constexpr size_t ROUTE = (size_t)BM * (EP + 1) * sizeof(float) +
                                  sizeof(float) * 8 * kMaxE + sizeof(int) * kMaxE;
  static constexpr size_t SCAN = sizeof(ScanSmem<kThreads>);
  static constexpr size_t SMEM = PIPE > ROUTE ? (PIPE > SCAN ? PIPE : SCAN)
                                              : (ROUTE > SCAN ? ROUTE : SCAN);
};

template <typename TIn, int TM, int TN>
__global__ void __launch_bounds__(kThreads) router_fused_kernel(const FusedArgs a) {
  using C = FusedCfg<TIn, TM, TN>;
  constexpr int BM = C::BM, EP = C::EP, LD = C::LD, CPR = C::CPR, EPC = C::EPC;
  constexpr int BK = kFuBK;
  extern __shared__ __align__(16) uint8_t fu_smem[];
  float* Af = reinterpret_cast<float*>(fu_smem);                    // [BK][BM+4]
  float* Bf = Af + BK * (BM + 4);                                   // [BK][EP+4]
  TIn* As = reinterpret_cast<TIn*>(Bf + BK * (EP + 4));             // [stages][BM][LD]
  TIn* Bs = As + kFuStages * BM * LD;                               // [stages][EP][LD]
  __shared__ int am_last;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * BM;
  const TIn* X = static_cast<const TIn*>(a.x);
  const TIn* Wr = static_cast<const TIn*>(a.W_r);
  pdl_wait();
  pdl_trigger();

  auto issue = [&](int stage, int k0) {
    TIn* as = As + stage * BM * LD;
    TIn* bs = Bs + stage * EP * LD;
    for (int c = tid; c < BM * CPR; c += kThreads) {
      const int r = c % BM, kc = (c / BM) * EPC;
      const int gm = m0 + r, gk = k0 + kc;
      const bool ok = gm < a.T && gk < a.d;
      cp_async16(as + r * LD + kc, X + (ok ? (size_t)gm * a.d + gk : 0), ok);
    }
    for (int c = tid; c < EP * CPR; c += kThreads) {
      const int r = c % EP, kc = (c / EP) * EPC;
      const int gk = k0 + kc;
      const bool ok = r < a.E && gk < a.d;
      cp_async16(bs + r * LD + kc, Wr + (ok ? (size_t)r * a.d + gk : 0), ok);
    }
  };
  auto convert = [&](int stage) {
    const TIn* as = As + stage * BM * LD;
    const TIn* bs = Bs + stage * EP * LD;
    for (int c = tid; c < BM * CPR; c += kThreads) {
      const int r = c % BM, kc = (c / BM) * EPC;
      float v[8];
      to_float8(*reinterpret_cast<const uint4*>(as + r * LD + kc), as, v);
#pragma unroll
      for (int i = 0; i < EPC; ++i) Af[(kc + i) * (BM + 4) + r] = v[i];
    }
    for (int c = tid; c < EP * CPR; c += kThreads) {
      const int r = c % EP, kc = (c / EP) * EPC;
      float v[8];
      to_float8(*reinterpret_cast<const uint4*>(bs + r * LD + kc), bs, v);
#pragma unroll
      for (int i = 0; i < EPC; ++i) Bf[(kc + i) * (EP + 4) + r] = v[i];
    }
  };

  float acc[TM][TN], part[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = part[i][j] = 0.f;
  const int nk = (a.d + BK - 1) / BK;
#pragma unroll
  for (int s = 0; s < kFuStages - 1; ++s) {
    if (s < nk) issue(s, s * BK);
    cp_async_commit();
  }
  for (int it = 0; it < nk; ++it) {
    cp_async_wait<kFuStages - 2>();
    __syncthreads();
    convert(it % kFuStages);
    {
      const int nxt = it + kFuStages - 1;
      if (nxt < nk) issue(nxt % kFuStages, nxt * BK);
      cp_async_commit();
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float av[TM], bv[TN];
      if (TM == 2) {
        const float2 a2 = *reinterpret_cast<const float2*>(Af + kk * (BM + 4) + ty * TM);
        av[0] = a2.x;
        av[TM - 1] = a2.y;
      } else {
        av[0] = Af[kk * (BM + 4) + ty];
      }
      if (TN >= 4) {
#pragma unroll
        for (int j = 0; j < TN; j += 4) {
          const float4 b4 = *reinterpret_cast<const float4*>(Bf + kk * (EP + 4) + tx * TN + j);
          bv[j] = b4.x;
          bv[j + 1] = b4.y;
          bv[j + 2] = b4.z;
          bv[j + 3] = b4.w;
        }
      } else {
        const float2 b2 = *reinterpret_cast<const float2*>(Bf + kk * (EP + 4) + tx * TN);
        bv[0] = b2.x;
        bv[TN - 1] = b2.y;
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
    }
    if ((it & 3) == 3 || it + 1 == nk) {   // fold every 128 k into the running sum
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          acc[i][j] += part[i][j];
          part[i][j] = 0.f;
        }
    }
  }
  cp_async_wait<0>();
  __syncthreads();                        // pipeline buffers become the routing area

  float* S = reinterpret_cast<float*>(fu_smem);                      // [BM][EP+1]
  float (*Pw)[kMaxE] = reinterpret_cast<float (*)[kMaxE]>(S + BM * (EP + 1));
  int* cnt = reinterpret_cast<int*>(Pw + 8);
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int m = ty * TM + i;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int e = tx * TN + j;
      if (e < a.E) {
        const float s = acc[i][j] + (a.logit_offset ? a.logit_offset[e] : 0.f);
        S[m * (EP + 1) + e] = s;
        if (a.scores_out && m0 + m < a.T) a.scores_out[(size_t)(m0 + m) * a.E + e] = s;
      }
    }
  }
  if (a.scores_out) return;
  for (int e = tid; e < a.E; e += kThreads) cnt[e] = 0;
  __syncthreads();

  constexpr int NPL = EP / 32 > 0 ? EP / 32 : 1;
  const int warp = tid >> 5, lane = tid & 31;
  float psum[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) psum[i] = 0.f;
  for (int tl = warp; tl < BM; tl += kThreads / 32) {
    const int t = m0 + tl;
    if (t >= a.T) break;
    float sv[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      sv[i] = e < a.E ? S[tl * (EP + 1) + e] : -INFINITY;
    }
    route_one_token<NPL>(sv, a.E, a.k, a.gate, a.sel_bias, a.topk_idx + (size_t)t * a.k,
                         a.topk_w + (size_t)t * a.k, cnt, psum);
  }
  __syncthreads();
  // Pw/cnt live in the routing area; the scan area overlaps it only after
  // publish_and_scan has read them (it synchronises before the scan).
  publish_and_scan<kThreads, NPL>(a.scan, psum, Pw, cnt,
                                  *reinterpret_cast<ScanSmem<kThreads>*>(fu_smem), &am_last);
}

template <typename TIn, int TN>
static cudaError_t launch_scores_t(const Plan& p, const ScoresArgs& a, cudaStream_t st) {
  constexpr int EPC = 16 / sizeof(TIn), LD = kScBK + EPC;
  const int smem = kScBK * (kScBM + 4 + 16 * TN + 4) * (int)sizeof(float) +
                   kScStages * (kScBM + 16 * TN) * LD * (int)sizeof(TIn);
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(attr_done.load(std::memory_order_acquire) & (1ull << (dev & 63)))) {
    e = cudaFuncSetAttribute(router_scores_kernel<TIn, TN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(1ull << (dev & 63), std::memory_order_release);
  }
  const dim3 grid(p.sc_mblocks, p.sc_nblocks, p.sc_splits);
  return launch_pdl(router_scores_kernel<TIn, TN>, grid, dim3(kThreads), (size_t)smem, st, a);
}

// Router logits into `scores` ([T][E], float32, offset included).
static cudaError_t launch_logits(const Plan& p, const void* x, const void* W_r,
                                 const float* logit_offset, float* scores, void* ws,
                                 cudaStream_t st);


template <typename TIn, int TM, int TN>
static cudaError_t launch_fused_t(const Plan& p, const FusedArgs& a, cudaStream_t st) {
  using C = FusedCfg<TIn, TM, TN>;
  static std::atomic<uint64_t> attr_done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(attr_done.load(std::memory_order_acquire) & (1ull << (dev & 63)))) {
    e = cudaFuncSetAttribute(router_fused_kernel<TIn, TM, TN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(1ull << (dev & 63), std::memory_order_release);
  }
  const int blocks = (p.cfg.T + C::BM - 1) / C::BM;
  return launch_pdl(router_fused_kernel<TIn, TM, TN>, dim3(blocks), dim3(kThreads), C::SMEM, st,
                    a);
}

template <typename TIn, int TM>
static cudaError_t launch_fused_tm(const Plan& p, const FusedArgs& a, cudaStream_t st) {
  switch (p.fu_tn) {
    case 2: return launch_fused_t<TIn, TM, 2>(p, a, st);
    case 4: return launch_fused_t<TIn, TM, 4>(p, a, st);
    case 8: return launch_fused_t<TIn, TM, 8>(p, a, st);
    case 16: return launch_fused_t<TIn, TM, 16>(p, a, st);
  }
  return cudaErrorInvalidValue;
}

static cudaError_t launch_fused(const Plan& p, const FusedArgs& a, cudaStream_t st) {
  if (p.cfg.dtype == MOE_BF16)
    return p.fu_tm == 2 ? launch_fused_tm<__nv_bfloat16, 2>(p, a, st)
                        : launch_fused_tm<__nv_bfloat16, 1>(p, a, st);
  return p.fu_tm == 2 ? launch_fused_tm<float, 2>(p, a, st) : launch_fused_tm<float, 1>(p, a, st);
}

cudaError_t launch_router(const Plan& p, const void* x, const void* W_r, const float* logit_offset,
                          const float* sel_bias, int32_t* topk_idx, float* topk_w, void* ws,
                          const ScanOutputs& so, cudaStream_t st, cudaEvent_t mid_event) {
  char* w = static_cast<char*>(ws);
  cudaError_t e;
  if (p.router_fused) {
    FusedArgs f;
    f.x = x;
    f.W_r = W_r;
    f.logit_offset = logit_offset;
    f.sel_bias = sel_bias;
    f.topk_idx = topk_idx;
    f.topk_w = topk_w;
    f.scores_out = nullptr;
    f.T = p.cfg.T;
    f.d = p.cfg.d;
    f.E = p.cfg.E;
    f.k = p.cfg.k;
    f.gate = p.cfg.gate;
    f.scan = scan_args(p, ws, so);
    e = launch_fused(p, f, st);
    if (e != cudaSuccess) return e;
    if (mid_event && (e = cudaEventRecord(mid_event, st)) != cudaSuccess) return e;
    return cudaSuccess;
  }
  float* scores = reinterpret_cast<float*>(w + p.ws.scores);
  e = launch_logits(p, x, W_r, logit_offset, scores, ws, st);
  if (e != cudaSuccess) return e;
  if (mid_event && (e = cudaEventRecord(mid_event, st)) != cudaSuccess) return e;
  TopkArgs t;
  t.scores = scores;
  t.sel_bias = sel_bias;
  t.topk_idx = topk_idx;
  t.topk_w = topk_w;
  t.T = p.cfg.T;
  t.E = p.cfg.E;
  t.k = p.cfg.k;
  t.BT = p.BT;
  t.gate = p.cfg.gate;
  t.scan = scan_args(p, ws, so);
  const dim3 g(p.nblk), b(kTopkThreads);
  const int npl = (p.cfg.E + 31) / 32;
  if (npl <= 1) return launch_pdl(router_topk_kernel<1>, g, b, 0, st, t);
  if (npl <= 2) return launch_pdl(router_topk_kernel<2>, g, b, 0, st, t);
  if (npl <= 4) return launch_pdl(router_topk_kernel<4>, g, b, 0, st, t);
  if (npl <= 8) return launch_pdl(router_topk_kernel<8>, g, b, 0, st, t);
  return launch_pdl(router_topk_kernel<16>, g, b, 0, st, t);
}

static cudaError_t launch_logits(const Plan& p, const void* x, const void* W_r,
                                 const float* logit_offset, float* scores, void* ws,
                                 cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  if (p.router_tc)
    return launch_router_tc(p, x, W_r, logit_offset, scores,
                            reinterpret_cast<uint32_t*>(w + p.ws.status), st);
  ScoresArgs a;
  a.x = x;
  a.W_r = W_r;
  a.logit_offset = logit_offset;
  a.part = reinterpret_cast<float*>(w + p.ws.score_parts);
  a.scores = scores;
  a.tile_counter = reinterpret_cast<unsigned int*>(w + p.ws.status + kTileCounterOffset);
  a.T = p.cfg.T;
  a.d = p.cfg.d;
  a.E = p.cfg.E;
  a.k_split = p.sc_ksplit;
  a.S = p.sc_splits;
  if (p.cfg.dtype == MOE_BF16)
    return p.sc_tn == 4 ? launch_scores_t<__nv_bfloat16, 4>(p, a, st)
                        : launch_scores_t<__nv_bfloat16, 2>(p, a, st);
  return p.sc_tn == 4 ? launch_scores_t<float, 4>(p, a, st) : launch_scores_t<float, 2>(p, a, st);
}

cudaError_t launch_router_scores(const Plan& p, const void* x, const void* W_r,
                                 const float* logit_offset, float* out, void* ws,
                                 cudaStream_t st) {
  if (tuning(MOE_TUNE_ROUTER) == MOE_ROUTER_FUSED && p.fu_tn > 0) {
    // the fused kernel's own logits, written out before its routing step
    FusedArgs f;
    std::memset(&f, 0, sizeof(f));
    f.x = x;
    f.W_r = W_r;
    f.logit_offset = logit_offset;
    f.scores_out = out;
    f.T = p.cfg.T;
    f.d = p.cfg.d;
    f.E = p.cfg.E;
    f.k = p.cfg.k;
    f.gate = p.cfg.gate;
    return launch_fused(p, f, st);
  }
  return launch_logits(p, x, W_r, logit_offset, out, ws, st);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Router logits without a caller workspace.
//
// For callers that cannot hand the library a workspace: a host framework that
// owns all device memory and gives none out per call, or code that must not
// enter the CUDA allocator on its latency path.  The router GEMM's scratch
// (split-K partial logits and the tile counters of its reduction) lives in the
// file-scope array below instead.  Each device on which this file's module is
// loaded (under CUDA's lazy module loading: by the first router call or the
// first no-workspace call on that device) holds kNoAllocScratchBytes of device
// memory for it until the process exits.
//
// Host code must not pass `g_noalloc_scratch` itself to a kernel: in host code
// that name is a host-side stand-in, not a device address.  The device address
// is looked up with cudaGetSymbolAddress once per CUDA context (the first call
// made with that context current) and cached under the context's unique id,
// so a device reset or another context gets its own lookup.
namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;       // 8 MiB
constexpr size_t kNoAllocCounterBytes = moe::kWsHeaderBytes;   // tile counters, zeroed per call

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_noalloc_mu;
constexpr int kNoAllocCacheSlots = 64;
unsigned long long g_noalloc_ctx[kNoAllocCacheSlots] = {};   // context ids (ids start at 1)
void* g_noalloc_addr[kNoAllocCacheSlots] = {};
int g_noalloc_next = 0;

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Device address of the scratch array in the current context; looked up once
// per context.  Also rejects devices that are not sm_103.
int noalloc_setup(void** addr) {
  static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_current || !get_id) return MOE_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_DEVICE;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return MOE_ERR_CUDA;
  if (ctx == nullptr) {   // no context yet: make the device's primary context current
    if (cudaSetDevice(dev) != cudaSuccess || get_current(&ctx) != CUDA_SUCCESS || !ctx)
      return MOE_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS || id == 0) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  for (int i = 0; i < kNoAllocCacheSlots; ++i) {
    if (g_noalloc_ctx[i] == id) {
      *addr = g_noalloc_addr[i];
      return MOE_OK;
    }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return MOE_ERR_CUDA;
  const int slot = g_noalloc_next;                 // oldest entry replaced when full
  g_noalloc_next = (g_noalloc_next + 1) % kNoAllocCacheSlots;
  g_noalloc_ctx[slot] = id;
  g_noalloc_addr[slot] = p;
  *addr = p;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_router_scores_noalloc(const moe_config* cfg, const void* x, const void* W_r,
                                         const float* logit_offset, float* scores,
                                         void* stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_ARG;
  Plan p;
  int rc = make_plan(cfg, WsKind::Route, &p);
  if (rc != MOE_OK) return rc;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !W_r || !scores) return MOE_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(W_r) & 15u) ||
      (reinterpret_cast<uintptr_t>(scores) & 3u))
    return MOE_ERR_ARG;
  // the same split of the reduction as moe_router_scores, which needs
  // S*T*E floats of partials next to the counters
  const size_t parts = p.sc_splits > 1 ? sizeof(float) * (size_t)p.sc_splits * cfg->T * cfg->E : 0;
  if (kNoAllocCounterBytes + parts > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* base = nullptr;
  rc = noalloc_setup(&base);
  if (rc != MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: start the counters at zero
  if (cudaMemsetAsync(base, 0, kNoAllocCounterBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
  ScoresArgs a;
  a.x = x;
  a.W_r = W_r;
  a.logit_offset = logit_offset;
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kNoAllocCounterBytes);
  a.scores = scores;
  a.tile_counter = static_cast<unsigned int*>(base);
  a.T = cfg->T;
  a.d = cfg->d;
  a.E = cfg->E;
  a.k_split = p.sc_ksplit;
  a.S = p.sc_splits;
  cudaError_t e;
  if (cfg->dtype == MOE_BF16)
    e = p.sc_tn == 4 ? launch_scores_t<__nv_bfloat16, 4>(p, a, st)
                     : launch_scores_t<__nv_bfloat16, 2>(p, a, st);
  else
    e = p.sc_tn == 4 ? launch_scores_t<float, 4>(p, a, st) : launch_scores_t<float, 2>(p, a, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
