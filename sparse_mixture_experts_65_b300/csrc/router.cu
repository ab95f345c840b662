// router.cu -- stage 1 and 2 of the layer in one kernel: router scores
// s = W_r x (+ o) with float32 accumulation, warp-level top-k with the
// selection bias, gate normalisation, the full router distribution for P_i,
// and per-block expert histograms.
//
// "Mixture of Experts" (llm-tutorial ch. 11) § Top-k routing: softmax over the
// k chosen logits; § Top-1 vs top-2: the full-softmax probability of a top-1
// choice; § Why MoE is hard: the router runs in float32 even when the model
// is bf16.  "Mixture of experts" (inside-the-model guide) § The computation
// and § Auxiliary-loss-free balancing: renormalised sigmoid gates and a bias
// that steers only the choice.
//
// One block owns BT tokens and all experts.  Phase 1 is a float32 FMA GEMM
// (bf16 x bf16 products are exact in float32) with the reduction split into
// KC-wide chunks summed separately, which keeps the rounding error of a
// d = 7168 dot product near 1e-7 relative.  Phase 2 gives each warp whole
// tokens: lanes hold E/32 scores, k rounds of warp arg-max pick the experts
// (larger score first, equal scores to the lower index).
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

struct RouterArgs {
  const void* x;
  const void* W_r;
  const float* logit_offset;
  const float* sel_bias;
  int32_t* topk_idx;
  float* topk_w;
  int* blk_cnt;
  float* blk_prob;
  int T, d, E, E_pad, k, BT, KC, gate;
};

template <typename TIn>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(const RouterArgs a) {
  extern __shared__ __align__(16) float sm[];
  constexpr int RT = kRouterRT;
  const int E_pad = a.E_pad, BT = a.BT, KC = a.KC;
  const int EC = E_pad < 256 ? E_pad : 256;   // experts per pass of the block
  const int EPT = (E_pad + 255) / 256;        // expert passes per thread (1 or 2)
  const int XS = BT + 4;                      // row stride of the x tile
  const int WS = E_pad + 1;                   // row stride of the W tile / scores
  float* xs = sm;                             // [KC][XS]
  float* wt = xs + KC * XS;                   // [KC][WS]
  float* S = wt + KC * WS;                    // [BT][WS]
  float* Pw = S + BT * WS;                    // [8][E_pad]
  int* cnt = reinterpret_cast<int*>(Pw + 8 * E_pad);  // [E_pad]

  const int tid = threadIdx.x;
  const int el = tid % EC, grp = tid / EC;
  const int t0 = blockIdx.x * BT;
  const TIn* x = static_cast<const TIn*>(a.x);
  const TIn* W = static_cast<const TIn*>(a.W_r);

  for (int e = tid; e < E_pad; e += kThreads) cnt[e] = 0;

  // ---- phase 1: scores ---------------------------------------------------
  float acc[2][RT];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int r = 0; r < RT; ++r) acc[c][r] = 0.f;

  for (int c0 = 0; c0 < a.d; c0 += KC) {
    for (int i = tid; i < BT * KC; i += kThreads) {
      const int tok = i / KC, kc = i - tok * KC;
      const int t = t0 + tok, c = c0 + kc;
      xs[kc * XS + tok] = (t < a.T && c < a.d) ? to_float(x[(size_t)t * a.d + c]) : 0.f;
    }
    for (int i = tid; i < E_pad * KC; i += kThreads) {
      const int e = i / KC, kc = i - e * KC;
      const int c = c0 + kc;
      wt[kc * WS + e] = (e < a.E && c < a.d) ? to_float(W[(size_t)e * a.d + c]) : 0.f;
    }
    __syncthreads();
    float part[2][RT];
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int r = 0; r < RT; ++r) part[c][r] = 0.f;
    const int kcn = min(KC, a.d - c0);
    for (int kc = 0; kc < kcn; ++kc) {
      const float4* xr = reinterpret_cast<const float4*>(xs + kc * XS + grp * RT);
      const float4 xa = xr[0], xb = xr[1];
      const float xv[RT] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c < EPT) {
          const float w = wt[kc * WS + el + c * 256];
#pragma unroll
          for (int r = 0; r < RT; ++r) part[c][r] = fmaf(w, xv[r], part[c][r]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int r = 0; r < RT; ++r) acc[c][r] += part[c][r];
    __syncthreads();
  }
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int e = el + c * 256;
    if (c < EPT && e < a.E) {
      const float off = a.logit_offset ? a.logit_offset[e] : 0.f;
#pragma unroll
      for (int r = 0; r < RT; ++r) S[(grp * RT + r) * WS + e] = acc[c][r] + off;
    }
  }
  __syncthreads();

  // ---- phase 2: top-k, gates, router distribution --------------------------
  const int warp = tid >> 5, lane = tid & 31;
  const int NPL = E_pad >> 5;   // scores per lane, <= 16
  float psum[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) psum[i] = 0.f;
  const bool sigm = a.gate == MOE_GATE_SIGMOID_RENORM;

  for (int tl = warp; tl < BT; tl += kThreads / 32) {
    const int t = t0 + tl;
    if (t >= a.T) break;
    const float* St = S + tl * WS;
    float sv[16], sel[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      sv[i] = -INFINITY;
      sel[i] = -INFINITY;
      const int e = lane + 32 * i;
      if (i < NPL && e < a.E) {
        const float s = St[e];
        sv[i] = s;
        float v = sigm ? sigmoidf_(s) : s;
        if (a.sel_bias) v += a.sel_bias[e];
        sel[i] = (v != v) ? -INFINITY : v;   // NaN never outranks a number
      }
    }
    uint32_t taken = 0;
    int my_idx = 0;
    for (int r = 0; r < a.k; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = lane + 32 * i;
        if (i < NPL && e < a.E && !((taken >> i) & 1u)) {
          if (sel[i] > bv || (sel[i] == bv && e < bi)) {
            bv = sel[i];
            bi = e;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (bi < a.E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == r) my_idx = bi < a.E ? bi : 0;
    }
    const bool mine = lane < a.k;
    const float s_me = mine ? St[my_idx] : -INFINITY;

    // full distribution over all experts
    float m_all = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i) m_all = fmaxf(m_all, sv[i]);
    m_all = warp_max(m_all);
    float z_all = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < NPL && lane + 32 * i < a.E) z_all += sigm ? sigmoidf_(sv[i]) : expf(sv[i] - m_all);
    }
    z_all = warp_sum(z_all);

    float g;
    if (a.gate == MOE_GATE_SOFTMAX_TOPK) {
      const float m_k = warp_max(s_me);
      const float ek = mine ? expf(s_me - m_k) : 0.f;
      g = ek / warp_sum(ek);
    } else if (sigm) {
      const float ak = mine ? sigmoidf_(s_me) : 0.f;
      g = ak / warp_sum(ak);
    } else {
      g = expf(s_me - m_all) / z_all;
    }
    if (mine) {
      a.topk_idx[(size_t)t * a.k + lane] = my_idx;
      a.topk_w[(size_t)t * a.k + lane] = g;
      atomicAdd(&cnt[my_idx], 1);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < NPL && lane + 32 * i < a.E)
        psum[i] += sigm ? sigmoidf_(sv[i]) / z_all : expf(sv[i] - m_all) / z_all;
    }
  }

  // ---- block statistics, fixed summation order ----------------------------
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (i < NPL) Pw[warp * E_pad + lane + 32 * i] = psum[i];
  __syncthreads();
  for (int e = tid; e < a.E; e += kThreads) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) s += Pw[w * E_pad + e];
    a.blk_prob[(size_t)blockIdx.x * a.E + e] = s;
    a.blk_cnt[(size_t)blockIdx.x * a.E + e] = cnt[e];
  }
}

size_t router_smem_bytes(const Plan& p) {
  const size_t f = (size_t)p.KC * (p.BT + 4) + (size_t)p.KC * (p.E_pad + 1) +
                   (size_t)p.BT * (p.E_pad + 1) + 8 * (size_t)p.E_pad;
  return f * sizeof(float) + (size_t)p.E_pad * sizeof(int);
}

cudaError_t launch_router(const Plan& p, const void* x, const void* W_r, const float* logit_offset,
                          const float* sel_bias, int32_t* topk_idx, float* topk_w, void* ws,
                          cudaStream_t st) {
  RouterArgs a;
  a.x = x;
  a.W_r = W_r;
  a.logit_offset = logit_offset;
  a.sel_bias = sel_bias;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.blk_cnt = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.blk_cnt);
  a.blk_prob = reinterpret_cast<float*>(static_cast<char*>(ws) + p.ws.blk_prob);
  a.T = p.cfg.T;
  a.d = p.cfg.d;
  a.E = p.cfg.E;
  a.E_pad = p.E_pad;
  a.k = p.cfg.k;
  a.BT = p.BT;
  a.KC = p.KC;
  a.gate = p.cfg.gate;
  const size_t smem = router_smem_bytes(p);
  if (p.cfg.dtype == MOE_BF16) {
    cudaError_t e = cudaFuncSetAttribute(router_topk_kernel<__nv_bfloat16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    router_topk_kernel<__nv_bfloat16><<<p.nblk, kThreads, smem, st>>>(a);
  } else {
    cudaError_t e = cudaFuncSetAttribute(router_topk_kernel<float>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    router_topk_kernel<float><<<p.nblk, kThreads, smem, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace moe
