// gemm_simt.cu -- stage 5 on the float32 path: grouped expert GEMMs over the
// ragged expert segments with plain float32 FMA (no TF32), so the output meets
// a 1e-5 relative tolerance.  Used for float32 layers, such as the 64 -> 256
// -> 64 toy layer of "Mixture-of-Experts" (neural networks visually), routing
// figure.
//
// Expert forms: "Mixture of Experts" (llm-tutorial ch. 11) § The mathematics
// (W2 act(W1 x), GELU or ReLU, no biases) and § Active vs total parameters
// (SwiGLU: gate W1, up W3, down W2); the shared expert of "Mixture of
// experts" (inside-the-model guide) § Fine-grained and shared experts is the
// last segment and reads x directly.
//
// Work items are (segment, M tile, N tile), read from the device-side tile
// prefix the scan kernel wrote; no host synchronisation is needed.
#include <climits>
#include <cmath>

#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"

namespace moe {

enum { SIMT_GELU = 0, SIMT_RELU = 1, SIMT_SWIGLU = 2, SIMT_NONE = 3 };

struct SimtArgs {
  const float* A;        // routed rows [R_cap][K]
  const float* A_sh;     // shared rows [A_sh_rows][K_sh]
  int A_sh_rows;
  const float* B0;       // routed weights [E][N][K]
  const float* B1;       // routed W3 (SwiGLU) or null
  const float* B0_sh;    // shared weights [N_sh][K_sh]
  const float* B1_sh;
  float* out;            // [R_cap][N]
  float* out_sh;         // [T_pad][N_sh]
  const int* tp;         // tile prefix [E+2]
  const int* seg_start;  // [E]
  const int* mtiles;     // [E+1]
  int E, has_shared;
  int N, K, N_sh, K_sh;
  int act;               // routed activation
  int act_sh;
  int R_cap;             // rows of the routed buffers
  uint32_t* status;
};

constexpr int SB_M = kSimtBM, SB_N = kSimtBN, SB_K = 16;

__device__ __forceinline__ float act_apply(int act, float a) {
  if (act == SIMT_GELU) return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f));
  if (act == SIMT_RELU) return fmaxf(a, 0.f);
  return a;
}

__global__ void __launch_bounds__(kThreads) simt_grouped_gemm(const SimtArgs a) {
  __shared__ __align__(16) float As[SB_K][SB_M + 4];
  __shared__ __align__(16) float Bs[SB_K][SB_N + 4];
  __shared__ __align__(16) float Cs[SB_K][SB_N + 4];   // second B operand (SwiGLU up)
  pdl_wait();
  pdl_trigger();
  const int nseg = a.E + a.has_shared;
  const int total = a.tp[nseg];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.tp[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int seg = lo;
    const bool sh = seg >= a.E;
    const int local = tile - a.tp[seg];
    const int mt = a.mtiles[seg];
    const int n_t = local / mt, m_t = local - n_t * mt;
    const int N = sh ? a.N_sh : a.N, K = sh ? a.K_sh : a.K;
    const int act = sh ? a.act_sh : a.act;
    const float* A = sh ? a.A_sh : a.A;
    const int row0 = sh ? m_t * SB_M : a.seg_start[seg] + m_t * SB_M;
    const int row_lim = sh ? a.A_sh_rows : a.R_cap;
    const float* B0 = sh ? a.B0_sh : a.B0 + (size_t)seg * N * K;
    const float* B1 = sh ? a.B1_sh : (a.B1 ? a.B1 + (size_t)seg * N * K : nullptr);
    const bool dual = act == SIMT_SWIGLU;
    float* out = sh ? a.out_sh : a.out;
    const int n0 = n_t * SB_N;

    float acc0[4][4], acc1[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += SB_K) {
      for (int i = threadIdx.x; i < SB_M * SB_K; i += kThreads) {
        const int r = i / SB_K, kk = i - r * SB_K;
        const int gr = row0 + r, gk = k0 + kk;
        As[kk][r] = (gr < row_lim && gk < K) ? A[(size_t)gr * K + gk] : 0.f;
      }
      for (int i = threadIdx.x; i < SB_N * SB_K; i += kThreads) {
        const int n = i / SB_K, kk = i - n * SB_K;
        const int gn = n0 + n, gk = k0 + kk;
        const bool ok = gn < N && gk < K;
        Bs[kk][n] = ok ? B0[(size_t)gn * K + gk] : 0.f;
        if (dual) Cs[kk][n] = ok ? B1[(size_t)gn * K + gk] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < SB_K; ++kk) {
        const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
        const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
        const float ar[4] = {av.x, av.y, av.z, av.w};
        const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc0[i][j] = fmaf(ar[i], br[j], acc0[i][j]);
        if (dual) {
          const float4 cv = *reinterpret_cast<const float4*>(&Cs[kk][tx * 4]);
          const float cr[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc1[i][j] = fmaf(ar[i], cr[j], acc1[i][j]);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int gr = row0 + ty * 4 + i;
      if (!sh && !in_bounds(gr >= 0 && gr < a.R_cap, a.status)) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int gn = n0 + tx * 4 + j;
        if (gn >= N) continue;
        float v;
        if (dual) {
          const float g = acc0[i][j];
          v = (g / (1.0f + expf(-g))) * acc1[i][j];
        } else {
          v = act_apply(act, acc0[i][j]);
        }
        out[(size_t)gr * N + gn] = v;
      }
    }
  }
}

static int simt_act(int act) {
  return act == MOE_ACT_GELU ? SIMT_GELU : act == MOE_ACT_RELU ? SIMT_RELU : SIMT_SWIGLU;
}

cudaError_t launch_experts_simt(const Plan& p, const void* x, const void* W1, const void* W3,
                                const void* W2, const void* Ws1, const void* Ws3,
                                const void* Ws2, void* ws, cudaStream_t st,
                                cudaEvent_t mid_event) {
  char* w = static_cast<char*>(ws);
  const Meta m = meta_ptrs(p, ws);
  const int grid_up = p.max_tiles_up < p.num_sms * 8 ? p.max_tiles_up : p.num_sms * 8;
  const int grid_dn = p.max_tiles_dn < p.num_sms * 8 ? p.max_tiles_dn : p.num_sms * 8;
  SimtArgs u;
  u.A = reinterpret_cast<const float*>(w + p.ws.xp);
  u.A_sh = static_cast<const float*>(x);
  u.A_sh_rows = p.cfg.T;
  u.B0 = static_cast<const float*>(W1);
  u.B1 = static_cast<const float*>(W3);
  u.B0_sh = static_cast<const float*>(Ws1);
  u.B1_sh = static_cast<const float*>(Ws3);
  u.out = reinterpret_cast<float*>(w + p.ws.h);
  u.out_sh = p.cfg.n_shared ? reinterpret_cast<float*>(w + p.ws.hs) : nullptr;
  u.tp = m.tp_up;
  u.seg_start = m.seg_start;
  u.mtiles = m.mtiles;
  u.E = p.cfg.E;
  u.has_shared = p.cfg.n_shared;
  u.N = p.cfg.f;
  u.K = p.cfg.d;
  u.N_sh = p.cfg.f_shared;
  u.K_sh = p.cfg.d;
  u.act = simt_act(p.cfg.act);
  u.act_sh = SIMT_SWIGLU;
  u.R_cap = p.R_cap;
  u.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  cudaError_t e = launch_pdl(simt_grouped_gemm, dim3(grid_up), dim3(kThreads), 0, st, u);
  if (e != cudaSuccess) return e;
  if (mid_event) {
    e = cudaEventRecord(mid_event, st);
    if (e != cudaSuccess) return e;
  }
  SimtArgs dn;
  dn.A = reinterpret_cast<const float*>(w + p.ws.h);
  dn.A_sh = p.cfg.n_shared ? reinterpret_cast<const float*>(w + p.ws.hs) : nullptr;
  dn.A_sh_rows = p.T_pad;
  dn.B0 = static_cast<const float*>(W2);
  dn.B1 = nullptr;
  dn.B0_sh = static_cast<const float*>(Ws2);
  dn.B1_sh = nullptr;
  dn.out = reinterpret_cast<float*>(w + p.ws.o);
  dn.out_sh = p.cfg.n_shared ? reinterpret_cast<float*>(w + p.ws.os) : nullptr;
  dn.tp = m.tp_dn;
  dn.seg_start = m.seg_start;
  dn.mtiles = m.mtiles;
  dn.E = p.cfg.E;
  dn.has_shared = p.cfg.n_shared;
  dn.N = p.cfg.d;
  dn.K = p.cfg.f;
  dn.N_sh = p.cfg.d;
  dn.K_sh = p.cfg.f_shared;
  dn.act = SIMT_NONE;
  dn.act_sh = SIMT_NONE;
  dn.R_cap = p.R_cap;
  dn.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  return launch_pdl(simt_grouped_gemm, dim3(grid_dn), dim3(kThreads), 0, st, dn);
}

}  // namespace moe
