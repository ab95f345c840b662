// route_scan.cuh -- stage 3 (capacity) and the balance statistics, run by the
// last routing block to finish, over the expert histograms every routing
// block published.
//
// "Mixture of Experts" (llm-tutorial ch. 11) § Expert capacity and dropped
// tokens, and "Mixture of experts" (inside-the-model guide) § Auxiliary loss:
// an expert takes at most C assignments; the rest skip it and travel on the
// residual path.  The order that decides who is dropped is the token-major key
// t*k + j, so the histogram of routing block b counts keys of tokens
// [b*BT, (b+1)*BT) and its exclusive scan over blocks gives every block the
// number of earlier keys per expert.  The guide's § Auxiliary loss and
// ch. 11 § The auxiliary loss give L = alpha * N * sum_i f_i P_i.
//
// Determinism: counts are integers; each float sum runs over a fixed
// partition of blocks in a fixed order, so repeated calls agree bitwise.
#pragma once

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

struct ScanArgs {
  int* blk_cnt;          // [nblk][E] in: histogram; out: exclusive scan over blocks
  float* blk_prob;       // [nblk][E]
  Meta m;
  int nblk, E, T, k, capacity, bm;
  int nt_up, nt_dn, nt_up_sh, nt_dn_sh, mt_sh, has_shared;
  float alpha;
  int32_t* expert_counts;
  float* aux_loss;
  int32_t* routed_counts;
  int32_t* offsets_out;
  float* f_out;
  float* P_out;
  unsigned int* done_counter;   // routing blocks finished (reset by the last one)
};

// Scan arguments of a layer call: workspace regions and caller outputs.
inline ScanArgs scan_args(const Plan& p, void* ws, const ScanOutputs& so) {
  char* w = static_cast<char*>(ws);
  ScanArgs c;
  c.blk_cnt = reinterpret_cast<int*>(w + p.ws.blk_cnt);
  c.blk_prob = reinterpret_cast<float*>(w + p.ws.blk_prob);
  c.m = meta_ptrs(p, ws);
  c.nblk = p.nblk;
  c.E = p.cfg.E;
  c.T = p.cfg.T;
  c.k = p.cfg.k;
  c.capacity = p.capacity;
  c.bm = p.bm;
  c.nt_up = p.nt_up;
  c.nt_dn = p.nt_dn;
  c.nt_up_sh = p.nt_up_sh;
  c.nt_dn_sh = p.nt_dn_sh;
  c.mt_sh = p.mt_sh;
  c.has_shared = p.cfg.n_shared;
  c.alpha = p.cfg.alpha;
  c.expert_counts = so.expert_counts;
  c.aux_loss = so.aux_loss;
  c.routed_counts = so.routed_counts;
  c.offsets_out = so.offsets;
  c.f_out = so.f_out;
  c.P_out = so.P_out;
  c.done_counter = reinterpret_cast<unsigned int*>(w + p.ws.status + kRouteDoneOffset);
  return c;
}

template <int NT>
struct ScanSmem {
  int scratch[4 * 33];
  int pc[NT];
  float pp[NT];
  int routed_s[kMaxE];
  float psum_s[kMaxE];
  double red[NT / 32];
};

// Exclusive prefix sums of four integers per thread over NT threads (NT a
// multiple of 32, <= 1024), in one pass.  `scratch` holds 4*33 ints.
template <int NT>
__device__ __forceinline__ int4 block_exscan4(int4 v, int* scratch, int4* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NW = NT / 32;
  int4 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, inc.x, o);
    const int ny = __shfl_up_sync(0xffffffffu, inc.y, o);
    const int nz = __shfl_up_sync(0xffffffffu, inc.z, o);
    const int nw = __shfl_up_sync(0xffffffffu, inc.w, o);
    if (lane >= o) {
      inc.x += nx;
      inc.y += ny;
      inc.z += nz;
      inc.w += nw;
    }
  }
  if (lane == 31) {
    scratch[warp] = inc.x;
    scratch[33 + warp] = inc.y;
    scratch[66 + warp] = inc.z;
    scratch[99 + warp] = inc.w;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int w = lane < NW ? scratch[33 * c + lane] : 0;
      int winc = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, winc, o);
        if (lane >= o) winc += n;
      }
      if (lane < NW) scratch[33 * c + lane] = winc - w;
      if (lane == 31) scratch[33 * c + 32] = winc;
    }
  }
  __syncthreads();
  const int4 out = make_int4(scratch[warp] + inc.x - v.x, scratch[33 + warp] + inc.y - v.y,
                             scratch[66 + warp] + inc.z - v.z, scratch[99 + warp] + inc.w - v.w);
  *total = make_int4(scratch[32], scratch[65], scratch[98], scratch[131]);
  return out;
}

// One block of NT threads, E <= NT (the split path runs it with 512 threads for
// E <= 512, the fused router with 256 threads for E <= 256).
// G = NT / next_pow2(E) threads share expert e:
// each sums a contiguous run of routing blocks, one thread per expert scans
// the G partial counts, and every thread then writes the exclusive per-block
// bases of its run.  Threads e < E then finish the per-expert values (kept
// count, segment start, tile counts, f_i, P_i) and the block-wide scans.
template <int NT>
__device__ void scan_block(const ScanArgs& a, ScanSmem<NT>& sm) {
  const int tid = threadIdx.x;
  int Epow = 1;
  while (Epow < a.E) Epow <<= 1;
  const int G = NT / Epow;
  {
    const int e = tid / G, g = tid - e * G;
    const int per = (a.nblk + G - 1) / G;
    const int b0 = min(a.nblk, g * per), b1 = min(a.nblk, b0 + per);
    int c = 0;
    float ps = 0.f;
    constexpr int U = 8;   // loads in flight per thread
    if (e < a.E) {
      for (int b = b0; b < b1; b += U) {
        int cv[U];
        float pv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool ok = b + u < b1;
          cv[u] = ok ? __ldcg(a.blk_cnt + (size_t)(b + u) * a.E + e) : 0;
          pv[u] = ok ? __ldcg(a.blk_prob + (size_t)(b + u) * a.E + e) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          c += cv[u];
          if (b + u < b1) ps += pv[u];
        }
      }
    }
    sm.pc[tid] = c;
    sm.pp[tid] = ps;
    __syncthreads();
    if (e < a.E && g == 0) {
      int run = 0;
      float pr = 0.f;
      for (int gg = 0; gg < G; ++gg) {
        const int v = sm.pc[tid + gg];
        sm.pc[tid + gg] = run;
        run += v;
        pr += sm.pp[tid + gg];
      }
      sm.routed_s[e] = run;
      sm.psum_s[e] = pr;
    }
    __syncthreads();
    if (e < a.E) {
      int run = sm.pc[tid];
      for (int b = b0; b < b1; b += U) {
        int cv[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          cv[u] = b + u < b1 ? __ldcg(a.blk_cnt + (size_t)(b + u) * a.E + e) : 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (b + u < b1) a.blk_cnt[(size_t)(b + u) * a.E + e] = run;
          run += cv[u];
        }
      }
    }
  }
  __syncthreads();
  {
    const int e = tid;
    int routed = 0, kept = 0, mt = 0;
    float P = 0.f, fr = 0.f;
    if (e < a.E) {
      routed = sm.routed_s[e];
      kept = routed < a.capacity ? routed : a.capacity;
      mt = (kept + a.bm - 1) / a.bm;
      P = a.T > 0 ? sm.psum_s[e] / (float)a.T : 0.f;
      fr = a.T > 0 ? (float)routed / (float)(a.T * a.k) : 0.f;
    }
    int4 tot;
    const int4 ex = block_exscan4<NT>(make_int4(kept, mt, mt * a.nt_up, mt * a.nt_dn),
                                      sm.scratch, &tot);
    const int ex_kept = ex.x, ex_mt = ex.y, ex_up = ex.z, ex_dn = ex.w;
    const int tot_kept = tot.x, tot_mt = tot.y, tot_up = tot.z, tot_dn = tot.w;
    if (e < a.E) {
      a.m.kept[e] = kept;
      a.m.offsets[e] = ex_kept;
      a.m.seg_start[e] = ex_mt * a.bm;
      a.m.mtiles[e] = mt;
      a.m.tp_up[e] = ex_up;
      a.m.tp_dn[e] = ex_dn;
      a.expert_counts[e] = kept;
      if (a.routed_counts) a.routed_counts[e] = routed;
      if (a.offsets_out) a.offsets_out[e] = ex_kept;
      if (a.f_out) a.f_out[e] = fr;
      if (a.P_out) a.P_out[e] = P;
    }
    if (tid == 0) {
      const int sh_up = a.has_shared ? a.mt_sh * a.nt_up_sh : 0;
      const int sh_dn = a.has_shared ? a.mt_sh * a.nt_dn_sh : 0;
      a.m.offsets[a.E] = tot_kept;
      a.m.seg_start[a.E] = tot_mt * a.bm;
      a.m.mtiles[a.E] = a.has_shared ? a.mt_sh : 0;
      a.m.tp_up[a.E] = tot_up;
      a.m.tp_up[a.E + 1] = tot_up + sh_up;
      a.m.tp_dn[a.E] = tot_dn;
      a.m.tp_dn[a.E + 1] = tot_dn + sh_dn;
      if (a.offsets_out) a.offsets_out[a.E] = tot_kept;
    }
    // L = alpha * E * sum_i f_i P_i in double: a fixed butterfly inside each
    // warp, then the warp sums in warp order.
    double l = (e < a.E) ? (double)fr * (double)P : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if ((tid & 31) == 0) sm.red[tid >> 5] = l;
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      for (int w = 0; w < NT / 32; ++w) t += sm.red[w];
      a.aux_loss[0] = (float)((double)a.alpha * (double)a.E * t);
    }
  }
}

}  // namespace moe
