// route.cu -- stage 3 (capacity and drops), stage 4 (permutation into
// expert-contiguous order) and the balance statistics of stage 6.
//
// "Mixture of Experts" (llm-tutorial ch. 11) § Expert capacity and dropped
// tokens, and "Mixture of experts" (inside-the-model guide) § Auxiliary loss:
// an expert takes at most C assignments; the rest skip it and travel on the
// residual path.  The order that decides who is dropped is the token-major key
// t*k + j: an assignment is kept iff fewer than C earlier keys went to the same
// expert.  "Chapter 33 — Mixture of Experts (MoE)" § Simple MoE Layer
// Implementation gathers each expert's tokens with a mask; here one stable
// counting sort over the keys produces the same groups without host syncs.
//
// Determinism: the histogram is an integer count, the scans run in a fixed
// order and every float sum has a fixed association, so repeated calls give
// bitwise-identical results.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "moe_internal.h"

namespace moe {

struct ScanArgs {
  int* blk_cnt;          // [nblk][E] in: histogram; out: exclusive scan over blocks
  const float* blk_prob; // [nblk][E]
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
};

// One block of 512 threads; thread e owns expert e.
__global__ void __launch_bounds__(512) scan_kernel(const ScanArgs a) {
  __shared__ int scratch[33];
  __shared__ double red[512];
  const int e = threadIdx.x;
  int routed = 0, kept = 0, mt = 0;
  float P = 0.f, fr = 0.f;
  if (e < a.E) {
    int* col = a.blk_cnt + e;
    int b = 0;
    for (; b + 4 <= a.nblk; b += 4) {
      const int c0 = col[(size_t)(b + 0) * a.E], c1 = col[(size_t)(b + 1) * a.E];
      const int c2 = col[(size_t)(b + 2) * a.E], c3 = col[(size_t)(b + 3) * a.E];
      col[(size_t)(b + 0) * a.E] = routed;
      col[(size_t)(b + 1) * a.E] = routed + c0;
      col[(size_t)(b + 2) * a.E] = routed + c0 + c1;
      col[(size_t)(b + 3) * a.E] = routed + c0 + c1 + c2;
      routed += c0 + c1 + c2 + c3;
    }
    for (; b < a.nblk; ++b) {
      const int c = col[(size_t)b * a.E];
      col[(size_t)b * a.E] = routed;
      routed += c;
    }
    float ps = 0.f;
    for (int bb = 0; bb < a.nblk; ++bb) ps += a.blk_prob[(size_t)bb * a.E + e];
    kept = routed < a.capacity ? routed : a.capacity;
    mt = (kept + a.bm - 1) / a.bm;
    P = a.T > 0 ? ps / (float)a.T : 0.f;
    fr = a.T > 0 ? (float)routed / (float)(a.T * a.k) : 0.f;
  }
  int tot_kept, tot_mt, tot_up, tot_dn;
  const int ex_kept = block_exclusive_scan(kept, scratch, &tot_kept);
  const int ex_mt = block_exclusive_scan(mt, scratch, &tot_mt);
  const int ex_up = block_exclusive_scan(mt * a.nt_up, scratch, &tot_up);
  const int ex_dn = block_exclusive_scan(mt * a.nt_dn, scratch, &tot_dn);
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
  if (e == 0) {
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
  // L = alpha * E * sum_i f_i P_i, summed as a fixed binary tree in double.
  red[e] = (e < a.E) ? (double)fr * (double)P : 0.0;
  __syncthreads();
  for (int s = 256; s > 0; s >>= 1) {
    if (e < s) red[e] += red[e + s];
    __syncthreads();
  }
  if (e == 0) a.aux_loss[0] = (float)((double)a.alpha * (double)a.E * red[0]);
}

struct PermuteArgs {
  const void* x;
  const int32_t* topk_idx;
  int32_t* slot_pos;
  int* key_row;
  const int* blk_base;   // [nblk][E] exclusive scan over blocks
  Meta m;
  void* xp;
  int T, d, E, k, BT, capacity, row_bytes;
  int copy;
};

// One block per routing block: rank every key among the earlier keys of the
// block that chose the same expert, add the block's base, apply the capacity
// test and write the row; then copy the kept token rows into expert order.
__global__ void __launch_bounds__(kThreads) permute_kernel(const PermuteArgs a) {
  extern __shared__ int smi[];
  const int b = blockIdx.x;
  const int t0 = b * a.BT;
  const int ntok = min(a.BT, a.T - t0);
  const int nk = ntok * a.k;
  int* e_s = smi;            // [BT*k]
  int* row_s = smi + a.BT * a.k;
  const size_t key0 = (size_t)t0 * a.k;
  for (int q = threadIdx.x; q < nk; q += kThreads) e_s[q] = a.topk_idx[key0 + q];
  __syncthreads();
  for (int q = threadIdx.x; q < nk; q += kThreads) {
    const int e = e_s[q];
    int rank = 0;
    for (int q2 = 0; q2 < q; ++q2) rank += (e_s[q2] == e);
    const int pos = a.blk_base[(size_t)b * a.E + e] + rank;
    const bool keep = pos < a.capacity;
    const int row = keep ? a.m.seg_start[e] + pos : -1;
    a.key_row[key0 + q] = row;
    if (a.slot_pos) a.slot_pos[key0 + q] = keep ? a.m.offsets[e] + pos : -1;
    row_s[q] = row;
  }
  __syncthreads();
  if (!a.copy) return;
  const int nvec = a.row_bytes / 16;
  const uint4* xs = static_cast<const uint4*>(a.x);
  uint4* xp = static_cast<uint4*>(a.xp);
  for (int i = threadIdx.x; i < nk * nvec; i += kThreads) {
    const int q = i / nvec, v = i - q * nvec;
    const int row = row_s[q];
    if (row >= 0) {
      const int t = t0 + q / a.k;
      xp[(size_t)row * nvec + v] = xs[(size_t)t * nvec + v];
    }
  }
}

Meta meta_ptrs(const Plan& p, void* ws) {
  int* base = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.meta);
  const int E = p.cfg.E;
  Meta m;
  m.kept = base;
  m.offsets = m.kept + E;
  m.seg_start = m.offsets + (E + 1);
  m.mtiles = m.seg_start + (E + 1);
  m.tp_up = m.mtiles + (E + 1);
  m.tp_dn = m.tp_up + (E + 2);
  return m;
}

cudaError_t launch_scan(const Plan& p, void* ws, int32_t* expert_counts, float* aux_loss,
                        int32_t* routed_counts, int32_t* offsets, float* f_out, float* P_out,
                        cudaStream_t st) {
  ScanArgs a;
  a.blk_cnt = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.blk_cnt);
  a.blk_prob = reinterpret_cast<const float*>(static_cast<char*>(ws) + p.ws.blk_prob);
  a.m = meta_ptrs(p, ws);
  a.nblk = p.nblk;
  a.E = p.cfg.E;
  a.T = p.cfg.T;
  a.k = p.cfg.k;
  a.capacity = p.capacity;
  a.bm = p.bm;
  a.nt_up = p.nt_up;
  a.nt_dn = p.nt_dn;
  a.nt_up_sh = p.nt_up_sh;
  a.nt_dn_sh = p.nt_dn_sh;
  a.mt_sh = p.mt_sh;
  a.has_shared = p.cfg.n_shared;
  a.alpha = p.cfg.alpha;
  a.expert_counts = expert_counts;
  a.aux_loss = aux_loss;
  a.routed_counts = routed_counts;
  a.offsets_out = offsets;
  a.f_out = f_out;
  a.P_out = P_out;
  scan_kernel<<<1, 512, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* topk_idx,
                           int32_t* slot_pos, bool copy_rows, void* ws, cudaStream_t st) {
  PermuteArgs a;
  a.x = x;
  a.topk_idx = topk_idx;
  a.slot_pos = slot_pos;
  a.key_row = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.key_row);
  a.blk_base = reinterpret_cast<const int*>(static_cast<char*>(ws) + p.ws.blk_cnt);
  a.m = meta_ptrs(p, ws);
  a.xp = static_cast<char*>(ws) + p.ws.xp;
  a.T = p.cfg.T;
  a.d = p.cfg.d;
  a.E = p.cfg.E;
  a.k = p.cfg.k;
  a.BT = p.BT;
  a.capacity = p.capacity;
  a.row_bytes = p.cfg.d * p.elem;
  a.copy = copy_rows ? 1 : 0;
  const size_t smem = 2 * sizeof(int) * (size_t)p.BT * p.cfg.k;
  permute_kernel<<<p.nblk, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
