// route.cu -- stage 4: positions of the kept assignments and the permutation
// of token rows into expert-contiguous order (the capacity scan that feeds it
// runs at the end of the top-k kernel, see route_scan.cuh).
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
#include "launch.cuh"
#include "moe_internal.h"

namespace moe {

struct PermuteArgs {
  const void* x;
  const int32_t* topk_idx;
  int32_t* slot_pos;
  int* key_row;
  const int* blk_base;   // [nblk][E] exclusive scan over blocks
  Meta m;
  void* xp;
  int* row_token;        // [R_cap]: token of each kept row
  int T, E, k, BT, capacity, nvec;   // nvec: 16-byte vectors per token row
  int copy;
};

// One block per routing block.  Warp 0 ranks every key among the earlier keys
// of the block that chose the same expert: keys go through in order, 32 at a
// time; __match_any_sync groups equal experts inside a chunk and a per-expert
// counter in shared memory carries the count across chunks.  Rank plus the
// block's base is the key's position; the capacity test and the row follow.
// Then all warps copy the kept token rows into expert order, one row per warp.
constexpr int kPermuteThreads = 512;

__global__ void __launch_bounds__(kPermuteThreads) permute_kernel(const PermuteArgs a) {
  extern __shared__ int smi[];
  int* cnt = smi;                 // [E]
  int* row_s = smi + a.E;         // [BT*k]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int t0 = b * a.BT;
  const int nk = min(a.BT, a.T - t0) * a.k;
  const size_t key0 = (size_t)t0 * a.k;
  for (int e = tid; e < a.E; e += kPermuteThreads) cnt[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  if (warp == 0) {
    const int* base = a.blk_base + (size_t)b * a.E;
    for (int c = 0; c < nk; c += 32) {
      const int q = c + lane;
      const bool valid = q < nk;
      const int e = valid ? a.topk_idx[key0 + q] : -1 - lane;   // invalid lanes never match
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int before = __popc(peers & ((1u << lane) - 1u));
      const int prior = valid ? cnt[e] : 0;
      __syncwarp();
      if (valid) {
        const int pos = base[e] + prior + before;
        const bool keep = pos < a.capacity;
        const int row = keep ? a.m.seg_start[e] + pos : -1;
        a.key_row[key0 + q] = row;
        if (a.slot_pos) a.slot_pos[key0 + q] = keep ? a.m.offsets[e] + pos : -1;
        if (keep) a.row_token[row] = t0 + q / a.k;
        row_s[q] = row;
        if (before == 0) cnt[e] = prior + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  if (!a.copy) return;
  // Row copies: (key, 16-byte vector) pairs spread over the block, four
  // independent loads in flight per thread before their stores.
  const uint4* xs = static_cast<const uint4*>(a.x);
  uint4* xp = static_cast<uint4*>(a.xp);
  const int total = nk * a.nvec;
  constexpr int U = 4;
  for (int i0 = tid; i0 < total; i0 += kPermuteThreads * U) {
    uint4 v[U];
    int dst_i[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kPermuteThreads;
      dst_i[u] = -1;
      if (i < total) {
        const int q = i / a.nvec, c = i - q * a.nvec;
        const int row = row_s[q];
        if (row >= 0) {
          v[u] = xs[(size_t)(t0 + q / a.k) * a.nvec + c];
          dst_i[u] = row;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kPermuteThreads;
      if (dst_i[u] >= 0) xp[(size_t)dst_i[u] * a.nvec + (i - (i / a.nvec) * a.nvec)] = v[u];
    }
  }
}

// Copy of the kept token rows into expert order after the one-launch router
// (key_row is final): grid-stride over (key, 16-byte vector), eight loads in
// flight per thread.
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(
    const uint4* x, uint4* xp, const int* key_row, int nkeys, int k, int nvec) {
  pdl_wait();
  pdl_trigger();
  const long long total = (long long)nkeys * nvec;
  const long long stride = (long long)gridDim.x * kGatherThreads;
  constexpr int U = 8;
  for (long long i0 = (long long)blockIdx.x * kGatherThreads + threadIdx.x; i0 < total;
       i0 += stride * U) {
    uint4 v[U];
    long long dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long i = i0 + u * stride;
      dst[u] = -1;
      if (i < total) {
        const int q = (int)(i / nvec);
        const int c = (int)(i - (long long)q * nvec);
        const int row = key_row[q];
        if (row >= 0) {
          v[u] = x[(size_t)(q / k) * nvec + c];
          dst[u] = (long long)row * nvec + c;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0) xp[dst[u]] = v[u];
  }
}

cudaError_t launch_gather_rows(const Plan& p, const void* x, void* ws, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  const int nkeys = p.cfg.T * p.cfg.k;
  const int nvec = p.cfg.d * p.elem / 16;
  const long long total = (long long)nkeys * nvec;
  long long blocks = (total + kGatherThreads * 8 - 1) / (kGatherThreads * 8);
  const long long cap = 8LL * p.num_sms;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(kGatherThreads), 0, st,
                    static_cast<const uint4*>(x), reinterpret_cast<uint4*>(w + p.ws.xp),
                    reinterpret_cast<const int*>(w + p.ws.key_row), nkeys, p.cfg.k, nvec);
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

cudaError_t launch_permute(const Plan& p, const void* x, const int32_t* topk_idx,
                           int32_t* slot_pos, bool copy_rows, void* ws, cudaStream_t st,
                           void* y) {
  PermuteArgs a;
  a.x = x;
  a.topk_idx = topk_idx;
  a.slot_pos = slot_pos;
  a.key_row = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.key_row);
  a.blk_base = reinterpret_cast<const int*>(static_cast<char*>(ws) + p.ws.blk_cnt);
  a.m = meta_ptrs(p, ws);
  a.xp = static_cast<char*>(ws) + p.ws.xp;
  a.row_token = reinterpret_cast<int*>(static_cast<char*>(ws) + p.ws.row_token);
  (void)y;
  a.T = p.cfg.T;
  a.E = p.cfg.E;
  a.k = p.cfg.k;
  a.BT = p.BT;
  a.capacity = p.capacity;
  a.nvec = p.cfg.d * p.elem / 16;
  a.copy = copy_rows ? 1 : 0;
  const size_t smem = sizeof(int) * ((size_t)p.cfg.E + (size_t)p.BT * p.cfg.k);
  return launch_pdl(permute_kernel, dim3(p.nblk), dim3(kPermuteThreads), smem, st, a);
}

}  // namespace moe
