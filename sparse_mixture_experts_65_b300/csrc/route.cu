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
#include <atomic>
#include <cfloat>
#include <climits>

#include "bulk_rows.cuh"
#include "check.cuh"
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
  uint32_t* status;
  int T, E, k, BT, capacity, nvec;   // nvec: 16-byte vectors per token row
  int R_cap;
  int copy;
};

// One block per routing block.  Warp 0 ranks every key among the earlier keys
// of the block that chose the same expert: keys go through in order, 32 at a
// time; __match_any_sync groups equal experts inside a chunk and a per-expert
// counter in shared memory carries the count across chunks.  Rank plus the
// block's base is the key's position; the capacity test and the row follow.
// Then all warps copy the kept token rows into expert order, one row per warp.
constexpr int kPermuteThreads = 512;
constexpr uint32_t kPermuteStage = 128u << 10;   // bulk-copy staging per block
constexpr uint64_t kPermuteTimeoutNs = 2000000000ull;

// Rows of at least 1 KB (and at most a quarter of the stage) move by bulk
// copies; shorter rows by 16-byte loads and stores.
__host__ __device__ inline bool permute_bulk(uint32_t row_bytes) {
  return row_bytes >= 1024u && row_bytes * 4u <= kPermuteStage;
}

// Shared memory: cnt[E] | row_s[BT*k] | (128-aligned) stage | kFanMaxSlots mbarriers.
__host__ __device__ inline size_t permute_stage_offset(int E, int keys) {
  return ((sizeof(int) * ((size_t)E + keys)) + 127) / 128 * 128;
}

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
      bool valid = q < nk;
      int e = valid ? a.topk_idx[key0 + q] : -1 - lane;   // invalid lanes never match
      if (valid && !in_bounds(e >= 0 && e < a.E, a.status)) {
        valid = false;
        row_s[q] = -1;
        e = -1 - lane;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int before = __popc(peers & ((1u << lane) - 1u));
      const int prior = valid ? cnt[e] : 0;
      __syncwarp();
      if (valid) {
        const int pos = base[e] + prior + before;
        bool keep = pos < a.capacity;
        int row = keep ? a.m.seg_start[e] + pos : -1;
        if (keep && !in_bounds(row >= 0 && row < a.R_cap, a.status)) {
          keep = false;
          row = -1;
        }
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
  const uint32_t row_bytes = (uint32_t)a.nvec * 16u;
  if (permute_bulk(row_bytes)) {
    // bulk copies through shared memory: each token row is read once and
    // stored to the segments of its kept slots, loads running ahead of stores
    uint8_t* stage = reinterpret_cast<uint8_t*>(smi) + permute_stage_offset(a.E, a.BT * a.k);
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage + kPermuteStage);
    const char* xs = static_cast<const char*>(a.x);
    char* xp = static_cast<char*>(a.xp);
    bulk_fanout_rows(
        nk / a.k, a.k, row_bytes,
        [&](int i) { return static_cast<const void*>(xs + (size_t)(t0 + i) * row_bytes); },
        [&](int i, int j) {
          const int row = row_s[i * a.k + j];
          return row >= 0 ? static_cast<void*>(xp + (size_t)row * row_bytes) : nullptr;
        },
        stage, kPermuteStage, bars, a.status, STATUS_TIMEOUT_ROUTE, kPermuteTimeoutNs);
    return;
  }
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
// (key_row is final): every block takes a contiguous range of tokens and
// copies each row once into shared memory and from there to the segments of
// the token's kept slots (rows too wide for three stage slots go key by key).
constexpr int kGatherThreads = 32 * kBulkIssuers;
constexpr uint32_t kGatherStage = 160u << 10;

__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(
    const char* x, char* xp, const int* key_row, int nkeys, int k, uint32_t row_bytes,
    int R_cap, uint32_t* status) {
  extern __shared__ __align__(128) uint8_t gsm[];
  pdl_wait();
  pdl_trigger();
  uint64_t* bars = reinterpret_cast<uint64_t*>(gsm + kGatherStage);
  if (row_bytes * 3u <= kGatherStage) {
    const int ntok = nkeys / k;
    const int per = (ntok + gridDim.x - 1) / gridDim.x;
    const int t0 = blockIdx.x * per;
    const int n = min(per, ntok - t0);
    if (n <= 0) return;
    bulk_fanout_rows(
        n, k, row_bytes,
        [&](int i) { return static_cast<const void*>(x + (size_t)(t0 + i) * row_bytes); },
        [&](int i, int j) {
          const int row = __ldg(key_row + (size_t)(t0 + i) * k + j);
          return row >= 0 && in_bounds(row < R_cap, status)
                     ? static_cast<void*>(xp + (size_t)row * row_bytes)
                     : nullptr;
        },
        gsm, kGatherStage, bars, status, STATUS_TIMEOUT_ROUTE, 2000000000ull);
    return;
  }
  const int per = (nkeys + gridDim.x - 1) / gridDim.x;
  const int q0 = blockIdx.x * per;
  const int n = min(per, nkeys - q0);
  if (n <= 0) return;
  bulk_copy_rows(
      n, row_bytes,
      [&](int i) { return static_cast<const void*>(x + (size_t)((q0 + i) / k) * row_bytes); },
      [&](int i) {
        const int row = __ldg(key_row + q0 + i);
        return row >= 0 && in_bounds(row < R_cap, status)
                   ? static_cast<void*>(xp + (size_t)row * row_bytes)
                   : nullptr;
      },
      gsm, kGatherStage, bars, status, STATUS_TIMEOUT_ROUTE, 2000000000ull);
}

cudaError_t launch_gather_rows(const Plan& p, const void* x, void* ws, cudaStream_t st) {
  char* w = static_cast<char*>(ws);
  const int nkeys = p.cfg.T * p.cfg.k;
  const uint32_t row_bytes = (uint32_t)p.cfg.d * p.elem;
  static std::atomic<uint64_t> attr_done{0};
  const size_t smem = kGatherStage + 8 * kFanMaxSlots;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_done.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(gather_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_release);
  }
  int blocks = p.num_sms;
  if (blocks > nkeys) blocks = nkeys > 0 ? nkeys : 1;
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(kGatherThreads), smem, st,
                    static_cast<const char*>(x), w + p.ws.xp,
                    reinterpret_cast<const int*>(w + p.ws.key_row), nkeys, p.cfg.k, row_bytes,
                    p.R_cap, reinterpret_cast<uint32_t*>(w + p.ws.status));
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
  a.R_cap = p.R_cap;
  a.copy = copy_rows ? 1 : 0;
  a.status = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + p.ws.status);
  const bool bulk = copy_rows && permute_bulk((uint32_t)a.nvec * 16u);
  const size_t ints = sizeof(int) * ((size_t)p.cfg.E + (size_t)p.BT * p.cfg.k);
  const size_t smem =
      bulk ? permute_stage_offset(p.cfg.E, p.BT * p.cfg.k) + kPermuteStage + 8 * kFanMaxSlots
           : ints;
  if (bulk) {
    static std::atomic<uint64_t> attr_done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_done.load(std::memory_order_acquire) & bit)) {
      e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               200 * 1024);
      if (e != cudaSuccess) return e;
      attr_done.fetch_or(bit, std::memory_order_release);
    }
  }
  return launch_pdl(permute_kernel, dim3(p.nblk), dim3(kPermuteThreads), smem, st, a);
}

}  // namespace moe
