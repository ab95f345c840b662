// gemm_tc.cu -- stage 5 on the bf16 path: the expert MLPs as grouped GEMMs
// over ragged expert segments on the 5th-generation tensor cores.
//
// Expert forms: "Mixture of Experts" (llm-tutorial ch. 11) § The mathematics
// (W2 act(W1 x): GELU in most production models, ReLU in the demo, no biases)
// and § Active vs total parameters (SwiGLU: gate W1, up W3, down W2).  Only
// chosen experts run: FLOPs per token scale with k (ch. 11 § The mathematics;
// "Mixture-of-Experts" (neural networks visually) § Show the math).  The shared
// expert of "Mixture of experts" (inside-the-model guide) § Fine-grained and
// shared experts is one more segment of the same launch, reading x directly.
//
// Kernel shape (one CTA per SM, persistent over work items):
//   warp 0    TMA producer: A tile (128 rows x 64 K) + B tile(s) (N rows x 64 K)
//             per stage, 128-byte swizzle, completion on a transaction barrier;
//   warp 1    allocates tensor memory; lane 0 issues tcgen05.mma (M=128,
//             N=MMA_N, K=16) into one of two TMEM accumulators and commits
//             stage releases and accumulator-ready signals;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator rows (one TMEM lane per
//             thread), activation (SwiGLU: silu(gate) * up from the two halves
//             of one N=2*BNH accumulator), bf16 or fp32 stores.
// Work items are (segment, M tile, N tile) read from a device tile prefix
// written by the scan kernel, N tiles outermost inside a segment so the CTAs
// that run together share the weight tile through L2.  Expert segments start
// on 128-row boundaries, so an M tile never mixes experts.
//
// Every wait is bounded: on a timeout the kernel records a status bit, tells
// the other roles to stop, drains its own copies and MMAs, frees tensor
// memory and returns.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "shared_out.cuh"
#include "tma_host.cuh"

namespace moe {

enum { EPI_SWIGLU = 0, EPI_GELU = 1, EPI_RELU = 2, EPI_OUT16 = 3, EPI_F32_CHUNKED = 4,
       EPI_COMBINE1 = 5, EPI_COMBINEK = 6 };

// EPI_OUT16 (down projection when the combine is a separate kernel): the
// expert output rows o are stored as bf16, rounded once from the float32
// accumulator; the combine sums g * o in float32 and rounds y once more.

// EPI_COMBINE1 (down projection of a top-1 layer without a shared expert):
// the combine is folded into the epilogue.  Row r of expert e holds the single
// kept slot of token t = row_token[r], so y[t] = bf16(g_t * acc) is written
// directly -- the same float32 product and the same single rounding as the
// separate combine kernel.  The epilogue warps also write y = 0 for the
// dropped tokens (key_row < 0).

// EPI_COMBINEK (down projection of every other tensor-core layer): the
// expert outputs o are stored as for EPI_OUT16, then each row counts itself in
// for its token and column slice (one counter per token and N tile; the
// shared expert's row counts too).  The row that completes the count sums the
// slice, y[t] = bf16(os[t] + sum_j g_tj * o[row(t, j)]) in float32 in the
// fixed order j = 0..k-1 over the kept slots -- the arithmetic of the
// separate combine kernel, so the result is the same bit for bit whichever
// row arrives last -- and re-arms the counter.  Tokens with no kept slot and
// no shared expert get y = 0 up front.

// EPI_F32_CHUNKED: the reduction runs in chunks of kChunkKB k-blocks (128 k),
// each accumulated by the tensor cores from zero; the epilogue adds the chunk
// results in float32, round to nearest, in chunk order.  The tensor cores'
// own float32 accumulation then spans at most 8 MMA steps, which keeps a
// 7168-wide dot product within ~2e-6 of exact (measured) instead of ~4e-5.
constexpr int kChunkKB = 2;

struct TcArgs {
  const int* tp;          // [E+2] tile prefix: routed segments, then the shared one
  const int* seg_start;   // [E] first row of each routed segment
  const int* mtiles;      // [E+1] M tiles per segment (index E: shared)
  const int* kept;        // [E] rows of each routed segment (padding rows follow)
  int rows_sh;            // rows of the shared segment (T)
  int static_mt;          // > 0: one dense segment of static_mt M tiles (no device schedule)
  int static_total;       // its tile count
  int E, has_shared;
  int N, K;               // routed output columns / reduction length
  int N_sh, K_sh;         // shared segment
  void* out;              // routed output rows [R_cap][ld_out]
  int ld_out;
  void* out_sh;           // shared output rows [T_pad][ld_out_sh]
  int ld_out_sh;
  int8_t* out_sh_exp = nullptr;   // down projection: the shared output's chunk exponents
  int ld_out_sh_exp = 0;          // [T_pad][ld_out_sh_exp]
  const float* col_bias;  // EPI_F32_CHUNKED: added per output column (may be null)
  int partial_rows;       // A tiles with at most this many real rows load 32-row boxes
  const int* row_token;   // token of each expert-ordered row (gather, EPI_COMBINE1)
  const float* gate;      // EPI_COMBINE1: topk_w, one gate per token
  void* y;                // EPI_COMBINE1: [T][ld_y] bf16 layer output
  int ld_y;
  const int* key_row;     // EPI_COMBINE1: [T] row of each token's slot, -1 if dropped
  int T_tokens;
  const char* gx;         // gathering up projection: x, rows of gx_row_bytes
  int gx_row_bytes;
  int early_b;            // the schedule predates the previous kernel: stream B before the wait
  const float* a_scale = nullptr;   // fp8 operands: scale of each A row (routed rows) ...
  const float* b0_scale = nullptr;  // ... and of each output column of B0 / B1, [E][N]
  const float* b1_scale = nullptr;
  int R_cap = 0;                    // rows of the routed output buffer
  int m64 = 0;                      // routed tiles of <= 64 rows multiply with M = 64
  unsigned* cmb_ctr = nullptr;      // EPI_COMBINEK: [T][cmb_nt] arrival counters
  int cmb_nt = 0;                   // N tiles per token row
  int k_slots = 1;                  // slots per token (key_row / gate are [T][k_slots])
  unsigned* zero_ctr = nullptr;     // cleared by this launch (the next launch's counters)
  int zero_ctr_n = 0;
  int T_x = 0;                      // rows of x (tokens): range of row_token entries
  int sched_bn = 0;                 // weights-as-M kernel: the column tile width that the
                                    // device tile prefix counts (N tiles per segment)
  uint32_t* status;
  uint64_t timeout_ns;
};

constexpr __host__ __device__ int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int BNH, bool DUAL, int EPI, bool F8 = false>
struct TcCfg {
  static constexpr int BM = kTcBM;
  static constexpr int ELEM = F8 ? 1 : 2;          // bytes per operand element
  static constexpr int BK = 128 / ELEM;            // k per stage: one 128-byte row
  static constexpr int BKX = 64;                   // the same in 16-bit tensor-map units
  static constexpr int KSTEPS = 4;                 // MMAs per stage, 32 bytes of k each
  static constexpr int MMA_N = DUAL ? 2 * BNH : BNH;
  static_assert(MMA_N % 16 == 0 && MMA_N >= 16 && MMA_N <= 256, "tcgen05 N for M=128");
  static_assert(BNH % 32 == 0, "epilogue walks 32-column chunks");
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = MMA_N * 128;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES_FIT = (200 * 1024) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int TMEM_COLS = pow2_at_least(2 * MMA_N);
  static_assert(TMEM_COLS <= 512, "two accumulators must fit in tensor memory");
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 16;
  // the device tile schedule, copied to shared memory once per CTA:
  // tp[E+2] | seg_start[E] | mtiles[E+1] | kept[E]
  static constexpr int SCHED_INTS = 4 * (kMaxE + 2);
  // row -> token tables of the four gathering producer warps (128 each)
  static constexpr int TOK_BYTES = 4 * 128 * 4;
  // fp8 operands: the output-column scales of the tile's two B halves
  static constexpr int CSCALE_BYTES = F8 ? 2 * 128 * 4 : 0;
  static constexpr int SMEM =
      1024 + STAGES * STAGE_BYTES + BAR_BYTES + 4 * SCHED_INTS + TOK_BYTES + CSCALE_BYTES;
  static constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(BM, MMA_N) : idesc_bf16_f32(BM, MMA_N);
  // M = 64 for routed tiles with at most 64 rows (the first half of the A tile)
  static constexpr uint32_t IDESC64 = F8 ? idesc_e4m3_f32(64, MMA_N) : idesc_bf16_f32(64, MMA_N);
};

struct TileInfo {
  int seg;
  bool shared;
  bool m64;     // at most 64 rows, multiplied with M = 64
  int a_row;    // first A row (and output row)
  int row_end;  // rows at or past this index are segment padding: not stored
  int n0;       // first output column
  int K, N;
};

// Tile schedule as seen by the kernel (shared-memory copies of the device
// arrays, or the global arrays in the static mode).
struct Sched {
  const int* tp;
  const int* seg_start;
  const int* mtiles;
  const int* kept;
};

__device__ __forceinline__ TileInfo decode_tile(const TcArgs& a, const Sched& sc, int tile,
                                                int bnh) {
  if (a.static_mt > 0) {   // dense GEMM: rows [0, rows_sh), tiles N-major
    TileInfo ti;
    ti.seg = 0;
    ti.shared = false;
    const int n_t = tile / a.static_mt, m_t = tile - n_t * a.static_mt;
    ti.a_row = m_t * kTcBM;
    ti.row_end = a.rows_sh;
    ti.n0 = n_t * bnh;
    ti.K = a.K;
    ti.N = a.N;
    ti.m64 = false;
    return ti;
  }
  const int nseg = a.E + a.has_shared;
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.tp[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.seg = lo;
  ti.shared = lo >= a.E;
  const int local = tile - sc.tp[lo];
  const int mt = sc.mtiles[lo];
  const int n_t = local / mt, m_t = local - n_t * mt;
  const int seg0 = ti.shared ? 0 : sc.seg_start[lo];
  ti.a_row = seg0 + m_t * kTcBM;
  ti.row_end = ti.shared ? a.rows_sh : seg0 + sc.kept[lo];
  ti.n0 = n_t * bnh;
  ti.K = ti.shared ? a.K_sh : a.K;
  ti.N = ti.shared ? a.N_sh : a.N;
  ti.m64 = a.m64 && !ti.shared && ti.row_end - ti.a_row <= 64;
  return ti;
}

// silu(g) * u with the hardware exponential and an approximate division
// (relative error ~1e-7, far below the bf16 rounding of h)
// Work item of a 2-CTA cluster: a pair of adjacent N tiles of one M tile;
// CTA rank r of the cluster takes N tile 2*np + r (past the segment's last N
// tile for an odd count: a phantom tile whose B loads fall outside the weight
// map -- zeros -- and whose results are never stored).  Pairs are numbered
// like tiles, N-major inside a segment; since every routed segment has the
// same number of N tiles, the pair prefix of segment s is (tp[s] / nt) * ntp.
__device__ __forceinline__ int pair_prefix(const TcArgs& a, const Sched& sc, int s, int nt,
                                           int ntp) {
  return (sc.tp[s] / nt) * ntp;
}

__device__ __forceinline__ int total_pairs(const TcArgs& a, const Sched& sc, int bnh) {
  const int nt = (a.N + bnh - 1) / bnh, ntp = (nt + 1) / 2;
  int tot = pair_prefix(a, sc, a.E, nt, ntp);
  if (a.has_shared) {
    const int nt_sh = (a.N_sh + bnh - 1) / bnh;
    tot += sc.mtiles[a.E] * ((nt_sh + 1) / 2);
  }
  return tot;
}

__device__ __forceinline__ TileInfo decode_pair(const TcArgs& a, const Sched& sc, int pair,
                                                int bnh, int rank) {
  const int nt = (a.N + bnh - 1) / bnh, ntp = (nt + 1) / 2;
  const int routed = pair_prefix(a, sc, a.E, nt, ntp);
  TileInfo ti;
  int local, mt;
  if (pair >= routed) {
    ti.seg = a.E;
    ti.shared = true;
    local = pair - routed;
    mt = sc.mtiles[a.E];
  } else {
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pair_prefix(a, sc, mid, nt, ntp) <= pair) lo = mid; else hi = mid - 1;
    }
    ti.seg = lo;
    ti.shared = false;
    local = pair - pair_prefix(a, sc, lo, nt, ntp);
    mt = sc.mtiles[lo];
  }
  const int np = local / mt, m_t = local - np * mt;
  const int seg0 = ti.shared ? 0 : sc.seg_start[ti.seg];
  ti.a_row = seg0 + m_t * kTcBM;
  ti.row_end = ti.shared ? a.rows_sh : seg0 + sc.kept[ti.seg];
  ti.n0 = (2 * np + rank) * bnh;
  ti.K = ti.shared ? a.K_sh : a.K;
  ti.N = ti.shared ? a.N_sh : a.N;
  ti.m64 = a.m64 && !ti.shared && ti.row_end - ti.a_row <= 64;
  return ti;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Epilogue of one accumulator: activation (or none, or the gate of a top-1
// combine), bf16 stores of this thread's row, masked at the segment's last
// row and the last column.
template <int BNH, bool DUAL, int EPI, bool F8 = false>
__device__ __forceinline__ void epilogue_tile(const TcArgs& a, const TileInfo& ti, uint32_t t_row,
                                              size_t orow, bool row_ok, float scale, int c_lo,
                                              int c_hi) {
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 32) {
    uint32_t r0[32];
    tmem_ld32(t_row + c, r0);
    uint32_t r1[32];
    if (DUAL) tmem_ld32(t_row + BNH + c, r1);
    tmem_ld_wait();
    const int col = ti.n0 + c;
    if ((EPI == EPI_OUT16 || EPI == EPI_COMBINEK) && ti.shared) {
      // the shared expert's output: fp16 scaled by 2^-e per 32-column chunk
      // (shared_out.cuh); columns past N hold zeros (their weights load as
      // zeros), so they do not move the chunk's maximum
      if (!row_ok || col >= ti.N) continue;   // past the last column: nothing to store
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(__uint_as_float(r0[i])));
      const int e = sh_chunk_exponent(amax);
      const float s = sh_pow2(-e);
      uint32_t ph[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        __half2 h2 = __floats2half2_rn(__uint_as_float(r0[2 * i]) * s,
                                       __uint_as_float(r0[2 * i + 1]) * s);
        ph[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      __half* dsth = static_cast<__half*>(a.out_sh) + orow * a.ld_out_sh + col;
      a.out_sh_exp[orow * a.ld_out_sh_exp + col / kShChunk] = static_cast<int8_t>(e);
      if (col + 32 <= ti.N) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
          reinterpret_cast<uint4*>(dsth)[v] =
              make_uint4(ph[4 * v], ph[4 * v + 1], ph[4 * v + 2], ph[4 * v + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (col + i < ti.N) {
            const uint32_t w = ph[i >> 1];
            reinterpret_cast<uint16_t*>(dsth)[i] =
                (i & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w);
          }
        }
      }
      continue;
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(
        EPI == EPI_COMBINE1 ? a.y : (ti.shared ? a.out_sh : a.out));
    const int ld = EPI == EPI_COMBINE1 ? a.ld_y : (ti.shared ? a.ld_out_sh : a.ld_out);
    __nv_bfloat16* dst = out + orow * ld + col;
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float v0 = __uint_as_float(r0[2 * i]), v1 = __uint_as_float(r0[2 * i + 1]);
      if (EPI == EPI_SWIGLU && F8) {
        // fp8 operands: gate and up accumulators times the row scale and the
        // column scales of W1 / W3 (N is a multiple of 4: a pair is in range
        // or out of it as a whole)
        const int cc = col + 2 * i;
        float2 sg = make_float2(0.f, 0.f), su = make_float2(0.f, 0.f);
        if (cc < ti.N) {
          const size_t si = (size_t)ti.seg * a.N + cc;
          sg = __ldg(reinterpret_cast<const float2*>(a.b0_scale + si));
          su = __ldg(reinterpret_cast<const float2*>(a.b1_scale + si));
        }
        v0 = silu_mul(v0 * (scale * sg.x), __uint_as_float(r1[2 * i]) * (scale * su.x));
        v1 = silu_mul(v1 * (scale * sg.y), __uint_as_float(r1[2 * i + 1]) * (scale * su.y));
      } else if (EPI == EPI_SWIGLU) {
        v0 = silu_mul(v0, __uint_as_float(r1[2 * i]));
        v1 = silu_mul(v1, __uint_as_float(r1[2 * i + 1]));
      } else if (EPI == EPI_RELU) {
        v0 = fmaxf(v0, 0.f);
        v1 = fmaxf(v1, 0.f);
      } else if (EPI == EPI_GELU) {
        v0 = 0.5f * v0 * (1.0f + erff(v0 * 0.70710678118654752f));
        v1 = 0.5f * v1 * (1.0f + erff(v1 * 0.70710678118654752f));
      } else if (EPI == EPI_COMBINE1) {
        v0 = fmaf(scale, v0, 0.f);
        v1 = fmaf(scale, v1, 0.f);
      }
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
      pk[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    if (!row_ok) {
    } else if (col + 32 <= ti.N) {
#pragma unroll
      for (int v = 0; v < 4; ++v)
        reinterpret_cast<uint4*>(dst)[v] =
            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (col + i < ti.N) {
          const uint32_t w = pk[i >> 1];
          reinterpret_cast<uint16_t*>(dst)[i] =
              (i & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w);
        }
      }
    }
  }
}

// A tiles with at most TcArgs::partial_rows real rows (small expert segments,
// decode batches) are loaded as ceil(rows / 32) boxes of 32 rows instead of
// one 128-row box: the rows left unloaded only feed accumulator rows that the
// epilogue never stores.
constexpr int kABox = 32;

// 32-row boxes a partial A tile loads (0: the whole 128-row box).
__device__ __forceinline__ int a_real_boxes(int rows, int partial_rows) {
  return rows > partial_rows ? 0 : (rows + kABox - 1) / kABox;
}
// Bytes the A loads of one stage deliver.
__device__ __forceinline__ uint32_t a_stage_bytes(int boxes, uint32_t full) {
  return boxes == 0 ? full : (uint32_t)boxes * kABox * 128u;
}
__device__ __forceinline__ void load_a_stage(uint32_t sa, const CUtensorMap* pA,
                                             const CUtensorMap* pA32, uint32_t bar, int kx,
                                             int a_row, int boxes) {
  if (boxes == 0) {
    tma_load_2d(sa, pA, bar, kx, a_row);
    return;
  }
  for (int b = 0; b < boxes; ++b) tma_load_2d(sa + b * kABox * 128, pA32, bar, kx, a_row + b * kABox);
}

// The A rows of one stage gathered from the token rows of x: 32 warp
// instructions of 4 whole 128-byte row pieces each (lanes 8r..8r+7 take the
// 8 16-byte chunks of row 4t + r), written in the 128-byte swizzle the MMA
// descriptors read (chunk c of row i at i*128 + (c ^ (i & 7))*16).  Rows whose
// token is -1 are skipped; with `in` false every copy reads nothing and writes
// zeros.
__device__ __forceinline__ void gather_stage(uint32_t sa, const int* tok_s, const char* gx,
                                          size_t row_bytes, int col, bool in, int sub,
                                          int chunk) {
#pragma unroll 8
  for (int t = 0; t < 32; ++t) {
    const int i = 4 * t + sub;
    const int tok = tok_s[i];
    if (tok >= 0)
      cp_async16_s(sa + i * 128 + ((chunk ^ (i & 7)) << 4),
                   in ? (const void*)(gx + (size_t)tok * row_bytes + (size_t)col * 2)
                      : (const void*)gx,
                   in ? 16u : 0u);
  }
  cp_async_commit_group();
}

// EPI_COMBINEK: count this row's output slice in for its token.  Returns the
// token when this row completed the count (its slice is then summed by the
// whole warp, combine_slice), else -1.
template <int BNH>
__device__ __forceinline__ int combine_arrive(const TcArgs& a, const TileInfo& ti, size_t orow,
                                              int parts) {
  const int t = ti.shared ? (int)orow : __ldg(a.row_token + orow);
  if (!in_bounds(t >= 0 && t < a.T_tokens, a.status)) return -1;
  const int* kr = a.key_row + (size_t)t * a.k_slots;
  int expect = a.has_shared;
  for (int j = 0; j < a.k_slots; ++j) expect += __ldg(kr + j) >= 0 ? 1 : 0;
  expect *= parts;                        // each row's slice arrives in `parts` column parts
  unsigned* ctr = a.cmb_ctr + (size_t)t * a.cmb_nt + ti.n0 / BNH;
  __threadfence();                        // this row's o slice before the count
  if (atomicAdd(ctr, 1u) + 1u != (unsigned)expect) return -1;
  __threadfence();                        // every counted slice before the reads
  *ctr = 0u;                              // re-armed (the up projection also clears)
  return t;
}

// y[t][n0 .. n0+BNH) of one token, by the whole warp: lane l takes the eight
// columns from n0 + 8l on (BNH <= 256), loads the shared expert's slice and the
// token's slot rows (all loads in flight together), and accumulates in the
// fixed order os, then j = 0..k-1 -- the separate combine kernel's arithmetic.
template <int BNH>
__device__ __forceinline__ void combine_slice(const TcArgs& a, const TileInfo& ti, int t,
                                              int lane) {
  static_assert(BNH <= 256, "one 8-column chunk per lane");
  const int c = lane * 8;
  const int ncol = ti.N - ti.n0 < BNH ? ti.N - ti.n0 : BNH;
  const bool act = c < ncol;
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.out);
  const __half* os = static_cast<const __half*>(a.out_sh);   // scaled fp16 shared output
  const int* kr = a.key_row + (size_t)t * a.k_slots;
  const float* gt = a.gate + (size_t)t * a.k_slots;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (a.has_shared && act) {
    const int col = ti.n0 + c;
    const uint4 u = __ldcg(reinterpret_cast<const uint4*>(os + (size_t)t * a.ld_out_sh + col));
    const int e = a.out_sh_exp[(size_t)t * a.ld_out_sh_exp + col / kShChunk];
    sh_decode8(u, e, acc);
  }
  for (int j0 = 0; j0 < a.k_slots; j0 += 8) {
    int r[8];
    float g[8];
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u;
      r[u] = j < a.k_slots ? __ldg(kr + j) : -1;
      if (r[u] >= 0 && !in_bounds(r[u] < a.R_cap, a.status)) r[u] = -1;
      g[u] = j < a.k_slots ? __ldg(gt + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = (act && r[u] >= 0)
                 ? __ldcg(reinterpret_cast<const uint4*>(o + (size_t)r[u] * a.ld_out + ti.n0 + c))
                 : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (r[u] < 0) continue;
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        acc[2 * i] = fmaf(g[u], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(g[u], f.y, acc[2 * i + 1]);
      }
    }
  }
  if (!act) return;
  uint4 pk;
  uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    pw[i] = *reinterpret_cast<uint32_t*>(&b2);
  }
  *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.y) + (size_t)t * a.ld_y + ti.n0 + c) =
      pk;
}

// Where the A rows of routed tiles come from:
//   AS_TMA  an expert-ordered buffer (xp, h, ...) by 2-D TMA tiles;
//   AS_CP   the token rows of x, gathered by four producer warps with cp.async;
//   AS_G4   the token rows of x, gathered by TMA (tile::gather4: four rows of
//           one 128-byte column slice per instruction, one instruction per lane
//           of the producer warp).
enum { AS_TMA = 0, AS_CP = 1, AS_G4 = 2 };

// Warp roles: producer warps (one TMA warp, or four gathering warps), one MMA
// warp, four epilogue warps.
template <int AS, int EPI>
struct TcWarps {
  static constexpr int PROD = AS == AS_CP ? 4 : 1;
  static constexpr int MMA = PROD;
  static constexpr int EPI0 = PROD + 1;
  // Epilogues with an activation (SwiGLU, GELU) have two warps per TMEM lane
  // quarter (warp w reads quarter w % 4), each taking half of a tile's
  // columns: with one warp per scheduler their dependent chains (TMEM loads,
  // exponentials, stores) put them on the critical path of short tiles
  // (e4m3 decode up projection 288 -> 157 us).  The light epilogues keep one
  // warp per quarter: extra waiting warps slowed the long-tile down
  // projection (DeepSeek-V3-shaped 1.61 -> 1.75 ms).
  static constexpr int EPIW = (EPI == EPI_SWIGLU || EPI == EPI_GELU) ? 8 : 4;
  static constexpr int THREADS = (PROD + 1 + EPIW) * 32;
};

template <int BNH, bool DUAL, int EPI, int AS, bool F8 = false, int CL = 1>
__global__ void __launch_bounds__(TcWarps<AS, EPI>::THREADS, 1)
tc_grouped_gemm(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mA_sh,
                const __grid_constant__ CUtensorMap mA32, const __grid_constant__ CUtensorMap mA32_sh,
                const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
                const __grid_constant__ CUtensorMap mB0_sh,
                const __grid_constant__ CUtensorMap mB1_sh, const TcArgs a) {
  using C = TcCfg<BNH, DUAL, EPI, F8>;
  constexpr bool GATHER = AS == AS_CP;
  // CL = 2: a cluster of two CTAs takes pairs of adjacent N tiles of one M
  // tile; each CTA loads half of the A rows and multicasts them to both, so
  // the A tile crosses from L2 once per pair; the stage's empty barrier then
  // waits for both CTAs' MMAs.
  static_assert(CL == 1 || (CL == 2 && AS == AS_TMA), "clusters: TMA-fed A tiles");
  const int cl_rank = CL == 2 ? (int)(blockIdx.x & 1) : 0;
  const int item0 = CL == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int istep = CL == 2 ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  static_assert(!F8 || (EPI == EPI_SWIGLU && AS == AS_TMA), "fp8 operands: SwiGLU up projection");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * C::STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem_base = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      // gathering: the transaction arrive of the stage's warp, then its
      // second arrive once the warp's row copies have landed
      mbar_init(full_bar(s), GATHER ? 2 : 1);
      mbar_init(empty_bar(s), CL);   // the MMA commit of every CTA that reads the stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 32 * TcWarps<AS, EPI>::EPIW);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mA32);
    tma_prefetch_desc(&mB0);
    if (DUAL) tma_prefetch_desc(&mB1);
    if (a.has_shared) {
      tma_prefetch_desc(&mA_sh);
      tma_prefetch_desc(&mA32_sh);
      tma_prefetch_desc(&mB0_sh);
      if (DUAL) tma_prefetch_desc(&mB1_sh);
    }
  }
  using Wr = TcWarps<AS, EPI>;
  if (warp == Wr::MMA) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CL == 2) cluster_sync();   // both CTAs' barriers exist before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The tile schedule is copied to shared memory.  With early_b it was
  // written two launches back (the routing kernel, which completed before the
  // previous grid could start us), so it is read before the wait and the
  // producer can stream the first stages' B tiles (weights) while the
  // previous kernel finishes; everything that kernel writes (A) waits.
  Sched sc;
  int* s_tp = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES);
  auto copy_sched = [&]() {
    int* s_seg = s_tp + (kMaxE + 2);
    int* s_mt = s_seg + (kMaxE + 2);
    int* s_kept = s_mt + (kMaxE + 2);
    if (a.static_mt == 0) {
      const int nseg = a.E + a.has_shared;
      for (int i = threadIdx.x; i <= nseg; i += blockDim.x) s_tp[i] = __ldg(a.tp + i);
      for (int i = threadIdx.x; i < nseg; i += blockDim.x) s_mt[i] = __ldg(a.mtiles + i);
      for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
        s_seg[i] = __ldg(a.seg_start + i);
        s_kept[i] = __ldg(a.kept + i);
      }
    }
    __syncthreads();
    sc.tp = s_tp;
    sc.seg_start = s_seg;
    sc.mtiles = s_mt;
    sc.kept = s_kept;
  };
  auto decode = [&](int item) -> TileInfo {
    if constexpr (CL == 2) return decode_pair(a, sc, item, BNH, cl_rank);
    else return decode_tile(a, sc, item, BNH);
  };
  auto count_items = [&]() -> int {
    if (a.static_mt > 0) return a.static_total;
    if constexpr (CL == 2) return total_pairs(a, sc, BNH);
    else return sc.tp[a.E + a.has_shared];
  };
  if (a.early_b) copy_sched();
  const int total = a.static_mt > 0 ? a.static_total : (a.early_b ? count_items() : 0);
  uint32_t npre = 0;   // uses whose B tiles were issued before the wait
  if (AS == AS_TMA && a.early_b && warp == 0 && lane == 0) {
    for (int tile = item0; tile < total && npre < (uint32_t)C::STAGES; tile += istep) {
      const TileInfo ti = decode(tile);
      const int e = ti.shared ? 0 : ti.seg;
      const int nk = (ti.K + C::BK - 1) / C::BK;
      const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
      const int a_boxes = CL == 2 ? 0 : a_real_boxes(rows, a.partial_rows);
      const uint32_t a_bytes =
          CL == 2 ? (ti.m64 ? (uint32_t)C::A_BYTES / 2 : (uint32_t)C::A_BYTES)
                  : a_stage_bytes(a_boxes, C::A_BYTES);
      for (int kb = 0; kb < nk && npre < (uint32_t)C::STAGES; ++kb, ++npre) {
        const uint32_t sb = smem_base + npre * C::STAGE_BYTES + C::A_BYTES;
        mbar_arrive_expect_tx(full_bar(npre), a_bytes + C::B_BYTES);
        tma_load_3d(sb, ti.shared ? &mB0_sh : &mB0, full_bar(npre), kb * C::BKX, ti.n0, e);
        if (DUAL)
          tma_load_3d(sb + BNH * 128, ti.shared ? &mB1_sh : &mB1, full_bar(npre), kb * C::BKX,
                      ti.n0, e);
      }
    }
  }
  pdl_wait();      // everything above ran while the previous kernel finished
  pdl_trigger();
  // counters the next launch (the down projection's combine) starts from
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.zero_ctr_n;
       i += gridDim.x * blockDim.x)
    a.zero_ctr[i] = 0u;
  if (!a.early_b) copy_sched();
  const int total_all = count_items();
  (void)total;

  auto give_up = [&]() {
    atomicOr(a.status, STATUS_TIMEOUT_GEMM);
    *abort_flag = 1;
  };

  if (warp < Wr::PROD) {
    if constexpr (GATHER) {
      // ---------------- gathering producers (four warps) ----------------
      // Warp w fills the stages of uses g = w, w + 4, ...  Routed tiles: the
      // 128 A rows come straight from the token rows of x (row_token), by
      // cp.async into the 128-byte-swizzled layout the MMA descriptors
      // expect (16-byte chunk c of row i at i*128 + (c ^ (i & 7))*16); one
      // warp instruction moves 4 whole 128-byte row segments (lanes 8r..8r+7
      // take the 8 chunks of row 4t + r).  The warp waits for its copies,
      // fences them for the tensor cores (generic -> async proxy) and
      // arrives; meanwhile the other three warps fill their stages.
      // Shared-expert tiles read x through the tensor map; B always by TMA.
      uint32_t g = 0;
      bool ok = true;
      const int sub = lane >> 3, chunk = lane & 7;
      for (int tile = item0; tile < total_all && ok; tile += istep) {
        const TileInfo ti = decode(tile);
        const int nk = (ti.K + C::BK - 1) / C::BK;
        // does this warp fill any stage of the tile?
        if (nk < Wr::PROD && (int)((uint32_t)(warp - (int)(g & 3u)) & 3u) >= nk) {
          g += nk;
          continue;
        }
        const bool gat = !ti.shared;
        const CUtensorMap* pB0 = ti.shared ? &mB0_sh : &mB0;
        const CUtensorMap* pB1 = ti.shared ? &mB1_sh : &mB1;
        const int e = ti.shared ? 0 : ti.seg;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = gat ? 0 : a_real_boxes(rows, a.partial_rows);
        const uint32_t a_bytes = gat ? 0u : a_stage_bytes(a_boxes, C::A_BYTES);
        // token of every row of the tile (-1 for padding rows), per warp;
        // loaded after the warp's first B tile of the tile is in flight
        int* tok_s = reinterpret_cast<int*>(smem + C::STAGES * C::STAGE_BYTES + C::BAR_BYTES +
                                            4 * C::SCHED_INTS) + warp * 128;
        bool tok_ready = !gat;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if ((int)(g & 3u) != warp) continue;
          const int s = g % C::STAGES;
          const uint32_t ph = (g / C::STAGES) & 1u;
          int okw = 1;
          if (lane == 0)
            okw = mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, a.timeout_ns, abort_flag) ? 1 : 0;
          okw = __shfl_sync(0xffffffffu, okw, 0);
          __syncwarp();
          if (!okw) {
            if (lane == 0) give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(full_bar(s), a_bytes + C::B_BYTES);
            if (!gat)
              load_a_stage(sa, &mA_sh, &mA32_sh, full_bar(s), kb * C::BKX, ti.a_row, a_boxes);
            tma_load_3d(sb, pB0, full_bar(s), kb * C::BKX, ti.n0, e);
            if (DUAL) tma_load_3d(sb + BNH * 128, pB1, full_bar(s), kb * C::BKX, ti.n0, e);
          }
          if (!tok_ready) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = ti.a_row + lane + 32 * j;
              int tk = r < ti.row_end ? __ldg(a.row_token + r) : -1;
              if (tk >= 0 && !in_bounds(tk < a.T_x, a.status)) tk = -1;
              tok_s[lane + 32 * j] = tk;
            }
            __syncwarp();
            tok_ready = true;
          }
          if (gat) {
            const int col = kb * C::BK + chunk * 8;
            gather_stage(sa, tok_s, a.gx, a.gx_row_bytes, col, col < ti.K, sub, chunk);
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
        }
      }
      // nothing asynchronous may still target shared memory at exit: warp 0
      // waits for the release (or, after a give-up, the landing) of the last
      // use of every stage
      if (warp == 0 && lane == 0) {
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
    } else if constexpr (AS == AS_G4) {
      // ---------------- TMA row-gather producer (whole warp) ----------------
      // Routed tiles: lane l gathers rows 4l .. 4l+3 of the tile (tokens
      // row_token[a_row + 4l + i]; rows past the segment's last kept row
      // repeat the tile's first token, they feed accumulator rows that are
      // never stored) with one tile::gather4 copy per stage, into bytes
      // 512l .. 512l+511 of the 128-byte-swizzled A tile -- the layout a
      // 128-row box load produces.  Lane 0 sets the stage's transaction count
      // and issues the B tiles (and the shared expert's A tiles) first.
      uint32_t g = 0;
      bool ok = true;
      for (int tile = item0; tile < total_all && ok; tile += istep) {
        const TileInfo ti = decode(tile);
        const CUtensorMap* pB0 = ti.shared ? &mB0_sh : &mB0;
        const CUtensorMap* pB1 = ti.shared ? &mB1_sh : &mB1;
        const int e = ti.shared ? 0 : ti.seg;
        const int nk = (ti.K + C::BK - 1) / C::BK;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = a_real_boxes(rows, a.partial_rows);
        const uint32_t a_sh_bytes = a_stage_bytes(a_boxes, C::A_BYTES);
        int tk0 = 0, tk1 = 0, tk2 = 0, tk3 = 0;
        if (!ti.shared) {
          int tk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = ti.a_row + 4 * lane + i;
            int v = r < ti.row_end ? __ldg(a.row_token + r) : -1;
            if (v >= 0 && !in_bounds(v < a.T_x, a.status)) v = -1;
            tk[i] = v;
          }
          int first = __shfl_sync(0xffffffffu, tk[0], 0);   // row a_row: always kept
          if (first < 0) first = 0;
          tk0 = tk[0] < 0 ? first : tk[0];
          tk1 = tk[1] < 0 ? first : tk[1];
          tk2 = tk[2] < 0 ? first : tk[2];
          tk3 = tk[3] < 0 ? first : tk[3];
        }
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % C::STAGES;
          const uint32_t ph = (g / C::STAGES) & 1u;
          int okw = 1;
          if (lane == 0)
            okw = mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, a.timeout_ns, abort_flag) ? 1 : 0;
          okw = __shfl_sync(0xffffffffu, okw, 0);
          if (!okw) {
            if (lane == 0) give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(full_bar(s),
                                  (ti.shared ? a_sh_bytes : (uint32_t)C::A_BYTES) + C::B_BYTES);
            if (ti.shared)
              load_a_stage(sa, &mA_sh, &mA32_sh, full_bar(s), kb * C::BKX, ti.a_row, a_boxes);
            tma_load_3d(sb, pB0, full_bar(s), kb * C::BKX, ti.n0, e);
            if (DUAL) tma_load_3d(sb + BNH * 128, pB1, full_bar(s), kb * C::BKX, ti.n0, e);
          }
          __syncwarp();
          if (!ti.shared)
            tma_gather4(sa + lane * 512u, &mA, full_bar(s), kb * C::BKX, tk0, tk1, tk2, tk3);
        }
      }
      // nothing asynchronous may still target shared memory at exit
      if (lane == 0) {
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
    } else if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t g = 0;
      bool ok = true;
      for (int tile = item0; tile < total_all && ok; tile += istep) {
        const TileInfo ti = decode(tile);
        const CUtensorMap* pA = ti.shared ? &mA_sh : &mA;
        const CUtensorMap* pA32 = ti.shared ? &mA32_sh : &mA32;
        const CUtensorMap* pB0 = ti.shared ? &mB0_sh : &mB0;
        const CUtensorMap* pB1 = ti.shared ? &mB1_sh : &mB1;
        const int e = ti.shared ? 0 : ti.seg;
        const int nk = (ti.K + C::BK - 1) / C::BK;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = CL == 2 ? 0 : a_real_boxes(rows, a.partial_rows);
        const uint32_t a_bytes =
            CL == 2 ? (ti.m64 ? (uint32_t)C::A_BYTES / 2 : (uint32_t)C::A_BYTES)
                    : a_stage_bytes(a_boxes, C::A_BYTES);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % C::STAGES;
          const uint32_t ph = (g / C::STAGES) & 1u;
          const bool pre = g < npre;   // B already in flight, transaction count set
          if (!pre && !mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          if (!pre) mbar_arrive_expect_tx(full_bar(s), a_bytes + C::B_BYTES);
          if constexpr (CL == 2) {
            // this CTA's half of the A rows (one 64-row box, the map's box in
            // cluster mode) to both CTAs; an M = 64 tile needs the first half only
            if (!(ti.m64 && cl_rank == 1))
              tma_load_2d_mc(sa + cl_rank * (kTcBM / 2) * 128, pA, full_bar(s), kb * C::BKX,
                             ti.a_row + cl_rank * (kTcBM / 2), 0x3);
          } else {
            load_a_stage(sa, pA, pA32, full_bar(s), kb * C::BKX, ti.a_row, a_boxes);
          }
          if (!pre) {
            tma_load_3d(sb, pB0, full_bar(s), kb * C::BKX, ti.n0, e);
            if (DUAL) tma_load_3d(sb + BNH * 128, pB1, full_bar(s), kb * C::BKX, ti.n0, e);
          }
        }
      }
      // Tail: on the normal path wait until the MMA warp has released every
      // stage (its last commits have landed); after a give-up, wait until
      // every copy already issued has landed.  Either way nothing asynchronous
      // still targets this block's shared memory when it exits.
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
  } else if (warp == Wr::MMA) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int tile = item0; tile < total_all && ok; tile += istep) {
        const TileInfo ti = decode(tile);
        const int nk = (ti.K + C::BK - 1) / C::BK;
        const int ck = EPI == EPI_F32_CHUNKED ? kChunkKB : nk;   // k-blocks per accumulator
        for (int kb0 = 0; kb0 < nk && ok; kb0 += ck, ++it) {
          const int ab = it & 1;
          const uint32_t aph = (it >> 1) & 1;
          if (!mbar_wait_sleep_bounded(tempty_bar(ab), aph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * C::MMA_N;
          const int kb1 = kb0 + ck < nk ? kb0 + ck : nk;
          const uint32_t idesc = ti.m64 ? C::IDESC64 : C::IDESC;
          for (int kb = kb0; kb < kb1; ++kb, ++g) {
            const int s = g % C::STAGES;
            const uint32_t ph = (g / C::STAGES) & 1u;
            if (!mbar_wait_sleep_bounded(full_bar(s), ph, a.timeout_ns, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_base + s * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
              const uint64_t ad = smem_desc_k128(sa + kk * 32);
              const uint64_t bd = smem_desc_k128(sb + kk * 32);
              if constexpr (F8)
                tc_mma_f8(d_tmem, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
              else
                tc_mma_bf16(d_tmem, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
            }
            if constexpr (CL == 2)
              tc_commit_mc(empty_bar(s), 0x3);   // both CTAs' copies of the stage are free
            else
              tc_commit(empty_bar(s));
          }
          if (!ok) break;
          tc_commit(tfull_bar(ab));
        }
      }
      if (!ok) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, a.timeout_ns, nullptr);
      }
    }
  } else {
    // ---------------- epilogue (the last eight warps) ----------------
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int row_in_tile = q * 32 + lane;
    const int ew = warp - Wr::EPI0;          // 0 .. EPIW-1
    // columns of this warp: a half of the tile when the halves are whole
    // 32-column chunks, else the first warp of the quarter takes all of them
    constexpr bool kSplit = Wr::EPIW == 8 && BNH % 64 == 0;
    const int half = ew >> 2;
    const int c_lo = kSplit ? half * (BNH / 2) : 0;
    const int c_hi = kSplit ? c_lo + BNH / 2 : (half == 0 ? BNH : 0);
    const bool has_cols = c_hi > c_lo;
    if constexpr (EPI == EPI_COMBINE1) {
      // a dropped token (key_row < 0, top-1) gets y = 0: its rows are spread
      // over all epilogue warps of the grid, written while the first
      // accumulator is still being computed
      uint4* y = static_cast<uint4*>(a.y);
      const int nvec = a.ld_y * 2 / 16;
      const int gw = blockIdx.x * Wr::EPIW + ew, nw = gridDim.x * Wr::EPIW;
      for (int t = gw; t < a.T_tokens; t += nw) {
        if (__ldg(a.key_row + t) < 0)
          for (int c = lane; c < nvec; c += 32) y[(size_t)t * nvec + c] = make_uint4(0, 0, 0, 0);
      }
    }
    if constexpr (EPI == EPI_COMBINEK) {
      // tokens that no row will count in for (every slot dropped, no shared
      // expert) get y = 0
      if (!a.has_shared) {
        uint4* y = static_cast<uint4*>(a.y);
        const int nvec = a.ld_y * 2 / 16;
        const int gw = blockIdx.x * Wr::EPIW + ew, nw = gridDim.x * Wr::EPIW;
        for (int t = gw; t < a.T_tokens; t += nw) {
          bool any = false;
          for (int j = 0; j < a.k_slots; ++j) any |= __ldg(a.key_row + (size_t)t * a.k_slots + j) >= 0;
          if (!any)
            for (int c = lane; c < nvec; c += 32) y[(size_t)t * nvec + c] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    int it = 0;
    bool ok = true;
    for (int tile = item0; tile < total_all && ok; tile += istep) {
      const TileInfo ti = decode(tile);
      // M = 64: rows 16q .. 16q+15 sit in the first 16 lanes of quarter q
      const int rit = !ti.m64 ? row_in_tile : (lane < 16 ? q * 16 + lane : kTcBM);
      const size_t orow = static_cast<size_t>(ti.a_row + rit);
      bool row_ok = rit < kTcBM && ti.a_row + rit < ti.row_end;
      if (row_ok && !ti.shared && a.static_mt == 0)
        row_ok = in_bounds((int)orow < a.R_cap, a.status);
      const int nk = (ti.K + C::BK - 1) / C::BK;
      const int ck = EPI == EPI_F32_CHUNKED ? kChunkKB : nk;
      float csum[EPI == EPI_F32_CHUNKED ? BNH : 1];
      if constexpr (EPI == EPI_F32_CHUNKED) {
#pragma unroll
        for (int i = 0; i < BNH; ++i) csum[i] = 0.f;
      }
      for (int kb0 = 0; kb0 < nk; kb0 += ck, ++it) {
        const int ab = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        // sleeping waits in every role (here, the producer's and the MMA
        // issuer's): a waiting warp takes no issue slots, nor power under the
        // cap (DeepSeek-V3-shaped 5.143 -> 5.128 ms per step for the
        // epilogue's, -> 5.099 ms for all of them)
        if (!mbar_wait_sleep_bounded(tfull_bar(ab), aph, a.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * C::MMA_N;
        if constexpr (EPI == EPI_F32_CHUNKED) {
          if (has_cols) {
#pragma unroll
            for (int c = 0; c < BNH; c += 32) {
              uint32_t r0[32];
              tmem_ld32(t_row + c, r0);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) csum[c + i] += __uint_as_float(r0[i]);
            }
          }
        } else if constexpr (EPI == EPI_COMBINE1) {
          // y row of the token this expert row belongs to, scaled by its gate
          int tok = row_ok ? __ldg(a.row_token + orow) : 0;
          const bool tok_ok = row_ok && in_bounds(tok >= 0 && tok < a.T_tokens, a.status);
          if (!tok_ok) tok = 0;
          const float g = tok_ok ? __ldg(a.gate + tok) : 0.f;
          epilogue_tile<BNH, DUAL, EPI>(a, ti, t_row, (size_t)tok, tok_ok, g, c_lo, c_hi);
        } else if constexpr (F8) {
          const float rs = row_ok ? __ldg(a.a_scale + orow) : 0.f;
          epilogue_tile<BNH, DUAL, EPI, true>(a, ti, t_row, orow, row_ok, rs, c_lo, c_hi);
        } else {
          epilogue_tile<BNH, DUAL, EPI>(a, ti, t_row, orow, row_ok, 1.f, c_lo, c_hi);
        }
        tc_fence_before();
        mbar_arrive(tempty_bar(ab));
        if constexpr (EPI == EPI_COMBINEK) {
          // rows that completed their token's count; the warp sums each one's
          // slice together
          const int tl = row_ok && has_cols ? combine_arrive<BNH>(a, ti, orow, kSplit ? 2 : 1) : -1;
          const unsigned am = __activemask();
          unsigned m = __ballot_sync(am, tl >= 0);
          while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1u;
            combine_slice<BNH>(a, ti, __shfl_sync(am, tl, src), lane);
          }
        }
      }
      if constexpr (EPI == EPI_F32_CHUNKED) {
        if (ok && row_ok && has_cols) {
          float* dst = static_cast<float*>(a.out) + orow * a.ld_out + ti.n0;
#pragma unroll
          for (int i = 0; i < BNH; ++i) {
            const int col = ti.n0 + i;
            if (col < ti.N) dst[i] = csum[i] + (a.col_bias ? a.col_bias[col] : 0.f);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Wr::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  // no CTA leaves while its peer may still multicast into it or commit to
  // its barriers
  if constexpr (CL == 2) cluster_sync();
}

// ---------------------------------------------------------------- up + down in one launch
// The up and down projections of a layer as one persistent launch over one
// work list: every up tile, then every down tile, dealt to the CTAs in turn.
// A down tile reads the h rows of its M tile, which exist once every up tile
// of that M tile has stored them: each up tile, after its stores, adds one to
// the M tile's counter (release), and the producer of a down tile issues its
// weight (W2) tiles for the first stages, waits for the count (acquire,
// bounded), then issues the h rows.  So W2 streams while the up projection's
// last wave finishes, and no SM idles between the two projections.  Deadlock
// cannot arise: every CTA runs all its up tiles before its first down tile,
// and the grid holds at most one CTA per SM (all resident).  The counters sit
// in the workspace header and the last CTA to finish clears them.
template <int BNH_, bool DUAL_, int EPI_>
struct TcPhase {
  static constexpr int BNH = BNH_;
  static constexpr bool DUAL = DUAL_;
  static constexpr int EPI = EPI_;
  using C = TcCfg<BNH_, DUAL_, EPI_>;
  static constexpr int EPIW = (EPI_ == EPI_SWIGLU || EPI_ == EPI_GELU) ? 8 : 4;
  // columns of an epilogue warp: a half of the tile for the activation
  // epilogues (when the halves are whole 32-column chunks), else all of them
  // for the first warp of each TMEM quarter
  static constexpr bool SPLIT = EPIW == 8 && BNH_ % 64 == 0;
};

template <class PU, class PD, int ASU>
struct UdCfg {
  static constexpr int SB = PU::C::STAGE_BYTES > PD::C::STAGE_BYTES ? PU::C::STAGE_BYTES
                                                                    : PD::C::STAGE_BYTES;
  static constexpr int A_BYTES = kTcBM * 128;
  static constexpr int STAGES_FIT = (200 * 1024) / SB;
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  static constexpr int ACC = PU::C::MMA_N > PD::C::MMA_N ? PU::C::MMA_N : PD::C::MMA_N;
  static constexpr int TMEM_COLS = pow2_at_least(2 * ACC);
  static_assert(TMEM_COLS <= 512, "two accumulators must fit in tensor memory");
  static constexpr int PROD = ASU == AS_CP ? 4 : 1;
  static constexpr int MMA = PROD;
  static constexpr int EPI0 = PROD + 1;
  static constexpr int EPIW = PU::EPIW > PD::EPIW ? PU::EPIW : PD::EPIW;
  static constexpr int THREADS = (PROD + 1 + EPIW) * 32;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 16;
  // tp_up[E+2] | tp_dn[E+2] | seg_start[E] | mtiles[E+1] | kept[E]
  static constexpr int SCHED_INTS = 5 * (kMaxE + 2);
  static constexpr int TOK_BYTES = 4 * 128 * 4;
  static constexpr int SMEM = 1024 + STAGES * SB + BAR_BYTES + 4 * SCHED_INTS + TOK_BYTES;
};

struct UdArgs {
  unsigned* done;    // [n_done] up tiles stored per M tile (routed M tiles, then shared)
  unsigned* up_all;  // up tiles stored in all
  unsigned* fin;     // CTAs finished (the last one clears the counters and itself)
  int n_done;
  int sh_base;       // index of the shared segment's first M tile (R_cap / 128)
  int nt_up, nt_up_sh;   // up tiles per routed / shared M tile
};

__device__ __forceinline__ int ud_mtile(const TileInfo& ti, int sh_base) {
  return (ti.shared ? sh_base : 0) + ti.a_row / kTcBM;
}

__device__ __forceinline__ void ud_epi_bar(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <class PU, class PD, int ASU>
__global__ void __launch_bounds__(UdCfg<PU, PD, ASU>::THREADS, 1)
tc_updown(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mA_sh,
          const __grid_constant__ CUtensorMap mA32, const __grid_constant__ CUtensorMap mA32_sh,
          const __grid_constant__ CUtensorMap mB0, const __grid_constant__ CUtensorMap mB1,
          const __grid_constant__ CUtensorMap mB0_sh, const __grid_constant__ CUtensorMap mB1_sh,
          const __grid_constant__ CUtensorMap mH, const __grid_constant__ CUtensorMap mH_sh,
          const __grid_constant__ CUtensorMap mH32, const __grid_constant__ CUtensorMap mH32_sh,
          const __grid_constant__ CUtensorMap mW2, const __grid_constant__ CUtensorMap mW2_sh,
          const TcArgs au, const TcArgs ad, const UdArgs ud) {
  using U = UdCfg<PU, PD, ASU>;
  constexpr bool GATHER = ASU == AS_CP;
  static_assert(ASU == AS_TMA || ASU == AS_CP, "up rows: TMA or cp.async gather");
  static_assert(!PD::DUAL && (PD::EPI == EPI_OUT16 || PD::EPI == EPI_COMBINE1), "down epilogues");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + U::STAGES * U::SB);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (U::STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * U::STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * U::STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * U::STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * U::STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_stop = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const uint32_t smem_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < U::STAGES; ++s) {
      mbar_init(full_bar(s), GATHER ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 32 * U::EPIW);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *s_stop = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mA32);
    tma_prefetch_desc(&mB0);
    if (PU::DUAL) tma_prefetch_desc(&mB1);
    tma_prefetch_desc(&mH);
    tma_prefetch_desc(&mH32);
    tma_prefetch_desc(&mW2);
    if (au.has_shared) {
      tma_prefetch_desc(&mA_sh);
      tma_prefetch_desc(&mA32_sh);
      tma_prefetch_desc(&mB0_sh);
      if (PU::DUAL) tma_prefetch_desc(&mB1_sh);
      tma_prefetch_desc(&mH_sh);
      tma_prefetch_desc(&mH32_sh);
      tma_prefetch_desc(&mW2_sh);
    }
  }
  if (warp == U::MMA) {
    tmem_alloc(smem_u32(tmem_slot), U::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();     // the schedule and the routed rows come from the routing kernels
  pdl_trigger();
  // both projections' tile schedules in shared memory (the segments are the
  // same; only the tile prefixes differ)
  int* s_tpu = reinterpret_cast<int*>(smem + U::STAGES * U::SB + U::BAR_BYTES);
  int* s_tpd = s_tpu + (kMaxE + 2);
  int* s_seg = s_tpd + (kMaxE + 2);
  int* s_mt = s_seg + (kMaxE + 2);
  int* s_kept = s_mt + (kMaxE + 2);
  const int nseg = au.E + au.has_shared;
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) {
    s_tpu[i] = __ldg(au.tp + i);
    s_tpd[i] = __ldg(ad.tp + i);
  }
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) s_mt[i] = __ldg(au.mtiles + i);
  for (int i = threadIdx.x; i < au.E; i += blockDim.x) {
    s_seg[i] = __ldg(au.seg_start + i);
    s_kept[i] = __ldg(au.kept + i);
  }
  __syncthreads();
  const Sched su{s_tpu, s_seg, s_mt, s_kept};
  const Sched sd{s_tpd, s_seg, s_mt, s_kept};
  const int n_up = s_tpu[nseg];
  const int total = n_up + s_tpd[nseg];
  auto decode = [&](int item, bool& dn) -> TileInfo {
    dn = item >= n_up;
    return dn ? decode_tile(ad, sd, item - n_up, PD::BNH) : decode_tile(au, su, item, PU::BNH);
  };
  auto give_up = [&]() {
    atomicOr(au.status, STATUS_TIMEOUT_GEMM);
    *abort_flag = 1;
  };
  // have the up tiles of a down tile's M tile stored its h rows?
  auto dep_met = [&](const TileInfo& ti) {
    return ld_acquire_gpu_u32(ud.done + ud_mtile(ti, ud.sh_base)) >=
           (unsigned)(ti.shared ? ud.nt_up_sh : ud.nt_up);
  };
  auto dep_wait = [&](const TileInfo& ti) -> bool {
    if (dep_met(ti)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
      if (dep_met(ti)) return true;
      if ((i & 63u) == 0) {
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > au.timeout_ns) return false;
      }
    }
  };

  if (warp < U::PROD) {
    if constexpr (GATHER) {
      // ---------------- four producer warps (gathered up rows) ----------------
      // As in tc_grouped_gemm: warp w fills the stages of uses g = w, w + 4, ...;
      // routed up tiles gather their rows of x with cp.async, every other tile
      // (the shared expert's up tiles, all down tiles) loads A by TMA.  A down
      // stage's weight tile goes out before the warp waits for the h rows.
      uint32_t g = 0;
      bool ok = true;
      bool all_up = false;   // (lane 0's view)
      const int sub = lane >> 3, chunk = lane & 7;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        bool dn;
        const TileInfo ti = decode(item, dn);
        const int nk = (ti.K + 63) / 64;
        if (nk < U::PROD && (int)((uint32_t)(warp - (int)(g & 3u)) & 3u) >= nk) {
          g += nk;
          continue;
        }
        const TcArgs& a = dn ? ad : au;
        const bool gat = !dn && !ti.shared;
        const CUtensorMap* pA = dn ? (ti.shared ? &mH_sh : &mH) : &mA_sh;
        const CUtensorMap* pA32 = dn ? (ti.shared ? &mH32_sh : &mH32) : &mA32_sh;
        const CUtensorMap* pB0 = dn ? (ti.shared ? &mW2_sh : &mW2) : (ti.shared ? &mB0_sh : &mB0);
        const CUtensorMap* pB1 = ti.shared ? &mB1_sh : &mB1;
        const bool dual = !dn && PU::DUAL;
        const int bnh = dn ? PD::BNH : PU::BNH;
        const uint32_t b_bytes = dn ? (uint32_t)PD::C::B_BYTES : (uint32_t)PU::C::B_BYTES;
        const int e = ti.shared ? 0 : ti.seg;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = gat ? 0 : a_real_boxes(rows, a.partial_rows);
        const uint32_t a_bytes = gat ? 0u : a_stage_bytes(a_boxes, U::A_BYTES);
        int* tok_s = reinterpret_cast<int*>(smem + U::STAGES * U::SB + U::BAR_BYTES +
                                            4 * U::SCHED_INTS) + warp * 128;
        bool tok_ready = !gat;
        bool dep_ok = !dn || all_up;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if ((int)(g & 3u) != warp) continue;
          const int s = g % U::STAGES;
          const uint32_t ph = (g / U::STAGES) & 1u;
          int okw = 1;
          if (lane == 0)
            okw = mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, au.timeout_ns, abort_flag) ? 1 : 0;
          okw = __shfl_sync(0xffffffffu, okw, 0);
          __syncwarp();
          if (!okw) {
            if (lane == 0) give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * U::SB;
          const uint32_t sb = sa + U::A_BYTES;
          if (lane == 0) {
            mbar_arrive_expect_tx(full_bar(s), a_bytes + b_bytes);
            tma_load_3d(sb, pB0, full_bar(s), kb * 64, ti.n0, e);
            if (dual) tma_load_3d(sb + bnh * 128, pB1, full_bar(s), kb * 64, ti.n0, e);
            if (!gat) {
              if (!dep_ok && ld_acquire_gpu_u32(ud.up_all) >= (unsigned)n_up) {
                fence_proxy_async_global();   // every up tile is stored: no more checks
                all_up = true;
                dep_ok = true;
              }
              if (!dep_ok) {
                // on a give-up the rows are loaded all the same (the call's
                // status reports the timeout), so that every issued stage completes
                if (!dep_wait(ti)) give_up();
                fence_proxy_async_global();
                dep_ok = true;
              }
              load_a_stage(sa, pA, pA32, full_bar(s), kb * 64, ti.a_row, a_boxes);
            }
          }
          if (!tok_ready) {
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = ti.a_row + lane + 32 * j;
              int tk = r < ti.row_end ? __ldg(au.row_token + r) : -1;
              if (tk >= 0 && !in_bounds(tk < au.T_x, au.status)) tk = -1;
              tok_s[lane + 32 * j] = tk;
            }
            __syncwarp();
            tok_ready = true;
          }
          if (gat) {
            const int col = kb * 64 + chunk * 8;
            gather_stage(sa, tok_s, au.gx, au.gx_row_bytes, col, col < ti.K, sub, chunk);
            cp_async_wait_group<0>();
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(s));
        }
      }
      if (warp == 0 && lane == 0) {
        for (int s = 0; s < U::STAGES; ++s) {
          if (g > static_cast<uint32_t>(s)) {
            const uint32_t issues = (g - 1 - s) / U::STAGES + 1;
            if (ok)
              mbar_wait_bounded(empty_bar(s), (issues - 1) & 1u, au.timeout_ns, abort_flag);
            else
              mbar_wait_bounded(full_bar(s), (issues - 1) & 1u, au.timeout_ns, nullptr);
          }
        }
      }
    } else if (lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t g = 0;   // stage uses issued
      bool ok = true;
      bool all_up = false;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        bool dn;
        const TileInfo ti = decode(item, dn);
        const TcArgs& a = dn ? ad : au;
        const CUtensorMap* pA = dn ? (ti.shared ? &mH_sh : &mH) : (ti.shared ? &mA_sh : &mA);
        const CUtensorMap* pA32 =
            dn ? (ti.shared ? &mH32_sh : &mH32) : (ti.shared ? &mA32_sh : &mA32);
        const CUtensorMap* pB0 = dn ? (ti.shared ? &mW2_sh : &mW2) : (ti.shared ? &mB0_sh : &mB0);
        const CUtensorMap* pB1 = ti.shared ? &mB1_sh : &mB1;
        const bool dual = !dn && PU::DUAL;
        const int bnh = dn ? PD::BNH : PU::BNH;
        const uint32_t b_bytes = dn ? (uint32_t)PD::C::B_BYTES : (uint32_t)PU::C::B_BYTES;
        const int e = ti.shared ? 0 : ti.seg;
        const int nk = (ti.K + 63) / 64;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = a_real_boxes(rows, a.partial_rows);
        const uint32_t a_bytes = a_stage_bytes(a_boxes, U::A_BYTES);
        int kb = 0;
        if (dn && !all_up) {
          // once every up tile is stored (observed through an acquire, then one
          // proxy fence), no down tile needs its own check
          if (ld_acquire_gpu_u32(ud.up_all) >= (unsigned)n_up) {
            fence_proxy_async_global();
            all_up = true;
          }
        }
        if (dn && !all_up) {
          if (!dep_met(ti)) {
            // the h rows are not all stored yet: the weight tiles of the first
            // stages go out now, their h rows after the wait (loaded even on a
            // give-up, so that every issued stage completes; the call's status
            // then reports the timeout)
            int nb = 0;
            for (; nb < nk && nb < U::STAGES; ++nb) {
              const uint32_t gg = g + nb;
              const int s = gg % U::STAGES;
              const uint32_t ph = (gg / U::STAGES) & 1u;
              if (!mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, au.timeout_ns, abort_flag)) {
                give_up();
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(full_bar(s), a_bytes + b_bytes);
              tma_load_3d(smem_base + s * U::SB + U::A_BYTES, pB0, full_bar(s), nb * 64, ti.n0, e);
            }
            if (ok && !dep_wait(ti)) give_up();
            fence_proxy_async_global();
            for (int j = 0; j < nb; ++j) {
              const int s = (g + j) % U::STAGES;
              load_a_stage(smem_base + s * U::SB, pA, pA32, full_bar(s), j * 64, ti.a_row, a_boxes);
            }
            kb = nb;
            if (!ok) {
              g += nb;
              break;
            }
          } else {
            fence_proxy_async_global();   // the count was observed through an acquire
          }
        }
        for (; kb < nk; ++kb) {
          const uint32_t gg = g + kb;
          const int s = gg % U::STAGES;
          const uint32_t ph = (gg / U::STAGES) & 1u;
          if (!mbar_wait_sleep_bounded(empty_bar(s), ph ^ 1u, au.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + s * U::SB;
          const uint32_t sb = sa + U::A_BYTES;
          mbar_arrive_expect_tx(full_bar(s), a_bytes + b_bytes);
          load_a_stage(sa, pA, pA32, full_bar(s), kb * 64, ti.a_row, a_boxes);
          tma_load_3d(sb, pB0, full_bar(s), kb * 64, ti.n0, e);
          if (dual) tma_load_3d(sb + bnh * 128, pB1, full_bar(s), kb * 64, ti.n0, e);
        }
        g += kb;
      }
      // nothing asynchronous may still target shared memory at exit
      for (int s = 0; s < U::STAGES; ++s) {
        if (g > static_cast<uint32_t>(s)) {
          const uint32_t issues = (g - 1 - s) / U::STAGES + 1;
          if (ok)
            mbar_wait_bounded(empty_bar(s), (issues - 1) & 1u, au.timeout_ns, abort_flag);
          else
            mbar_wait_bounded(full_bar(s), (issues - 1) & 1u, au.timeout_ns, nullptr);
        }
      }
    }
  } else if (warp == U::MMA) {
    if (lane == 0) {
      // ---------------- MMA issuer: one accumulator per tile ----------------
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++it) {
        bool dn;
        const TileInfo ti = decode(item, dn);
        const int nk = (ti.K + 63) / 64;
        const int ab = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_sleep_bounded(tempty_bar(ab), aph ^ 1u, au.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * U::ACC;
        const uint32_t idesc = dn ? (ti.m64 ? PD::C::IDESC64 : PD::C::IDESC)
                                  : (ti.m64 ? PU::C::IDESC64 : PU::C::IDESC);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % U::STAGES;
          const uint32_t ph = (g / U::STAGES) & 1u;
          if (!mbar_wait_sleep_bounded(full_bar(s), ph, au.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + s * U::SB;
          const uint32_t sb = sa + U::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d_tmem, smem_desc_k128(sa + kk * 32), smem_desc_k128(sb + kk * 32), idesc,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          tc_commit(empty_bar(s));
        }
        if (!ok) break;
        tc_commit(tfull_bar(ab));
      }
      if (!ok) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, au.timeout_ns, nullptr);
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    const int ew = warp - U::EPI0;
    const int ep_tid = ew * 32 + lane;
    const int half = ew >> 2;
    const int cu_lo = PU::SPLIT ? half * (PU::BNH / 2) : 0;
    const int cu_hi = PU::SPLIT ? cu_lo + PU::BNH / 2 : (half == 0 ? PU::BNH : 0);
    const int cd_lo = PD::SPLIT ? half * (PD::BNH / 2) : 0;
    const int cd_hi = PD::SPLIT ? cd_lo + PD::BNH / 2 : (half == 0 ? PD::BNH : 0);
    if constexpr (PD::EPI == EPI_COMBINE1) {
      // a dropped token (key_row < 0, top-1) gets y = 0
      uint4* y = static_cast<uint4*>(ad.y);
      const int nvec = ad.ld_y * 2 / 16;
      const int gw = blockIdx.x * U::EPIW + ew, nw = gridDim.x * U::EPIW;
      for (int t = gw; t < ad.T_tokens; t += nw) {
        if (__ldg(ad.key_row + t) < 0)
          for (int c = lane; c < nvec; c += 32) y[(size_t)t * nvec + c] = make_uint4(0, 0, 0, 0);
      }
    }
    int it = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++it) {
      bool dn;
      const TileInfo ti = decode(item, dn);
      const TcArgs& a = dn ? ad : au;
      const int rit = !ti.m64 ? row_in_tile : (lane < 16 ? q * 16 + lane : kTcBM);
      const size_t orow = static_cast<size_t>(ti.a_row + rit);
      bool row_ok = rit < kTcBM && ti.a_row + rit < ti.row_end;
      if (row_ok && !ti.shared) row_ok = in_bounds((int)orow < a.R_cap, a.status);
      const int ab = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      bool ok = mbar_wait_sleep_bounded(tfull_bar(ab), aph, au.timeout_ns, abort_flag);
      if (!ok) give_up();
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * U::ACC;
      if (ok) {
        if (dn) {
          if constexpr (PD::EPI == EPI_COMBINE1) {
            int tok = row_ok ? __ldg(ad.row_token + orow) : 0;
            const bool tok_ok = row_ok && in_bounds(tok >= 0 && tok < ad.T_tokens, ad.status);
            if (!tok_ok) tok = 0;
            const float gt = tok_ok ? __ldg(ad.gate + tok) : 0.f;
            epilogue_tile<PD::BNH, false, PD::EPI>(ad, ti, t_row, (size_t)tok, tok_ok, gt, cd_lo,
                                                   cd_hi);
          } else {
            epilogue_tile<PD::BNH, false, PD::EPI>(ad, ti, t_row, orow, row_ok, 1.f, cd_lo, cd_hi);
          }
        } else {
          epilogue_tile<PU::BNH, PU::DUAL, PU::EPI>(au, ti, t_row, orow, row_ok, 1.f, cu_lo,
                                                    cu_hi);
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(ab));
      if (!dn) {
        // this up tile's h rows are stored: count them in for their M tile
        // (every epilogue thread's stores, then one release); all epilogue
        // threads stop together if any role gave up
        __threadfence();
        ud_epi_bar(32 * U::EPIW);
        if (ep_tid == 0) {
          if (*abort_flag == 0) {
            red_add_release_gpu(ud.done + ud_mtile(ti, ud.sh_base), 1u);
            red_add_release_gpu(ud.up_all, 1u);
          }
          *s_stop = *abort_flag;
        }
        ud_epi_bar(32 * U::EPIW);
        if (*s_stop) break;
      } else if (!ok) {
        break;   // down tiles have no barriers: leave at once
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == U::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, U::TMEM_COLS);
  }
  // the last CTA to finish clears the counters for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ud.fin, 1u) == gridDim.x - 1u) {
      for (int i = 0; i < ud.n_done; ++i) ud.done[i] = 0u;
      *ud.up_all = 0u;
      __threadfence();
      *ud.fin = 0u;
    }
  }
}

// ---------------------------------------------------------------- down projection, e4m3 weights
// o = h W2^T with W2 stored as e4m3 codes and one float32 scale per output
// channel (W2[e][n][c] = W2s[e][n] * e4m3(W2q[e][n][c])).  The tensor cores
// take no bf16 x e4m3 product, and quantising h would add rounding decisions
// on activations, so the codes are expanded to bf16 on chip -- exactly: every
// e4m3 value is a bf16 value -- and the product runs as the bf16 kernel's,
// the channel scale multiplying the float32 accumulator in the epilogue.  The
// weights then stream at one byte each.
//
// Three rings per CTA, each with its own depth: the codes (64 bytes per
// weight row and K block, no swizzle; loaded by the code producer, the only
// HBM stream that matters, so the deepest ring and issued ahead of the
// previous kernel's end), the h rows (bf16, 128-byte swizzle; loaded by the
// A producer, mostly L2 hits) and the expanded bf16 weight tiles (written by
// four converter warps in the layout the MMA descriptors read).  A code
// stage is freed as soon as the converters have read it, so the code ring
// does not wait for the tensor cores; the MMA's commits free the A and bf16
// stages.
template <int BNH, int EPI>
struct F8wCfg {
  static constexpr int A_BYTES = kTcBM * 128;
  static constexpr int B_BYTES = BNH * 128;       // expanded weights, bf16
  static constexpr int R_BYTES = BNH * 64;        // codes
  static constexpr int AST = 4;
  static constexpr int BST = 2;
  static constexpr int RING_BUDGET = 208 * 1024;
  static constexpr int CST_FIT = (RING_BUDGET - AST * A_BYTES - BST * B_BYTES) / R_BYTES;
  static constexpr int CST = CST_FIT > 12 ? 12 : CST_FIT;
  static constexpr int R_OFF = 0;
  static constexpr int A_OFF = CST * R_BYTES;
  static constexpr int B_OFF = A_OFF + AST * A_BYTES;
  static constexpr int RING_BYTES = B_OFF + BST * B_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BNH);
  static constexpr int EPIW = 4;
  static constexpr int CONVW = 4;
  static constexpr int EPI0 = 2;
  static constexpr int CONV0 = EPI0 + EPIW;
  static constexpr int APROD = CONV0 + CONVW;     // the A producer's warp
  static constexpr int THREADS = (APROD + 1) * 32;
  static constexpr int NBARS = 2 * (CST + AST + BST) + 5;
  static constexpr int BAR_BYTES = 8 * NBARS + 16;
  static constexpr int SCHED_INTS = 4 * (kMaxE + 2);
  static constexpr int SMEM = 1024 + RING_BYTES + BAR_BYTES + 4 * SCHED_INTS;
  static constexpr uint32_t IDESC = idesc_bf16_f32(kTcBM, BNH);
  static constexpr uint32_t IDESC64 = idesc_bf16_f32(64, BNH);
  static_assert(BNH % 32 == 0 && BNH <= 256, "tile width");
  static_assert(CST >= 4, "code ring depth");
  static_assert(R_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0,
                "swizzled tiles start on 1024-byte boundaries");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Four e4m3 codes (one 32-bit word, lowest byte first) as two bf16 pairs
// (codes 0, 1 and codes 2, 3; lower code in the lower half), exactly, on the
// integer and FMA pipes.  A byte permute spreads each code into its own
// sign-extended 16-bit half; shifted left by 4 and masked, the half keeps the
// sign in bit 15 and the code's 4 exponent and 3 mantissa bits in bits 10..4:
// the bf16 whose value is the code's value times 2^-120 (the bf16 exponent is
// the e4m3 one, bias 127 instead of 7; an e4m3 subnormal, exponent 0, lands
// on the bf16 subnormal of the same mantissa).  One bf16 multiply by 2^120
// (exact: every e4m3 value is a normal bf16 value) gives the value.  The NaN
// codes 0x7F / 0xFF come out as +-480.
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
  uint32_t lo, hi;
  asm("prmt.b32 %0, %1, 0, 0x9180;" : "=r"(lo) : "r"(w));   // s(c1) c1 s(c0) c0
  asm("prmt.b32 %0, %1, 0, 0xB3A2;" : "=r"(hi) : "r"(w));   // s(c3) c3 s(c2) c2
  lo = (lo << 4) & 0x87F087F0u;
  hi = (hi << 4) & 0x87F087F0u;
  uint2 r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r.x) : "r"(lo), "r"(0x7B807B80u), "r"(0x80008000u));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r.y) : "r"(hi), "r"(0x7B807B80u), "r"(0x80008000u));
  return r;
}

// Epilogue of the e4m3-weight down projection: the accumulator times the
// output channel's scale, then as epilogue_tile (bf16 o rows, or the top-1
// combine y = bf16(g * value)).
template <int BNH, int EPI>
__device__ __forceinline__ void epilogue_tile_f8w(const TcArgs& a, const TileInfo& ti,
                                                  uint32_t t_row, size_t orow, bool row_ok,
                                                  float gate, int c_lo, int c_hi) {
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 32) {
    uint32_t r0[32];
    tmem_ld32(t_row + c, r0);
    tmem_ld_wait();
    const int col = ti.n0 + c;
    __nv_bfloat16* out =
        static_cast<__nv_bfloat16*>(EPI == EPI_COMBINE1 ? a.y : a.out);
    const int ld = EPI == EPI_COMBINE1 ? a.ld_y : a.ld_out;
    __nv_bfloat16* dst = out + orow * ld + col;
    const float* cs = a.b0_scale + (size_t)ti.seg * a.N;
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int cc = col + 2 * i;
      const float s0 = cc < ti.N ? __ldg(cs + cc) : 0.f;
      const float s1 = cc + 1 < ti.N ? __ldg(cs + cc + 1) : 0.f;
      float v0 = __uint_as_float(r0[2 * i]) * s0, v1 = __uint_as_float(r0[2 * i + 1]) * s1;
      if (EPI == EPI_COMBINE1) {
        v0 = fmaf(gate, v0, 0.f);
        v1 = fmaf(gate, v1, 0.f);
      }
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v0, v1);
      pk[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    if (!row_ok) {
    } else if (col + 32 <= ti.N) {
#pragma unroll
      for (int v = 0; v < 4; ++v)
        reinterpret_cast<uint4*>(dst)[v] =
            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (col + i < ti.N) {
          const uint32_t w = pk[i >> 1];
          reinterpret_cast<uint16_t*>(dst)[i] =
              (i & 1) ? static_cast<uint16_t>(w >> 16) : static_cast<uint16_t>(w);
        }
      }
    }
  }
}

template <int BNH, int EPI>
__global__ void __launch_bounds__(F8wCfg<BNH, EPI>::THREADS, 1)
tc_down_f8w(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mA32,
            const __grid_constant__ CUtensorMap mW, const TcArgs a) {
  using C = F8wCfg<BNH, EPI>;
  static_assert(EPI == EPI_OUT16 || EPI == EPI_COMBINE1, "down epilogues");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  // barriers: codes full / empty, A full / empty, bf16 tiles full / empty,
  // accumulators full / empty, drain
  auto cfull = [&](int s) { return bar0 + 8u * s; };
  auto cempty = [&](int s) { return bar0 + 8u * (C::CST + s); };
  auto afull = [&](int s) { return bar0 + 8u * (2 * C::CST + s); };
  auto aempty = [&](int s) { return bar0 + 8u * (2 * C::CST + C::AST + s); };
  auto bfull = [&](int s) { return bar0 + 8u * (2 * (C::CST + C::AST) + s); };
  auto bempty = [&](int s) { return bar0 + 8u * (2 * (C::CST + C::AST) + C::BST + s); };
  const uint32_t tb0 = bar0 + 8u * (2 * (C::CST + C::AST + C::BST));
  auto tfull_bar = [&](int b) { return tb0 + 8u * b; };
  auto tempty_bar = [&](int b) { return tb0 + 8u * (2 + b); };
  const uint32_t drain_bar = tb0 + 8u * 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto stage_r = [&](int s) { return smem_base + C::R_OFF + s * C::R_BYTES; };
  auto stage_a = [&](int s) { return smem_base + C::A_OFF + s * C::A_BYTES; };
  auto stage_b = [&](int s) { return smem_base + C::B_OFF + s * C::B_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::CST; ++s) {
      mbar_init(cfull(s), 1);
      mbar_init(cempty(s), C::CONVW);
    }
    for (int s = 0; s < C::AST; ++s) {
      mbar_init(afull(s), 1);
      mbar_init(aempty(s), 1);
    }
    for (int s = 0; s < C::BST; ++s) {
      mbar_init(bfull(s), C::CONVW);
      mbar_init(bempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 32 * C::EPIW);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mA32);
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
  // The tile schedule was written by the routing kernel, two launches back
  // (complete before the previous grid could start this one): it is read
  // before the wait, and the code producer streams the first stages' codes
  // meanwhile; h (written by the previous kernel) waits.
  int* s_tp = reinterpret_cast<int*>(smem + C::RING_BYTES + C::BAR_BYTES);
  int* s_seg = s_tp + (kMaxE + 2);
  int* s_mt = s_seg + (kMaxE + 2);
  int* s_kept = s_mt + (kMaxE + 2);
  // The prefix counts sched_bn-wide column tiles per M tile, the same number
  // for every segment (no shared segment on this path), so the prefix of this
  // kernel's BNH-wide tiles is (tp / nt_sched) * nt.
  const int nseg = a.E;
  const int nt_sched = (a.N + a.sched_bn - 1) / a.sched_bn;
  const int nt = (a.N + BNH - 1) / BNH;
  for (int i = threadIdx.x; i <= nseg; i += blockDim.x) s_tp[i] = (__ldg(a.tp + i) / nt_sched) * nt;
  for (int i = threadIdx.x; i < nseg; i += blockDim.x) s_mt[i] = __ldg(a.mtiles + i);
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
    s_seg[i] = __ldg(a.seg_start + i);
    s_kept[i] = __ldg(a.kept + i);
  }
  __syncthreads();
  const Sched sc{s_tp, s_seg, s_mt, s_kept};
  const int total = s_tp[nseg];
  auto give_up = [&]() {
    atomicOr(a.status, STATUS_TIMEOUT_GEMM);
    *abort_flag = 1;
  };
  // Waits until every load this thread issued into a ring has landed: on the
  // consumers' release of each stage's last use when all went well, else on
  // the load itself.
  auto drain_ring = [&](uint32_t issued, int depth, auto full, auto empty, bool ok) {
    for (int s = 0; s < depth; ++s) {
      if (issued > static_cast<uint32_t>(s)) {
        const uint32_t uses = (issued - 1 - s) / depth + 1;
        if (ok)
          mbar_wait_sleep_bounded(empty(s), (uses - 1) & 1u, a.timeout_ns, abort_flag);
        else
          mbar_wait_bounded(full(s), (uses - 1) & 1u, a.timeout_ns, nullptr);
      }
    }
  };
  uint32_t npre = 0;   // code stages issued before the wait
  if (warp == 0 && lane == 0) {
    for (int tile = blockIdx.x; tile < total && npre < (uint32_t)C::CST; tile += gridDim.x) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int nk = (ti.K + 63) / 64;
      for (int kb = 0; kb < nk && npre < (uint32_t)C::CST; ++kb, ++npre) {
        mbar_arrive_expect_tx(cfull(npre), C::R_BYTES);
        tma_load_3d(stage_r(npre), &mW, cfull(npre), kb * 32, ti.n0, ti.seg);
      }
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- code producer ----------------
      uint32_t g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(a, sc, tile, BNH);
        const int nk = (ti.K + 63) / 64;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          if (g < npre) continue;   // in flight since the prologue
          const int s = g % C::CST;
          const uint32_t ph = (g / C::CST) & 1u;
          if (!mbar_wait_sleep_bounded(cempty(s), ph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(cfull(s), C::R_BYTES);
          tma_load_3d(stage_r(s), &mW, cfull(s), kb * 32, ti.n0, ti.seg);
        }
      }
      drain_ring(g, C::CST, cfull, cempty, ok);
    }
  } else if (warp == C::APROD) {
    if (lane == 0) {
      // ---------------- A (h rows) producer ----------------
      uint32_t g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(a, sc, tile, BNH);
        const int nk = (ti.K + 63) / 64;
        const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
        const int a_boxes = a_real_boxes(rows, a.partial_rows);
        const uint32_t a_bytes = a_stage_bytes(a_boxes, C::A_BYTES);
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % C::AST;
          const uint32_t ph = (g / C::AST) & 1u;
          if (!mbar_wait_sleep_bounded(aempty(s), ph ^ 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(afull(s), a_bytes);
          load_a_stage(stage_a(s), &mA, &mA32, afull(s), kb * 64, ti.a_row, a_boxes);
        }
      }
      drain_ring(g, C::AST, afull, aempty, ok);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
        const TileInfo ti = decode_tile(a, sc, tile, BNH);
        const int nk = (ti.K + 63) / 64;
        const int ab = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_sleep_bounded(tempty_bar(ab), aph ^ 1u, a.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * BNH;
        const uint32_t idesc = ti.m64 ? C::IDESC64 : C::IDESC;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int sa = g % C::AST, sb = g % C::BST;
          // the stage's h rows have landed and its weights are expanded
          if (!mbar_wait_sleep_bounded(afull(sa), (g / C::AST) & 1u, a.timeout_ns, abort_flag) ||
              !mbar_wait_sleep_bounded(bfull(sb), (g / C::BST) & 1u, a.timeout_ns, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_bf16(d_tmem, smem_desc_k128(stage_a(sa) + kk * 32),
                        smem_desc_k128(stage_b(sb) + kk * 32), idesc,
                        (kb != 0 || kk != 0) ? 1u : 0u);
          tc_commit(aempty(sa));
          tc_commit(bempty(sb));
        }
        if (!ok) break;
        tc_commit(tfull_bar(ab));
      }
      if (!ok) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, a.timeout_ns, nullptr);
      }
    }
  } else if (warp >= C::CONV0) {
    // ---------------- converter warps ----------------
    // item i of a stage: weight row i / 8, 16-byte chunk i % 8 of its bf16
    // row (eight codes); the bf16 tile is written in the 128-byte swizzle
    // (chunk c of row n at n*128 + (c ^ (n & 7))*16)
    const int ct = (warp - C::CONV0) * 32 + lane;
    uint32_t g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int nk = (ti.K + 63) / 64;
      for (int kb = 0; kb < nk; ++kb, ++g) {
        const int sr = g % C::CST, sb = g % C::BST;
        // every lane waits (it reads what the TMA wrote and overwrites what
        // the tensor cores read)
        const bool okl =
            mbar_wait_sleep_bounded(cfull(sr), (g / C::CST) & 1u, a.timeout_ns, abort_flag) &&
            mbar_wait_sleep_bounded(bempty(sb), ((g / C::BST) & 1u) ^ 1u, a.timeout_ns,
                                    abort_flag);
        if (!__all_sync(0xffffffffu, okl)) {
          if (lane == 0) give_up();
          ok = false;
          break;
        }
        const uint32_t raw = stage_r(sr);
        const uint32_t bt = stage_b(sb);
        constexpr int PER = (BNH * 8) / (C::CONVW * 32);
        static_assert(PER * C::CONVW * 32 == BNH * 8, "items per converter thread");
        uint2 codes[PER];
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int i = ct + j * 32 * C::CONVW;
          codes[j] = lds_u2(raw + (i >> 3) * 64 + (i & 7) * 8);
        }
        // the codes are in registers: the code stage can be refilled
        __syncwarp();
        if (lane == 0) mbar_arrive(cempty(sr));
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const int i = ct + j * 32 * C::CONVW;
          const int n = i >> 3, c = i & 7;
          const uint2 b01 = e4m3x4_to_bf16x4(codes[j].x), b23 = e4m3x4_to_bf16x4(codes[j].y);
          sts_u4(bt + n * 128 + ((c ^ (n & 7)) << 4), make_uint4(b01.x, b01.y, b23.x, b23.y));
        }
        fence_proxy_async_smem();   // the tensor cores read what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(bfull(sb));
      }
    }
  } else {
    // ---------------- epilogue (four warps, one per TMEM lane quarter) ----------------
    const int q = warp & 3;
    const int row_in_tile = q * 32 + lane;
    if constexpr (EPI == EPI_COMBINE1) {
      // a dropped token (key_row < 0, top-1) gets y = 0
      uint4* y = static_cast<uint4*>(a.y);
      const int nvec = a.ld_y * 2 / 16;
      const int gw = blockIdx.x * C::EPIW + (warp - C::EPI0), nw = gridDim.x * C::EPIW;
      for (int t = gw; t < a.T_tokens; t += nw) {
        if (__ldg(a.key_row + t) < 0)
          for (int c = lane; c < nvec; c += 32) y[(size_t)t * nvec + c] = make_uint4(0, 0, 0, 0);
      }
    }
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int rit = !ti.m64 ? row_in_tile : (lane < 16 ? q * 16 + lane : kTcBM);
      const size_t orow = static_cast<size_t>(ti.a_row + rit);
      bool row_ok = rit < kTcBM && ti.a_row + rit < ti.row_end;
      if (row_ok) row_ok = in_bounds((int)orow < a.R_cap, a.status);
      const int ab = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!mbar_wait_sleep_bounded(tfull_bar(ab), aph, a.timeout_ns, abort_flag)) {
        give_up();
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * BNH;
      if constexpr (EPI == EPI_COMBINE1) {
        int tok = row_ok ? __ldg(a.row_token + orow) : 0;
        const bool tok_ok = row_ok && in_bounds(tok >= 0 && tok < a.T_tokens, a.status);
        if (!tok_ok) tok = 0;
        const float gt = tok_ok ? __ldg(a.gate + tok) : 0.f;
        epilogue_tile_f8w<BNH, EPI>(a, ti, t_row, (size_t)tok, tok_ok, gt, 0, BNH);
      } else {
        epilogue_tile_f8w<BNH, EPI>(a, ti, t_row, orow, row_ok, 1.f, 0, BNH);
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(ab));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- e4m3 down weights, weights as M
// The same product for decode-sized segments, with the operands swapped:
// o^T = W2 h^T, the 128 output channels of a tile as the MMA's M and the
// segment's token rows as its N (32 per pass).  An expert segment of a decode
// batch holds a few rows, so the weights-as-B form multiplies M = 64 rows, one
// or two of them real, against every channel; here the tensor work per stage
// shrinks by the row ratio, and the h rows of a stage (two 32-row boxes, 8 KB)
// travel in the same stage as its codes (128 rows of 128 bytes: whole DRAM
// lines, 16 KB), so they are requested as early as the codes are.  One ring
// of code + h stages (the producer's), a ring of expanded bf16 weight tiles
// (two 64-wide panels per stage, the converters'), two 32-column
// accumulators.
// A stage is free once the converters have read its codes and the MMAs that
// read its h rows have completed.  Segments of more than 32 rows take one
// pass per 32 rows, each re-streaming the tile's weights: the plan uses this
// kernel where segments average at most one row in eight.
constexpr int kSwN = 32;   // token rows per pass (the MMA's N)
template <int EPI>
struct F8sCfg {
  static constexpr int BNH = 128;                   // output channels per tile (the MMA's M)
  static constexpr int KB = 128;                    // K per stage: whole 128-byte code rows
  static constexpr int PANEL = 64;                  // K per 128-byte bf16 panel
  static constexpr int R_BYTES = BNH * KB;          // codes of one K block
  static constexpr int H_PANEL = kSwN * 128;        // h rows of one panel (a 32-row box)
  static constexpr int H_BYTES = 2 * H_PANEL;
  static constexpr int STAGE_BYTES = R_BYTES + H_BYTES;
  static constexpr int W_PANEL = BNH * 128;         // expanded bf16 weights of one panel
  static constexpr int W_BYTES = 2 * W_PANEL;
  static constexpr int WST = 2;
  static constexpr int RING_BUDGET = 208 * 1024;
  static constexpr int ST_FIT = (RING_BUDGET - WST * W_BYTES) / STAGE_BYTES;
  static constexpr int ST = ST_FIT > 16 ? 16 : ST_FIT;
  static constexpr int W_OFF = ST * STAGE_BYTES;
  static constexpr int RING_BYTES = W_OFF + WST * W_BYTES;
  static constexpr int TMEM_COLS = 2 * kSwN;        // two accumulators of kSwN columns
  static constexpr int EPIW = 4;
  static constexpr int CONVW = 4;
  static constexpr int EPI0 = 2;
  static constexpr int CONV0 = EPI0 + EPIW;
  static constexpr int THREADS = (CONV0 + CONVW) * 32;
  static constexpr int NBARS = 2 * (ST + WST) + 5;
  static constexpr int BAR_BYTES = 8 * NBARS + 16;
  static constexpr int SCHED_INTS = 4 * (kMaxE + 2);
  static constexpr int SMEM = 1024 + RING_BYTES + BAR_BYTES + 4 * SCHED_INTS;
  static constexpr uint32_t IDESC = idesc_bf16_f32(BNH, kSwN);
  static_assert(R_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0,
                "swizzled tiles start on 1024-byte boundaries");
  static_assert(ST >= 5, "stage ring depth");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int EPI>
__global__ void __launch_bounds__(F8sCfg<EPI>::THREADS, 1)
tc_down_f8s(const __grid_constant__ CUtensorMap mA32, const __grid_constant__ CUtensorMap mW,
            const TcArgs a) {
  using C = F8sCfg<EPI>;
  static_assert(EPI == EPI_OUT16 || EPI == EPI_COMBINE1, "down epilogues");
  constexpr int BNH = C::BNH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  // barriers: stages full / empty, bf16 weight tiles full / empty,
  // accumulators full / empty, drain
  auto sfull = [&](int s) { return bar0 + 8u * s; };
  auto sempty = [&](int s) { return bar0 + 8u * (C::ST + s); };
  auto wfull = [&](int s) { return bar0 + 8u * (2 * C::ST + s); };
  auto wempty = [&](int s) { return bar0 + 8u * (2 * C::ST + C::WST + s); };
  const uint32_t tb0 = bar0 + 8u * (2 * (C::ST + C::WST));
  auto tfull_bar = [&](int b) { return tb0 + 8u * b; };
  auto tempty_bar = [&](int b) { return tb0 + 8u * (2 + b); };
  const uint32_t drain_bar = tb0 + 8u * 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t smem_base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto stage_r = [&](int s) { return smem_base + s * C::STAGE_BYTES; };
  auto stage_h = [&](int s) { return smem_base + s * C::STAGE_BYTES + C::R_BYTES; };
  auto stage_w = [&](int s) { return smem_base + C::W_OFF + s * C::W_BYTES; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(sfull(s), 1);
      mbar_init(sempty(s), C::CONVW + 1);   // the converters' reads and the MMAs' commit
    }
    for (int s = 0; s < C::WST; ++s) {
      mbar_init(wfull(s), C::CONVW);
      mbar_init(wempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 32 * C::EPIW);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA32);
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
  // The tile schedule (written by the routing kernel, two launches back) is
  // read before the wait.  Its prefix counts sched_bn-wide column tiles per
  // M tile; every routed segment has the same count, so the prefix of this
  // kernel's 128-wide tiles is (tp / nt_sched) * nt.
  int* s_tp = reinterpret_cast<int*>(smem + C::RING_BYTES + C::BAR_BYTES);
  int* s_seg = s_tp + (kMaxE + 2);
  int* s_mt = s_seg + (kMaxE + 2);
  int* s_kept = s_mt + (kMaxE + 2);
  const int nt_sched = (a.N + a.sched_bn - 1) / a.sched_bn;
  const int nt = (a.N + BNH - 1) / BNH;
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_tp[i] = (__ldg(a.tp + i) / nt_sched) * nt;
  for (int i = threadIdx.x; i < a.E; i += blockDim.x) {
    s_mt[i] = __ldg(a.mtiles + i);
    s_seg[i] = __ldg(a.seg_start + i);
    s_kept[i] = __ldg(a.kept + i);
  }
  __syncthreads();
  const Sched sc{s_tp, s_seg, s_mt, s_kept};
  const int total = s_tp[a.E];
  auto give_up = [&]() {
    atomicOr(a.status, STATUS_TIMEOUT_GEMM);
    *abort_flag = 1;
  };
  // passes (32-row groups) of a tile
  auto passes_of = [&](const TileInfo& ti) {
    const int rows = ti.row_end - ti.a_row < kTcBM ? ti.row_end - ti.a_row : kTcBM;
    return rows > 0 ? (rows + kSwN - 1) / kSwN : 0;
  };
  uint32_t npre = 0;   // stages whose codes were issued before the wait
  if (warp == 0 && lane == 0) {
    for (int tile = blockIdx.x; tile < total && npre < (uint32_t)C::ST; tile += gridDim.x) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int nk = (ti.K + C::KB - 1) / C::KB;
      const int np = passes_of(ti);
      for (int ps = 0; ps < np && npre < (uint32_t)C::ST; ++ps)
        for (int kb = 0; kb < nk && npre < (uint32_t)C::ST; ++kb, ++npre) {
          mbar_arrive_expect_tx(sfull(npre), C::STAGE_BYTES);
          tma_load_3d(stage_r(npre), &mW, sfull(npre), kb * (C::KB / 2), ti.n0, ti.seg);
        }
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer: codes and h rows of each stage ----------------
      uint32_t g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(a, sc, tile, BNH);
        const int nk = (ti.K + C::KB - 1) / C::KB;
        const int np = passes_of(ti);
        for (int ps = 0; ps < np && ok; ++ps) {
          for (int kb = 0; kb < nk; ++kb, ++g) {
            const int s = g % C::ST;
            if (g >= npre) {
              if (!mbar_wait_sleep_bounded(sempty(s), ((g / C::ST) & 1u) ^ 1u, a.timeout_ns,
                                           abort_flag)) {
                give_up();
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(sfull(s), C::STAGE_BYTES);
              tma_load_3d(stage_r(s), &mW, sfull(s), kb * (C::KB / 2), ti.n0, ti.seg);
            }
            const int row = ti.a_row + ps * kSwN;
            tma_load_2d(stage_h(s), &mA32, sfull(s), kb * C::KB, row);
            tma_load_2d(stage_h(s) + C::H_PANEL, &mA32, sfull(s), kb * C::KB + C::PANEL, row);
          }
        }
      }
      // every load issued has landed before the block exits
      for (int s = 0; s < C::ST; ++s) {
        if (g > static_cast<uint32_t>(s)) {
          const uint32_t uses = (g - 1 - s) / C::ST + 1;
          if (ok)
            mbar_wait_sleep_bounded(sempty(s), (uses - 1) & 1u, a.timeout_ns, abort_flag);
          else
            mbar_wait_bounded(sfull(s), (uses - 1) & 1u, a.timeout_ns, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t g = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const TileInfo ti = decode_tile(a, sc, tile, BNH);
        const int nk = (ti.K + C::KB - 1) / C::KB;
        const int np = passes_of(ti);
        for (int ps = 0; ps < np && ok; ++ps, ++it) {
          const int ab = it & 1;
          if (!mbar_wait_sleep_bounded(tempty_bar(ab), ((it >> 1) & 1) ^ 1u, a.timeout_ns,
                                       abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + ab * kSwN;
          for (int kb = 0; kb < nk; ++kb, ++g) {
            const int s = g % C::ST, w = g % C::WST;
            // the stage's h rows have landed and its weights are expanded
            if (!mbar_wait_sleep_bounded(sfull(s), (g / C::ST) & 1u, a.timeout_ns, abort_flag) ||
                !mbar_wait_sleep_bounded(wfull(w), (g / C::WST) & 1u, a.timeout_ns,
                                         abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int pn = 0; pn < 2; ++pn)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma_bf16(d_tmem, smem_desc_k128(stage_w(w) + pn * C::W_PANEL + kk * 32),
                            smem_desc_k128(stage_h(s) + pn * C::H_PANEL + kk * 32), C::IDESC,
                            (kb != 0 || pn != 0 || kk != 0) ? 1u : 0u);
            tc_commit(sempty(s));
            tc_commit(wempty(w));
          }
          if (!ok) break;
          tc_commit(tfull_bar(ab));
        }
      }
      if (!ok) {
        tc_commit(drain_bar);
        mbar_wait_bounded(drain_bar, 0, a.timeout_ns, nullptr);
      }
    }
  } else if (warp >= C::CONV0) {
    // ---------------- converter warps ----------------
    // item i of a stage: weight row i / 16, eight codes i % 16 of its 128-byte
    // code row: 16-byte chunk (i % 16) % 8 of the row's bf16 panel (i % 16) / 8,
    // written in the 128-byte swizzle
    const int ct = (warp - C::CONV0) * 32 + lane;
    constexpr int PER = (BNH * 16) / (C::CONVW * 32);
    static_assert(PER * C::CONVW * 32 == BNH * 16, "items per converter thread");
    uint32_t g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int nk = (ti.K + C::KB - 1) / C::KB;
      const int np = passes_of(ti);
      for (int ps = 0; ps < np && ok; ++ps) {
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % C::ST, w = g % C::WST;
          const bool okl =
              mbar_wait_sleep_bounded(sfull(s), (g / C::ST) & 1u, a.timeout_ns, abort_flag) &&
              mbar_wait_sleep_bounded(wempty(w), ((g / C::WST) & 1u) ^ 1u, a.timeout_ns,
                                      abort_flag);
          if (!__all_sync(0xffffffffu, okl)) {
            if (lane == 0) give_up();
            ok = false;
            break;
          }
          const uint32_t raw = stage_r(s);
          const uint32_t wt = stage_w(w);
          uint2 codes[PER];
#pragma unroll
          for (int j = 0; j < PER; ++j) {
            const int i = ct + j * 32 * C::CONVW;
            codes[j] = lds_u2(raw + (i >> 4) * 128 + (i & 15) * 8);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty(s));   // the codes are in registers
#pragma unroll
          for (int j = 0; j < PER; ++j) {
            const int i = ct + j * 32 * C::CONVW;
            const int n = i >> 4, pn = (i >> 3) & 1, c = i & 7;
            const uint2 b01 = e4m3x4_to_bf16x4(codes[j].x), b23 = e4m3x4_to_bf16x4(codes[j].y);
            sts_u4(wt + pn * C::W_PANEL + n * 128 + ((c ^ (n & 7)) << 4),
                   make_uint4(b01.x, b01.y, b23.x, b23.y));
          }
          fence_proxy_async_smem();   // the tensor cores read what these threads wrote
          __syncwarp();
          if (lane == 0) mbar_arrive(wfull(w));
        }
      }
    }
  } else {
    // ---------------- epilogue (four warps, one per TMEM lane quarter) ----------------
    // thread = output channel (TMEM lane), its 32 accumulator columns = the
    // pass's 32 token rows
    const int q = warp & 3;
    if constexpr (EPI == EPI_COMBINE1) {
      // a dropped token (key_row < 0, top-1) gets y = 0
      uint4* y = static_cast<uint4*>(a.y);
      const int nvec = a.ld_y * 2 / 16;
      const int gw = blockIdx.x * C::EPIW + (warp - C::EPI0), nw = gridDim.x * C::EPIW;
      for (int t = gw; t < a.T_tokens; t += nw) {
        if (__ldg(a.key_row + t) < 0)
          for (int c = lane; c < nvec; c += 32) y[(size_t)t * nvec + c] = make_uint4(0, 0, 0, 0);
      }
    }
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile(a, sc, tile, BNH);
      const int np = passes_of(ti);
      const int ch = ti.n0 + q * 32 + lane;
      const bool ch_ok = ch < ti.N;
      const float sc_ch = ch_ok ? __ldg(a.b0_scale + (size_t)ti.seg * a.N + ch) : 0.f;
      for (int ps = 0; ps < np; ++ps, ++it) {
        const int ab = it & 1;
        if (!mbar_wait_sleep_bounded(tfull_bar(ab), (it >> 1) & 1, a.timeout_ns, abort_flag)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[kSwN];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ab * kSwN, r);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(tempty_bar(ab));
        const int row0 = ti.a_row + ps * kSwN;
        int rend = ti.row_end - row0 < kSwN ? ti.row_end - row0 : kSwN;
        if (rend > 0 && !in_bounds(row0 + rend <= a.R_cap, a.status))
          rend = a.R_cap - row0 > 0 ? a.R_cap - row0 : 0;
        if (!ch_ok) continue;
        // unrolled over the pass's 32 columns (register-resident accumulator
        // values), predicated on the real rows
#pragma unroll
        for (int j = 0; j < kSwN; ++j) {
          if (j < rend) {
            const int row = row0 + j;
            const float v = __uint_as_float(r[j]) * sc_ch;
            if constexpr (EPI == EPI_COMBINE1) {
              const int tok = __ldg(a.row_token + row);
              if (in_bounds(tok >= 0 && tok < a.T_tokens, a.status)) {
                const float gt = __ldg(a.gate + tok);
                static_cast<__nv_bfloat16*>(a.y)[(size_t)tok * a.ld_y + ch] =
                    __float2bfloat16_rn(fmaf(gt, v, 0.f));
              }
            } else {
              static_cast<__nv_bfloat16*>(a.out)[(size_t)row * a.ld_out + ch] =
                  __float2bfloat16_rn(v);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
struct TcMaps {
  CUtensorMap A, A_sh, A32, A32_sh, B0, B1, B0_sh, B1_sh;
};

template <int BNH, bool DUAL, int EPI, int AS = AS_TMA, bool F8 = false, int CL = 1>
static cudaError_t run_tc(const TcMaps& m, const TcArgs& a, int grid, cudaStream_t st) {
  using C = TcCfg<BNH, DUAL, EPI, F8>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = tc_grouped_gemm<BNH, DUAL, EPI, AS, F8, CL>;
  cudaError_t e = smem_attr_once(kern, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  if constexpr (CL == 1) {
    return launch_pdl(kern, dim3(grid), dim3(TcWarps<AS, EPI>::THREADS), C::SMEM, st, m.A,
                      m.A_sh, m.A32, m.A32_sh, m.B0, m.B1, m.B0_sh, m.B1_sh, a);
  } else {
    // clusters of CL CTAs along x (the grid a multiple of CL), with
    // programmatic dependent launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid < CL ? CL : (grid / CL) * CL);
    cfg.blockDim = dim3(TcWarps<AS, EPI>::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, m.A, m.A_sh, m.A32, m.A32_sh, m.B0, m.B1, m.B0_sh,
                              m.B1_sh, a);
  }
}

template <int AS>
static cudaError_t dispatch_up_t(int bn, int act, const TcMaps& m, const TcArgs& a, int grid,
                                 cudaStream_t st, bool cl2 = false) {
  if constexpr (AS == AS_TMA) {
    if (cl2 && act == MOE_ACT_SWIGLU && bn == 128)
      return run_tc<128, true, EPI_SWIGLU, AS_TMA, false, 2>(m, a, grid, st);
  }
  if (act == MOE_ACT_SWIGLU) {
    switch (bn) {
      case 128: return run_tc<128, true, EPI_SWIGLU, AS>(m, a, grid, st);
      case 96: return run_tc<96, true, EPI_SWIGLU, AS>(m, a, grid, st);
      case 64: return run_tc<64, true, EPI_SWIGLU, AS>(m, a, grid, st);
      case 32: return run_tc<32, true, EPI_SWIGLU, AS>(m, a, grid, st);
    }
  } else if (act == MOE_ACT_RELU) {
    switch (bn) {
      case 256: return run_tc<256, false, EPI_RELU, AS>(m, a, grid, st);
      case 128: return run_tc<128, false, EPI_RELU, AS>(m, a, grid, st);
      case 96: return run_tc<96, false, EPI_RELU, AS>(m, a, grid, st);
      case 64: return run_tc<64, false, EPI_RELU, AS>(m, a, grid, st);
    }
  } else {
    switch (bn) {
      case 256: return run_tc<256, false, EPI_GELU, AS>(m, a, grid, st);
      case 128: return run_tc<128, false, EPI_GELU, AS>(m, a, grid, st);
      case 96: return run_tc<96, false, EPI_GELU, AS>(m, a, grid, st);
      case 64: return run_tc<64, false, EPI_GELU, AS>(m, a, grid, st);
    }
  }
  return cudaErrorInvalidValue;
}

// fp8 (e4m3) A and B: the SwiGLU up projection of a layer with fp8 gate/up weights
static cudaError_t dispatch_up_f8(int bn, const TcMaps& m, const TcArgs& a, int grid,
                                  cudaStream_t st) {
  switch (bn) {
    case 128: return run_tc<128, true, EPI_SWIGLU, AS_TMA, true>(m, a, grid, st);
    case 96: return run_tc<96, true, EPI_SWIGLU, AS_TMA, true>(m, a, grid, st);
    case 64: return run_tc<64, true, EPI_SWIGLU, AS_TMA, true>(m, a, grid, st);
    case 32: return run_tc<32, true, EPI_SWIGLU, AS_TMA, true>(m, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

static cudaError_t dispatch_up(int as, int bn, int act, const TcMaps& m, const TcArgs& a,
                               int grid, cudaStream_t st, bool cl2) {
  return as == AS_CP   ? dispatch_up_t<AS_CP>(bn, act, m, a, grid, st)
         : as == AS_G4 ? dispatch_up_t<AS_G4>(bn, act, m, a, grid, st)
                       : dispatch_up_t<AS_TMA>(bn, act, m, a, grid, st, cl2);
}

static cudaError_t dispatch_down(int bn, bool combine1, bool combinek, const TcMaps& m,
                                 const TcArgs& a, int grid, cudaStream_t st, bool cl2 = false) {
  if (cl2 && !combinek) {
    if (combine1) {
      if (bn == 256) return run_tc<256, false, EPI_COMBINE1, AS_TMA, false, 2>(m, a, grid, st);
      if (bn == 192) return run_tc<192, false, EPI_COMBINE1, AS_TMA, false, 2>(m, a, grid, st);
    } else {
      if (bn == 256) return run_tc<256, false, EPI_OUT16, AS_TMA, false, 2>(m, a, grid, st);
      if (bn == 192) return run_tc<192, false, EPI_OUT16, AS_TMA, false, 2>(m, a, grid, st);
    }
  }
  if (combinek) {
    switch (bn) {
      case 256: return run_tc<256, false, EPI_COMBINEK>(m, a, grid, st);
      case 192: return run_tc<192, false, EPI_COMBINEK>(m, a, grid, st);
      case 128: return run_tc<128, false, EPI_COMBINEK>(m, a, grid, st);
      case 96: return run_tc<96, false, EPI_COMBINEK>(m, a, grid, st);
      case 64: return run_tc<64, false, EPI_COMBINEK>(m, a, grid, st);
    }
    return cudaErrorInvalidValue;
  }
  if (combine1) {
    switch (bn) {
      case 256: return run_tc<256, false, EPI_COMBINE1>(m, a, grid, st);
      case 192: return run_tc<192, false, EPI_COMBINE1>(m, a, grid, st);
      case 128: return run_tc<128, false, EPI_COMBINE1>(m, a, grid, st);
      case 96: return run_tc<96, false, EPI_COMBINE1>(m, a, grid, st);
      case 64: return run_tc<64, false, EPI_COMBINE1>(m, a, grid, st);
    }
    return cudaErrorInvalidValue;
  }
  switch (bn) {
    case 256: return run_tc<256, false, EPI_OUT16>(m, a, grid, st);
    case 192: return run_tc<192, false, EPI_OUT16>(m, a, grid, st);
    case 128: return run_tc<128, false, EPI_OUT16>(m, a, grid, st);
    case 96: return run_tc<96, false, EPI_OUT16>(m, a, grid, st);
    case 64: return run_tc<64, false, EPI_OUT16>(m, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

constexpr uint64_t kGemmTimeoutNs = 2000000000ull;   // 2 s

// ---- the down projection with e4m3 weights ----
template <int BNH, int EPI>
static cudaError_t run_f8w(const TcMaps& m, const CUtensorMap& mW, const TcArgs& a, int grid,
                           cudaStream_t st) {
  using C = F8wCfg<BNH, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = tc_down_f8w<BNH, EPI>;
  cudaError_t e = smem_attr_once(kern, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM, st, m.A, m.A32, mW, a);
}

template <int EPI>
static cudaError_t run_f8s(const TcMaps& m, const CUtensorMap& mW, const TcArgs& a, int grid,
                           cudaStream_t st) {
  using C = F8sCfg<EPI>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = tc_down_f8s<EPI>;
  cudaError_t e = smem_attr_once(kern, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM, st, m.A32, mW, a);
}

static cudaError_t dispatch_down_f8w(int bn, bool combine1, const TcMaps& m, const CUtensorMap& mW,
                                     const TcArgs& a, int grid, cudaStream_t st) {
  if (combine1) {
    switch (bn) {
      case 256: return run_f8w<256, EPI_COMBINE1>(m, mW, a, grid, st);
      case 192: return run_f8w<192, EPI_COMBINE1>(m, mW, a, grid, st);
      case 128: return run_f8w<128, EPI_COMBINE1>(m, mW, a, grid, st);
      case 96: return run_f8w<96, EPI_COMBINE1>(m, mW, a, grid, st);
      case 64: return run_f8w<64, EPI_COMBINE1>(m, mW, a, grid, st);
    }
    return cudaErrorInvalidValue;
  }
  switch (bn) {
    case 256: return run_f8w<256, EPI_OUT16>(m, mW, a, grid, st);
    case 192: return run_f8w<192, EPI_OUT16>(m, mW, a, grid, st);
    case 128: return run_f8w<128, EPI_OUT16>(m, mW, a, grid, st);
    case 96: return run_f8w<96, EPI_OUT16>(m, mW, a, grid, st);
    case 64: return run_f8w<64, EPI_OUT16>(m, mW, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

// ---- up + down in one launch: the compiled forms ----
template <class PU, class PD, int ASU>
static cudaError_t run_ud(const TcMaps& mu, const TcMaps& md, const TcArgs& au, const TcArgs& ad,
                          const UdArgs& ud, int grid, cudaStream_t st) {
  using U = UdCfg<PU, PD, ASU>;
  static std::atomic<uint64_t> attr_done{0};
  auto kern = tc_updown<PU, PD, ASU>;
  cudaError_t e = smem_attr_once(kern, U::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(U::THREADS), U::SMEM, st, mu.A, mu.A_sh, mu.A32,
                    mu.A32_sh, mu.B0, mu.B1, mu.B0_sh, mu.B1_sh, md.A, md.A_sh, md.A32,
                    md.A32_sh, md.B0, md.B0_sh, au, ad, ud);
}

using UdSw128 = TcPhase<128, true, EPI_SWIGLU>;
using UdSw96 = TcPhase<96, true, EPI_SWIGLU>;
using UdRelu256 = TcPhase<256, false, EPI_RELU>;
using UdOut256 = TcPhase<256, false, EPI_OUT16>;
using UdOut192 = TcPhase<192, false, EPI_OUT16>;
using UdOut96 = TcPhase<96, false, EPI_OUT16>;
using UdCmb256 = TcPhase<256, false, EPI_COMBINE1>;
using UdCmb192 = TcPhase<192, false, EPI_COMBINE1>;

// The forms compiled for one launch (the tilings the bench workloads take:
// SwiGLU up tiles of 128 columns fed by TMA or gathered, of 96 for the
// smallest decode batch; ReLU up tiles of 256 gathered, with the combine in
// the down epilogue); any other layer runs the two launches.
bool updown_compiled(int as, int act, int up_bn, int dn_bn, bool combine1) {
  if (act == MOE_ACT_SWIGLU && !combine1) {
    if (up_bn == 128 && (as == AS_TMA || as == AS_CP)) return dn_bn == 256 || dn_bn == 192;
    if (up_bn == 96 && as == AS_TMA) return dn_bn == 96;
  }
  if (act == MOE_ACT_RELU && combine1 && up_bn == 256 && as == AS_CP)
    return dn_bn == 192 || dn_bn == 256;
  return false;
}

static cudaError_t dispatch_updown(int as, int act, int up_bn, int dn_bn, bool combine1,
                                   const TcMaps& mu, const TcMaps& md, const TcArgs& au,
                                   const TcArgs& ad, const UdArgs& ud, int grid, cudaStream_t st) {
  if (act == MOE_ACT_SWIGLU && !combine1 && up_bn == 128) {
    if (as == AS_TMA) {
      if (dn_bn == 256) return run_ud<UdSw128, UdOut256, AS_TMA>(mu, md, au, ad, ud, grid, st);
      if (dn_bn == 192) return run_ud<UdSw128, UdOut192, AS_TMA>(mu, md, au, ad, ud, grid, st);
    } else if (as == AS_CP) {
      if (dn_bn == 256) return run_ud<UdSw128, UdOut256, AS_CP>(mu, md, au, ad, ud, grid, st);
      if (dn_bn == 192) return run_ud<UdSw128, UdOut192, AS_CP>(mu, md, au, ad, ud, grid, st);
    }
  }
  if (act == MOE_ACT_SWIGLU && !combine1 && up_bn == 96 && as == AS_TMA && dn_bn == 96)
    return run_ud<UdSw96, UdOut96, AS_TMA>(mu, md, au, ad, ud, grid, st);
  if (act == MOE_ACT_RELU && combine1 && up_bn == 256 && as == AS_CP) {
    if (dn_bn == 192) return run_ud<UdRelu256, UdCmb192, AS_CP>(mu, md, au, ad, ud, grid, st);
    if (dn_bn == 256) return run_ud<UdRelu256, UdCmb256, AS_CP>(mu, md, au, ad, ud, grid, st);
  }
  return cudaErrorInvalidValue;
}

int updown_counters(const Plan& p) { return p.R_cap / kTcBM + p.mt_sh; }

bool updown_eligible(const Plan& p) {
  if (!p.tc || p.fp8 || p.combine_k || p.cluster2_up || p.cluster2_dn || p.gather4) return false;
  if (updown_counters(p) > kMaxTileCounters) return false;   // the counters live in the header
  return updown_compiled(p.gather ? AS_CP : AS_TMA, p.cfg.act, p.up_bn, p.dn_bn,
                         p.combine_in_down);
}

// The form that measures faster as one launch (same box, A/B in one call):
// the gathered ReLU up projection with the combine in the down epilogue
// (Switch-shaped layer 95.0 -> 89.5 us per step).  The 128-column SwiGLU
// forms do not (DeepSeek-V3-shaped +0.5 %, Mixtral-shaped +1.3 %, gpt-oss-
// shaped T = 16 +1.2 %): those layers run under the power cap, where closing
// the idle gap between the projections saves no energy and so no time.  The
// 96-column decode form did at first (gpt-oss-shaped T = 1: 65.2 -> 64.6 us),
// but with the current kernels two launches are ahead (63.4 against 62.5 us
// per step, three calls).
bool updown_default(const Plan& p) {
  return p.cfg.act == MOE_ACT_RELU && p.combine_in_down;
}

cudaError_t launch_experts_tc(const Plan& p, const void* x, const void* W1, const void* W3,
                              const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                              void* ws, cudaStream_t st, cudaEvent_t mid_event, void* y,
                              const float* topk_w, const float* W1s, const float* W3s,
                              const float* W2s) {
  const moe_config& c = p.cfg;
  char* w = static_cast<char*>(ws);
  const Meta meta = meta_ptrs(p, ws);
  const bool sh = c.n_shared != 0;
  const bool dual = c.act == MOE_ACT_SWIGLU;
  uint32_t* status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  const void* h = w + p.ws.h;
  const void* hs = sh ? static_cast<const void*>(w + p.ws.hs) : h;

  // ---- up projection: h = act(xp W1^T) or silu(xp W1^T) * (xp W3^T), where
  // xp holds the routed rows of x in expert order: either gathered through
  // row_token inside the kernel, or copied beforehand and read by TMA; the
  // shared expert reads x itself ----
  // (fp8 gate/up weights: A is the e4m3 copy xq of the routed rows, one
  // scale per row in xs; B holds e4m3 codes with one scale per column)
  const int el = p.fp8 ? 1 : 2;
  const bool from_x = p.gather || p.gather4;
  const void* a_src = p.fp8 ? static_cast<const void*>(w + p.ws.xq)
                      : from_x ? x : static_cast<const void*>(w + p.ws.xp);
  const uint64_t a_rows = from_x ? (uint64_t)c.T : (uint64_t)p.R_cap;
  TcMaps mu;
  // the row-gathering TMA reads boxes one row high
  // (2-CTA clusters load A in halves of 64 rows, each CTA one half)
  const uint32_t a_box = p.gather4 ? 1u : (p.cluster2_up ? (uint32_t)kTcBM / 2 : (uint32_t)kTcBM);
  bool ok = encode_2d(&mu.A, a_src, a_rows, c.d, a_box, el);
  ok = ok && encode_2d(&mu.A32, a_src, a_rows, c.d, kABox, el);
  ok = ok && encode_3d(&mu.B0, W1, c.E, c.f, c.d, p.up_bn, el);
  ok = ok && encode_3d(&mu.B1, dual ? W3 : W1, c.E, c.f, c.d, p.up_bn, el);
  if (sh) {
    // the shared expert's rows are x itself, loaded as 128-row boxes (64-row
    // halves in cluster mode) whatever the routed rows' source
    const uint32_t a_box_sh = p.cluster2_up ? (uint32_t)kTcBM / 2 : (uint32_t)kTcBM;
    ok = ok && encode_2d(&mu.A_sh, x, c.T, c.d, a_box_sh);
    ok = ok && encode_2d(&mu.A32_sh, x, c.T, c.d, kABox);
    ok = ok && encode_3d(&mu.B0_sh, Ws1, 1, c.f_shared, c.d, p.up_bn);
    ok = ok && encode_3d(&mu.B1_sh, Ws3, 1, c.f_shared, c.d, p.up_bn);
  } else {
    mu.A_sh = mu.A;
    mu.A32_sh = mu.A32;
    mu.B0_sh = mu.B0;
    mu.B1_sh = mu.B1;
  }
  if (!ok) return cudaErrorInvalidValue;
  TcArgs au;
  au.tp = meta.tp_up;
  au.seg_start = meta.seg_start;
  au.mtiles = meta.mtiles;
  au.kept = meta.kept;
  au.rows_sh = c.T;
  au.static_mt = 0;
  au.static_total = 0;
  au.col_bias = nullptr;
  au.partial_rows = p.partial_rows_up;
  au.row_token = reinterpret_cast<const int*>(w + p.ws.row_token);
  au.gx = static_cast<const char*>(x);
  au.gx_row_bytes = c.d * 2;
  au.early_b = 0;
  au.a_scale = p.fp8 ? reinterpret_cast<const float*>(w + p.ws.xs) : nullptr;
  au.b0_scale = W1s;
  au.b1_scale = W3s;
  au.gate = nullptr;
  au.y = nullptr;
  au.ld_y = 0;
  au.key_row = nullptr;
  au.T_tokens = 0;
  au.E = c.E;
  au.has_shared = sh ? 1 : 0;
  au.N = c.f;
  au.K = c.d;
  au.N_sh = sh ? c.f_shared : 0;
  au.K_sh = c.d;
  au.out = w + p.ws.h;
  au.ld_out = c.f;
  au.out_sh = sh ? static_cast<void*>(w + p.ws.hs) : nullptr;
  au.ld_out_sh = sh ? c.f_shared : 0;
  au.R_cap = p.R_cap;
  au.T_x = c.T;
  au.m64 = p.m64 ? 1 : 0;
  unsigned* cmb_ctr = p.combine_k ? reinterpret_cast<unsigned*>(w + p.ws.cmb_ctr) : nullptr;
  au.zero_ctr = cmb_ctr;
  au.zero_ctr_n = p.combine_k ? c.T * p.nt_dn : 0;
  au.status = status;
  au.timeout_ns = kGemmTimeoutNs;
  const int grid_up = p.max_tiles_up < p.num_sms ? p.max_tiles_up : p.num_sms;
  const int as = p.gather ? AS_CP : p.gather4 ? AS_G4 : AS_TMA;

  // ---- down projection: o = h W2^T (fp32) ----
  TcMaps md;
  ok = encode_2d(&md.A, h, p.R_cap, c.f, p.cluster2_dn ? kTcBM / 2 : kTcBM);
  ok = ok && encode_2d(&md.A32, h, p.R_cap, c.f, kABox);
  ok = ok && encode_3d(&md.B0, W2, c.E, c.d, c.f, p.dn_bn);
  md.B1 = md.B0;
  if (sh) {
    ok = ok && encode_2d(&md.A_sh, hs, p.T_pad, c.f_shared, p.cluster2_dn ? kTcBM / 2 : kTcBM);
    ok = ok && encode_2d(&md.A32_sh, hs, p.T_pad, c.f_shared, kABox);
    ok = ok && encode_3d(&md.B0_sh, Ws2, 1, c.d, c.f_shared, p.dn_bn);
  } else {
    md.A_sh = md.A;
    md.A32_sh = md.A32;
    md.B0_sh = md.B0;
  }
  md.B1_sh = md.B0_sh;
  if (!ok) return cudaErrorInvalidValue;
  TcArgs ad = au;
  ad.partial_rows = p.partial_rows;
  ad.early_b = 1;   // the schedule comes from the routing kernel, two launches back
  ad.zero_ctr = nullptr;
  ad.zero_ctr_n = 0;
  if (p.combine_in_down || p.combine_k) {
    ad.row_token = reinterpret_cast<const int*>(w + p.ws.row_token);
    ad.gate = topk_w;
    ad.y = y;
    ad.ld_y = c.d;
    ad.key_row = reinterpret_cast<const int*>(w + p.ws.key_row);
    ad.T_tokens = c.T;
    ad.k_slots = c.k;
    ad.cmb_ctr = cmb_ctr;
    ad.cmb_nt = p.nt_dn;
  }
  ad.tp = meta.tp_dn;
  ad.N = c.d;
  ad.K = c.f;
  ad.N_sh = sh ? c.d : 0;
  ad.K_sh = sh ? c.f_shared : 0;
  ad.out = w + p.ws.o;
  ad.ld_out = c.d;
  ad.out_sh = sh ? static_cast<void*>(w + p.ws.os) : nullptr;
  ad.ld_out_sh = sh ? c.d : 0;
  ad.out_sh_exp = sh ? reinterpret_cast<int8_t*>(w + p.ws.os_exp) : nullptr;
  ad.ld_out_sh_exp = sh ? (c.d + kShChunk - 1) / kShChunk : 0;
  const int grid_dn = p.max_tiles_dn < p.num_sms ? p.max_tiles_dn : p.num_sms;
  if (W2s != nullptr) {
    // e4m3 down weights: the codes by 64-byte tiles, expanded on chip
    if (sh || p.fused || p.combine_k) return cudaErrorInvalidValue;
    // the weights-as-N form takes 256-column tiles whatever the bf16 tiling:
    // it is bound by the MMA instructions it issues, and wider tiles carry
    // more weight bytes per instruction (gpt-oss-shaped T = 16: 139 -> 130 us,
    // T = 256: 283 -> 266 us against 192 columns)
    constexpr int kF8wBn = 256;
    CUtensorMap mW;
    if (!encode_3d_codes(&mW, W2, c.E, c.d, c.f, kF8wBn)) return cudaErrorInvalidValue;
    TcArgs a8 = ad;
    a8.b0_scale = W2s;
    a8.sched_bn = p.dn_bn;
    CUtensorMap mWs;
    if (p.dn_swap && !encode_3d_codes(&mWs, W2, c.E, c.d, c.f, F8sCfg<EPI_OUT16>::BNH,
                                      F8sCfg<EPI_OUT16>::KB))
      return cudaErrorInvalidValue;
    cudaError_t e = p.fp8 ? dispatch_up_f8(p.up_bn, mu, au, grid_up, st)
                          : dispatch_up(as, p.up_bn, c.act, mu, au, grid_up, st, p.cluster2_up);
    if (e != cudaSuccess) return e;
    if (mid_event && (e = cudaEventRecord(mid_event, st)) != cudaSuccess) return e;
    if (p.dn_swap) {
      // tiles of 128 output channels: the down tile count scaled to that width
      const int nt_s = (c.d + F8sCfg<EPI_OUT16>::BNH - 1) / F8sCfg<EPI_OUT16>::BNH;
      const long long tiles = (long long)(p.R_cap / kTcBM) * nt_s;
      const int grid = tiles < p.num_sms ? (int)tiles : p.num_sms;
      return p.combine_in_down ? run_f8s<EPI_COMBINE1>(md, mWs, a8, grid, st)
                               : run_f8s<EPI_OUT16>(md, mWs, a8, grid, st);
    }
    const long long tiles_w = (long long)(p.R_cap / kTcBM) * ((c.d + kF8wBn - 1) / kF8wBn);
    const int grid_w = tiles_w < p.num_sms ? (int)tiles_w : p.num_sms;
    return dispatch_down_f8w(kF8wBn, p.combine_in_down, md, mW, a8, grid_w, st);
  }
  if (p.fused) {
    // both projections in one launch; the up stage event then covers both
    UdArgs ud;
    ud.done = reinterpret_cast<unsigned*>(w + p.ws.status + kTileCounterOffset);
    ud.fin = reinterpret_cast<unsigned*>(w + p.ws.status + kUpDownFinOffset);
    ud.up_all = reinterpret_cast<unsigned*>(w + p.ws.status + kUpDownAllOffset);
    ud.n_done = updown_counters(p);
    ud.sh_base = p.R_cap / kTcBM;
    ud.nt_up = p.nt_up;
    ud.nt_up_sh = p.nt_up_sh;
    const long long tiles = (long long)p.max_tiles_up + p.max_tiles_dn;
    const int grid = tiles < p.num_sms ? (int)tiles : p.num_sms;
    cudaError_t e = dispatch_updown(as, c.act, p.up_bn, p.dn_bn, p.combine_in_down, mu, md, au,
                                    ad, ud, grid, st);
    if (e != cudaSuccess) return e;
    return mid_event ? cudaEventRecord(mid_event, st) : cudaSuccess;
  }
  cudaError_t e = p.fp8 ? dispatch_up_f8(p.up_bn, mu, au, grid_up, st)
                        : dispatch_up(as, p.up_bn, c.act, mu, au, grid_up, st, p.cluster2_up);
  if (e != cudaSuccess) return e;
  if (mid_event) {
    e = cudaEventRecord(mid_event, st);
    if (e != cudaSuccess) return e;
  }
  return dispatch_down(p.dn_bn, p.combine_in_down, p.combine_k, md, ad, grid_dn, st,
                       p.cluster2_dn);
}

// ---------------------------------------------------------------- router
// Router logits s = x W_r^T (+ offset) on the tensor cores: bf16 operands
// (their products are exact), each 128-wide chunk of the reduction
// accumulated in tensor memory, the chunks added in float32 by the epilogue,
// float32 output [T][E].

cudaError_t launch_router_tc(const Plan& p, const void* x, const void* W_r,
                             const float* logit_offset, float* scores, uint32_t* status,
                             cudaStream_t st) {
  const moe_config& c = p.cfg;
  // experts per tile: 32 for small E (twice the tiles), else 64
  const int bn = c.E <= 64 ? 32 : 64;
  TcMaps m;
  bool ok = encode_2d(&m.A, x, c.T, c.d, kTcBM);
  ok = ok && encode_2d(&m.A32, x, c.T, c.d, kABox);
  ok = ok && encode_3d(&m.B0, W_r, 1, c.E, c.d, bn);
  if (!ok) return cudaErrorInvalidValue;
  m.A_sh = m.A;
  m.A32_sh = m.A32;
  m.B1 = m.B0_sh = m.B1_sh = m.B0;
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.E = 1;
  a.N = c.E;
  a.K = c.d;
  a.out = scores;
  a.ld_out = c.E;
  a.rows_sh = c.T;
  a.static_mt = (c.T + kTcBM - 1) / kTcBM;
  a.static_total = a.static_mt * ((c.E + bn - 1) / bn);
  a.col_bias = logit_offset;
  a.partial_rows = p.partial_rows;
  a.row_token = nullptr;
  a.gate = nullptr;
  a.y = nullptr;
  a.ld_y = 0;
  a.key_row = nullptr;
  a.T_tokens = 0;
  a.gx = nullptr;
  a.gx_row_bytes = 0;
  a.early_b = 0;
  a.status = status;
  a.timeout_ns = kGemmTimeoutNs;
  const int grid = a.static_total < p.num_sms ? a.static_total : p.num_sms;
  return bn == 32 ? run_tc<32, false, EPI_F32_CHUNKED>(m, a, grid, st)
                  : run_tc<64, false, EPI_F32_CHUNKED>(m, a, grid, st);
}

// ---------------------------------------------------------------- self-test
// One block waits on a barrier that nothing completes; the bounded wait gives
// up after wait_ns, records the timeout bit and the block returns normally.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t wait_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(smem_u32(&bar), 0, wait_ns, nullptr))
      atomicOr(status, STATUS_TIMEOUT_SELFTEST);
  }
}

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t wait_ns, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(status, wait_ns);
  return cudaGetLastError();
}

}  // namespace moe
