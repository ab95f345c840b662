// combine.cu -- stage 6: y[t] = shared(x_t) + sum_j g_tj * o[row(t, j)],
// over the kept slots, accumulated in float32 in the fixed order j = 0..k-1
// (no atomics), then rounded once to the output dtype.  The routed expert
// outputs o arrive in the layer dtype (bf16 on the tensor-core path, float32
// on the float32 path), the shared expert's in float32 on the float32 path
// and as scaled fp16 on the tensor-core path (shared_out.cuh).
//
// "Mixture of Experts" (llm-tutorial ch. 11) § The mathematics and
// "Mixture-of-Experts" (neural networks visually) § Show the math: the layer
// output is the gate-weighted sum over the chosen experts only; dropped
// slots contribute nothing (ch. 11 § Expert capacity and dropped tokens).
#include "check.cuh"
#include "common.cuh"
#include "launch.cuh"
#include "moe_internal.h"
#include "shared_out.cuh"

namespace moe {

struct CombineArgs {
  const void* o;         // [R_cap][d] TOut
  const void* os;        // [T_pad][d]: float32 (float32 path) or scaled fp16; or null
  const int8_t* os_exp;  // [T_pad][ld_exp] chunk exponents of the scaled fp16 form
  int ld_exp;
  const int* key_row;    // [T*k]
  const float* topk_w;   // [T*k]
  void* y;               // [T][d]
  int T, d, k, R_cap;
  uint32_t* status;
};

__device__ __forceinline__ void store4(float* y, size_t i, float4 v) {
  *reinterpret_cast<float4*>(y + i) = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* y, size_t i, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(y + i) = u;
}

__device__ __forceinline__ float4 load4(const float* p, size_t i) {
  return *reinterpret_cast<const float4*>(p + i);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, size_t i) {
  const uint2 u = *reinterpret_cast<const uint2*>(p + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename TOut>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineArgs a) {
  __shared__ int rows[kMaxK];
  __shared__ float gates[kMaxK];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < a.k) {
    const int r = a.key_row[(size_t)t * a.k + threadIdx.x];
    rows[threadIdx.x] = r >= 0 && in_bounds(r < a.R_cap, a.status) ? r : -1;
    gates[threadIdx.x] = a.topk_w[(size_t)t * a.k + threadIdx.x];
  }
  __syncthreads();
  const TOut* o = static_cast<const TOut*>(a.o);
  TOut* y = static_cast<TOut*>(a.y);
  for (int c = threadIdx.x * 4; c < a.d; c += kThreads * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (a.os) {
      if constexpr (sizeof(TOut) == 4) {
        acc = load4(static_cast<const float*>(a.os), (size_t)t * a.d + c);
      } else {
        // four scaled fp16 values of one 32-column chunk
        const uint2 u =
            *reinterpret_cast<const uint2*>(static_cast<const __half*>(a.os) + (size_t)t * a.d + c);
        const float s = sh_pow2(a.os_exp[(size_t)t * a.ld_exp + c / kShChunk]);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        acc = make_float4(f0.x * s, f0.y * s, f1.x * s, f1.y * s);
      }
    }
    for (int j = 0; j < a.k; ++j) {
      const int r = rows[j];
      if (r < 0) continue;
      const float g = gates[j];
      const float4 v = load4(o, (size_t)r * a.d + c);
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    }
    store4(y, (size_t)t * a.d + c, acc);
  }
}

// bf16 rows (d a multiple of 8): 16-byte loads, and every kept slot's row of
// one 8-column chunk is requested before the first of them is used (U slots
// at a time), so that each thread keeps up to U + 1 loads in flight.  The arithmetic and its order are those of
// combine_kernel.
template <int U>
__global__ void __launch_bounds__(kThreads) combine_bf16x8_kernel(const CombineArgs a) {
  __shared__ int rows[kMaxK];
  __shared__ float gates[kMaxK];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < a.k) {
    const int r = a.key_row[(size_t)t * a.k + threadIdx.x];
    rows[threadIdx.x] = r >= 0 && in_bounds(r < a.R_cap, a.status) ? r : -1;
    gates[threadIdx.x] = a.topk_w[(size_t)t * a.k + threadIdx.x];
  }
  __syncthreads();
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(a.o);
  const __half* os = static_cast<const __half*>(a.os);
  __nv_bfloat16* y = static_cast<__nv_bfloat16*>(a.y);
  for (int c = threadIdx.x * 8; c < a.d; c += blockDim.x * 8) {
    float acc[8];
    if (os) {
      const uint4 u = *reinterpret_cast<const uint4*>(os + (size_t)t * a.d + c);
      sh_decode8(u, a.os_exp[(size_t)t * a.ld_exp + c / kShChunk], acc);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    }
    for (int j0 = 0; j0 < a.k; j0 += U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u;
        const int r = j < a.k ? rows[j] : -1;
        v[u] = r >= 0 ? *reinterpret_cast<const uint4*>(o + (size_t)r * a.d + c)
                      : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u;
        if (j >= a.k || rows[j] < 0) continue;
        const float g = gates[j];
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(b[i]);
          acc[2 * i] = fmaf(g, f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(g, f.y, acc[2 * i + 1]);
        }
      }
    }
    uint4 pk;
    uint32_t* pw = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      pw[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(y + (size_t)t * a.d + c) = pk;
  }
}

cudaError_t launch_combine(const Plan& p, const float* topk_w, void* y, void* ws,
                           cudaStream_t st) {
  CombineArgs a;
  char* w = static_cast<char*>(ws);
  a.o = w + p.ws.o;
  a.os = p.cfg.n_shared ? static_cast<const void*>(w + p.ws.os) : nullptr;
  a.os_exp = p.cfg.n_shared && p.tc ? reinterpret_cast<const int8_t*>(w + p.ws.os_exp) : nullptr;
  a.ld_exp = (p.cfg.d + kShChunk - 1) / kShChunk;
  a.key_row = reinterpret_cast<const int*>(w + p.ws.key_row);
  a.topk_w = topk_w;
  a.y = y;
  a.T = p.cfg.T;
  a.d = p.cfg.d;
  a.k = p.cfg.k;
  a.R_cap = p.R_cap;
  a.status = reinterpret_cast<uint32_t*>(w + p.ws.status);
  if (p.cfg.dtype == MOE_BF16) {
    // many slots per token: all of a chunk's slot rows in flight at once
    // (DeepSeek-V3-shaped layer 126 -> 120 us); with few slots the plain
    // kernel measured faster (Mixtral-shaped 48 vs 52 us, gpt-oss-shaped
    // decode 8 vs 10 us)
    const dim3 g(p.cfg.T), b(kThreads);
    // 128 threads per token row for the many-slot kernel: more blocks resident
    // per SM to cover the slot rows' latency (DeepSeek-V3-shaped 118.0 ->
    // 115.8 us; 64 threads: 117.5)
    if (p.cfg.k >= 8) return launch_pdl(combine_bf16x8_kernel<8>, g, dim3(128), 0, st, a);
    return launch_pdl(combine_kernel<__nv_bfloat16>, g, b, 0, st, a);
  }
  return launch_pdl(combine_kernel<float>, dim3(p.cfg.T), dim3(kThreads), 0, st, a);
}

}  // namespace moe
