// quant.cu -- the token rows entering an fp8 up projection, in e4m3.
//
// A layer whose gate and up expert weights are stored as fp8 (e4m3) runs its
// up projection with fp8 operands on both sides, so every routed row of x is
// quantised first.  Row r of an expert segment (the kept slot (t, j) with
// key_row[t*k + j] = r) gets
//   xs[r]    = s_t = 2^q, q the smallest integer (not below -126) with
//              max_c |x[t][c]| / 2^q <= 448, the largest e4m3 magnitude
//              (s_t = 1 for an all-zero row);
//   xq[r][c] = e4m3(x[t][c] / s_t), rounded to nearest even.
// Dividing by a power of two is exact, so the codes depend only on x.  The
// pages use no 8-bit formats; this is the definition of the fp8-weight
// variant of the layer (the expert weights' own scales are inputs).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "check.cuh"
#include "launch.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kQuantThreads = 128;

// Exponent of the row scale: with amax = f * 2^q, f in [0.5, 1), the bound
// amax / 2^e <= 448 = 1.75 * 2^8 first holds at e = q - 9, or at q - 8 when
// f > 0.875; never below -126 (2^-126 is the smallest normal float).
__device__ __forceinline__ int row_scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int q = 0;
  const float f = frexpf(amax, &q);
  const int e = q - 9 + (f > 0.875f ? 1 : 0);
  return e < -126 ? -126 : e;
}

__global__ void __launch_bounds__(kQuantThreads)
    quant_rows_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ key_row,
                      int k, int d, uint8_t* __restrict__ xq, float* __restrict__ xs,
                      int R_cap, uint32_t* status) {
  __shared__ float red[kQuantThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int key = blockIdx.x;
  const int row = key_row[key];
  if (row < 0) return;                      // dropped slot: no row
  if (!in_bounds(row < R_cap, status)) return;
  const int t = key / k;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);   // 8 values each
  const int nv = d / 8;
  float amax = 0.f;
  for (int i = threadIdx.x; i < nv; i += kQuantThreads) {
    const uint4 u = __ldg(src + i);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(v.x), fabsf(v.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const int e = row_scale_exponent(amax);
  const float inv = ldexpf(1.f, -e);        // x * 2^-e is exactly x / 2^e
  if (threadIdx.x == 0) xs[row] = ldexpf(1.f, e);
  uint2* dst = reinterpret_cast<uint2*>(xq + (size_t)row * d);
  for (int i = threadIdx.x; i < nv; i += kQuantThreads) {
    const uint4 u = __ldg(src + i);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&u);
    uint32_t packed[2];
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      float2 v0 = __bfloat1622float2(b[j]), v1 = __bfloat1622float2(b[j + 1]);
      v0.x *= inv;
      v0.y *= inv;
      v1.x *= inv;
      v1.y *= inv;
      // two values per conversion, the first in the low byte
      const uint32_t c0 = __nv_cvt_float2_to_fp8x2(v0, __NV_SATFINITE, __NV_E4M3);
      const uint32_t c1 = __nv_cvt_float2_to_fp8x2(v1, __NV_SATFINITE, __NV_E4M3);
      packed[j / 2] = (c0 & 0xffffu) | (c1 << 16);
    }
    dst[i] = make_uint2(packed[0], packed[1]);
  }
}

cudaError_t launch_quant_rows(const Plan& p, const void* x, void* ws, cudaStream_t st) {
  const moe_config& c = p.cfg;
  char* w = static_cast<char*>(ws);
  const int keys = c.T * c.k;
  return launch_pdl(quant_rows_kernel, dim3(keys), dim3(kQuantThreads), 0, st,
                    static_cast<const __nv_bfloat16*>(x),
                    reinterpret_cast<const int*>(w + p.ws.key_row), c.k, c.d,
                    reinterpret_cast<uint8_t*>(w + p.ws.xq), reinterpret_cast<float*>(w + p.ws.xs),
                    p.R_cap, reinterpret_cast<uint32_t*>(w + p.ws.status));
}

}  // namespace moe
