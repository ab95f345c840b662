// shared_out.cuh -- the storage of the shared expert's output between the
// down projection and the combine (tensor-core path).
//
// The shared expert's output enters y with weight 1, so its rounding goes into
// y nearly whole; stored as bf16 it put a test layer's output 0.033 off the
// float64 layer, above the 3e-2 bar, and as float32 it costs twice the bytes.
// It is stored as fp16 (11 significant bits) scaled by a power of two per
// 32-column chunk of a row: 2^-e brings the chunk's largest magnitude into
// [2^14, 2^15), where fp16 cannot overflow; the exponents e are int8, one per
// chunk.  The scaling is exact, so the one rounding is the fp16 one.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace moe {

constexpr int kShChunk = 32;   // output columns per exponent

// e for a chunk whose largest magnitude is amax (0 for zeros and fp32
// subnormals; at least -126 so that 2^-e stays a normal fp32 value).
__device__ __forceinline__ int sh_chunk_exponent(float amax) {
  const int b = (__float_as_int(amax) >> 23) & 0xFF;   // biased exponent
  if (b == 0) return 0;
  const int e = b - 127 - 14;
  return e < -126 ? -126 : e;
}

// 2^e for -126 <= e <= 127, exactly.
__device__ __forceinline__ float sh_pow2(int e) { return __int_as_float((e + 127) << 23); }

// Eight stored values (one 16-byte load) back to float32, times 2^e.
__device__ __forceinline__ void sh_decode8(uint4 u, int e, float* out) {
  const float s = sh_pow2(e);
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    out[2 * i] = f.x * s;
    out[2 * i + 1] = f.y * s;
  }
}

}  // namespace moe
