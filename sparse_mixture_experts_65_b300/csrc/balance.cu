// balance.cu -- two load-balancing controls that sit next to the layer call.
//
//   * Router z-loss.  "Mixture of Experts" (llm-tutorial ch. 11) § Why MoE is
//     hard names the ST-MoE router z-loss, a penalty on large router logits
//     that keeps the softmax well conditioned, without printing its formula.
//     Computed here in the ST-MoE form, the batch mean of each token's squared
//     log-partition function:  z = (1/T) sum_t (log sum_e exp s_te)^2,  over
//     the logits the layer routes with (moe_router_scores), coefficient left
//     to the caller.
//   * One step of auxiliary-loss-free balancing.  "Mixture of experts"
//     (inside-the-model guide) § Auxiliary-loss-free balancing: every expert
//     keeps a bias that only steers the choice, lowered by gamma after a step
//     in which the expert was overloaded and raised by gamma when it was
//     underloaded.  Load = routed (pre-drop) count; overloaded means above
//     the mean T*k/E, compared exactly in integers (routed_i * E vs T * k).
//
// The z-loss runs as one cluster of kZlCluster CTAs: each thread takes whole
// tokens (a fixed token -> thread map), the per-token terms are summed in
// double in a fixed order (thread, warp shuffle tree, warps in order, CTAs in
// rank order through distributed shared memory), so the result is the same
// bit for bit on every run.  No global scratch and no atomics.
#include <cmath>
#include <cstdint>

#include "launch.cuh"
#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kZlCluster = 8;     // CTAs of the one cluster (portable size)
constexpr int kZlThreads = 512;

// Every thread of every CTA of the cluster arrives; release/acquire order the
// shared-memory writes before the barrier with the reads after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release;\n\t"
      "barrier.cluster.wait.acquire;" ::: "memory");
}

// Read a double from the same shared-memory variable of CTA `rank` of the
// cluster.
__device__ __forceinline__ double ld_cluster_f64(const double* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote)
               : "r"(smem_u32(local)), "r"(rank));
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(remote) : "memory");
  return v;
}

// log sum_e exp(row[e]) in one pass: the running maximum m is taken out of
// the exponentials, and the partial sum is rescaled whenever m grows.
template <bool VEC>
__device__ __forceinline__ float token_logsumexp(const float* __restrict__ row, int E) {
  float m = -INFINITY, sum = 0.f;
  if constexpr (VEC) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int c = 0; c < E / 4; ++c) {
      const float4 v = __ldg(r4 + c);
      const float cm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
      if (cm > m) {
        sum *= expf(m - cm);
        m = cm;
      }
      sum += (expf(v.x - m) + expf(v.y - m)) + (expf(v.z - m) + expf(v.w - m));
    }
  } else {
#pragma unroll 4
    for (int e = 0; e < E; ++e) {
      const float v = __ldg(row + e);
      if (v > m) {
        sum *= expf(m - v);
        m = v;
      }
      sum += expf(v - m);
    }
  }
  return m + logf(sum);
}

__global__ void __launch_bounds__(kZlThreads)
    router_z_loss_kernel(const float* __restrict__ s, int T, int E, int vec, float* out) {
  __shared__ double warp_part[kZlThreads / 32];
  __shared__ double cta_part;
  pdl_wait();
  pdl_trigger();
  const uint32_t rank = cluster_ctarank();
  double acc = 0.0;
  for (int t = (int)rank * kZlThreads + (int)threadIdx.x; t < T; t += kZlCluster * kZlThreads) {
    const float* row = s + (size_t)t * E;
    const float lse = vec ? token_logsumexp<true>(row, E) : token_logsumexp<false>(row, E);
    acc += (double)lse * (double)lse;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double c = 0.0;
    for (int w = 0; w < kZlThreads / 32; ++w) c += warp_part[w];
    cta_part = c;
  }
  cluster_barrier();   // every CTA's part is in its shared memory
  if (rank == 0 && threadIdx.x == 0) {
    double z = 0.0;
    for (uint32_t r = 0; r < (uint32_t)kZlCluster; ++r) z += ld_cluster_f64(&cta_part, r);
    *out = T > 0 ? (float)(z / (double)T) : 0.f;
  }
  cluster_barrier();   // no CTA exits while rank 0 may still read its part
}

__global__ void __launch_bounds__(kMaxE)
    bias_update_kernel(const int32_t* __restrict__ routed, int E, long long mean_scaled,
                       float gamma, float* bias) {
  pdl_wait();
  pdl_trigger();
  const int i = threadIdx.x;
  if (i >= E) return;
  const long long load_scaled = (long long)routed[i] * E;
  const float b = bias[i];
  if (load_scaled > mean_scaled)
    bias[i] = __fsub_rn(b, gamma);
  else if (load_scaled < mean_scaled)
    bias[i] = __fadd_rn(b, gamma);
}

cudaError_t launch_router_z_loss(const float* scores, int T, int E, float* z_loss,
                                 cudaStream_t st) {
  const int vec = (E % 4 == 0) && ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kZlCluster);
  cfg.blockDim = dim3(kZlThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kZlCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_z_loss_kernel, scores, T, E, vec, z_loss);
}

cudaError_t launch_bias_update(const int32_t* routed_counts, int E, int T, int k, float gamma,
                               float* sel_bias, cudaStream_t st) {
  const int threads = (E + 31) / 32 * 32;
  return launch_pdl(bias_update_kernel, dim3(1), dim3(threads), 0, st, routed_counts, E,
                    (long long)T * (long long)k, gamma, sel_bias);
}

}  // namespace moe
