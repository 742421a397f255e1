// routing_stats.cu -- routing statistics of the expert assignments
// ("Mixtral of Experts" section 5, Routing analysis): per-expert counts split
// by choice (Fig. 7 and Fig. 9: the share of tokens routed to each expert as
// first or second choice) and the repeat counts of Table 5 (consecutive tokens
// t and t+1 with the same first choice; with at least one expert in common
// among their K choices).
//
// One thread per token: it adds its K choices to a shared [K][n] histogram and
// compares its ids with those of token t+1.  Per-block totals are added to the
// outputs with integer atomics, so the results do not depend on the order.
#include "device.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(256) routing_stats_kernel(const int32_t* __restrict__ ids, int T,
                                                            int K, int n,
                                                            int32_t* __restrict__ slot_counts,
                                                            int32_t* __restrict__ repeats) {
  extern __shared__ int s_hist[];  // [K][n]
  __shared__ int s_rep[2];
  for (int i = threadIdx.x; i < K * n; i += blockDim.x) s_hist[i] = 0;
  if (threadIdx.x < 2) s_rep[threadIdx.x] = 0;
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  int first = 0, any = 0;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    const int32_t* a = ids + (size_t)t * K;
    for (int k = 0; k < K; ++k) {
      const int e = a[k];
      if ((unsigned)e < (unsigned)n) atomicAdd(&s_hist[k * n + e], 1);
    }
    if (t + 1 < T) {
      const int32_t* b = a + K;
      first += (a[0] == b[0]) ? 1 : 0;
      bool shared = false;
      for (int k = 0; k < K && !shared; ++k)
        for (int j = 0; j < K; ++j)
          if (a[k] == b[j]) {
            shared = true;
            break;
          }
      any += shared ? 1 : 0;
    }
  }
  // warp totals, then one shared atomic per warp
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    first += __shfl_xor_sync(0xffffffffu, first, o);
    any += __shfl_xor_sync(0xffffffffu, any, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (first) atomicAdd(&s_rep[0], first);
    if (any) atomicAdd(&s_rep[1], any);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < K * n; i += blockDim.x)
    if (s_hist[i] != 0) atomicAdd(&slot_counts[i], s_hist[i]);
  if (threadIdx.x < 2 && s_rep[threadIdx.x] != 0) atomicAdd(&repeats[threadIdx.x], s_rep[threadIdx.x]);
}

cudaError_t launch_routing_stats(const moe_shape& s, const int32_t* ids, int32_t* slot_counts,
                                 int32_t* repeats, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(slot_counts, 0, sizeof(int32_t) * s.top_k * s.n_experts, st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(repeats, 0, 2 * sizeof(int32_t), st);
  if (e != cudaSuccess || s.T == 0) return e;
  int64_t blocks = (s.T + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 4;
  if (blocks > cap) blocks = cap;
  const size_t smem = sizeof(int) * (size_t)s.top_k * s.n_experts;
  return launch_pdl(routing_stats_kernel, dim3((unsigned)blocks), dim3(256), smem, st, ids, s.T,
                    s.top_k, s.n_experts, slot_counts, repeats);
}

}  // namespace moe
