// combine.cu -- gated combine ("Mixtral of Experts" section 2.1: the layer
// output is the gate-weighted sum of the selected experts' outputs).
//
// y[t] = bf16( sum_{k<K} gates[t,k] * y_perm[slot_row[t*K+k]]  (+ residual[t]) )
// 16-byte vector loads of the K expert rows, fp32 accumulation in slot order
// k = 0..K-1 (a fixed order, so the result does not depend on scheduling),
// residual added last.
#include "device.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ void unpack8c(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One thread per 16-byte slice of an output row: thread i of the flat grid
// writes slice i % (dim/8) of token i / (dim/8), with the loads of KC slots
// at a time in flight together (KC: the smallest of 2, 4, 8 that covers K, so
// top-2 keeps the registers, hence the occupancy, of a two-slot loop).
template <int KC>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_perm,
                                                      const int32_t* __restrict__ slot_row,
                                                      const float* __restrict__ gates,
                                                      const uint16_t* __restrict__ residual,
                                                      int T, int K, int d, int R,
                                                      uint16_t* __restrict__ y) {
  const int vec = d >> 3;
  const int64_t total = (int64_t)T * vec;
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / vec);
    const int v = (int)(i - (int64_t)t * vec);
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    // KC slots at a time: their row indices and gates, then their row
    // slices, are all requested before the first is used; the sum still runs
    // k = 0, 1, ... in order
    for (int k0 = 0; k0 < K; k0 += KC) {
      int row[KC];
      float g[KC];
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        const int k = k0 + j;
        row[j] = k < K ? __ldg(slot_row + (size_t)t * K + k) : -1;
        g[j] = k < K ? __ldg(gates + (size_t)t * K + k) : 0.0f;
      }
      uint4 val[KC];
#pragma unroll
      for (int j = 0; j < KC; ++j)
        val[j] = (unsigned)row[j] < (unsigned)R
                     ? __ldg(reinterpret_cast<const uint4*>(y_perm + (size_t)row[j] * d) + v)
                     : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        if ((unsigned)row[j] < (unsigned)R) {
          float f[8];
          unpack8c(val[j], f);
#pragma unroll
          for (int u = 0; u < 8; ++u) acc[u] = fmaf(g[j], f[u], acc[u]);
        }
      }
    }
    if (residual != nullptr) {
      float r[8];
      unpack8c(__ldg(reinterpret_cast<const uint4*>(residual + (size_t)t * d) + v), r);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += r[j];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + (size_t)t * d)[v] = o;
  }
}

cudaError_t launch_combine(const moe_shape& s, const uint16_t* y_perm, const int32_t* slot_row,
                           const float* gates, const uint16_t* residual, uint16_t* y,
                           cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  const int64_t total = (int64_t)s.T * (s.dim / 8);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 16;
  if (blocks > cap) blocks = cap;
  auto kern = s.top_k <= 2 ? combine_kernel<2> : (s.top_k <= 4 ? combine_kernel<4> : combine_kernel<8>);
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(256), 0, st, y_perm, slot_row, gates,
                    residual, s.T, s.top_k, s.dim, s.T * s.top_k, y);
}

}  // namespace moe
