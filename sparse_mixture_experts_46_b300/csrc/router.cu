// router.cu -- router logits, top-K selection and gate softmax
// ("Mixtral of Experts" section 2.1, G(x) = Softmax(TopK(x . W_g))).
//
// One warp owns TPW tokens at a time.  Each lane walks the feature dimension
// in 8-element (16-byte) slices, so a warp reads 512 contiguous bytes of every
// token row per step; W_g rows are read through L1 and shared by the TPW
// tokens.  Logits accumulate in fp32 (bf16 x bf16 products are exact in fp32)
// and are reduced across the warp with butterfly shuffles, after which every
// lane holds all n logits of its tokens.  Lane 0 then selects the top K
// (strictly greater wins, scanning experts in ascending order, so ties go to
// the lower index), computes the softmax of the selected logits and writes
// ids / gates.  Per-expert counts are gathered in a shared histogram and
// added to global memory once per block (integer atomics: order-free).
//
// Optional RMSNorm (residual-stack workload): u = bf16(x / sqrt(mean(x^2)+eps))
// is written out and the logits are taken on u, exactly as the expert FFN
// will see it.
#include "device.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int NE, int TPW>
__global__ void __launch_bounds__(256) router_topk_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int T, int d, int n, int K,
    int32_t* __restrict__ ids, float* __restrict__ gates, int32_t* __restrict__ counts,
    uint16_t* __restrict__ u_out, float eps) {
  __shared__ int s_hist[kMaxExperts];
  if (threadIdx.x < kMaxExperts) s_hist[threadIdx.x] = 0;
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const bool norm = (u_out != nullptr);

  for (int t0 = (blockIdx.x * (blockDim.x >> 5) + warp) * TPW; t0 < T; t0 += warps_total * TPW) {
    float rs[TPW];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) rs[tt] = 1.0f;
    if (norm) {
      float ss[TPW];
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) ss[tt] = 0.0f;
      for (int j0 = lane * 8; j0 < d; j0 += 256) {
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt) {
          if (t0 + tt < T) {
            float v[8];
            unpack8(*reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d + j0), v);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss[tt] = fmaf(v[i], v[i], ss[tt]);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) {
        ss[tt] = warp_sum(ss[tt]);
        rs[tt] = 1.0f / sqrtf(ss[tt] / (float)d + eps);
      }
    }

    float acc[TPW][NE];
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int e = 0; e < NE; ++e) acc[tt][e] = 0.0f;

    for (int j0 = lane * 8; j0 < d; j0 += 256) {
      float xv[TPW][8];
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) {
        if (t0 + tt < T) {
          const size_t off = (size_t)(t0 + tt) * d + j0;
          unpack8(*reinterpret_cast<const uint4*>(x + off), xv[tt]);
          if (norm) {
            uint32_t pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              pk[i] = pack_bf16x2(xv[tt][2 * i] * rs[tt], xv[tt][2 * i + 1] * rs[tt]);
              xv[tt][2 * i] = __uint_as_float(pk[i] << 16);
              xv[tt][2 * i + 1] = __uint_as_float(pk[i] & 0xFFFF0000u);
            }
            *reinterpret_cast<uint4*>(u_out + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) xv[tt][i] = 0.0f;
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        float w[NE];
        const uint16_t* row = wg + (size_t)(j0 + jj) * n;
        if (n == NE) {
#pragma unroll
          for (int q = 0; q < NE / 8; ++q) {
            float f[8];
            unpack8(__ldg(reinterpret_cast<const uint4*>(row) + q), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) w[q * 8 + i] = f[i];
          }
        } else {
#pragma unroll
          for (int e = 0; e < NE; ++e) w[e] = (e < n) ? bf16_bits_to_f32(__ldg(row + e)) : 0.0f;
        }
#pragma unroll
        for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
          for (int e = 0; e < NE; ++e) acc[tt][e] = fmaf(xv[tt][jj], w[e], acc[tt][e]);
      }
    }

#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int e = 0; e < NE; ++e) acc[tt][e] = warp_sum(acc[tt][e]);

    if (lane == 0) {
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) {
        const int t = t0 + tt;
        if (t >= T) break;
        uint32_t taken = 0;
        float v0 = 0.0f, denom = 0.0f;
        // pass 1: select in order, accumulate the softmax denominator
        for (int k = 0; k < K; ++k) {
          float best = 0.0f;
          int bi = -1;
#pragma unroll
          for (int e = 0; e < NE; ++e) {
            if (e < n && !((taken >> e) & 1u) && (bi < 0 || acc[tt][e] > best)) {
              best = acc[tt][e];
              bi = e;
            }
          }
          taken |= 1u << bi;
          if (k == 0) v0 = best;
          denom += expf(best - v0);
          ids[(size_t)t * K + k] = bi;
          atomicAdd(&s_hist[bi], 1);
        }
        // pass 2: the same selection again, now writing normalised gates
        taken = 0;
        const float inv = 1.0f / denom;
        for (int k = 0; k < K; ++k) {
          float best = 0.0f;
          int bi = -1;
#pragma unroll
          for (int e = 0; e < NE; ++e) {
            if (e < n && !((taken >> e) & 1u) && (bi < 0 || acc[tt][e] > best)) {
              best = acc[tt][e];
              bi = e;
            }
          }
          taken |= 1u << bi;
          gates[(size_t)t * K + k] = expf(best - v0) * inv;
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < n && s_hist[threadIdx.x] != 0) atomicAdd(&counts[threadIdx.x], s_hist[threadIdx.x]);
}

template <int NE, int TPW>
static cudaError_t launch_router_t(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                   int32_t* ids, float* gates, int32_t* counts, uint16_t* u_out,
                                   float eps, cudaStream_t st) {
  const int warps_needed = (s.T + TPW - 1) / TPW;
  int blocks = (warps_needed + 7) / 8;
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  router_topk_kernel<NE, TPW><<<blocks, 256, 0, st>>>(x, wg, s.T, s.dim, s.n_experts, s.top_k,
                                                      ids, gates, counts, u_out, eps);
  return cudaGetLastError();
}

cudaError_t launch_router(const moe_shape& s, const uint16_t* x, const uint16_t* wg, int32_t* ids,
                          float* gates, int32_t* counts, uint16_t* u_out, float eps,
                          cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.n_experts, st);
  if (e != cudaSuccess) return e;
  if (s.T == 0) return cudaSuccess;
  if (s.n_experts <= 8) return launch_router_t<8, 4>(s, x, wg, ids, gates, counts, u_out, eps, st);
  if (s.n_experts <= 16) return launch_router_t<16, 2>(s, x, wg, ids, gates, counts, u_out, eps, st);
  return launch_router_t<32, 1>(s, x, wg, ids, gates, counts, u_out, eps, st);
}

}  // namespace moe
