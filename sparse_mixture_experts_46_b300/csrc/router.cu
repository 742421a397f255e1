// router.cu -- router logits, top-K selection and gate softmax
// ("Mixtral of Experts" section 2.1, G(x) = Softmax(TopK(x . W_g))).
//
// A 256-thread block owns TPB consecutive tokens at a time.  The feature
// dimension is split across all threads of the block in 8-element (16-byte)
// slices, so a token row is read by the whole block at once and every thread
// issues its loads independently (no long per-thread dependency chain).  When
// W_g fits (n*dim*2 <= 96 KB, 64 KB for Mixtral) and the batch has at least four
// token groups per persistent block, the blocks are persistent and first copy
// W_g transposed ([n][dim]) into shared memory, so the W_g slice a
// thread needs is one conflict-free 16-byte read per expert; otherwise each
// thread reads its W_g rows from global memory.  Every W_g value a thread
// loads is shared by the TPB tokens.  Products of
// bf16 values are exact in fp32 and accumulate in fp32.  Partial logits are
// reduced with warp butterflies, then across the 8 warps in a fixed order
// (deterministic).  Thread tt < TPB then selects the top K of token tt:
// strictly-greater wins while scanning experts in ascending order, so ties go
// to the lower index; gates are the softmax of the selected logits.
// When counts are requested they are gathered in a shared histogram and added
// to global memory once per block (integer atomics: order-free).
//
// Optional RMSNorm (residual-stack workload): u = bf16(x / sqrt(mean(x^2)+eps))
// is written out and the logits are taken on u, exactly as the expert FFN
// will see it.
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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

}  // namespace

template <int NE, int TPB, bool STAGED>
__global__ void __launch_bounds__(kThreads) router_topk_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int T, int d, int n, int K,
    int32_t* __restrict__ ids, float* __restrict__ gates, int32_t* __restrict__ counts,
    uint16_t* __restrict__ u_out, float eps) {
  __shared__ float s_part[kWarps][TPB * NE];
  __shared__ float s_logit[TPB * NE];
  __shared__ float s_rs[TPB];
  __shared__ int s_hist[kMaxExperts];
  extern __shared__ __align__(16) uint16_t s_wgt[];  // STAGED: W_g transposed, [n][d]

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nvec = d >> 3;  // 16-byte slices per row
  const bool norm = (u_out != nullptr);
  if (tid < kMaxExperts) s_hist[tid] = 0;

  pdl_wait();  // x (and W_g) may be written by the previous kernel
  pdl_launch_dependents();
  if constexpr (STAGED) {
    // one W_g row (n values) per thread and step, 16-byte loads when n == NE
    if (n == NE) {
#pragma unroll 4
      for (int j = tid; j < d; j += kThreads) {
#pragma unroll
        for (int q = 0; q < NE / 8; ++q) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)j * NE) + q);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            s_wgt[(size_t)(q * 8 + 2 * i) * d + j] = (uint16_t)(w[i] & 0xFFFFu);
            s_wgt[(size_t)(q * 8 + 2 * i + 1) * d + j] = (uint16_t)(w[i] >> 16);
          }
        }
      }
    } else {
      for (int j = tid; j < d; j += kThreads) {
#pragma unroll
        for (int e = 0; e < NE; ++e)
          if (e < n) s_wgt[(size_t)e * d + j] = __ldg(wg + (size_t)j * n + e);
      }
    }
    __syncthreads();
  }

  const int ngroups = (T + TPB - 1) / TPB;
  for (int g = blockIdx.x; g < ngroups; g += gridDim.x) {
  const int t0 = g * TPB;

  // ---- RMSNorm scale per token (sum of squares over the whole block)
  if (norm) {
    float ss[TPB];
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) ss[tt] = 0.0f;
#pragma unroll 2
    for (int v = tid; v < nvec; v += kThreads) {
#pragma unroll
      for (int tt = 0; tt < TPB; ++tt) {
        if (t0 + tt < T) {
          float f[8];
          unpack8(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d) + v), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) ss[tt] = fmaf(f[i], f[i], ss[tt]);
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) {
      const float w = warp_sum(ss[tt]);
      if (lane == 0) s_part[warp][tt] = w;
    }
    __syncthreads();
    if (tid < TPB) {
      float s = 0.0f;
      for (int w = 0; w < kWarps; ++w) s += s_part[w][tid];
      s_rs[tid] = 1.0f / sqrtf(s / (float)d + eps);
    }
    __syncthreads();
  }

  // ---- partial logits over this thread's slices
  float acc[TPB][NE];
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt)
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[tt][e] = 0.0f;

#pragma unroll 2
  for (int v = tid; v < nvec; v += kThreads) {
    const int j0 = v * 8;
    float xv[TPB][8];
#pragma unroll
    for (int tt = 0; tt < TPB; ++tt) {
      if (t0 + tt < T) {
        const size_t off = (size_t)(t0 + tt) * d + j0;
        unpack8(__ldg(reinterpret_cast<const uint4*>(x + off)), xv[tt]);
        if (norm) {
          const float rs = s_rs[tt];
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pk[i] = pack_bf16x2(xv[tt][2 * i] * rs, xv[tt][2 * i + 1] * rs);
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
    if constexpr (STAGED) {
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        if (e < n) {
          float w[8];
          unpack8(*reinterpret_cast<const uint4*>(s_wgt + (size_t)e * d + j0), w);
#pragma unroll
          for (int tt = 0; tt < TPB; ++tt)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[tt][e] = fmaf(xv[tt][jj], w[jj], acc[tt][e]);
        }
      }
    } else {
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
        for (int tt = 0; tt < TPB; ++tt)
#pragma unroll
          for (int e = 0; e < NE; ++e) acc[tt][e] = fmaf(xv[tt][jj], w[e], acc[tt][e]);
      }
    }
  }

  // ---- block reduction in a fixed order: warp butterflies, then warps 0..7
#pragma unroll
  for (int tt = 0; tt < TPB; ++tt)
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const float s = warp_sum(acc[tt][e]);
      if (lane == 0) s_part[warp][tt * NE + e] = s;
    }
  __syncthreads();
  if (tid < TPB * NE) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += s_part[w][tid];
    s_logit[tid] = s;
  }
  __syncthreads();

  // ---- selection and gates: thread tt owns token t0 + tt
  if (tid < TPB && t0 + tid < T) {
    const int t = t0 + tid;
    const float* l = s_logit + tid * NE;
    uint32_t taken = 0;
    float v0 = 0.0f, denom = 0.0f;
    for (int k = 0; k < K; ++k) {  // selection order = slot order
      float best = 0.0f;
      int bi = -1;
      for (int e = 0; e < n; ++e) {
        const float le = l[e] == l[e] ? l[e] : -INFINITY;  // NaN counts as -inf
        if (!((taken >> e) & 1u) && (bi < 0 || le > best)) {
          best = le;
          bi = e;
        }
      }
      taken |= 1u << bi;
      if (k == 0) v0 = best;
      denom += expf(best - v0);
      ids[(size_t)t * K + k] = bi;
      if (counts != nullptr) atomicAdd(&s_hist[bi], 1);
    }
    // gates: the same selection again (cheaper than re-reading ids from memory)
    const float inv = 1.0f / denom;
    taken = 0;
    for (int k = 0; k < K; ++k) {
      float best = 0.0f;
      int bi = -1;
      for (int e = 0; e < n; ++e) {
        const float le = l[e] == l[e] ? l[e] : -INFINITY;  // NaN counts as -inf
        if (!((taken >> e) & 1u) && (bi < 0 || le > best)) {
          best = le;
          bi = e;
        }
      }
      taken |= 1u << bi;
      gates[(size_t)t * K + k] = expf(best - v0) * inv;
    }
  }
  __syncthreads();  // s_part, s_logit and s_rs are reused by the next token group
  }  // token groups
  if (counts != nullptr && tid < n && s_hist[tid] != 0) atomicAdd(&counts[tid], s_hist[tid]);
}

constexpr size_t kStagedMaxBytes = 96 * 1024;

template <int NE, int TPB>
static cudaError_t launch_router_t(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                   int32_t* ids, float* gates, int32_t* counts, uint16_t* u_out,
                                   float eps, cudaStream_t st) {
  const int groups = (s.T + TPB - 1) / TPB;
  const size_t wbytes = (size_t)s.n_experts * s.dim * 2;
  // staging pays off once every persistent block has several token groups
  if (wbytes <= kStagedMaxBytes && groups >= 4 * num_sms()) {
    auto kern = router_topk_kernel<NE, TPB, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStagedMaxBytes);
    if (e != cudaSuccess) return e;
    int blocks = num_sms() * 2;
    if (blocks > groups) blocks = groups;
    return launch_pdl(kern, dim3(blocks), dim3(kThreads), wbytes, st, x, wg, s.T, s.dim,
                      s.n_experts, s.top_k, ids, gates, counts, u_out, eps);
  }
  return launch_pdl(router_topk_kernel<NE, TPB, false>, dim3(groups), dim3(kThreads), 0, st, x,
                    wg, s.T, s.dim, s.n_experts, s.top_k, ids, gates, counts, u_out, eps);
}

cudaError_t launch_router(const moe_shape& s, const uint16_t* x, const uint16_t* wg, int32_t* ids,
                          float* gates, int32_t* counts, uint16_t* u_out, float eps,
                          uint32_t* err, cudaStream_t st) {
  if (counts != nullptr) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.n_experts, st);
    if (e != cudaSuccess) return e;
  }
  if (s.T == 0) return cudaSuccess;
  if (router_tc_supported(s) || router_wide_supported(s)) {
    // tensor-core logits; the RMSNorm (if any) runs first as its own kernel
    if (u_out != nullptr) {
      cudaError_t e = launch_rmsnorm(s, x, eps, u_out, st);
      if (e != cudaSuccess) return e;
      x = u_out;
    }
    return router_tc_supported(s) ? launch_router_tc(s, x, wg, ids, gates, counts, err, st)
                                  : launch_router_wide(s, x, wg, ids, gates, counts, err, st);
  }
  if (s.n_experts <= 8) return launch_router_t<8, 4>(s, x, wg, ids, gates, counts, u_out, eps, st);
  if (s.n_experts <= 16) return launch_router_t<16, 2>(s, x, wg, ids, gates, counts, u_out, eps, st);
  return launch_router_t<32, 1>(s, x, wg, ids, gates, counts, u_out, eps, st);
}

}  // namespace moe
