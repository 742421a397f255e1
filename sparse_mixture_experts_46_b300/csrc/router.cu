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
        if (!((taken >> e) & 1u) && (bi < 0 || l[e] > best)) {
          best = l[e];
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
        if (!((taken >> e) & 1u) && (bi < 0 || l[e] > best)) {
          best = l[e];
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

// ---------------------------------------------------------------------------
// Large-batch router: one warp owns TPW = 32 / NE consecutive tokens.
//
// W_g is staged once per block in shared memory as [NE/8][8][d/8] rows of 8
// experts (16 bytes): row (q, jj, c) holds W_g[8c + jj][8q .. 8q + 7], so the
// 32 lanes of a warp, which own consecutive 8-element slices c of the token
// row, read consecutive 16-byte rows (no bank conflicts).  Every lane keeps
// TPW x NE = 32 fp32 partial logits; a butterfly reduce-scatter (31 shuffles,
// a fixed tree, deterministic) leaves lane l with the logit of token
// t0 + l / NE and expert l % NE.  The top K are then chosen inside each group
// of NE lanes by K argmax butterflies (strictly greater wins, ties go to the
// lower expert index), and the gates are the softmax of the selected logits
// in slot order.
template <int NE>
__global__ void __launch_bounds__(128) router_warp_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int T, int d, int n, int K,
    int32_t* __restrict__ ids, float* __restrict__ gates, int32_t* __restrict__ counts,
    uint16_t* __restrict__ u_out, float eps) {
  constexpr int TPW = 32 / NE;
  constexpr int NQ = NE / 8;
  extern __shared__ __align__(16) uint4 s_w[];  // [NQ][8][d/8] rows of 8 bf16
  __shared__ int s_hist[kMaxExperts];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int nchunks = d >> 3;
  const bool norm = (u_out != nullptr);
  if (tid < kMaxExperts) s_hist[tid] = 0;

  pdl_wait();  // x and W_g may be written by the previous kernel
  pdl_launch_dependents();
  if (n == NE) {
    // asynchronous 16-byte copies: every row of the block's share is in flight at once
    for (int i = tid; i < d * NQ; i += blockDim.x) {
      const int j = i % d;  // W_g row
      const int q = i / d;  // group of 8 experts
      const uint32_t dst = smem_u32(&s_w[(size_t)(q * 8 + (j & 7)) * nchunks + (j >> 3)]);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                   "l"(reinterpret_cast<const uint4*>(wg + (size_t)j * NE) + q)
                   : "memory");
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // n < NE: scalar loads, the padding experts get zero weights
    for (int i = tid; i < d * NQ; i += blockDim.x) {
      const int j = i % d;
      const int q = i / d;
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const int e0 = q * 8 + 2 * h;
        const uint32_t lo = e0 < n ? __ldg(wg + (size_t)j * n + e0) : 0u;
        const uint32_t hi = e0 + 1 < n ? __ldg(wg + (size_t)j * n + e0 + 1) : 0u;
        w[h] = lo | (hi << 16);
      }
      s_w[(size_t)(q * 8 + (j & 7)) * nchunks + (j >> 3)] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  __syncthreads();

  const int gw = blockIdx.x * (blockDim.x >> 5) + (tid >> 5);
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int ngroups = (T + TPW - 1) / TPW;

  // x slices of the group's TPW tokens, streamed through a PF-deep register
  // ring: the loads of slice c + 32*PF are issued before slice c is used, so
  // PF global loads per token are always in flight.
  constexpr int PF = 4;
  auto load_slice = [&](uint4* dst, int t0, int c) {
#pragma unroll
    for (int t = 0; t < TPW; ++t)
      dst[t] = (c < nchunks && t0 + t < T)
                   ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * d) + c)
                   : make_uint4(0u, 0u, 0u, 0u);
  };
  auto for_each_slice = [&](int t0, auto&& body) {
    uint4 ring[PF][TPW];
#pragma unroll
    for (int p = 0; p < PF; ++p) load_slice(ring[p], t0, lane + 32 * p);
    for (int base = 0; base < nchunks; base += 32 * PF) {
#pragma unroll
      for (int p = 0; p < PF; ++p) {
        const int c = base + lane + 32 * p;
        if (c < nchunks) {
          uint4 cur[TPW];
#pragma unroll
          for (int t = 0; t < TPW; ++t) cur[t] = ring[p][t];
          load_slice(ring[p], t0, c + 32 * PF);
          body(cur, c);
        }
      }
    }
  };

  for (int g = gw; g < ngroups; g += nw) {
    const int t0 = g * TPW;
    float rs[TPW];
#pragma unroll
    for (int t = 0; t < TPW; ++t) rs[t] = 1.0f;
    if (norm) {
      float ss[TPW];
#pragma unroll
      for (int t = 0; t < TPW; ++t) ss[t] = 0.0f;
      for_each_slice(t0, [&](const uint4* cur, int) {
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
          float f[8];
          unpack8(cur[t], f);
#pragma unroll
          for (int i = 0; i < 8; ++i) ss[t] = fmaf(f[i], f[i], ss[t]);
        }
      });
#pragma unroll
      for (int t = 0; t < TPW; ++t) rs[t] = 1.0f / sqrtf(warp_sum(ss[t]) / (float)d + eps);
    }

    float acc[TPW][NE];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int e = 0; e < NE; ++e) acc[t][e] = 0.0f;
    for_each_slice(t0, [&](const uint4* cur, int c) {
      float xv[TPW][8];
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        unpack8(cur[t], xv[t]);
        if (norm && t0 + t < T) {
          const size_t off = (size_t)(t0 + t) * d + (size_t)c * 8;
          uint32_t pk[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pk[i] = pack_bf16x2(xv[t][2 * i] * rs[t], xv[t][2 * i + 1] * rs[t]);
            xv[t][2 * i] = __uint_as_float(pk[i] << 16);
            xv[t][2 * i + 1] = __uint_as_float(pk[i] & 0xFFFF0000u);
          }
          *reinterpret_cast<uint4*>(u_out + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float w[8];
          unpack8(s_w[(size_t)(q * 8 + jj) * nchunks + c], w);
#pragma unroll
          for (int t = 0; t < TPW; ++t)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              acc[t][q * 8 + i] = fmaf(xv[t][jj], w[i], acc[t][q * 8 + i]);
        }
      }
    });

    // reduce-scatter of the 32 partial sums: lane l ends with value index l
    float* v = &acc[0][0];
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
      const bool upper = (lane & s) != 0;
#pragma unroll
      for (int i = 0; i < s; ++i) {
        const float send = upper ? v[i] : v[i + s];
        const float keep = upper ? v[i + s] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
      }
    }
    const int t = t0 + lane / NE;
    const int e = lane % NE;
    float lv = v[0];
    if (e >= n || !(lv == lv)) lv = -INFINITY;  // padding and NaN never beat a real logit

    // top-K inside the NE-lane group; every lane follows the selection
    float v0 = 0.0f, denom = 0.0f, mine = 0.0f;
    int my_slot = -1;
    float cur = lv;
    for (int k = 0; k < K; ++k) {
      float bv = cur;
      int be = (my_slot < 0) ? e : kMaxExperts;  // taken lanes cannot win again
      if (my_slot >= 0) bv = -INFINITY;
#pragma unroll
      for (int o = 1; o < NE; o <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if (k == 0) v0 = bv;
      denom += expf(bv - v0);
      if (be == e) {
        my_slot = k;
        mine = bv;
      }
    }
    if (t < T && my_slot >= 0) {
      ids[(size_t)t * K + my_slot] = e;
      gates[(size_t)t * K + my_slot] = expf(mine - v0) / denom;
      if (counts != nullptr) atomicAdd(&s_hist[e], 1);
    }
  }
  if (counts != nullptr) {
    __syncthreads();
    if (tid < n && s_hist[tid] != 0) atomicAdd(&counts[tid], s_hist[tid]);
  }
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

// The warp router takes batches of at least this many tokens whose W_g
// (padded to 8 or 16 experts) fits in shared memory.
constexpr int kWarpRouterMinT = 512;
constexpr size_t kWarpRouterMaxBytes = 128 * 1024;

template <int NE>
static cudaError_t launch_router_warp(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                                      int32_t* ids, float* gates, int32_t* counts,
                                      uint16_t* u_out, float eps, size_t wbytes, cudaStream_t st) {
  auto kern = router_warp_kernel<NE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kWarpRouterMaxBytes);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, wbytes);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int groups = (s.T + (32 / NE) - 1) / (32 / NE);
  int blocks = (groups + 3) / 4;  // four warps per block, one token group each
  if (blocks > per_sm * num_sms()) blocks = per_sm * num_sms();
  return launch_pdl(kern, dim3(blocks), dim3(128), wbytes, st, x, wg, s.T, s.dim, s.n_experts,
                    s.top_k, ids, gates, counts, u_out, eps);
}

cudaError_t launch_router(const moe_shape& s, const uint16_t* x, const uint16_t* wg, int32_t* ids,
                          float* gates, int32_t* counts, uint16_t* u_out, float eps,
                          cudaStream_t st) {
  if (counts != nullptr) {
    cudaError_t e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * s.n_experts, st);
    if (e != cudaSuccess) return e;
  }
  if (s.T == 0) return cudaSuccess;
  if (s.T >= kWarpRouterMinT && s.n_experts <= 16) {
    const int ne = s.n_experts <= 8 ? 8 : 16;
    const size_t wbytes = (size_t)s.dim * ne * 2;
    if (wbytes <= kWarpRouterMaxBytes) {
      return ne == 8 ? launch_router_warp<8>(s, x, wg, ids, gates, counts, u_out, eps, wbytes, st)
                     : launch_router_warp<16>(s, x, wg, ids, gates, counts, u_out, eps, wbytes, st);
    }
  }
  if (s.n_experts <= 8) return launch_router_t<8, 4>(s, x, wg, ids, gates, counts, u_out, eps, st);
  if (s.n_experts <= 16) return launch_router_t<16, 2>(s, x, wg, ids, gates, counts, u_out, eps, st);
  return launch_router_t<32, 1>(s, x, wg, ids, gates, counts, u_out, eps, st);
}

}  // namespace moe
