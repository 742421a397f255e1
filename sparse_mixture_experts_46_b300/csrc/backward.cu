// backward.cu -- the layer backward's CUDA-core kernels: the gradients of the
// gated combine and of the router, the transposes that feed the weight-gradient
// GEMMs, and the final input gradient ("Mixtral of Experts" section 2.1; the
// gradient of y = sum_k G(x)_k E_k(x) with the routing held fixed).
//
//   combine:  dO[row(t,k)] = g[t,k] dy[t]            (bf16, grouped rows)
//             dg[t,k]     = <dy[t], y_perm[row(t,k)]> (fp32, fixed lane order)
//   router:   dl[t,k] = g[t,k] (dg[t,k] - sum_j g[t,j] dg[t,j])
//             dW_g[:, e] = sum over the rows r of expert e of x_perm[r] dl[r]
//   input:    dx[t] = sum_k (dx_perm[row(t,k)] + dl[t,k] W_g[:, e_k])
//   transposes with each expert's rows padded to a multiple of 64 (zeros), so
//   that a weight gradient sum_r P[r] Q[r]^T over an expert's rows is a GEMM
//   over whole 64-row K blocks.
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ void unpack8b(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8b(const float* f) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

}  // namespace

// poff[e] = sum over e' < e of round_up(count_e', 64); poff[n] = total padded rows.
__global__ void __launch_bounds__(kMaxExperts) pad_offsets_kernel(const int32_t* __restrict__ offsets,
                                                                  int n, int R,
                                                                  int32_t* __restrict__ poff) {
  __shared__ int s_scan[33];
  pdl_wait();
  pdl_launch_dependents();
  const int e = threadIdx.x;
  int padded = 0;
  if (e < n) {
    const int lo = min(max(offsets[e], 0), R);
    const int hi = min(max(offsets[e + 1], lo), R);
    padded = (hi - lo + 63) & ~63;
  }
  int total = 0;
  const int ex = block_exclusive_scan(padded, s_scan, &total);
  if (e < n) poff[e] = ex;
  if (e == 0) poff[n] = total;
}

// Grouped activations [R, C] (expert e's rows at [offsets[e], offsets[e+1]))
// -> dst [C, Rpad] with expert e's rows at columns [poff[e], poff[e] + count)
// and zeros up to poff[e+1].  Grid: (C / 64, Rpad_max / 64).
__global__ void __launch_bounds__(256) transpose_grouped_kernel(const uint16_t* __restrict__ src,
                                                                int C, int src_ld,
                                                                const int32_t* __restrict__ offsets,
                                                                const int32_t* __restrict__ poff,
                                                                int n, int R,
                                                                uint16_t* __restrict__ dst,
                                                                int dst_ld) {
  __shared__ uint16_t tile[64][66];
  pdl_wait();
  pdl_launch_dependents();
  const int c0 = blockIdx.x * 64, p0 = blockIdx.y * 64;
  if (p0 >= poff[n]) return;  // beyond the padded rows of this call
  const int e = find_expert(poff, n, p0);
  const int lo = min(max(offsets[e], 0), R);
  const int hi = min(max(offsets[e + 1], lo), R);
  const int r0 = lo + (p0 - poff[e]);  // first source row of this 64-row tile
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int r = i >> 6, c = i & 63;
    tile[r][c] = (r0 + r < hi && c0 + c < C) ? src[(int64_t)(r0 + r) * src_ld + c0 + c] : 0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int c = i >> 6, r = i & 63;
    if (c0 + c < C) dst[(int64_t)(c0 + c) * dst_ld + p0 + r] = tile[r][c];
  }
}

// One warp per assignment (t, k): dO[row] = bf16(g dy[t]), dg[t,k] = <dy[t], y_perm[row]>.
__global__ void __launch_bounds__(256) combine_bwd_kernel(const uint16_t* __restrict__ dy,
                                                          const uint16_t* __restrict__ y_perm,
                                                          const int32_t* __restrict__ slot_row,
                                                          const float* __restrict__ gates, int T,
                                                          int K, int d, int R,
                                                          uint16_t* __restrict__ dO,
                                                          float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  const int nvec = d >> 3;
  for (int a = blockIdx.x * 8 + (threadIdx.x >> 5); a < T * K; a += gridDim.x * 8) {
    const int t = a / K;
    const int row = slot_row[a];
    const float g = gates[a];
    float acc = 0.0f;
    if ((unsigned)row < (unsigned)R) {
      const uint4* dyr = reinterpret_cast<const uint4*>(dy + (size_t)t * d);
      const uint4* yr = reinterpret_cast<const uint4*>(y_perm + (size_t)row * d);
      uint4* outr = reinterpret_cast<uint4*>(dO + (size_t)row * d);
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float fy[8], fo[8], o[8];
        unpack8b(__ldg(dyr + v), fy);
        unpack8b(__ldg(yr + v), fo);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc = fmaf(fy[i], fo[i], acc);
          o[i] = g * fy[i];
        }
        outr[v] = pack8b(o);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) dg[a] = acc;
  }
}

// dl[t,k] = g_k (dg_k - sum_j g_j dg_j); also scattered to the grouped rows.
__global__ void __launch_bounds__(256) router_bwd_kernel(const float* __restrict__ gates,
                                                         const float* __restrict__ dg,
                                                         const int32_t* __restrict__ slot_row,
                                                         int T, int K, int R,
                                                         float* __restrict__ dl,
                                                         float* __restrict__ dl_perm) {
  pdl_wait();
  pdl_launch_dependents();
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int k = 0; k < K; ++k) s = fmaf(gates[t * K + k], dg[t * K + k], s);
    for (int k = 0; k < K; ++k) {
      const float v = gates[t * K + k] * (dg[t * K + k] - s);
      dl[t * K + k] = v;
      const int row = slot_row[t * K + k];
      if ((unsigned)row < (unsigned)R) dl_perm[row] = v;
    }
  }
}

// dW_g[j][e] = sum over the rows r of expert e, ascending, of x_perm[r][j] dl_perm[r].
// Grid: (d / 256, n); thread j of the block owns one column.
__global__ void __launch_bounds__(256) router_wgrad_kernel(const uint16_t* __restrict__ x_perm,
                                                           const float* __restrict__ dl_perm,
                                                           const int32_t* __restrict__ offsets,
                                                           int d, int n, int R,
                                                           float* __restrict__ dwg) {
  pdl_wait();
  pdl_launch_dependents();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int e = blockIdx.y;
  if (j >= d) return;
  const int lo = min(max(offsets[e], 0), R);
  const int hi = min(max(offsets[e + 1], lo), R);
  float acc = 0.0f;
#pragma unroll 8
  for (int r = lo; r < hi; ++r)
    acc = fmaf(__uint_as_float((uint32_t)x_perm[(size_t)r * d + j] << 16), dl_perm[r], acc);
  dwg[(size_t)j * n + e] = acc;
}

// dx[t] = bf16( sum_k (dx_perm[row(t,k)] + dl[t,k] W_g[:, e_k]) ), k ascending.
__global__ void __launch_bounds__(256) input_grad_kernel(const uint16_t* __restrict__ dx_perm,
                                                         const int32_t* __restrict__ slot_row,
                                                         const int32_t* __restrict__ ids,
                                                         const float* __restrict__ dl,
                                                         const uint16_t* __restrict__ wg, int T,
                                                         int K, int d, int n, int R,
                                                         uint16_t* __restrict__ dx) {
  pdl_wait();
  pdl_launch_dependents();
  const int nvec = d >> 3;
  const int64_t total = (int64_t)T * nvec;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / nvec);
    const int v = (int)(i - (int64_t)t * nvec);
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int row = slot_row[t * K + k];
      const int e = ids[t * K + k];
      const float l = dl[t * K + k];
      float f[8];
      if ((unsigned)row < (unsigned)R) {
        unpack8b(__ldg(reinterpret_cast<const uint4*>(dx_perm + (size_t)row * d) + v), f);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] += f[u];
      }
      if ((unsigned)e < (unsigned)n) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          acc[u] = fmaf(l, __uint_as_float((uint32_t)__ldg(wg + (size_t)(v * 8 + u) * n + e) << 16),
                        acc[u]);
      }
    }
    reinterpret_cast<uint4*>(dx + (size_t)t * d)[v] = pack8b(acc);
  }
}

// ------------------------------------------------------------------ host ---

static int cap_blocks(int64_t want) {
  const int64_t cap = (int64_t)num_sms() * 16;
  return (int)(want < 1 ? 1 : (want > cap ? cap : want));
}

cudaError_t launch_pad_offsets(const int32_t* offsets, int n, int R, int32_t* poff,
                               cudaStream_t st) {
  return launch_pdl(pad_offsets_kernel, dim3(1), dim3(kMaxExperts), 0, st, offsets, n, R, poff);
}

cudaError_t launch_transpose_grouped(const uint16_t* src, int C, int src_ld,
                                     const int32_t* offsets, const int32_t* poff, int n, int R,
                                     int rpad_max, uint16_t* dst, int dst_ld, cudaStream_t st) {
  const dim3 grid((unsigned)((C + 63) / 64), (unsigned)(rpad_max / 64));
  return launch_pdl(transpose_grouped_kernel, grid, dim3(256), 0, st, src, C, src_ld, offsets,
                    poff, n, R, dst, dst_ld);
}

cudaError_t launch_combine_bwd(const moe_shape& s, const uint16_t* dy, const uint16_t* y_perm,
                               const int32_t* slot_row, const float* gates, uint16_t* dO,
                               float* dg, cudaStream_t st) {
  const int A = s.T * s.top_k;
  return launch_pdl(combine_bwd_kernel, dim3((unsigned)cap_blocks((A + 7) / 8)), dim3(256), 0, st,
                    dy, y_perm, slot_row, gates, s.T, s.top_k, s.dim, A, dO, dg);
}

cudaError_t launch_router_bwd(const moe_shape& s, const float* gates, const float* dg,
                              const int32_t* slot_row, float* dl, float* dl_perm,
                              cudaStream_t st) {
  return launch_pdl(router_bwd_kernel, dim3((unsigned)cap_blocks((s.T + 255) / 256)), dim3(256), 0,
                    st, gates, dg, slot_row, s.T, s.top_k, s.T * s.top_k, dl, dl_perm);
}

cudaError_t launch_router_wgrad(const moe_shape& s, const uint16_t* x_perm, const float* dl_perm,
                                const int32_t* offsets, float* dwg, cudaStream_t st) {
  const dim3 grid((unsigned)((s.dim + 255) / 256), (unsigned)s.n_experts);
  return launch_pdl(router_wgrad_kernel, grid, dim3(256), 0, st, x_perm, dl_perm, offsets, s.dim,
                    s.n_experts, s.T * s.top_k, dwg);
}

cudaError_t launch_input_grad(const moe_shape& s, const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* ids, const float* dl, const uint16_t* wg, uint16_t* dx,
                              cudaStream_t st) {
  const int64_t total = (int64_t)s.T * (s.dim / 8);
  return launch_pdl(input_grad_kernel, dim3((unsigned)cap_blocks((total + 255) / 256)), dim3(256),
                    0, st, dx_perm, slot_row, ids, dl, wg, s.T, s.top_k, s.dim, s.n_experts,
                    s.T * s.top_k, dx);
}

}  // namespace moe
