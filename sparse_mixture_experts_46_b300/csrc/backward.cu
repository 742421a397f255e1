// backward.cu -- the layer backward's CUDA-core kernels: the gradients of the
// gated combine and of the router, the zeroing of the padding rows between the
// expert groups, and the final input gradient ("Mixtral of Experts" section 2.1; the
// gradient of y = sum_k G(x)_k E_k(x) with the routing held fixed).
//
//   combine:  dO[row(t,k)] = g[t,k] dy[t]            (bf16, grouped rows)
//             dg[t,k]     = <dy[t], y_perm[row(t,k)]> (fp32, fixed lane order)
//   router:   dl[t,k] = g[t,k] (dg[t,k] - sum_j g[t,j] dg[t,j])
//             dW_g[:, e] = sum over the rows r of expert e of x_perm[r] dl[r]
//   input:    dx[t] = sum_k (dx_perm[row(t,k)] + dl[t,k] W_g[:, e_k])
// The backward groups its rows with every expert's group starting on a
// multiple of 64 rows; the padding rows of the grouped activations are zeroed
// here, so that a weight gradient sum_r P[r]^T Q[r] over an expert's group is
// a GEMM over whole 64-row K blocks.
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

// Zero rows [offsets[e] + counts[e], offsets[e+1]) of each buffer (<= 63 rows
// per expert).  Grid: (n * 64, 3): block (e, i) clears padding row i of expert
// e (if there is one) in the buffer blockIdx.y picks.
struct PadBufs {
  uint16_t* p[3];
  int cols[3];
};

__global__ void __launch_bounds__(256) zero_pad_rows_kernel(const int32_t* __restrict__ offsets,
                                                            const int32_t* __restrict__ counts,
                                                            int rows, const PadBufs bufs) {
  pdl_wait();
  pdl_launch_dependents();
  const int e = blockIdx.x >> 6;
  uint16_t* base = bufs.p[blockIdx.y];
  const int cols = bufs.cols[blockIdx.y];
  if (base == nullptr) return;
  const int lo = min(max(offsets[e] + counts[e], 0), rows);
  const int hi = min(max(offsets[e + 1], lo), rows);
  const int r = lo + (int)(blockIdx.x & 63);
  if (r >= hi) return;
  uint4* row = reinterpret_cast<uint4*>(base + (size_t)r * cols);
  for (int i = threadIdx.x; i < (cols >> 3); i += blockDim.x) row[i] = make_uint4(0u, 0u, 0u, 0u);
}

// wgT[e][j] = wg[j][e]: the router weight with each expert's column as a
// contiguous row, for the input gradient's 16-byte loads.
__global__ void __launch_bounds__(256) transpose_wg_kernel(const uint16_t* __restrict__ wg, int d,
                                                           int n, uint16_t* __restrict__ wgT) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d * n; i += gridDim.x * blockDim.x) {
    const int e = i / d, j = i - e * d;
    wgT[i] = wg[(size_t)j * n + e];
  }
}

// One warp per assignment (t, k): dO[row] = bf16(g dy[t]), dg[t,k] = <dy[t], y_perm[row]>.
__global__ void __launch_bounds__(256) combine_bwd_kernel(const uint16_t* __restrict__ dy,
                                                          const uint16_t* __restrict__ y_perm,
                                                          const int32_t* __restrict__ slot_row,
                                                          const float* __restrict__ gates, int T,
                                                          int K, int d, int rows,
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
    if ((unsigned)row < (unsigned)rows) {
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
                                                         int T, int K, int rows,
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
      if ((unsigned)row < (unsigned)rows) dl_perm[row] = v;
    }
  }
}

// dW_g[j][e] = sum over the rows r of expert e's group of x_perm[r][j] dl_perm[r].
// Grid: (d / 256, n), 512 threads: warp w takes rows lo + w, lo + w + 16, ...
// of the group, each lane 8 consecutive columns (one 16-byte load per row);
// the 16 warps' partial sums are then added in warp order, so the result does
// not depend on timing.
constexpr int kRwgWarps = 16;

__global__ void __launch_bounds__(kRwgWarps * 32) router_wgrad_kernel(
    const uint16_t* __restrict__ x_perm, const float* __restrict__ dl_perm,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ counts, int d, int n,
    int rows, float* __restrict__ dwg) {
  __shared__ float part[kRwgWarps][256];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int e = blockIdx.y;
  const int j0 = blockIdx.x * 256 + lane * 8;  // this lane's 8 columns
  const int lo = min(max(offsets[e], 0), rows);
  const int hi = min(lo + max(counts[e], 0), rows);
  float acc[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) acc[u] = 0.0f;
  if (j0 < d) {
#pragma unroll 4
    for (int r = lo + w; r < hi; r += kRwgWarps) {
      float f[8];
      unpack8b(__ldg(reinterpret_cast<const uint4*>(x_perm + (size_t)r * d + j0)), f);
      const float l = __ldg(dl_perm + r);
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = fmaf(f[u], l, acc[u]);
    }
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) part[w][lane * 8 + u] = acc[u];
  __syncthreads();
  if (threadIdx.x < 256) {
    const int j = blockIdx.x * 256 + threadIdx.x;
    float sum = 0.0f;
#pragma unroll
    for (int v = 0; v < kRwgWarps; ++v) sum += part[v][threadIdx.x];
    if (j < d) dwg[(size_t)j * n + e] = sum;
  }
}

// dx[t] = bf16( sum_k (dx_perm[row(t,k)] + dl[t,k] W_g[:, e_k]) ), k ascending
// (wgT: W_g transposed, [n, d]).
__global__ void __launch_bounds__(256) input_grad_kernel(const uint16_t* __restrict__ dx_perm,
                                                         const int32_t* __restrict__ slot_row,
                                                         const int32_t* __restrict__ ids,
                                                         const float* __restrict__ dl,
                                                         const uint16_t* __restrict__ wgT, int T,
                                                         int K, int d, int n, int rows,
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
      if ((unsigned)row < (unsigned)rows) {
        unpack8b(__ldg(reinterpret_cast<const uint4*>(dx_perm + (size_t)row * d) + v), f);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] += f[u];
      }
      if ((unsigned)e < (unsigned)n) {
        float w[8];
        unpack8b(__ldg(reinterpret_cast<const uint4*>(wgT + (size_t)e * d) + v), w);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = fmaf(l, w[u], acc[u]);
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

cudaError_t launch_zero_pad_rows(const int32_t* offsets, const int32_t* counts, int n, int rows,
                                 uint16_t* b0, int c0, uint16_t* b1, int c1, uint16_t* b2, int c2,
                                 cudaStream_t st) {
  if (c0 % 8 != 0 || c1 % 8 != 0 || c2 % 8 != 0) return cudaErrorInvalidValue;
  const PadBufs bufs{{b0, b1, b2}, {c0, c1, c2}};
  return launch_pdl(zero_pad_rows_kernel, dim3((unsigned)n * 64, 3), dim3(256), 0, st, offsets,
                    counts, rows, bufs);
}

cudaError_t launch_combine_bwd(const moe_shape& s, const uint16_t* dy, const uint16_t* y_perm,
                               const int32_t* slot_row, const float* gates, int rows,
                               uint16_t* dO, float* dg, cudaStream_t st) {
  const int A = s.T * s.top_k;
  return launch_pdl(combine_bwd_kernel, dim3((unsigned)cap_blocks((A + 7) / 8)), dim3(256), 0, st,
                    dy, y_perm, slot_row, gates, s.T, s.top_k, s.dim, rows, dO, dg);
}

cudaError_t launch_router_bwd(const moe_shape& s, const float* gates, const float* dg,
                              const int32_t* slot_row, int rows, float* dl, float* dl_perm,
                              cudaStream_t st) {
  return launch_pdl(router_bwd_kernel, dim3((unsigned)cap_blocks((s.T + 255) / 256)), dim3(256), 0,
                    st, gates, dg, slot_row, s.T, s.top_k, rows, dl, dl_perm);
}

cudaError_t launch_router_wgrad(const moe_shape& s, const uint16_t* x_perm, const float* dl_perm,
                                const int32_t* offsets, const int32_t* counts, int rows,
                                float* dwg, cudaStream_t st) {
  if (s.dim % 8 != 0) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((s.dim + 255) / 256), (unsigned)s.n_experts);
  return launch_pdl(router_wgrad_kernel, grid, dim3(kRwgWarps * 32), 0, st, x_perm, dl_perm,
                    offsets, counts, s.dim, s.n_experts, rows, dwg);
}

cudaError_t launch_input_grad(const moe_shape& s, const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* ids, const float* dl, const uint16_t* wg,
                              uint16_t* wgT, int rows, uint16_t* dx, cudaStream_t st) {
  const int dn = s.dim * s.n_experts;
  cudaError_t e = launch_pdl(transpose_wg_kernel, dim3((unsigned)cap_blocks((dn + 255) / 256)),
                             dim3(256), 0, st, wg, s.dim, s.n_experts, wgT);
  if (e != cudaSuccess) return e;
  const int64_t total = (int64_t)s.T * (s.dim / 8);
  return launch_pdl(input_grad_kernel, dim3((unsigned)cap_blocks((total + 255) / 256)), dim3(256),
                    0, st, dx_perm, slot_row, ids, dl, (const uint16_t*)wgT, s.T, s.top_k, s.dim,
                    s.n_experts, rows, dx);
}

}  // namespace moe
