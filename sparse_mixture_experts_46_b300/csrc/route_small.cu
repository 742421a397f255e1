// route_small.cu -- routing of a small batch in one launch: router logits,
// top-K selection and gate softmax ("Mixtral of Experts" section 2.1,
// G(x) = Softmax(TopK(x . W_g))), then the expert grouping of the T*K
// assignments and the gather of the grouped rows.
//
// For a decode-sized batch (T <= 32 tokens, n <= 8 experts) the router, the
// grouping and the gather are each a chain of latencies, not of bandwidth
// (x is 128 KB and W_g 64 KB at Mixtral dims); run as three kernels they cost
// about 20 us.  Here one cluster of 8 CTAs does all of it:
//   1. CTA r takes the model-dimension slice [r*d/8, (r+1)*d/8) (its W_g rows
//      are requested into L2 before the kernel waits for its predecessor).
//      Warp w owns tokens w, w+8, w+16, w+24; lane l walks the 16-byte slices
//      l, l+32, ... of the CTA's dimension range, two at a time (every load
//      of both in flight), multiplying the token rows with the 8 W_g rows of
//      the slice (bf16 products are exact in fp32, accumulation in fp32).  A
//      butterfly reduce-scatter over the warp's lanes leaves lane l with the
//      warp's sum for (token slot l/8, expert l%8).
//   2. Every CTA stores its partial logits into slot r of EVERY CTA's shared
//      memory (distributed shared memory); one cluster barrier later each CTA
//      holds all 8 partials and, with no further exchange, adds them in rank
//      order (a fixed order: the 8 CTAs run the same arithmetic on the same
//      values, so they agree bit for bit), and one thread per token selects
//      the top K: scanning experts in ascending order, strictly greater wins,
//      so ties go to the lower index and a NaN logit never beats a real one;
//      the gates are the softmax of the selected logits, accumulated in slot
//      order.
//   3. Every CTA groups the assignments a = t*K + k by expert, stably (tokens
//      ascending inside a group); CTA 0 writes ids, gates, offsets, slot_row
//      and perm_src.
//   4. Each CTA copies its share of the grouped rows x_perm[r] = x[perm_src[r]]
//      with 16-byte moves, from its own copy of the grouping.
// No wait in this kernel spins on memory: the only synchronisation is one
// hardware cluster barrier, after which no CTA touches a peer's shared memory.
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kRsThreads = 256;
constexpr int kRsCluster = 8;
constexpr int kRsMaxT = 32;
constexpr int kRsNE = 8;                       // experts handled (n <= 8)
constexpr int kRsMaxR = kRsMaxT * kRsNE;       // assignments (K <= n <= 8)

__device__ __forceinline__ void unpack8r(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Request the 128-byte line holding `p` into L2.  Nothing is read into
// registers or L1, and L2 is the point of coherence, so the prefetch may be
// issued before pdl_wait(): a line the predecessor writes afterwards is
// updated in L2 like any other.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void st_cluster_f32r(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

}  // namespace

__global__ void __launch_bounds__(kRsThreads, 1)
    route_small_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wg, int T,
                       int d, int n, int K, int32_t* __restrict__ ids,
                       float* __restrict__ gates, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ perm_src, int32_t* __restrict__ slot_row,
                       uint16_t* __restrict__ x_perm) {
  __shared__ float s_part[kRsCluster][kRsMaxT * kRsNE];  // rank c's partial logits [token][expert]
  __shared__ float s_logit[kRsMaxT * kRsNE];
  __shared__ int s_ids[kRsMaxR];              // expert of assignment a
  __shared__ int s_perm[kRsMaxR];             // token of grouped row r
  __shared__ int s_wcnt[kRsThreads / 32][kRsNE];
  __shared__ int s_base[kRsNE];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int R = T * K;
  const int dc = d / kRsCluster;  // dimensions of this CTA (a multiple of 16)
  const int d0 = (int)rank * dc;
  const int slices = dc >> 3;

  {  // this CTA's W_g rows into L2 while the predecessor finishes
    const char* w0 = reinterpret_cast<const char*>(wg + (size_t)d0 * n);
    const int bytes = dc * n * 2;
    for (int o = tid * 128; o < bytes; o += kRsThreads * 128) prefetch_l2(w0 + o);
  }
  if (tid < kRsNE * (kRsThreads / 32)) s_wcnt[tid / kRsNE][tid % kRsNE] = 0;
  pdl_wait();  // x and W_g may be written by the previous kernel
  pdl_launch_dependents();

  // ---- 1. partial logits of this CTA's dimension slice
  float acc[4][kRsNE];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < kRsNE; ++e) acc[i][e] = 0.0f;
  // one 16-byte slice at dd: W_g rows dd..dd+7 (8 experts each) times the
  // warp's 4 token rows
  auto fma_slice = [&](const uint4* wv, const uint4* xv) {
    float w[8][kRsNE];
#pragma unroll
    for (int j = 0; j < 8; ++j) unpack8r(wv[j], w[j]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float xf[8];
      unpack8r(xv[i], xf);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < kRsNE; ++e) acc[i][e] = fmaf(xf[j], w[j][e], acc[i][e]);
    }
  };
  auto load_x = [&](int dd, uint4* xv) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = warp + 8 * i;
      xv[i] = t < T ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + dd))
                    : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (n == kRsNE) {
    // slices s and s + 32 per round: all 24 loads issued before the first use
    for (int s = lane; s < slices; s += 64) {
      const bool two = s + 32 < slices;
      uint4 wv[2][8], xv[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int dd = d0 + (s + 32 * h) * 8;
        if (h == 0 || two) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            wv[h][j] = __ldg(reinterpret_cast<const uint4*>(wg + (size_t)(dd + j) * kRsNE));
          load_x(dd, xv[h]);
        }
      }
      fma_slice(wv[0], xv[0]);
      if (two) fma_slice(wv[1], xv[1]);
    }
  } else {
    // n < 8: W_g rows of n bf16 are not 16-byte aligned; experts >= n are zero
    for (int s = lane; s < slices; s += 32) {
      const int dd = d0 + s * 8;
      uint4 wv[8], xv[4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        uint32_t u[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e0 = 2 * q, e1 = 2 * q + 1;
          const uint32_t lo = e0 < n ? (uint32_t)__ldg(wg + (size_t)(dd + j) * n + e0) : 0u;
          const uint32_t hi = e1 < n ? (uint32_t)__ldg(wg + (size_t)(dd + j) * n + e1) : 0u;
          u[q] = lo | (hi << 16);
        }
        wv[j] = make_uint4(u[0], u[1], u[2], u[3]);
      }
      load_x(dd, xv);
      fma_slice(wv, xv);
    }
  }
  // butterfly reduce-scatter of the 32 values over the warp: lane l keeps the
  // warp's sum of value l (token slot l / 8, expert l % 8)
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int e = 0; e < kRsNE; ++e) v[i * kRsNE + e] = acc[i][e];
#pragma unroll
  for (int half = 16; half >= 1; half >>= 1) {
    const bool up = (lane & half) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
    }
  }

  // ---- 2. this CTA's partials into slot `rank` of every CTA of the cluster
  {
    const int t = warp + 8 * (lane >> 3);  // rows t >= T hold zeros and are never read
    const uint32_t local = smem_u32(&s_part[rank][t * kRsNE + (lane & 7)]);
#pragma unroll
    for (int c = 0; c < kRsCluster; ++c) st_cluster_f32r(smem_map_rank(local, (uint32_t)c), v[0]);
  }
  cluster_sync_all();  // every CTA holds all partials; no DSMEM access after this

  if (tid < T * kRsNE) {
    float sum = 0.0f;
#pragma unroll
    for (int c = 0; c < kRsCluster; ++c) sum += s_part[c][tid];  // rank order
    s_logit[tid] = sum;
  }
  __syncthreads();
  if (tid < T) {
    float l[kRsNE];
#pragma unroll
    for (int e = 0; e < kRsNE; ++e) {
      const float lv = s_logit[tid * kRsNE + e];
      l[e] = (e < n && lv == lv) ? lv : -INFINITY;
    }
    float v0 = 0.0f, denom = 0.0f;
    float sel[kRsNE];
    uint32_t taken = 0;
    for (int k = 0; k < K; ++k) {
      float best = 0.0f;
      int bi = -1;
#pragma unroll
      for (int e = 0; e < kRsNE; ++e)
        if (e < n && !((taken >> e) & 1u) && (bi < 0 || l[e] > best)) {
          best = l[e];
          bi = e;
        }
      taken |= 1u << bi;
      if (k == 0) v0 = best;
      sel[k] = best;
      denom += expf(best - v0);
      s_ids[tid * K + k] = bi;
      if (rank == 0) ids[(size_t)tid * K + k] = bi;
    }
    if (rank == 0)
      for (int k = 0; k < K; ++k) gates[(size_t)tid * K + k] = expf(sel[k] - v0) / denom;
  }
  __syncthreads();

  // ---- 3. stable grouping of the R <= 256 assignments (one per thread)
  const int e = tid < R ? s_ids[tid] : -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned lower = peers & ((1u << lane) - 1u);
  if (e >= 0 && lower == 0) s_wcnt[warp][e] = __popc(peers);
  __syncthreads();
  if (warp == 0) {
    // lane x: the size of expert x's group, then an exclusive scan over lanes
    int cnt = 0;
    if (lane < kRsNE)
#pragma unroll
      for (int w = 0; w < kRsThreads / 32; ++w) cnt += s_wcnt[w][lane];
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kRsNE; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane < kRsNE) s_base[lane] = incl - cnt;
    if (rank == 0 && lane <= n) offsets[lane] = lane < n ? incl - cnt : R;
  }
  __syncthreads();
  if (e >= 0) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_wcnt[w][e];
    const int row = s_base[e] + before + __popc(lower);
    s_perm[row] = tid / K;
    if (rank == 0) {
      slot_row[tid] = row;
      perm_src[row] = tid / K;
    }
  }
  __syncthreads();

  // ---- 4. gather: x_perm[r] = x[perm_src[r]], rows split over the cluster
  const int vec = d >> 3;
  const int total = R * vec;
  const int stride = kRsCluster * kRsThreads;
  for (int i0 = (int)rank * kRsThreads + tid; i0 < total; i0 += 4 * stride) {
    uint4 val[4];
    int r[4], c[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * stride;
      r[u] = i < total ? i / vec : -1;
      c[u] = i < total ? i - r[u] * vec : 0;
      val[u] = r[u] >= 0 ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)s_perm[r[u]] * d) + c[u])
                         : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (r[u] >= 0) reinterpret_cast<uint4*>(x_perm + (size_t)r[u] * d)[c[u]] = val[u];
  }
}

bool route_small_supported(const moe_shape& s) {
  return s.T >= 1 && s.T <= kRsMaxT && s.n_experts <= kRsNE && s.top_k <= s.n_experts &&
         s.dim % (kRsCluster * 16) == 0;
}

cudaError_t launch_route_small(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                               int32_t* ids, float* gates, int32_t* offsets, int32_t* perm_src,
                               int32_t* slot_row, uint16_t* x_perm, cudaStream_t st) {
  if (!route_small_supported(s)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kRsCluster);
  cfg.blockDim = dim3(kRsThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRsCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, route_small_kernel, x, wg, s.T, s.dim, s.n_experts, s.top_k,
                            ids, gates, offsets, perm_src, slot_row, x_perm);
}

}  // namespace moe
