// permute.cu -- expert grouping of the T*K assignments (the per-expert token
// groups of "Mixtral of Experts" section 2.1: experts receive different
// numbers of tokens and each group is processed as one dense block).
//
// The grouped order is the stable sort of the flat assignments a = t*K + k by
// expert id.  It is built without any order-dependent atomics, so it is
// bit-reproducible:
//   1. hist:    every block of kPermuteChunk assignments counts its experts;
//   2. scan:    one block turns the [chunk, expert] counts into per-expert
//               totals, offsets (exclusive prefix over experts) and each
//               chunk's first row inside every expert group;
//   3. scatter: every block ranks its assignments inside their expert
//               (warp match + popcount, then a prefix over the block's warps),
//               writing slot_row[a] and perm_src[row];
//   4. gather:  x_perm[row] = x[perm_src[row]], 16-byte vector moves, one
//               thread per slice.
// For small T*K (decode batches) steps 1-3 run as one single-block kernel, and
// up to 8192 assignments (a Mixtral prefill batch of 4096 tokens) as one
// cluster of up to 8 blocks.
// With pad > 1 every expert's group starts on a multiple of `pad` rows
// (offsets are then the padded starts and the group of e ends at
// offsets[e] + counts[e]); the padding rows get perm_src = -1 and are written
// as zeros by the gather.
#include "device.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(kPermuteChunk) permute_hist_kernel(const int32_t* __restrict__ ids,
                                                                     int R, int n,
                                                                     int32_t* __restrict__ hist) {
  __shared__ int s[kMaxExperts];
  for (int e = threadIdx.x; e < n; e += blockDim.x) s[e] = 0;
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  const int a = blockIdx.x * kPermuteChunk + threadIdx.x;
  if (a < R) {
    const int e = ids[a];
    if ((unsigned)e < (unsigned)n) atomicAdd(&s[e], 1);  // ids outside [0, n) are ignored
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) hist[(size_t)blockIdx.x * n + e] = s[e];
}

// One block of kMaxExperts threads: thread e owns expert e.
__global__ void __launch_bounds__(kMaxExperts) permute_scan_kernel(const int32_t* __restrict__ hist,
                                                                   int nchunks, int n, int pad,
                                                                   int32_t* __restrict__ counts,
                                                                   int32_t* __restrict__ offsets,
                                                                   int32_t* __restrict__ chunk_base,
                                                                   int32_t* __restrict__ perm_src) {
  __shared__ int s_scan[33];
  const int e = threadIdx.x;
  int total = 0;
  pdl_wait();
  pdl_launch_dependents();
  if (e < n) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = hist[(size_t)c * n + e];
      chunk_base[(size_t)c * n + e] = total;  // rank of the chunk's first row inside expert e
      total += v;
    }
  }
  // exclusive prefix over experts (threads >= n contribute 0)
  const int seg = (total + pad - 1) / pad * pad;
  int all = 0;
  const int excl = block_exclusive_scan(seg, s_scan, &all);
  if (e < n) {
    if (counts) counts[e] = total;
    offsets[e] = excl;
    for (int c = 0; c < nchunks; ++c) chunk_base[(size_t)c * n + e] += excl;
    for (int r = excl + total; r < excl + seg; ++r) perm_src[r] = -1;  // padding rows
  }
  if (e == 0) offsets[n] = all;
}

__global__ void __launch_bounds__(kPermuteChunk) permute_scatter_kernel(
    const int32_t* __restrict__ ids, int R, int K, int n, const int32_t* __restrict__ chunk_base,
    int32_t* __restrict__ perm_src, int32_t* __restrict__ slot_row) {
  constexpr int kWarps = kPermuteChunk / 32;
  __shared__ int wcnt[kWarps][kMaxExperts];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kWarps * kMaxExperts; i += blockDim.x) (&wcnt[0][0])[i] = 0;
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();

  const int a = blockIdx.x * kPermuteChunk + threadIdx.x;
  int e = (a < R) ? ids[a] : -1;
  if ((unsigned)e >= (unsigned)n) e = -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned lower = peers & ((1u << lane) - 1u);
  const int rank_in_warp = __popc(lower);
  if (e >= 0 && lower == 0) wcnt[warp][e] = __popc(peers);  // group leader
  __syncthreads();
  if (e >= 0) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += wcnt[w][e];
    const int row = chunk_base[(size_t)blockIdx.x * n + e] + before + rank_in_warp;
    slot_row[a] = row;
    perm_src[row] = a / K;
  }
}

// x_perm[r, :] = x[perm_src[r], :]; one thread per 16-byte slice of a row
// (flat grid), four slices in flight per thread.  Rows whose perm_src
// is not a token (padding; or ids outside [0, n)) are written as zeros.  With
// `rows_used` (device, padded groups) rows at or past *rows_used are skipped.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ perm_src,
                                                          int R, int d, int T,
                                                          const int32_t* __restrict__ rows_used,
                                                          uint16_t* __restrict__ x_perm) {
  const int vec = d >> 3;
  pdl_wait();
  pdl_launch_dependents();
  const int rows = rows_used != nullptr ? min(max(*rows_used, 0), R) : R;
  const int64_t total = (int64_t)rows * vec;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // 4 slices per round (i, i + stride, ...): their source rows, then their
  // 16 bytes, are all requested before the first store
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    int r[4], v[4], t[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      r[u] = i < total ? (int)(i / vec) : -1;
      v[u] = i < total ? (int)(i - (int64_t)r[u] * vec) : 0;
      t[u] = r[u] >= 0 ? __ldg(perm_src + r[u]) : -1;
    }
    uint4 val[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      val[u] = (unsigned)t[u] < (unsigned)T
                   ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)t[u] * d) + v[u])
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (r[u] >= 0) reinterpret_cast<uint4*>(x_perm + (size_t)r[u] * d)[v[u]] = val[u];
  }
}

// Steps 1-3 in one block of 1024 threads, for small T*K (<= kSmallPermute):
// a shared histogram gives counts and offsets; the assignments are then
// ranked 1024 at a time (warp match + popcount, prefix over the 32 warps, and
// a running row base per expert carried from one 1024-slice to the next).
constexpr int kSmallPermute = 2048;

__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* __restrict__ ids,
                                                            int R, int K, int n, int pad,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ perm_src,
                                                            int32_t* __restrict__ slot_row) {
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_wcnt[32][kMaxExperts];
  __shared__ int s_scan[33];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  if (tid < kMaxExperts) s_cnt[tid] = 0;
  for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  for (int a = tid; a < R; a += blockDim.x) {
    const int e = ids[a];
    if ((unsigned)e < (unsigned)n) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  {
    const int total = tid < n ? s_cnt[tid] : 0;
    const int seg = (total + pad - 1) / pad * pad;
    int all = 0;
    const int excl = block_exclusive_scan(seg, s_scan, &all);
    if (tid < n) {
      s_base[tid] = excl;
      offsets[tid] = excl;
      if (counts) counts[tid] = total;
      for (int r = excl + total; r < excl + seg; ++r) perm_src[r] = -1;  // padding rows
    }
    if (tid == 0) offsets[n] = all;
  }
  __syncthreads();
  for (int c0 = 0; c0 < R; c0 += blockDim.x) {
    const int a = c0 + tid;
    int e = (a < R) ? ids[a] : -1;
    if ((unsigned)e >= (unsigned)n) e = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (e >= 0 && lower == 0) s_wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_wcnt[w][e];
      const int row = s_base[e] + before + __popc(lower);
      slot_row[a] = row;
      perm_src[row] = a / K;
    }
    __syncthreads();
    if (tid < n) {
      int add = 0;
      for (int w = 0; w < 32; ++w) {
        add += s_wcnt[w][tid];
        s_wcnt[w][tid] = 0;
      }
      s_base[tid] += add;
    }
    __syncthreads();
  }
}

// Steps 1-3 for kSmallPermute < T*K <= kClusterPermute, pad == 1: one cluster
// of ceil(T*K / 1024) blocks, one assignment per thread (block r takes the
// slice [1024 r, 1024 (r+1))).  Each block counts its slice's experts (warp
// match + popcount) and stores the counts into slot r of EVERY block's shared
// memory (distributed shared memory); after the launch's one full cluster
// barrier each block derives on its own the expert totals, the offsets (their
// exclusive prefix) and where its slice starts inside every expert group (the
// slices before it, in rank order), then ranks its assignments -- the same
// stable order as the other paths.  Block 0 writes counts and offsets.
constexpr int kClusterPermuteCtas = 8;
constexpr int kClusterPermute = kClusterPermuteCtas * 1024;

__device__ __forceinline__ void st_cluster_s32p(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__global__ void __launch_bounds__(1024) permute_cluster_kernel(const int32_t* __restrict__ ids,
                                                              int R, int K, int n,
                                                              int32_t* __restrict__ counts,
                                                              int32_t* __restrict__ offsets,
                                                              int32_t* __restrict__ perm_src,
                                                              int32_t* __restrict__ slot_row) {
  __shared__ int s_wcnt[32][kMaxExperts];
  __shared__ int s_slice[kClusterPermuteCtas][kMaxExperts];  // each block's counts
  __shared__ int s_base[kMaxExperts];
  __shared__ int s_scan[33];
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int nct = (int)gridDim.x;  // the whole grid is one cluster
  // this block is running: peers may store into it once they have waited on
  // this phase (just before their first remote store)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  for (int i = tid; i < 32 * kMaxExperts; i += blockDim.x) (&s_wcnt[0][0])[i] = 0;
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();
  const int a = (int)rank * 1024 + tid;
  int e = (a < R) ? ids[a] : -1;
  if ((unsigned)e >= (unsigned)n) e = -1;  // ids outside [0, n) are ignored
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const unsigned lower = peers & ((1u << lane) - 1u);
  if (e >= 0 && lower == 0) s_wcnt[warp][e] = __popc(peers);
  __syncthreads();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every block is running
  if (tid < n) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += s_wcnt[w][tid];
    const uint32_t local = smem_u32(&s_slice[rank][tid]);
    for (int q = 0; q < nct; ++q) st_cluster_s32p(smem_map_rank(local, (uint32_t)q), c);
  }
  cluster_sync_all();  // every block's counts everywhere; no remote access after this
  int total = 0, before = 0;
  if (tid < n) {
    for (int q = 0; q < nct; ++q) {
      const int v = s_slice[q][tid];
      total += v;
      if (q < (int)rank) before += v;
    }
  }
  int all = 0;
  const int excl = block_exclusive_scan(total, s_scan, &all);
  if (tid < n) {
    s_base[tid] = excl + before;
    if (rank == 0) {
      offsets[tid] = excl;
      if (counts) counts[tid] = total;
    }
  }
  if (rank == 0 && tid == 0) offsets[n] = all;
  __syncthreads();
  if (e >= 0) {
    int bw = 0;
    for (int w = 0; w < warp; ++w) bw += s_wcnt[w][e];
    const int row = s_base[e] + bw + __popc(lower);
    slot_row[a] = row;
    perm_src[row] = a / K;
  }
}

cudaError_t launch_permute(const moe_shape& s, const uint16_t* x, const int32_t* ids,
                           int32_t* counts_out, int32_t* offsets, int32_t* chunk_hist,
                           int32_t* chunk_base, int32_t* perm_src, int32_t* slot_row,
                           uint16_t* x_perm, int nchunks, cudaStream_t st, int pad,
                           int rows_alloc) {
  const int R = s.T * s.top_k;
  if (pad < 1) return cudaErrorInvalidValue;
  if (pad > 1 && rows_alloc < permute_padded_rows(R, s.n_experts, pad))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (R <= kSmallPermute) {
    e = launch_pdl(permute_small_kernel, dim3(1), dim3(1024), 0, st, ids, R, s.top_k, s.n_experts,
                   pad, counts_out, offsets, perm_src, slot_row);
    if (e != cudaSuccess) return e;
  } else if (R <= kClusterPermute && pad == 1) {
    const int nct = (R + 1023) / 1024;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nct);
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nct;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, permute_cluster_kernel, ids, R, s.top_k, s.n_experts, counts_out,
                           offsets, perm_src, slot_row);
    if (e != cudaSuccess) return e;
  } else {
    e = launch_pdl(permute_hist_kernel, dim3(nchunks), dim3(kPermuteChunk), 0, st, ids, R,
                   s.n_experts, chunk_hist);
    if (e != cudaSuccess) return e;
    e = launch_pdl(permute_scan_kernel, dim3(1), dim3(kMaxExperts), 0, st, (const int32_t*)chunk_hist,
                   nchunks, s.n_experts, pad, counts_out, offsets, chunk_base, perm_src);
    if (e != cudaSuccess) return e;
    e = launch_pdl(permute_scatter_kernel, dim3(nchunks), dim3(kPermuteChunk), 0, st, ids, R,
                   s.top_k, s.n_experts, (const int32_t*)chunk_base, perm_src, slot_row);
    if (e != cudaSuccess) return e;
  }
  if (R == 0) return cudaSuccess;
  if (x_perm != nullptr) {
    const int rows = pad > 1 ? rows_alloc : R;
    const int64_t total = (int64_t)rows * (s.dim / 8);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    e = launch_pdl(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, x,
                   (const int32_t*)perm_src, rows, s.dim, s.T,
                   pad > 1 ? (const int32_t*)(offsets + s.n_experts) : (const int32_t*)nullptr,
                   x_perm);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
