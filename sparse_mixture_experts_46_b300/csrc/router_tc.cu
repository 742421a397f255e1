// router_tc.cu -- router logits on the tensor cores, top-K selection and gate
// softmax ("Mixtral of Experts" section 2.1, G(x) = Softmax(TopK(x . W_g))),
// plus the RMSNorm of the residual-stack workload.
//
// The logits l = x . W_g are a skinny GEMM (n <= 16 columns): on CUDA cores
// it costs one FMA and most of an unpack per weight per token, and the warps
// that issue them cannot keep enough loads in flight to stream x at HBM rate.
// Here a CTA owns 128 tokens and a K range of the model dimension:
//   * x tiles (128 tokens x 64 features, bf16, 128-byte swizzle) arrive by TMA
//     through a shared-memory ring of up to 8 stages; the first stages are
//     requested before the W_g slice below is built, so both overlap;
//   * the CTA's slice of W_g is written once, by its threads, transposed into
//     the K-major 128-byte-swizzled layout of a 16-row MMA operand (experts
//     n..15 are zero), so no transposed copy of W_g is needed;
//   * one thread issues tcgen05.mma M=128 x N=16 x K=16 into a 16-column fp32
//     TMEM accumulator (bf16 products are exact, accumulation in fp32);
//   * when the K range is split over a cluster of `split` CTAs (so that enough
//     SMs stream x), CTA r selects for tokens [r*128/split, (r+1)*128/split):
//     every CTA stores its partial logits of those tokens straight into CTA
//     r's shared memory (distributed shared memory, one slot per source rank;
//     the first store waits only for the cluster-barrier phase that every CTA
//     arrives at when it starts), and after one full cluster barrier CTA r sums
//     its slots in rank order (a fixed order: deterministic) without any
//     remote load;
//   * one thread per token selects the top K: scanning experts in ascending
//     order, strictly greater wins, so ties go to the lower index; the gates
//     are the softmax of the selected logits, accumulated in slot order.
// Every wait is bounded; an expired wait records the error word.
#include <cudaTypedefs.h>

#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace moe {

// Error word of the router calls that have no workspace (moe_router_topk);
// moe_check_error reads and clears it together with the workspace word.
__device__ uint32_t g_router_err = 0;

namespace {

constexpr int kRtThreads = 128;
constexpr int kRtMaxStages = 12;
constexpr size_t kRtSmemBudget = 227 * 1024;
constexpr int kRtTileBytes = 128 * 128;  // 128 tokens x 64 bf16
constexpr int kRtWBytes = 16 * 128;      // 16 expert rows x 64 bf16, per K block
constexpr int kRtPartStride = 20;        // floats per partial row (16-byte rows, no bank conflicts)
constexpr int kRtMaxKbPerCta = 64;
constexpr uint32_t kRtIdesc = idesc_bf16_f32(128, 16);

__device__ __forceinline__ void tmem_ld_16(uint32_t ta, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Request the 128-byte line holding `p` into L2.  Nothing is read into
// registers or L1, and L2 is the point of coherence, so the prefetch may be
// issued before pdl_wait(): a line the predecessor writes afterwards is
// updated in L2 like any other.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The two halves of a cluster barrier: arrive without ordering any memory
// access (it only announces that this CTA is running), and wait with acquire
// semantics.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 16-byte store into a cluster peer's shared memory (addr 16-byte aligned).
__device__ __forceinline__ void st_cluster_f32x4(uint32_t addr, float a, float b, float c,
                                                 float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
// 16-byte load from a cluster peer's shared memory (addr 16-byte aligned).
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Top-K of one token's logits l[0..16) (entries >= n are ignored) and the
// softmax of the selected ones; writes ids / gates of token t.
__device__ __forceinline__ void select_topk(const float* l_in, int n, int K, int t,
                                            int32_t* ids, float* gates, int* hist) {
  float l[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float v = l_in[e];
    l[e] = (e < n && v == v) ? v : -INFINITY;  // padding and NaN never beat a real logit
  }
  // two passes of the same selection: ids and the softmax denominator, then
  // the gates (keeps every array statically indexed, i.e. in registers)
  float v0 = 0.0f, denom = 0.0f;
  for (int pass = 0; pass < 2; ++pass) {
    uint32_t taken = 0;
    for (int k = 0; k < K; ++k) {
      float best = 0.0f;
      int bi = -1;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        if (e < n && !((taken >> e) & 1u) && (bi < 0 || l[e] > best)) {
          best = l[e];
          bi = e;
        }
      }
      taken |= 1u << bi;
      if (pass == 0) {
        if (k == 0) v0 = best;
        denom += expf(best - v0);
        ids[(size_t)t * K + k] = bi;
        if (hist != nullptr) atomicAdd(&hist[bi], 1);
      } else {
        gates[(size_t)t * K + k] = expf(best - v0) / denom;
      }
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const uint16_t* __restrict__ wg,
                     int T, int d, int n, int K, int split, int kb_per_cta, int stages,
                     int32_t* __restrict__ ids, float* __restrict__ gates,
                     int32_t* __restrict__ counts, uint32_t* err, uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* bw = ring + stages * kRtTileBytes;                           // [kb][16][128 B]
  float* part = reinterpret_cast<float*>(bw + (size_t)kb_per_cta * kRtWBytes);  // [128][17]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + 128 * kRtPartStride);
  uint64_t* empty = full + kRtMaxStages;
  uint64_t* tfull = empty + kRtMaxStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* hist = abort_flag + 1;  // [kMaxExperts]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = split > 1 ? cluster_ctarank() : 0u;
  const int tile = blockIdx.x / split;
  const int kb0 = (int)rank * kb_per_cta;
  // this CTA is running: peers may store into its partial buffer once they
  // have waited on this phase (just before their first remote store)
  if (split > 1) cluster_arrive_relaxed();

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int e = tid; e < kMaxExperts; e += kRtThreads) hist[e] = 0;
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm_x);
  if (warp == 1) tmem_alloc(tmem_slot, 32);
  {  // this CTA's W_g rows into L2 while the predecessor finishes
    const char* w0 = reinterpret_cast<const char*>(wg + (size_t)kb0 * 64 * n);
    const int bytes = kb_per_cta * 64 * n * 2;
    for (int o = tid * 128; o < bytes; o += kRtThreads * 128) prefetch_l2(w0 + o);
  }

  pdl_wait();  // x and W_g may be written by the previous kernel
  pdl_launch_dependents();
  __syncthreads();  // barriers initialised before the first TMA completes on them
  const int first = kb_per_cta < stages ? kb_per_cta : stages;
  if (tid == 0) {
    // the ring starts filling now; the rest of the x tiles follow below
    for (int kb = 0; kb < first; ++kb) {
      mbar_arrive_expect_tx(&full[kb], kRtTileBytes);
      tma_load_2d(ring + kb * kRtTileBytes, &tm_x, (kb0 + kb) * 64, tile * 128, &full[kb]);
    }
  }

  // W_g rows [64*kb0, 64*(kb0 + kb_per_cta)) transposed into the MMA's B
  // operand: expert e, feature kk of K block kb at byte
  //   kb*2048 + e*128 + ((kk/8) ^ (e%8))*16 + (kk%8)*2,
  // so the 8 features kk..kk+7 (kk a multiple of 8) of one expert are one
  // 16-byte vector.
  const int rows = kb_per_cta * 64;
  if (n == 8 || n == 16) {
    // a thread takes 8 consecutive rows (its loads all in flight), transposes
    // them in registers and writes one 16-byte vector per expert
    for (int g = tid; g < rows / 8; g += kRtThreads) {
      const int i = g * 8;
      uint4 v[8][2];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 2; ++q)
          v[j][q] = q * 8 < n ? __ldg(reinterpret_cast<const uint4*>(wg + (size_t)(kb0 * 64 + i + j) * n) + q)
                              : make_uint4(0u, 0u, 0u, 0u);
      uint8_t* base = bw + (size_t)(i >> 6) * kRtWBytes;
      const int chunk = (i & 63) >> 3;
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint4 a = v[2 * p][e >> 3], b = v[2 * p + 1][e >> 3];
          const uint32_t wa = ((e & 7) >> 1) == 0 ? a.x : ((e & 7) >> 1) == 1 ? a.y : ((e & 7) >> 1) == 2 ? a.z : a.w;
          const uint32_t wb = ((e & 7) >> 1) == 0 ? b.x : ((e & 7) >> 1) == 1 ? b.y : ((e & 7) >> 1) == 2 ? b.z : b.w;
          const uint32_t lo = (e & 1) ? (wa >> 16) : (wa & 0xFFFFu);
          const uint32_t hi = (e & 1) ? (wb >> 16) : (wb & 0xFFFFu);
          w[p] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(base + e * 128 + ((chunk ^ (e & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  } else {
    for (int i = tid; i < rows; i += kRtThreads) {
      const int k = kb0 * 64 + i;
      const int kb = i >> 6, kk = i & 63;
      uint8_t* base = bw + (size_t)kb * kRtWBytes + (kk & 7) * 2;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        *reinterpret_cast<uint16_t*>(base + e * 128 + ((((kk >> 3) ^ (e & 7))) << 4)) =
            e < n ? __ldg(wg + (size_t)k * n + e) : (uint16_t)0;
    }
  }
  // the generic-proxy writes above are read by the tensor core (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem = *tmem_slot;
  const WaitCtl wctl{abort_flag, err, limit_ns};

  if (warp == 0 && lane == 0) {
    // TMA producer: the rest of the x tiles of the CTA's K range
    for (int kb = first; kb < kb_per_cta; ++kb) {
      const int s = kb % stages;
      const uint32_t ph = (uint32_t)(kb / stages) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) break;
      mbar_arrive_expect_tx(&full[s], kRtTileBytes);
      tma_load_2d(ring + s * kRtTileBytes, &tm_x, (kb0 + kb) * 64, tile * 128, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // MMA issuer
    for (int kb = 0; kb < kb_per_cta; ++kb) {
      const int s = kb % stages;
      const uint32_t ph = (uint32_t)(kb / stages) & 1u;
      if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) break;
      tc_fence_after_sync();
      const uint32_t sa = smem_u32(ring + s * kRtTileBytes);
      const uint32_t sb = smem_u32(bw + (size_t)kb * kRtWBytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ss(tmem, sdesc_kmajor_sw128(sa + kk * 32), sdesc_kmajor_sw128(sb + kk * 32),
                    kRtIdesc, (kb | kk) != 0 ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    mma_commit(tfull);  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // epilogue: every warp reads its 32 TMEM lanes (= tokens)
  int ok = 0;
  if (lane == 0) ok = mbar_wait(tfull, 0, wctl, kErrTimeoutEpilogue) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  float lg[16];
  if (ok) {
    tc_fence_after_sync();
    tmem_ld_16(tmem + ((uint32_t)(warp * 32) << 16), lg);
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) lg[e] = 0.0f;
  }
  const int r = warp * 32 + lane;  // token row inside the tile
  int* h = counts != nullptr ? hist : nullptr;
  if (split == 1) {
    const int t = tile * 128 + r;
    if (ok && t < T) select_topk(lg, n, K, t, ids, gates, h);
  } else {
    // token row r belongs to CTA r / per; its partials land in that CTA's
    // slot (this rank, r % per).  The stores are fire-and-forget; the barrier
    // (release / acquire at cluster scope) makes them visible, and after it no
    // CTA touches a peer's shared memory, so none has to wait for the others
    // before leaving.
    const int per = 128 / split;
    cluster_wait();  // every peer of the cluster is running
    const uint32_t dst = smem_map_rank(
        smem_u32(part + ((int)rank * per + r % per) * kRtPartStride), (uint32_t)(r / per));
#pragma unroll
    for (int q = 0; q < 4; ++q)
      st_cluster_f32x4(dst + 16u * q, lg[4 * q], lg[4 * q + 1], lg[4 * q + 2], lg[4 * q + 3]);
    cluster_sync_all();
    if (tid < per) {
      float sum[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) sum[e] = 0.0f;
      for (int c = 0; c < split; ++c) {  // rank order: a fixed summation order
        const float4* src = reinterpret_cast<const float4*>(part + (c * per + tid) * kRtPartStride);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 v = src[q];
          sum[4 * q] += v.x;
          sum[4 * q + 1] += v.y;
          sum[4 * q + 2] += v.z;
          sum[4 * q + 3] += v.w;
        }
      }
      const int t = tile * 128 + (int)rank * per + tid;
      if (t < T && !*abort_flag) select_topk(sum, n, K, t, ids, gates, h);
    }
  }

  __syncthreads();
  if (counts != nullptr && tid < n && hist[tid] != 0) atomicAdd(&counts[tid], hist[tid]);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 32);
  }
}

// ---------------------------------------------------------------------------
// Wide router: 32 < n <= 256 experts (fine-grained MoE, e.g. top 8 of 160).
// W_g tiles arrive by TMA straight from its [dim, n] layout: a box of 64
// experts x 64 features lands as 64 rows (features) of 128 bytes (experts),
// 128-byte swizzled, i.e. the MN-major operand layout; the MMA is M=128 tokens
// x N=round_up(n, 16) x K=16, B marked MN-major in the instruction descriptor
// (matrix descriptor: 1024 bytes between 8-row feature groups, 8 KB between
// 64-expert blocks).  One CTA per 128 tokens, or, when there are too few
// token tiles to cover the SMs (decode batches), a cluster of `split` CTAs
// per tile, each reducing 1/split of the model dimension: every CTA writes
// its 128 x n fp32 partial logits over its (by then idle) operand ring, and
// CTA r adds rows [r*128/split, (r+1)*128/split) of all the cluster's partials
// in rank order (a fixed order) through distributed shared memory.  The thread
// of each token then walks its n logits in ascending expert order and keeps a
// sorted top-K list (strictly greater displaces, so ties keep the lower index).
constexpr int kRwThreads = 128;
constexpr int kRwStages = 4;
constexpr int kRwMaxK = 8;

// Order of the top-K lists: larger logit first, equal logits by lower index.
__device__ __forceinline__ bool rw_before(float a, int ia, float b, int ib) {
  return a > b || (a == b && ia < ib);
}
// A top-K list is kRwMaxK sorted slots whose first kRwMaxK - K hold (+inf, -1),
// which nothing displaces: the K kept entries are the last slots, so the
// current K-th best is always the last slot and most candidates are turned
// away by one comparison (an insertion is a chain through every slot).
__device__ __forceinline__ void rw_init(float* tv, int* ti, int K) {
#pragma unroll
  for (int j = 0; j < kRwMaxK; ++j) {
    const bool pinned = j < kRwMaxK - K;
    tv[j] = pinned ? INFINITY : -INFINITY;
    ti[j] = pinned ? -1 : 0x7fffffff;
  }
}
// Insertion without a chain through the slots: "slot j keeps its entry"
// (the entry is before the candidate) holds for a prefix of the sorted list,
// so every slot's new entry follows from the old list alone -- its own entry,
// the candidate, or the entry one slot up.
__device__ __forceinline__ void rw_insert(float* tv, int* ti, float val, int e) {
  if (!rw_before(val, e, tv[kRwMaxK - 1], ti[kRwMaxK - 1])) return;
  bool keep[kRwMaxK];
#pragma unroll
  for (int j = 0; j < kRwMaxK; ++j) keep[j] = !rw_before(val, e, tv[j], ti[j]);
#pragma unroll
  for (int j = kRwMaxK - 1; j >= 0; --j) {
    if (!keep[j]) {
      const bool here = j == 0 || keep[j - 1];
      tv[j] = here ? val : tv[j > 0 ? j - 1 : 0];
      ti[j] = here ? e : ti[j > 0 ? j - 1 : 0];
    }
  }
}

__global__ void __launch_bounds__(kRwThreads, 1)
    router_tc_wide_kernel(const __grid_constant__ CUtensorMap tm_x,
                          const __grid_constant__ CUtensorMap tm_w, int T, int d, int n, int K,
                          int nblk, int split, int kb_per_cta, int32_t* __restrict__ ids,
                          float* __restrict__ gates, int32_t* __restrict__ counts, uint32_t* err,
                          uint64_t limit_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int stage_bytes = kRtTileBytes + nblk * 8192;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRwStages * stage_bytes);
  uint64_t* empty = full + kRwStages;
  uint64_t* tfull = empty + kRwStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* hist = abort_flag + 1;  // [kMaxExperts]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = split > 1 ? cluster_ctarank() : 0u;
  const int tile = blockIdx.x / split;
  const int kb0 = (int)rank * kb_per_cta;
  const int npad = (n + 15) & ~15;
  const int pstride = npad + 4;  // floats per token row of the partials (16-byte rows)
  float* part = reinterpret_cast<float*>(ring);  // [128][pstride], over the ring once it is idle

  if (tid == 0) {
    for (int s = 0; s < kRwStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int e = tid; e < kMaxExperts; e += kRwThreads) hist[e] = 0;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 256);

  pdl_wait();  // x and W_g may be written by the previous kernel
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wctl{abort_flag, err, limit_ns};

  if (warp == 0 && lane == 0) {
    for (int kb = 0; kb < kb_per_cta; ++kb) {
      const int s = kb % kRwStages;
      const uint32_t ph = (uint32_t)(kb / kRwStages) & 1u;
      if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) break;
      uint8_t* st = ring + s * stage_bytes;
      mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
      tma_load_2d(st, &tm_x, (kb0 + kb) * 64, tile * 128, &full[s]);
      for (int b = 0; b < nblk; ++b)
        tma_load_2d(st + kRtTileBytes + b * 8192, &tm_w, b * 64, (kb0 + kb) * 64, &full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)npad) | (1u << 16);  // B MN-major
    for (int kb = 0; kb < kb_per_cta; ++kb) {
      const int s = kb % kRwStages;
      const uint32_t ph = (uint32_t)(kb / kRwStages) & 1u;
      if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) break;
      tc_fence_after_sync();
      const uint32_t sa = smem_u32(ring + s * stage_bytes);
      const uint32_t sb = sa + kRtTileBytes;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ss(tmem, sdesc_kmajor_sw128(sa + kk * 32),
                    sdesc_mnmajor_sw128(sb + kk * 2048, 8192, 1024), idesc,
                    (kb | kk) != 0 ? 1u : 0u);
      mma_commit(&empty[s]);
    }
    mma_commit(tfull);
  }
  __syncwarp();

  int ok = 0;
  if (lane == 0) ok = mbar_wait(tfull, 0, wctl, kErrTimeoutEpilogue) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  const int r = warp * 32 + lane;  // token row inside the tile = TMEM lane
  // every token row's logits into the partial buffer over the (idle) ring:
  // every MMA, hence every operand read, has completed
  if (ok) tc_fence_after_sync();
  for (int c0 = 0; c0 < npad; c0 += 16) {
    float v[16];
    if (ok) {
      tmem_ld_16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);  // warp-collective
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 16; i += 4)
      *reinterpret_cast<float4*>(part + r * pstride + c0 + i) =
          make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
  }
  const int per = 128 / split;  // token rows this CTA selects for
  const int row0 = (int)rank * per;
  if (split > 1) {
    // every CTA's partials are visible cluster-wide (and every peer, having
    // arrived here, is running)
    cluster_sync_all();
    // this CTA's token rows: the sum over the cluster in rank order, written
    // back over its own rows (no peer reads them); one item = 4 experts of a
    // row, every peer's 16 bytes requested before the sum
    const int n4 = npad >> 2;
    for (int i = tid; i < per * n4; i += kRwThreads) {
      const int rr = row0 + i / n4;
      const int e = (i - (i / n4) * n4) * 4;
      const uint32_t local = smem_u32(part + rr * pstride + e);
      float4 pv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (c < split) pv[c] = ld_cluster_f32x4(smem_map_rank(local, (uint32_t)c));
      float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        if (c < split) {  // rank order: a fixed summation order
          sum.x += pv[c].x;
          sum.y += pv[c].y;
          sum.z += pv[c].z;
          sum.w += pv[c].w;
        }
      }
      *reinterpret_cast<float4*>(part + rr * pstride + e) = sum;
    }
  }
  __syncthreads();
  // selection: `split` threads per token row (G = 128 / per); thread g keeps
  // the top K of experts g, g + G, ... (NaN counts as -inf), then the G lists
  // are merged into thread 0's; the list order is total, so the result does
  // not depend on the order of the merge
  {
    const int G = split;
    const int rl = tid / G, g = tid - (tid / G) * G;
    const float* row = part + (row0 + rl) * pstride;
    float tv[kRwMaxK];
    int ti[kRwMaxK];
    rw_init(tv, ti, K);
    for (int e = g; e < n; e += G) {
      const float x = row[e];
      rw_insert(tv, ti, x == x ? x : -INFINITY, e);
    }
    // merge the row's G lists (consecutive lanes of one warp) as a tree of
    // shuffles: at distance d, lane g (g % 2d == 0) takes the kept entries of
    // lane g + d
    for (int d = 1; d < G; d <<= 1) {
#pragma unroll
      for (int j = 0; j < kRwMaxK; ++j) {
        const float pv = __shfl_down_sync(0xffffffffu, tv[j], d);
        const int pi = __shfl_down_sync(0xffffffffu, ti[j], d);
        if ((g & (2 * d - 1)) == 0 && j >= kRwMaxK - K) rw_insert(tv, ti, pv, pi);
      }
    }
    const int t = tile * 128 + row0 + rl;
    if (g == 0 && ok && t < T && !*abort_flag) {
      // slot k of the output is list slot kRwMaxK - K + k
      // the largest kept logit (the list is sorted and holds no NaN)
      float v0 = -INFINITY;
#pragma unroll
      for (int j = 0; j < kRwMaxK; ++j)
        if (j >= kRwMaxK - K) v0 = fmaxf(v0, tv[j]);
      float denom = 0.0f;
#pragma unroll
      for (int j = 0; j < kRwMaxK; ++j)
        if (j >= kRwMaxK - K) denom += expf(tv[j] - v0);
#pragma unroll
      for (int j = 0; j < kRwMaxK; ++j) {
        if (j >= kRwMaxK - K) {
          const int k = j - (kRwMaxK - K);
          ids[(size_t)t * K + k] = ti[j];
          gates[(size_t)t * K + k] = expf(tv[j] - v0) / denom;
          if (counts != nullptr) atomicAdd(&hist[ti[j]], 1);
        }
      }
    }
  }
  if (split > 1) cluster_sync_all();  // no CTA leaves while a peer may still read its partials
  __syncthreads();
  if (counts != nullptr)
    for (int e = tid; e < n; e += kRwThreads)
      if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

// u = bf16(x / sqrt(mean(x^2) + eps)), one warp per token: the sum of squares
// over the row (fixed lane order, warp butterfly), then the scaled row.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* __restrict__ x, int T,
                                                      int d, float eps,
                                                      uint16_t* __restrict__ u) {
  const int lane = threadIdx.x & 31;
  const int nchunks = d >> 3;
  pdl_wait();
  pdl_launch_dependents();
  for (int t = blockIdx.x * 8 + (threadIdx.x >> 5); t < T; t += gridDim.x * 8) {
    const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)t * d);
    float ss = 0.0f;
#pragma unroll 8
    for (int c = lane; c < nchunks; c += 32) {
      const uint4 v = __ldg(row + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rs = 1.0f / sqrtf(ss / (float)d + eps);
    uint4* out = reinterpret_cast<uint4*>(u + (size_t)t * d);
#pragma unroll 8
    for (int c = lane; c < nchunks; c += 32) {
      const uint4 v = __ldg(row + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        p[i] = pack_bf16x2(__uint_as_float(w[i] << 16) * rs,
                           __uint_as_float(w[i] & 0xFFFF0000u) * rs);
      out[c] = make_uint4(p[0], p[1], p[2], p[3]);
    }
  }
}

// ------------------------------------------------------------------ host ---

static PFN_cuTensorMapEncodeTiled_v12000 rt_tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool router_wide_supported(const moe_shape& s) {
  return s.n_experts > 32 && s.n_experts <= kMaxExperts && s.n_experts % 8 == 0 &&
         s.top_k <= kRwMaxK && s.dim % 64 == 0;
}

bool router_tc_supported(const moe_shape& s) {
  if (s.n_experts > 16 || s.dim % 64 != 0) return false;
  const int kb = s.dim / 64;
  int split = 1;
  while (kb / split > kRtMaxKbPerCta && split < 8) split *= 2;
  return kb % split == 0 && kb / split <= kRtMaxKbPerCta;
}

static cudaError_t router_err_word(uint32_t** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_router_err);
}

cudaError_t router_err_read_clear(uint32_t* word) {
  uint32_t* p = nullptr;
  cudaError_t e = router_err_word(&p);
  if (e != cudaSuccess) return e;
  e = cudaMemcpy(word, p, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess || *word == 0) return e;
  const uint32_t zero = 0;
  return cudaMemcpy(p, &zero, sizeof(uint32_t), cudaMemcpyHostToDevice);
}

cudaError_t launch_router_tc(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                             int32_t* ids, float* gates, int32_t* counts, uint32_t* err,
                             cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  if (err == nullptr) {
    cudaError_t e = router_err_word(&err);
    if (e != cudaSuccess) return e;
  }
  auto enc = rt_tensor_map_encoder();
  if (enc == nullptr) return cudaErrorInvalidValue;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {(cuuint64_t)s.dim, (cuuint64_t)s.T};
  const cuuint64_t strides[1] = {(cuuint64_t)s.dim * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  // split the K range over a cluster until the grid covers the SMs (and the
  // CTA's W_g slice fits in shared memory)
  const int tiles = (s.T + 127) / 128;
  const int kb = s.dim / 64;
  int split = 1;
  while (split < 8 && kb % (split * 2) == 0 &&
         (tiles * split * 2 <= num_sms() || kb / split > kRtMaxKbPerCta))
    split *= 2;
  const int kb_per = kb / split;
  const size_t fixed = 1024 + (size_t)kb_per * kRtWBytes + 128 * kRtPartStride * 4 + 2048;
  int stages = (int)((kRtSmemBudget - fixed) / kRtTileBytes);
  if (stages > kRtMaxStages) stages = kRtMaxStages;
  if (stages > kb_per) stages = kb_per;
  if (stages < 2) stages = 2;
  const size_t smem = fixed + (size_t)stages * kRtTileBytes;
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * split));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_tc_kernel, tm, wg, s.T, s.dim, s.n_experts, s.top_k,
                            split, kb_per, stages, ids, gates, counts, err, kWaitLimitNs);
}

cudaError_t launch_router_wide(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                               int32_t* ids, float* gates, int32_t* counts, uint32_t* err,
                               cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  if (err == nullptr) {
    cudaError_t e = router_err_word(&err);
    if (e != cudaSuccess) return e;
  }
  auto enc = rt_tensor_map_encoder();
  if (enc == nullptr) return cudaErrorInvalidValue;
  CUtensorMap tm_x, tm_w;
  const cuuint32_t estr[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)s.dim, (cuuint64_t)s.T};
    const cuuint64_t strides[1] = {(cuuint64_t)s.dim * 2};
    const cuuint32_t box[2] = {64, 128};
    if (enc(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // W_g [dim, n]: experts are the contiguous (inner) dimension
    const cuuint64_t dims[2] = {(cuuint64_t)s.n_experts, (cuuint64_t)s.dim};
    const cuuint64_t strides[1] = {(cuuint64_t)s.n_experts * 2};
    const cuuint32_t box[2] = {64, 64};
    if (enc(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(wg), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int nblk = (s.n_experts + 63) / 64;
  const size_t ring = (size_t)kRwStages * (kRtTileBytes + nblk * 8192);
  // the partial logits [128][npad + 4] fp32 reuse the ring
  static_assert((size_t)kRwStages * (kRtTileBytes + 8192) >= 128 * (64 + 4) * 4, "partials");
  // + barriers, flags and the count histogram
  const size_t smem = 1024 + ring + 2048;
  cudaError_t e = cudaFuncSetAttribute(router_tc_wide_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // split the model dimension over a cluster until the grid covers the SMs
  const int tiles = (s.T + 127) / 128;
  const int kb = s.dim / 64;
  int split = 1;
  while (split < 8 && kb % (split * 2) == 0 && tiles * split * 2 <= num_sms()) split *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * split));
  cfg.blockDim = dim3(kRwThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, router_tc_wide_kernel, tm_x, tm_w, s.T, s.dim, s.n_experts,
                            s.top_k, nblk, split, kb / split, ids, gates, counts, err,
                            kWaitLimitNs);
}

cudaError_t launch_rmsnorm(const moe_shape& s, const uint16_t* x, float eps, uint16_t* u,
                           cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  int64_t blocks = (s.T + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(rmsnorm_kernel, dim3((unsigned)blocks), dim3(256), 0, st, x, s.T, s.dim, eps,
                    u);
}

}  // namespace moe
