// device.cuh -- sm_103a building blocks written as inline PTX: shared-memory
// mbarriers with bounded waits, TMA tiled loads, and the tcgen05 tensor-core
// instructions (TMEM allocation, MMA issue/commit, TMEM -> register loads).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// Workspace error word bits (OR-ed in by kernels, read by moe_check_error).
enum : uint32_t {
  kErrTimeoutProducer = 1u << 0,
  kErrTimeoutMma = 1u << 1,
  kErrTimeoutEpilogue = 1u << 2,
  kErrTimeoutDrain = 1u << 3,
  kErrTimeoutSelftest = 1u << 4,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ mbarrier ---

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Control block of the bounded waits of one CTA.
struct WaitCtl {
  volatile int* abort;    // shared flag: set once any wait of the CTA expired
  uint32_t* err;          // global error word
  uint64_t limit_ns;      // per-wait limit
};

// Wait until the phase of parity `parity` of `bar` has completed.  Returns
// false (and records `code`) if it did not complete within w.limit_ns, or if
// another role of the CTA already gave up.  Never traps, never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*w.abort) return false;
      if (global_timer_ns() - t0 > w.limit_ns) {
        atomicOr(w.err, code);
        *w.abort = 1;
        return false;
      }
    }
  }
}

// Exclusive prefix sum of v over the threads of the block (blockDim.x a
// multiple of 32, at most 1024); every thread must call it.  *total receives
// the sum over the block.  s_scan: 33 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_scan, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_scan[warp] = incl;  // warp totals
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? s_scan[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_scan[lane] = wi - w;           // exclusive prefix of the warp totals
    if (lane == 31) s_scan[32] = wi;  // block total
  }
  __syncthreads();
  const int r = incl - v + s_scan[warp];
  *total = s_scan[32];
  __syncthreads();  // s_scan may be reused by the caller
  return r;
}

// Tile schedule of a grouped GEMM from the device-resident offsets: expert e
// owns rows [s_off[e], s_end[e]) (clamped into [0, rows_total]), split into
// s_tiles[e] token tiles of `tok_tile` rows; its work units are
// s_start[e] .. s_start[e+1] (tiles x `w_units` weight tiles, expert-major).
// The group of expert e ends at offsets[e + 1], or, with `counts` (groups
// padded apart), at offsets[e] + counts[e].
// With s_span (nullable): s_span[e] = token tiles per L2 block of expert e --
// all of its tiles when its activation rows (row_bytes each) fit in
// `l2_budget` bytes, else the fewest equal blocks that do (see pair_gemm.cu).
// Every thread of the block calls it; s_scan is 33 ints of shared memory.
__device__ __forceinline__ void build_tile_schedule(const int32_t* offsets, int n, int rows_total,
                                                    int tok_tile, int w_units, int* s_off,
                                                    int* s_end, int* s_tiles, int* s_start,
                                                    int* s_scan, const int32_t* counts = nullptr,
                                                    int* s_span = nullptr, int64_t row_bytes = 0,
                                                    int64_t l2_budget = 0) {
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int e = base + (int)threadIdx.x;
    int units = 0;
    if (e < n) {
      const int lo = min(max(offsets[e], 0), rows_total);
      const int end = counts != nullptr ? lo + max(counts[e], 0) : offsets[e + 1];
      const int hi = min(max(end, lo), rows_total);
      const int tt = (hi - lo + tok_tile - 1) / tok_tile;
      s_off[e] = lo;
      s_end[e] = hi;
      s_tiles[e] = tt;
      units = tt * w_units;
      if (s_span != nullptr) {
        const int64_t bytes = (int64_t)(hi - lo) * row_bytes;
        int64_t blocks = l2_budget > 0 ? (bytes + l2_budget - 1) / l2_budget : 1;
        if (blocks > tt) blocks = tt;
        if (blocks < 1) blocks = 1;
        const int nb = (int)blocks;
        s_span[e] = tt > 0 ? (tt + nb - 1) / nb : 1;
      }
    }
    int total = 0;
    const int ex = block_exclusive_scan(units, s_scan, &total);
    if (e < n) s_start[e] = carry + ex;
    carry += total;
  }
  if (threadIdx.x == 0) s_start[n] = carry;
  __syncthreads();
}

// Expert owning work unit t: the largest e with s_start[e] <= t (t < s_start[n]).
__device__ __forceinline__ int find_expert(const int* s_start, int n, int t) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_start[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Bounded wait that ignores the abort flag: lets copies and MMAs that are
// already in flight land before a CTA exits (records kErrTimeoutDrain).
__device__ __forceinline__ void pair_drain_wait_shared(uint64_t* bar, uint32_t parity,
                                                       uint32_t* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrTimeoutDrain);
      return;
    }
  }
}

// ----------------------------------------------------------------- TMA ---

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes on
// `bar`.  c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int32_t c0,
                                            int32_t c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (createpolicy encoding).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* tm, int32_t c0,
                                                 int32_t c1, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------- tcgen05 ---

// Allocate `ncols` TMEM columns (power of two >= 32); executed by one full warp.
// The base address is written to shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major, shape M x N (x K=16).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4)               // D format: f32
         | (1u << 7)             // A format: bf16
         | (1u << 10)            // B format: bf16
         | ((N >> 3) << 17)      // N / 8
         | ((M >> 4) << 24);     // M / 16
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes (64 bf16 of K), 8-row swizzle
// atoms of 1024 bytes stacked along M/N (stride byte offset 1024).  The tile
// must start on a 1024-byte boundary; advancing `addr` by 32 bytes selects the
// next K=16 slice inside the 128-byte row.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);          // start address
  d |= static_cast<uint64_t>(1u) << 16;                         // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                 // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                         // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                         // 128-byte swizzle
  return d;
}

// TMA tensor store from shared memory (bulk-group completion), and the group
// waits: `.read` returns once the source shared memory may be rewritten.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, const void* src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(tm),
      "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Generic-proxy shared-memory writes made visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// MN-major operand, 128-byte swizzle: rows of 128 bytes hold 64 consecutive
// M (or N) elements of one K index; `lbo` bytes separate 64-element M/N
// blocks and `sbo` bytes separate groups of 8 K rows.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t addr, uint32_t lbo,
                                                        uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T, single CTA; `accumulate` = 0 overwrites.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every previously issued tcgen05.mma of this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Load 16 consecutive fp32 columns of this thread's TMEM lane at each of two
// addresses (warp-collective), and wait for completion.
__device__ __forceinline__ void tmem_ld_2x16(uint32_t ta, uint32_t tb, float* a, float* b) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[16 + i]);
  }
}

// ---------------------------------------------------------------- misc ---

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float silu_mul(float a, float g) {
  // SiLU(a) * g = a * g / (1 + exp(-a))
  return a * g / (1.0f + __expf(-a));
}

}  // namespace moe

namespace moe {

// Programmatic dependent launch.  Kernels of the layer are launched with the
// programmatic-stream-serialization attribute: a kernel may start (and run
// its prologue) while its predecessor is still finishing, and pdl_wait()
// blocks until the predecessor grid has completed and its writes are visible.
// Every kernel calls pdl_wait() before its first global-memory access that
// depends on earlier work, and writes no global memory before it.  Without
// the attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace moe

namespace moe {

// ------------------------------------------------- CTA pairs (cluster of 2) ---
// A CTA pair runs one tcgen05 MMA of M = 256 rows: each CTA holds 128 rows of
// A and its own 128-lane slice of the accumulator, and half of the N columns
// of B; the MMA is issued by the even CTA of the pair for both.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the object at shared::cta address `a` in CTA
// `rank` of this cluster.
__device__ __forceinline__ uint32_t smem_map_rank(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Every thread of both CTAs: release this CTA's prior shared-memory writes and
// wait until all threads of the cluster have arrived.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive (release, cluster scope) on the mbarrier at shared::cluster address
// `bar`, which may belong to the other CTA of the pair.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory; the bytes are counted on
// the mbarrier at shared::cluster address `bar`, which may be the pair peer's.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, int32_t c0,
                                                 int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// TMEM allocation shared by the pair: one warp of EACH CTA executes it with the
// same column count; both receive the same base address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A * B^T over the pair (M = 256): A and B descriptors address the
// same shared-memory offsets in both CTAs.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at the same offset in every CTA of `mask` when
// all previously issued pair MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective)
// and wait for completion.
__device__ __forceinline__ void tmem_ld_32(uint32_t ta, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(ta)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier over the `nthreads` threads that use id `id` (1..15).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace moe
