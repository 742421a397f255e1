// wgrad_gemm.cu -- weight gradients of the expert SwiGLU FFN on CTA pairs
// (tcgen05 cta_group::2): for every expert e
//   C_e[m][n] = sum over the rows r of expert e of P[r][m] * Q[r][n]   (fp32)
// ("Mixtral of Experts" section 2.1: dW2_e = dO_e^T H_e, dW1_e = dA_e^T X_e,
// dW3_e = dG_e^T X_e, the expert weights' gradients summed over the tokens
// routed to the expert).
//
// Both operands are read as the grouped activations themselves, P [rows, M]
// and Q [rows, N], in which every expert's group starts on a multiple of 64
// rows and is followed by zero rows up to the next group ([offsets[e],
// offsets[e+1])): the reduction over an expert's tokens is a run of whole
// 64-row K blocks, each landing by TMA as 64 rows of 128 bytes (64 columns),
// 128-byte swizzled -- the MN-major operand layout for both A and B, so no
// transposed copy is made.  A pair owns a 256 x 256
// output tile (each CTA 128 rows of P and half of the 256 rows of Q, the MMA
// M = 256 spread over both); the accumulator (2 x 256 TMEM columns, double
// buffered) is drained by four epilogue warps, each owning 32 output rows:
// 32 accumulator columns at a time go to a per-warp shared-memory tile (fp32,
// 128-byte swizzled, double buffered) that a TMA tensor store writes to the
// gradient, so the 4-byte-per-element output leaves as full coalesced lines
// while the next tile's MMAs run.
// Work units: (expert, 256-row block of M, 256-column block of N), round robin
// over the pairs.  An expert without tokens writes zeros.
#include <cudaTypedefs.h>

#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace moe {

struct WgradArgs {
  const int32_t* offsets;  // [n + 1] group starts (multiples of 64); padding rows are zero
  // rows m < m_split go to out0[e][m][:], the rest to out1[e][m - m_split][:]
  // (the output tensor maps view them as [n * rows, N])
  int m_split;
  int m_rest;           // M - m_split
  int m_blocks;         // M / 256
  int n_blocks;         // N / 256
  int N;                // output row length
  int n_experts;
  uint32_t* err;
  uint64_t limit_ns;
};

constexpr int kWgStages = 6;
constexpr int kWgStageBytes = 2 * 128 * 128;  // 128 columns of P + 128 of Q (64 K rows each)
constexpr int kWgStagingBytes = 4 * 2 * 32 * 128;  // per warp: 2 x [32 rows][32 fp32]
constexpr int kWgSmemBytes = kWgStages * kWgStageBytes + kWgStagingBytes + 1024 + 1024;
static_assert(kWgSmemBytes <= 232448, "shared memory");

__global__ void __launch_bounds__(192, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tm_p,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_o0,
                      const __grid_constant__ CUtensorMap tm_o1, const WgradArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* staging = reinterpret_cast<float*>(tiles + kWgStages * kWgStageBytes);
  uint8_t* aux = tiles + kWgStages * kWgStageBytes + kWgStagingBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + kWgStages;
  uint64_t* tfull = empty + kWgStages;  // [2]
  uint64_t* tempty = tfull + 2;         // [2]
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_ok = abort_flag + 1;  // [2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int per_expert = args.m_blocks * args.n_blocks;
  const int total = args.n_experts * per_expert;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWgStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 2);
    mbar_init(&tempty[1], 2);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_p);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_o0);
    tma_prefetch_desc(&tm_o1);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);

  pdl_wait();  // the operands and the offsets are written by earlier kernels
  pdl_launch_dependents();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl wctl{abort_flag, args.err, args.limit_ns};
  // unit -> expert, M block, N block, K blocks [kb0, kb0 + nkb)
  auto decode = [&](int u, int& e, int& mb, int& nb, int& kb0, int& nkb) {
    e = u / per_expert;
    const int local = u - e * per_expert;
    mb = local / args.n_blocks;
    nb = local - mb * args.n_blocks;
    kb0 = args.offsets[e] >> 6;
    nkb = max(args.offsets[e + 1] - args.offsets[e], 0) >> 6;
  };

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = pair; ok && u < total; u += npairs) {
        int e, mb, nb, kb0, nkb;
        decode(u, e, mb, nb, kb0, nkb);
        const int prow = mb * 256 + (int)rank * 128;
        const int qrow = nb * 256 + (int)rank * 128;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWgStages;
          const uint32_t ph = (uint32_t)(it / kWgStages) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * kWgStageBytes);
          const uint32_t bar = smem_map_rank(smem_u32(&full[s]), 0);
          uint8_t* st = tiles + s * kWgStageBytes;
          const int ky = (kb0 + kb) * 64;  // 64 grouped rows = one K block
          tma_load_2d_pair(st, &tm_p, prow, ky, bar);
          tma_load_2d_pair(st + 64 * 128, &tm_p, prow + 64, ky, bar);
          tma_load_2d_pair(st + 128 * 128, &tm_q, qrow, ky, bar);
          tma_load_2d_pair(st + 192 * 128, &tm_q, qrow + 64, ky, bar);
        }
      }
      if (rank == 0)
        for (int j = (it > kWgStages ? it - kWgStages : 0); j < it; ++j)
          pair_drain_wait_shared(&full[j % kWgStages], (uint32_t)(j / kWgStages) & 1u, args.err,
                                 args.limit_ns);
    }
  } else if (warp == 1) {
    if (rank == 0 && lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      // A and B both MN-major
      const uint32_t idesc = idesc_bf16_f32(256, 256) | (1u << 15) | (1u << 16);
      for (int u = pair; ok && u < total; u += npairs, ++lt) {
        int e, mb, nb, kb0, nkb;
        decode(u, e, mb, nb, kb0, nkb);
        const int b = lt & 1;
        const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(&tempty[b], tph ^ 1u, wctl, kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(b * 256);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kWgStages;
          const uint32_t ph = (uint32_t)(it / kWgStages) & 1u;
          if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(tiles + s * kWgStageBytes);
          const uint32_t sb = sa + 128 * 128;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_pair(d0, sdesc_mnmajor_sw128(sa + kk * 2048, 64 * 128, 1024),
                          sdesc_mnmajor_sw128(sb + kk * 2048, 64 * 128, 1024), idesc,
                          (kb | kk) != 0 ? 1u : 0u);
          mma_commit_pair_mc(&empty[s], 0x3);
        }
        if (!ok) break;
        mma_commit_pair_mc(&tfull[b], 0x3);  // with no K block: arrives at once
      }
      mma_commit_pair_mc(drain, 0x1);
      pair_drain_wait_shared(drain, 0, args.err, args.limit_ns);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter = this warp's 32 output rows
    const int et = threadIdx.x - 64;
    float* stg = staging + q * (2 * 32 * 32);  // [2][32][32], 1024-byte aligned halves
    uint32_t chunk = 0;                        // stores issued by this warp so far
    int lt = 0;
    for (int u = pair; u < total; u += npairs, ++lt) {
      const int b = lt & 1;
      const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
      if (et == 0) s_ok[b] = mbar_wait(&tfull[b], tph, wctl, kErrTimeoutEpilogue) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!s_ok[b]) break;
      tc_fence_after_sync();
      int e, mb, nb, kb0, nkb;
      decode(u, e, mb, nb, kb0, nkb);
      const int m0 = mb * 256 + (int)rank * 128 + q * 32;  // this warp's first output row
      const bool lo = m0 < args.m_split;
      const CUtensorMap* tmo = lo ? &tm_o0 : &tm_o1;
      const int y = lo ? e * args.m_split + m0 : e * args.m_rest + (m0 - args.m_split);
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
#pragma unroll 1
      for (int c0 = 0; c0 < 256; c0 += 32, ++chunk) {
        float* buf = stg + (chunk & 1u) * (32 * 32);
        // the store issued from this buffer two chunks ago has read it
        if (chunk >= 2 && lane == 0) bulk_wait_read_le1();
        __syncwarp();
        float v[32];
        if (nkb > 0) {
          tmem_ld_32(tacc + (uint32_t)c0, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        }
        // row `lane` of the tile, 16-byte pieces at the 128-byte swizzle slots
        float* row = buf + lane * 32;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 2)) =
              make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tmo, buf, nb * 256 + c0, y);
          bulk_commit();
        }
      }
      tc_fence_before_sync();
      named_bar_sync(1, 128);
      if (et == 0) mbar_arrive_cluster(smem_map_rank(smem_u32(&tempty[b]), 0));
    }
    if (lane == 0) bulk_wait_all();  // the gradient is written before the CTA exits
  }

  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host ---

static PFN_cuTensorMapEncodeTiled_v12000 wg_encoder() {
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

// Grouped bf16 activations [rows, cols], boxes of 64 columns x 64 rows.
static bool wg_encode(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows) {
  auto enc = wg_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 gradient [rows, cols] stored by 32 x 32 tiles, 128-byte swizzle.
static bool wg_encode_out(CUtensorMap* tm, float* base, uint64_t cols, uint64_t rows) {
  auto enc = wg_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// C_e = P_e^T Q_e for every expert: p [rows, M], q [rows, N] (bf16, expert
// e's group at rows [offsets[e], offsets[e+1]), offsets multiples of 64, the
// rows past the group's tokens zero), M and N multiples of 256.  Rows
// m < m_split of C_e go to out0 ([n, m_split, N] fp32), the others to out1
// ([n, M - m_split, N]); m_split is a multiple of 128.
cudaError_t launch_wgrad(const uint16_t* p, const uint16_t* q, int M, int N, int rows,
                         const int32_t* offsets, int n, float* out0, float* out1, int m_split,
                         uint32_t* err, cudaStream_t st) {
  if (M % 256 != 0 || N % 256 != 0 || rows % 64 != 0 || rows <= 0) return cudaErrorInvalidValue;
  if (m_split <= 0 || m_split > M || m_split % 128 != 0) return cudaErrorInvalidValue;
  const int m_rest = M - m_split;
  CUtensorMap tm_p, tm_q, tm_o0, tm_o1;
  if (!wg_encode(&tm_p, p, M, rows) || !wg_encode(&tm_q, q, N, rows) ||
      !wg_encode_out(&tm_o0, out0, N, (uint64_t)n * m_split) ||
      !wg_encode_out(&tm_o1, m_rest > 0 ? out1 : out0, N,
                     (uint64_t)n * (m_rest > 0 ? m_rest : m_split)))
    return cudaErrorInvalidValue;
  static int grids[64] = {0};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int& grid = grids[dev];
  if (grid == 0) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kWgSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = kWgSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, wgrad_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    grid = 2 * clusters < (num_sms() & ~1) ? 2 * clusters : (num_sms() & ~1);
  }
  const WgradArgs a{offsets, m_split, m_rest, M / 256, N / 256, N, n, err, kWaitLimitNs};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = kWgSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, wgrad_pair_kernel, tm_p, tm_q, tm_o0, tm_o1, a);
}

}  // namespace moe
