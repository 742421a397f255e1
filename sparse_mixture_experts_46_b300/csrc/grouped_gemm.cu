// grouped_gemm.cu -- expert SwiGLU FFN as two grouped GEMMs over variable-size
// expert groups, on the 5th-generation tensor cores (tcgen05 + TMEM), fed by
// TMA ("Mixtral of Experts" section 2.1: each selected expert is a SwiGLU
// feed-forward block; the per-expert token groups have different sizes).
//
//   pass 1 (gate/up, GLU):  H[r]      = bf16(SiLU(X[r] W1_e^T) * (X[r] W3_e^T))
//   pass 2 (down):          Y_perm[r] = bf16(H[r] W2_e^T)
// for every grouped row r of expert e (rows [offsets[e], offsets[e+1])).
//
// One persistent kernel template, two operand layouts:
//  * tokens on M (SWAP = false; large T): the MMA is 128 token rows x N weight
//    rows.  In pass 1 the B tile stacks 128 rows of W1 over the same 128 rows
//    of W3, so one M128xN256 MMA produces both halves of the gate in TMEM and
//    the epilogue applies SiLU(a)*g column-pair-wise.  In pass 2 B is 256 (or
//    128) rows of W2.
//  * weights on M (SWAP = true; small T): the MMA is 128 weight rows x N = 32
//    token rows, so every weight byte is streamed from HBM exactly once per
//    32-token chunk of an expert; pass 1 issues two MMAs per K-slice (W1 and
//    W3 tiles against the same token tile) into two TMEM accumulators.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (one thread): fills a STAGES-deep shared-memory
//               ring, one mbarrier pair (full/empty) per stage;
//   warp 1      TMEM owner + MMA issuer (one thread): tcgen05.mma per 16-wide
//               K slice, tcgen05.commit frees the ring slot and, after the
//               last K block, signals the accumulator;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane TMEM quarter, SwiGLU /
//               convert, bf16 stores; double-buffered accumulators let the
//               epilogue of tile i overlap the main loop of tile i+1.
// Tiles are scheduled from the device-resident offsets (the host never sees
// the per-expert counts): tile t -> expert e, weight tile wt, token tile at,
// ordered expert-major, then weight tile, then token tile, so CTAs working at
// the same time share weight tiles through L2.
//
// Every wait is bounded (device.cuh): on expiry the CTA records the error
// word, lets its in-flight TMA copies and MMAs land, frees TMEM and exits.
#include <cudaTypedefs.h>

#include <cmath>

#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace moe {

struct GemmArgs {
  const int32_t* offsets;  // [n + 1] grouped-row offsets (device)
  uint16_t* out;           // H [R, hidden] (pass 1) or y_perm [R, dim] (pass 2)
  uint32_t* err;           // workspace error word
  uint64_t limit_ns;       // bounded-wait limit
  int n_experts;
  int k_blocks;            // reduction length / 64
  int w_tiles;             // weight tiles per expert
  int w_rows_per_expert;   // rows of one expert's weight matrix (hidden or dim)
  int out_ld;              // output row stride in elements
  int rows_total;          // R: grouped rows (offsets are clamped to [0, R])
};

template <bool SWAP, bool GLU, int BN, int STAGES>
struct GemmCfg {
  static constexpr int BK = 64;                                // bf16 per 128-byte row
  static constexpr int A_BYTES = 128 * 128;                    // one 128-row operand tile
  static constexpr int NUM_A = (SWAP && GLU) ? 2 : 1;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = NUM_A * A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = (SWAP && GLU) ? 2 * BN : BN;  // fp32 columns per buffer
  static constexpr int TMEM_COLS = (2 * ACC_COLS <= 32)    ? 32
                                   : (2 * ACC_COLS <= 64)  ? 64
                                   : (2 * ACC_COLS <= 128) ? 128
                                   : (2 * ACC_COLS <= 256) ? 256
                                                           : 512;
  static constexpr int ACT_ROWS = SWAP ? BN : 128;             // token rows per tile
  static constexpr int W_ROWS = SWAP ? 128 : (GLU ? BN / 2 : BN);  // weight rows per matrix
  static constexpr uint32_t IDESC = idesc_bf16_f32(128, BN);
  // barriers and flags (1 KB), then the tile schedule: 4 tables of kMaxExperts + 1
  static constexpr int AUX_BYTES = 1024 + 4 * (kMaxExperts + 1) * 4 + 33 * 4;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + AUX_BYTES + 1024;  // + alignment slack
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert(2 * ACC_COLS <= 512, "TMEM columns");
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(!(!SWAP && GLU) || BN == 256, "gate/up pass stacks two 128-row weight tiles");
};

// Bounded wait that ignores the abort flag: used to let copies / MMAs that are
// already in flight complete before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
                                           uint64_t limit_ns) {
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

template <bool SWAP, bool GLU, int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_act,
                        const __grid_constant__ CUtensorMap tm_w0,
                        const __grid_constant__ CUtensorMap tm_w1, const GemmArgs args) {
  using C = GemmCfg<SWAP, GLU, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* aux = tiles + STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_tile_start = reinterpret_cast<int*>(aux + 1024);  // [kMaxExperts + 1]
  int* s_act_tiles = s_tile_start + kMaxExperts + 1;         // [kMaxExperts + 1]
  int* s_off = s_act_tiles + kMaxExperts + 1;                // [kMaxExperts + 1]
  int* s_end = s_off + kMaxExperts + 1;                      // [kMaxExperts + 1]
  int* s_scan = s_end + kMaxExperts + 1;                     // [33]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n = args.n_experts;

  // Prologue independent of earlier kernels: barriers, TMEM, descriptor prefetch.
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_act);
    tma_prefetch_desc(&tm_w0);
    if (GLU) tma_prefetch_desc(&tm_w1);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);

  // The offsets and the activations are written by earlier kernels.
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  build_tile_schedule(args.offsets, n, args.rows_total, C::ACT_ROWS, args.w_tiles, s_off, s_end,
                      s_act_tiles, s_tile_start, s_scan);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_tile_start[n];
  const WaitCtl wctl{abort_flag, args.err, args.limit_ns};

  auto decode_tile = [&](int t, int& e, int& at, int& wt) {
    e = find_expert(s_tile_start, n, t);
    const int local = t - s_tile_start[e];
    const int na = s_act_tiles[e];
    wt = local / na;
    at = local - wt * na;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x) {
        int e, at, wt;
        decode_tile(t, e, at, wt);
        const int act_row = s_off[e] + at * C::ACT_ROWS;
        const int w_row = e * args.w_rows_per_expert + wt * C::W_ROWS;
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          const int kx = kb * C::BK;
          if (!SWAP) {
            tma_load_2d(st, &tm_act, kx, act_row, &full[s]);
            tma_load_2d(st + C::A_BYTES, &tm_w0, kx, w_row, &full[s]);
            if (GLU) tma_load_2d(st + C::A_BYTES + (BN / 2) * 128, &tm_w1, kx, w_row, &full[s]);
          } else {
            tma_load_2d(st, &tm_w0, kx, w_row, &full[s]);
            if (GLU) tma_load_2d(st + C::A_BYTES, &tm_w1, kx, w_row, &full[s]);
            tma_load_2d(st + C::NUM_A * C::A_BYTES, &tm_act, kx, act_row, &full[s]);
          }
        }
      }
      // Let every issued copy land before the CTA can exit.
      for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
        drain_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, args.err, args.limit_ns);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total_tiles; t += gridDim.x, ++lt) {
        const int b = lt & 1;
        const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(&tempty[b], tph ^ 1u, wctl, kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(b * C::ACC_COLS);
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(tiles + s * C::STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            const uint32_t accum = (kb | kk) != 0 ? 1u : 0u;
            if (!SWAP) {
              mma_bf16_ss(d0, sdesc_kmajor_sw128(sa + kk * 32),
                          sdesc_kmajor_sw128(sa + C::A_BYTES + kk * 32), C::IDESC, accum);
            } else {
              const uint32_t sb = sa + C::NUM_A * C::A_BYTES;
              mma_bf16_ss(d0, sdesc_kmajor_sw128(sa + kk * 32), sdesc_kmajor_sw128(sb + kk * 32),
                          C::IDESC, accum);
              if (GLU)
                mma_bf16_ss(d0 + BN, sdesc_kmajor_sw128(sa + C::A_BYTES + kk * 32),
                            sdesc_kmajor_sw128(sb + kk * 32), C::IDESC, accum);
            }
          }
          mma_commit(&empty[s]);  // ring slot free once these MMAs have read it
        }
        if (!ok) break;
        mma_commit(&tfull[b]);    // accumulator b complete
      }
      // Every MMA must have completed before TMEM is released.
      mma_commit(drain);
      drain_wait(drain, 0, args.err, args.limit_ns);
    }
  } else {
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;  // this warp's TMEM lane quarter
    int lt = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++lt) {
      const int b = lt & 1;
      const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&tfull[b], tph, wctl, kErrTimeoutEpilogue) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      int e, at, wt;
      decode_tile(t, e, at, wt);
      const int act_row0 = s_off[e] + at * C::ACT_ROWS;
      const int act_end = s_end[e];
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      if (!SWAP) {
        const int row = act_row0 + q * 32 + lane;
        const bool valid = row < act_end;
        uint16_t* orow = args.out + (size_t)(valid ? row : 0) * args.out_ld;
        if (GLU) {
          const int col0 = wt * (BN / 2);
#pragma unroll 1
          for (int c = 0; c < BN / 2; c += 16) {
            float a[16], g[16];
            tmem_ld_2x16(tacc + c, tacc + BN / 2 + c, a, g);
            if (valid) {
              uint32_t p[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                p[i] = pack_bf16x2(silu_mul(a[2 * i], g[2 * i]), silu_mul(a[2 * i + 1], g[2 * i + 1]));
              uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
              dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
              dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
            }
          }
        } else {
          const int col0 = wt * BN;
#pragma unroll 1
          for (int c = 0; c < BN; c += 32) {
            float a[16], g[16];
            tmem_ld_2x16(tacc + c, tacc + c + 16, a, g);
            if (valid) {
              uint32_t p[16];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                p[i] = pack_bf16x2(a[2 * i], a[2 * i + 1]);
                p[8 + i] = pack_bf16x2(g[2 * i], g[2 * i + 1]);
              }
              uint4* dst = reinterpret_cast<uint4*>(orow + col0 + c);
              dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
              dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
              dst[2] = make_uint4(p[8], p[9], p[10], p[11]);
              dst[3] = make_uint4(p[12], p[13], p[14], p[15]);
            }
          }
        }
      } else {
        // lane <-> weight row j (output column); TMEM columns <-> token rows
        const int j = wt * 128 + q * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < BN; c += 16) {
          float a[16], g[16];
          tmem_ld_2x16(tacc + c, tacc + (GLU ? BN : 0) + c, a, g);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int row = act_row0 + c + i;
            if (row < act_end) {
              const float v = GLU ? silu_mul(a[i], g[i]) : a[i];
              const __nv_bfloat16 hv = __float2bfloat16_rn(v);
              args.out[(size_t)row * args.out_ld + j] = *reinterpret_cast<const uint16_t*>(&hv);
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Weight stream, stream-K schedule (small T).  The weight tiles of one pass
// (expert x 128 weight rows, over the whole reduction) do not divide evenly
// into the SMs (e.g. 896 gate/up tiles on 148 SMs is 6.05 tiles each), and
// the pass is HBM-bound, so a whole-tile round robin leaves most SMs idle in
// the last round.  Here the pass is a list of units (tile, 64-wide K block)
// and CTA c streams the contiguous units [c*U/G, (c+1)*U/G): every SM moves
// the same number of weight bytes.  A tile that a CTA covers completely gets
// the usual epilogue.  A tile split between CTAs: every contributor writes its
// fp32 accumulator slice to its partial slot in the workspace, publishes it
// (fence, then an atomic increment of the tile's counter), and the contributor
// that arrives last sums all slices in CTA order (a fixed order:
// deterministic), applies the epilogue and resets the counter to zero.  No CTA
// waits for another.
struct StreamKArgs {
  const int32_t* offsets;  // [n + 1] grouped-row offsets (device)
  uint16_t* out;           // H [R, hidden] (gate/up) or y_perm [R, dim] (down)
  uint32_t* err;           // workspace error word
  uint64_t limit_ns;       // bounded-wait limit
  int n_experts;
  int k_blocks;            // reduction length / 64
  int w_tiles;             // weight tiles (128 rows) per expert
  int w_rows_per_expert;   // rows of one expert's weight matrix
  int out_ld;              // output row stride in elements
  int rows_total;          // R
  float* partials;         // [gridDim][2][128][ACC_COLS] fp32 accumulator slices
  int* counters;           // [tiles] arrivals per split tile; zero on entry and exit
  int presumed_units;      // units of the presumed schedule requested into L2 before
                           // the dependency wait (0: none)
};

// L2 prefetch of the box at (x, y) of a tiled tensor map.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* tm, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
}

template <bool GLU, int STAGES>
__global__ void __launch_bounds__(192, 1)
    stream_k_kernel(const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_w0,
                    const __grid_constant__ CUtensorMap tm_w1, const StreamKArgs args) {
  using C = GemmCfg<true, GLU, kStreamTokens, STAGES>;
  constexpr int BN = kStreamTokens;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* aux = tiles + STAGES * C::STAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_ok = abort_flag + 1;   // [2] wait decisions, alternating by segment
  int* s_last = s_ok + 2;       // last-arriver flag of the current split tile
  int* s_tile_start = reinterpret_cast<int*>(aux + 1024);  // [kMaxExperts + 1]
  int* s_act_tiles = s_tile_start + kMaxExperts + 1;
  int* s_off = s_act_tiles + kMaxExperts + 1;
  int* s_end = s_off + kMaxExperts + 1;
  int* s_scan = s_end + kMaxExperts + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n = args.n_experts;
  const int G = gridDim.x;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 4);
    mbar_init(&tempty[1], 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_act);
    tma_prefetch_desc(&tm_w0);
    if (GLU) tma_prefetch_desc(&tm_w1);
    // The weights do not depend on the kernel that runs before this pass
    // (the routing before pass 1, pass 1 before pass 2), so the stream can
    // start while it finishes: the first units of this CTA's range under the
    // presumed schedule -- every expert touched, with one activation tile
    // (true whenever T <= 32) -- are requested into L2.
    // A prefetch is only a hint: a wrong presumption costs the bandwidth of
    // lines nobody reads, never a wrong result, and L2 is the point of
    // coherence, so nothing stale can be read.
    if (args.presumed_units > 0) {
      const int64_t Up = (int64_t)n * args.w_tiles * args.k_blocks;
      const int64_t p0 = (int64_t)cta * Up / G;
      int64_t p1 = (int64_t)(cta + 1) * Up / G;
      if (p1 > p0 + args.presumed_units) p1 = p0 + args.presumed_units;
      for (int64_t u = p0; u < p1; ++u) {
        const int t = (int)(u / args.k_blocks);
        const int kb = (int)(u - (int64_t)t * args.k_blocks);
        const int e = t / args.w_tiles, wt = t - e * args.w_tiles;
        const int w_row = e * args.w_rows_per_expert + wt * C::W_ROWS;
        tma_prefetch_l2_2d(&tm_w0, kb * C::BK, w_row);
        if (GLU) tma_prefetch_l2_2d(&tm_w1, kb * C::BK, w_row);
      }
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);

  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  build_tile_schedule(args.offsets, n, args.rows_total, C::ACT_ROWS, args.w_tiles, s_off, s_end,
                      s_act_tiles, s_tile_start, s_scan);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int KB = args.k_blocks;
  const int64_t U = (int64_t)s_tile_start[n] * KB;  // units of the pass
  auto range_start = [&](int c) -> int64_t { return (int64_t)c * U / G; };
  const int64_t u0 = range_start(cta), u1 = range_start(cta + 1);
  const WaitCtl wctl{abort_flag, args.err, args.limit_ns};

  auto decode_tile = [&](int t, int& e, int& at, int& wt) {
    e = find_expert(s_tile_start, n, t);
    const int local = t - s_tile_start[e];
    const int na = s_act_tiles[e];
    wt = local / na;
    at = local - wt * na;
  };
  // segments of this CTA's range: tile t, K blocks [kb_lo, kb_hi)
  const int t_first = u0 < u1 ? (int)(u0 / KB) : 0;
  const int t_stop = u0 < u1 ? (int)((u1 - 1) / KB) + 1 : 0;
  auto seg_bounds = [&](int t, int& kb_lo, int& kb_hi) {
    const int64_t base = (int64_t)t * KB;
    kb_lo = u0 > base ? (int)(u0 - base) : 0;
    kb_hi = u1 < base + KB ? (int)(u1 - base) : KB;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = t_first; ok && t < t_stop; ++t) {
        int e, at, wt, kb_lo, kb_hi;
        decode_tile(t, e, at, wt);
        seg_bounds(t, kb_lo, kb_hi);
        const int act_row = s_off[e] + at * C::ACT_ROWS;
        const int w_row = e * args.w_rows_per_expert + wt * C::W_ROWS;
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + s * C::STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
          const int kx = kb * C::BK;
          tma_load_2d(st, &tm_w0, kx, w_row, &full[s]);
          if (GLU) tma_load_2d(st + C::A_BYTES, &tm_w1, kx, w_row, &full[s]);
          tma_load_2d(st + C::NUM_A * C::A_BYTES, &tm_act, kx, act_row, &full[s]);
        }
      }
      for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
        drain_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, args.err, args.limit_ns);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer ---
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = t_first; ok && t < t_stop; ++t, ++lt) {
        int kb_lo, kb_hi;
        seg_bounds(t, kb_lo, kb_hi);
        const int b = lt & 1;
        const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(&tempty[b], tph ^ 1u, wctl, kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(b * C::ACC_COLS);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(tiles + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::NUM_A * C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk) {
            const uint32_t accum = (kb != kb_lo || kk != 0) ? 1u : 0u;
            mma_bf16_ss(d0, sdesc_kmajor_sw128(sa + kk * 32), sdesc_kmajor_sw128(sb + kk * 32),
                        C::IDESC, accum);
            if (GLU)
              mma_bf16_ss(d0 + BN, sdesc_kmajor_sw128(sa + C::A_BYTES + kk * 32),
                          sdesc_kmajor_sw128(sb + kk * 32), C::IDESC, accum);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&tfull[b]);
      }
      mma_commit(drain);
      drain_wait(drain, 0, args.err, args.limit_ns);
    }
  } else {
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;            // this warp's TMEM lane quarter
    const int et = threadIdx.x - 64;   // 0..127
    const int r = q * 32 + lane;       // accumulator row (weight row inside the tile)
    auto cta_of_unit = [&](int64_t u) {
      int c = (int)(u * G / U);
      while (c + 1 < G && range_start(c + 1) <= u) ++c;
      while (c > 0 && range_start(c) > u) --c;
      return c;
    };
    int lt = 0;
    for (int t = t_first; t < t_stop; ++t, ++lt) {
      const int b = lt & 1;
      const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
      // one thread decides for all four warps (they then meet the same barriers);
      // the decision slot alternates so the next write cannot overtake a read
      if (et == 0) s_ok[b] = mbar_wait(&tfull[b], tph, wctl, kErrTimeoutEpilogue) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!s_ok[b]) break;
      tc_fence_after_sync();
      int e, at, wt, kb_lo, kb_hi;
      decode_tile(t, e, at, wt);
      seg_bounds(t, kb_lo, kb_hi);
      const int act_row0 = s_off[e] + at * C::ACT_ROWS;
      const int act_end = s_end[e];
      const int j = wt * 128 + r;  // output column
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      float acc[C::ACC_COLS];
#pragma unroll
      for (int c = 0; c < C::ACC_COLS; c += 32) {
        float v0[16], v1[16];
        tmem_ld_2x16(tacc + c, tacc + c + 16, v0, v1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc[c + i] = v0[i];
          acc[c + 16 + i] = v1[i];
        }
      }
      bool emit = (kb_lo == 0 && kb_hi == KB);  // this CTA covers the whole tile
      if (!emit) {
        // publish this CTA's slice, then count the arrival
        const int64_t base = (int64_t)t * KB;
        const int slot = u0 > base ? 0 : 1;
        float4* dst = reinterpret_cast<float4*>(
            args.partials + ((size_t)(cta * 2 + slot) * 128 + r) * C::ACC_COLS);
#pragma unroll
        for (int c = 0; c < C::ACC_COLS; c += 4)
          dst[c / 4] = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
        __threadfence();
        named_bar_sync(1, 128);
        // contributors: the CTAs from the one holding the tile's first unit to the
        // one holding its last, skipping those whose range is empty
        const int c_first = cta_of_unit(base), c_last = cta_of_unit(base + KB - 1);
        if (et == 0) {
          int parts = 0;
          int64_t lo = range_start(c_first);
          for (int cc = c_first; cc <= c_last; ++cc) {
            const int64_t hi = range_start(cc + 1);
            parts += hi > lo ? 1 : 0;
            lo = hi;
          }
          const int old = atomicAdd(&args.counters[t], 1);
          *s_last = (old == parts - 1) ? 1 : 0;
        }
        named_bar_sync(1, 128);
        emit = *s_last != 0;
        if (emit) {
          __threadfence();
          // every contributor's slice, in CTA order
#pragma unroll
          for (int c = 0; c < C::ACC_COLS; ++c) acc[c] = 0.0f;
          int64_t lo = range_start(c_first);
          for (int cc = c_first; cc <= c_last; ++cc) {
            const int64_t hi = range_start(cc + 1);
            const bool contributes = hi > lo;
            const int sl = lo > base ? 0 : 1;
            lo = hi;
            if (!contributes) continue;
            const float4* src = reinterpret_cast<const float4*>(
                args.partials + ((size_t)(cc * 2 + sl) * 128 + r) * C::ACC_COLS);
#pragma unroll
            for (int c = 0; c < C::ACC_COLS; c += 4) {
              const float4 v = __ldcg(src + c / 4);
              acc[c] += v.x;
              acc[c + 1] += v.y;
              acc[c + 2] += v.z;
              acc[c + 3] += v.w;
            }
          }
          if (et == 0) args.counters[t] = 0;  // ready for the next call
        }
      }
      if (emit) {
        // lane <-> weight row j (output column); accumulator columns <-> token rows
#pragma unroll
        for (int i = 0; i < BN; ++i) {
          const int row = act_row0 + i;
          if (row < act_end) {
            const float v = GLU ? silu_mul(acc[i], acc[BN + i]) : acc[i];
            const __nv_bfloat16 hv = __float2bfloat16_rn(v);
            args.out[(size_t)row * args.out_ld + j] = *reinterpret_cast<const uint16_t*>(&hv);
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

__global__ void wait_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl w{&abort_flag, err, limit_ns};
    (void)mbar_wait(&bar, 0, w, kErrTimeoutSelftest);  // nothing ever arrives
  }
}

// ------------------------------------------------------------------ host ---

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Row-major bf16 matrix [rows, cols], box of box_cols x box_rows, 128-byte swizzle.
static bool encode_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                      uint32_t box_cols, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool SWAP, bool GLU, int BN, int STAGES>
static cudaError_t run_gemm(const CUtensorMap& a, const CUtensorMap& w0, const CUtensorMap& w1,
                            const GemmArgs& args, int grid, cudaStream_t st) {
  using C = GemmCfg<SWAP, GLU, BN, STAGES>;
  auto kern = grouped_gemm_kernel<SWAP, GLU, BN, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(192), C::SMEM_BYTES, st, a, w0, w1, args);
}

// Units of a pass each CTA requests into L2 before the dependency wait (24
// units are 768 KB per CTA in pass 1, 384 KB in pass 2; 48 measured slower,
// 6 and 12 gained less).
constexpr int kPresumedUnits = 24;

template <bool GLU, int STAGES>
static cudaError_t run_stream_k(const CUtensorMap& a, const CUtensorMap& w0,
                                const CUtensorMap& w1, const StreamKArgs& args, int grid,
                                cudaStream_t st) {
  using C = GemmCfg<true, GLU, kStreamTokens, STAGES>;
  auto kern = stream_k_kernel<GLU, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(192), C::SMEM_BYTES, st, a, w0, w1, args);
}

cudaError_t launch_expert_ffn(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets,
                              const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                              uint16_t* h, uint16_t* y_perm, int path, uint32_t* err,
                              float* partials, int* counters, cudaStream_t st) {
  const int R = s.T * s.top_k;
  if (R == 0) return cudaSuccess;
  const int d = s.dim, hd = s.hidden, n = s.n_experts;
  const bool stream = path == MOE_FFN_WEIGHT_STREAM ||
                      (path == MOE_FFN_AUTO && s.T <= kAutoStreamMaxT);
  if (path == MOE_FFN_PAIR_GEMM || (path == MOE_FFN_AUTO && !stream && pair_ffn_supported(s)))
    return launch_expert_ffn_pair(s, x_perm, offsets, w1, w3, w2, h, y_perm, err, st);
  const int grid = num_sms();
  CUtensorMap tm_x, tm_w1, tm_w3, tm_h, tm_w2;
  GemmArgs a1{offsets, h, err, kWaitLimitNs, n, d / 64, hd / 128, hd, hd, R};
  GemmArgs a2{offsets, y_perm, err, kWaitLimitNs, n, hd / 64, 0, d, d, R};
  cudaError_t e;
  if (!stream) {
    if (!encode_2d(&tm_x, x_perm, d, R, 64, 128) ||
        !encode_2d(&tm_w1, w1, d, (uint64_t)n * hd, 64, 128) ||
        !encode_2d(&tm_w3, w3, d, (uint64_t)n * hd, 64, 128) ||
        !encode_2d(&tm_h, h, hd, R, 64, 128))
      return cudaErrorInvalidValue;
    e = run_gemm<false, true, 256, 4>(tm_x, tm_w1, tm_w3, a1, grid, st);
    if (e != cudaSuccess) return e;
    if (d % 256 == 0) {
      if (!encode_2d(&tm_w2, w2, hd, (uint64_t)n * d, 64, 256)) return cudaErrorInvalidValue;
      a2.w_tiles = d / 256;
      return run_gemm<false, false, 256, 4>(tm_h, tm_w2, tm_w2, a2, grid, st);
    }
    if (!encode_2d(&tm_w2, w2, hd, (uint64_t)n * d, 64, 128)) return cudaErrorInvalidValue;
    a2.w_tiles = d / 128;
    return run_gemm<false, false, 128, 6>(tm_h, tm_w2, tm_w2, a2, grid, st);
  }
  if (!encode_2d(&tm_x, x_perm, d, R, 64, kStreamTokens) ||
      !encode_2d(&tm_w1, w1, d, (uint64_t)n * hd, 64, 128) ||
      !encode_2d(&tm_w3, w3, d, (uint64_t)n * hd, 64, 128) ||
      !encode_2d(&tm_h, h, hd, R, 64, kStreamTokens) ||
      !encode_2d(&tm_w2, w2, hd, (uint64_t)n * d, 64, 128))
    return cudaErrorInvalidValue;
  // stream-K when the tiles of a pass surely fit the counters: an expert with
  // c rows has ceil(c / 32) token tiles, so a pass has at most
  // (R / 32 + n) * (weight tiles per expert) tiles
  const int64_t max_tiles = ((int64_t)R / kStreamTokens + n) * ((d > hd ? d : hd) / 128);
  if (partials != nullptr && counters != nullptr && max_tiles <= kStreamKCounters &&
      grid <= kStreamKMaxCtas) {
    // Before pass 1 the HBM idles while the routing finishes, before pass 2
    // while the last CTAs of pass 1 finish; each pass then starts streaming
    // its first units by presuming every expert touched (see the kernel).
    // Only where that presumption nearly always holds: with T tokens choosing
    // K of n experts uniformly, an expert stays untouched with probability
    // (1 - K/n)^T (Mixtral decode, T=16: 0.01; 8 of 160: 0.44).
    const bool presume =
        s.T <= kStreamTokens && std::pow(1.0 - (double)s.top_k / n, (double)s.T) <= 0.05;
    const StreamKArgs k1{offsets, h, err, kWaitLimitNs, n, d / 64, hd / 128, hd, hd, R,
                         partials, counters, presume ? kPresumedUnits : 0};
    e = run_stream_k<true, 6>(tm_x, tm_w1, tm_w3, k1, grid, st);
    if (e != cudaSuccess) return e;
    const StreamKArgs k2{offsets, y_perm, err, kWaitLimitNs, n, hd / 64, d / 128, d, d, R,
                         partials, counters, presume ? kPresumedUnits : 0};
    return run_stream_k<false, 10>(tm_h, tm_w2, tm_w2, k2, grid, st);
  }
  e = run_gemm<true, true, kStreamTokens, 6>(tm_x, tm_w1, tm_w3, a1, grid, st);
  if (e != cudaSuccess) return e;
  a2.w_tiles = d / 128;
  return run_gemm<true, false, kStreamTokens, 10>(tm_h, tm_w2, tm_w2, a2, grid, st);
}

cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
