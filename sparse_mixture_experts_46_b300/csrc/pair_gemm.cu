// pair_gemm.cu -- expert SwiGLU FFN as two grouped GEMMs on CTA pairs
// (tcgen05 cta_group::2), weights on the MMA M side, tokens on N
// ("Mixtral of Experts" section 2.1: each selected expert is a SwiGLU
// feed-forward block; the per-expert token groups have different sizes).
//
//   pass 1 (gate/up, GLU):  H[r]      = bf16(SiLU(X[r] W1_e^T) * (X[r] W3_e^T))
//   pass 2 (down):          Y_perm[r] = bf16(H[r] W2_e^T)
// for every grouped row r of expert e (rows [offsets[e], offsets[e+1])).
//
// One MMA covers M = 256 weight rows x N token rows x K = 16, split over the
// two CTAs of a cluster: each CTA stages 128 weight rows (A) and N/2 token rows
// (B) per 64-wide K block, and holds its 128 x N slice of the fp32 accumulator
// in its own TMEM.  Compared with one CTA computing 128 x 256 alone, every SM
// streams a third less operand data per MMA (32 KB instead of 48 KB per K
// block).  Because tokens sit on N, the last token tile of an expert shrinks
// its MMA to N = (remaining rows rounded up to 16): no 128-row padding.
//   * gate/up: each CTA's A tile stacks 64 rows of W1 over the same 64 rows of
//     W3, so TMEM lanes 0-63 hold x.W1 and lanes 64-127 hold x.W3 of the same
//     hidden units; the epilogue pairs them through shared memory.
//   * down: each CTA's A tile is 128 rows of W2.
//
// Warp roles (192 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      TMA producer (one thread) in both CTAs: fills a STAGES-deep
//               ring; every load completes on the EVEN CTA's full barrier
//               (cta_group::2 form), which expects both CTAs' bytes;
//   warp 1      TMEM (512 columns, allocated by both CTAs as a pair) and, in
//               the even CTA only, the MMA issuer: one thread waits on full,
//               issues the pair MMAs and commits to the empty barriers and the
//               accumulator barriers of BOTH CTAs (multicast commit);
//   warps 2..5  epilogue in both CTAs: tcgen05.ld of 32 accumulator columns,
//               staged through shared memory as [token][weight row] fp32, then
//               SwiGLU / convert and coalesced bf16 stores of token rows.
// The accumulator is double-buffered (2 x 256 TMEM columns), so the epilogue
// of tile i overlaps the main loop of tile i+1.  Tiles (expert, weight tile,
// token tile) are scheduled from the device-resident offsets, expert-major,
// then weight tile, then token tile, round-robin over the pairs.  An expert
// whose activation rows exceed an L2 budget (kL2Budget: a skewed routing can
// send tens of thousands of rows to one expert) has its token tiles split into
// equal blocks that fit, walked block by block (block, weight tile, token
// tile): each block's rows stay in L2 while every weight tile passes over
// them, instead of all the expert's rows being re-read from HBM once per
// weight tile.
//
// The same kernel serves the activation-gradient GEMMs of the backward pass
// with the weights read in their stored layout (AMN): there the reduction
// runs over the weight matrix's ROWS (dH = dO W2_e, dX = dA W1_e + dG W3_e),
// so each CTA's A tile is taken as two boxes of 64 weight columns x 64 weight
// rows -- the MN-major operand layout -- and marked MN-major in the
// instruction descriptor; no transposed copy of any weight is made.
//
// Every wait is bounded (device.cuh); an expired wait records the error word
// and the CTA winds down through the same exit path.
#include <cudaTypedefs.h>

#include <mutex>

#include "device.cuh"
#include "internal.h"

namespace moe {

// Epilogue of a pass: what the accumulator (out[r][j] = sum_k act[r][k] W_e[j][k])
// becomes.
enum : int {
  kEpiPlain = 0,      // out = bf16(acc)
  kEpiGlu = 1,        // W1/W3 stacked: out = bf16(SiLU(a) * g)
  kEpiGluSave = 2,    // as kEpiGlu, and save[r] = [bf16(a) | bf16(g)] (pre-activations)
  kEpiSwigluBwd = 3,  // acc = dH; from saved a, g: out[r] = [dA | dG] (SwiGLU backward)
};

struct PairArgs {
  const int32_t* offsets;  // [n + 1] grouped-row offsets (device)
  uint16_t* out;           // H [R, hidden] (gate/up) or y_perm [R, dim] (down)
  uint32_t* err;           // workspace error word
  uint64_t limit_ns;       // bounded-wait limit
  int n_experts;
  int k_blocks;            // reduction length / 64
  int w_tiles;             // weight tiles (of the pair) per expert
  int w_rows_per_expert;   // rows of one expert's weight matrix (hidden or dim)
  int out_ld;              // output row stride in elements
  int rows_total;          // R: grouped rows (offsets are clamped to [0, R])
  uint16_t* save;          // kEpiGluSave: [R, 2 * out_ld] pre-activations a | g
  const uint16_t* saved;   // kEpiSwigluBwd: [R, out_ld] pre-activations a | g (out_ld = 2h)
  // AMN only: the reduction walks w_k_rows rows of tm_w0's expert block for
  // K blocks [0, k_split), then the same rows of tm_w1's for the rest
  int k_split;
  int w_k_rows;
  const int32_t* counts;   // nullable: padded groups end at offsets[e] + counts[e]
};

// Activation bytes of one expert that the tile order keeps resident in L2
// (about a third of the 126 MB L2; weights in flight and outputs share it).
constexpr int64_t kL2Budget = 40ll << 20;

template <bool GLU, int STAGES>
struct PairCfg {
  static constexpr int BK = 64;                  // bf16 per 128-byte row
  static constexpr int A_BYTES = 128 * 128;      // 128 weight rows of one CTA
  static constexpr int B_BYTES = 128 * 128;      // up to 128 token rows of one CTA
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TOK_TILE = 256;           // token rows per pair tile (max MMA N)
  static constexpr int W_ROWS = GLU ? 64 : 128;  // rows per weight matrix per CTA
  static constexpr int OUT_COLS = GLU ? 64 : 128;  // output columns per CTA and tile
  static constexpr int ACC_COLS = 256;           // TMEM columns per accumulator buffer
  static constexpr int CHUNK = 32;               // accumulator columns per epilogue step
  static constexpr int STAGING_BYTES = CHUNK * 128 * 4;
  // barriers and flags (1 KB), then the tile schedule: 5 tables of kMaxExperts + 1
  static constexpr int AUX_BYTES = 1024 + 5 * (kMaxExperts + 1) * 4 + 33 * 4;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING_BYTES + AUX_BYTES + 1024;
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void pair_drain_wait(uint64_t* bar, uint32_t parity, uint32_t* err,
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

template <int EPI, int STAGES, bool AMN>
__global__ void __launch_bounds__(192, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap tm_act,
                     const __grid_constant__ CUtensorMap tm_w0,
                     const __grid_constant__ CUtensorMap tm_w1, const PairArgs args) {
  constexpr bool GLU = EPI == kEpiGlu || EPI == kEpiGluSave;
  static_assert(!(AMN && GLU), "stored-layout weights serve the plain and SwiGLU-backward passes");
  using C = PairCfg<GLU, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  // Both CTAs of the pair place every tile at the same shared-memory offset:
  // the pair MMA addresses the peer's operands through the issuer's offsets.
  uint8_t* tiles = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* staging = reinterpret_cast<float*>(tiles + STAGES * C::STAGE_BYTES);  // [32][128]
  uint8_t* aux = tiles + STAGES * C::STAGE_BYTES + C::STAGING_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(aux);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;   // [2]
  uint64_t* tempty = tfull + 2;       // [2]
  uint64_t* drain = tempty + 2;       // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_ok = abort_flag + 1;
  int* s_tile_start = reinterpret_cast<int*>(aux + 1024);  // [kMaxExperts + 1]
  int* s_tok_tiles = s_tile_start + kMaxExperts + 1;         // [kMaxExperts + 1]
  int* s_off = s_tok_tiles + kMaxExperts + 1;                // [kMaxExperts + 1]
  int* s_end = s_off + kMaxExperts + 1;                      // [kMaxExperts + 1]
  int* s_span = s_end + kMaxExperts + 1;                     // [kMaxExperts + 1]
  int* s_scan = s_span + kMaxExperts + 1;                    // [33]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n = args.n_experts;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs of the pair
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;

  // Prologue independent of earlier kernels: barriers, TMEM, descriptors.
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&tfull[0], 1);
    mbar_init(&tfull[1], 1);
    mbar_init(&tempty[0], 2);  // one arrival from each CTA's epilogue
    mbar_init(&tempty[1], 2);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_act);
    tma_prefetch_desc(&tm_w0);
    if (GLU) tma_prefetch_desc(&tm_w1);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 2 * C::ACC_COLS);

  // The offsets and the activations are written by earlier kernels.
  pdl_wait();
  pdl_launch_dependents();
  build_tile_schedule(args.offsets, n, args.rows_total, C::TOK_TILE, args.w_tiles, s_off, s_end,
                      s_tok_tiles, s_tile_start, s_scan, args.counts, s_span,
                      (int64_t)args.k_blocks * C::BK * 2, kL2Budget);
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after_sync();

  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = s_tile_start[n];
  const WaitCtl wctl{abort_flag, args.err, args.limit_ns};

  // tile -> expert e, weight tile wt, first token row, valid rows, MMA N;
  // the expert's tiles are blocks of s_span[e] token tiles (the last block may
  // be shorter), each walked weight tile by weight tile
  auto decode_tile = [&](int t, int& e, int& wt, int& row0, int& rows, int& N) {
    e = find_expert(s_tile_start, n, t);
    const int local = t - s_tile_start[e];
    const int ntt = s_tok_tiles[e];
    const int span = s_span[e];
    const int per_block = args.w_tiles * span;
    const int blk = local / per_block;
    const int rem = local - blk * per_block;
    const int bs = min(span, ntt - blk * span);  // token tiles in this block
    wt = rem / bs;
    const int tt = blk * span + (rem - wt * bs);
    row0 = s_off[e] + tt * C::TOK_TILE;
    rows = min(C::TOK_TILE, s_end[e] - row0);
    N = (rows + 15) & ~15;
  };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = pair; ok && t < total_tiles; t += npairs) {
        int e, wt, row0, rows, N;
        decode_tile(t, e, wt, row0, rows, N);
        const int act_row = row0 + (int)rank * (N >> 1);
        const int w_row = e * args.w_rows_per_expert + wt * 2 * C::W_ROWS + (int)rank * C::W_ROWS;
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&empty[s], ph ^ 1u, wctl, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          // both CTAs' bytes complete on the even CTA's full barrier
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * C::STAGE_BYTES);
          const uint32_t bar = smem_map_rank(smem_u32(&full[s]), 0);
          uint8_t* st = tiles + s * C::STAGE_BYTES;
          const int kx = kb * C::BK;
          if (AMN) {
            // weight rows are the reduction: two 64-column boxes of 64 rows
            const bool hi = kb >= args.k_split;
            const CUtensorMap* tw = hi ? &tm_w1 : &tm_w0;
            const int ky = e * args.w_k_rows + (hi ? kb - args.k_split : kb) * C::BK;
            const int m0 = wt * 2 * C::W_ROWS + (int)rank * C::W_ROWS;
            tma_load_2d_pair(st, tw, m0, ky, bar);
            tma_load_2d_pair(st + C::A_BYTES / 2, tw, m0 + 64, ky, bar);
          } else {
            tma_load_2d_pair(st, &tm_w0, kx, w_row, bar);
            if (GLU) tma_load_2d_pair(st + C::A_BYTES / 2, &tm_w1, kx, w_row, bar);
          }
          tma_load_2d_pair(st + C::A_BYTES, &tm_act, kx, act_row, bar);
        }
      }
      // the even CTA can observe the loads landing: let them land before exit
      if (rank == 0)
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          pair_drain_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, args.err,
                          args.limit_ns);
    }
  } else if (warp == 1) {
    // -------------------------------------------- MMA issuer (even CTA) ---
    if (rank == 0 && lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int t = pair; ok && t < total_tiles; t += npairs, ++lt) {
        int e, wt, row0, rows, N;
        decode_tile(t, e, wt, row0, rows, N);
        const int b = lt & 1;
        const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
        if (!mbar_wait(&tempty[b], tph ^ 1u, wctl, kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(b * C::ACC_COLS);
        const uint32_t idesc = idesc_bf16_f32(256, (uint32_t)N) | (AMN ? (1u << 15) : 0u);
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          if (!mbar_wait(&full[s], ph, wctl, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(tiles + s * C::STAGE_BYTES);
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            mma_bf16_pair(d0,
                          AMN ? sdesc_mnmajor_sw128(sa + kk * 2048, C::A_BYTES / 2, 1024)
                              : sdesc_kmajor_sw128(sa + kk * 32),
                          sdesc_kmajor_sw128(sb + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          mma_commit_pair_mc(&empty[s], 0x3);  // ring slot free in both CTAs
        }
        if (!ok) break;
        mma_commit_pair_mc(&tfull[b], 0x3);    // accumulator b complete in both CTAs
      }
      // every MMA must have completed before either CTA releases TMEM or exits
      mma_commit_pair_mc(drain, 0x1);
      pair_drain_wait(drain, 0, args.err, args.limit_ns);
    }
  } else {
    // ---------------------------------------------------------- epilogue ---
    const int q = warp & 3;              // this warp's TMEM lane quarter
    const int et = threadIdx.x - 64;     // 0..127
    int lt = 0;
    for (int t = pair; t < total_tiles; t += npairs, ++lt) {
      const int b = lt & 1;
      const uint32_t tph = (uint32_t)(lt >> 1) & 1u;
      // one thread decides for all four warps (they then meet the same barriers)
      if (et == 0) *s_ok = mbar_wait(&tfull[b], tph, wctl, kErrTimeoutEpilogue) ? 1 : 0;
      named_bar_sync(1, 128);
      if (!*s_ok) break;
      tc_fence_after_sync();
      int e, wt, row0, rows, N;
      decode_tile(t, e, wt, row0, rows, N);
      const int col0 = wt * 2 * C::OUT_COLS + (int)rank * C::OUT_COLS;  // output column base
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * C::ACC_COLS);
      // SwiGLU backward: this thread's saved pre-activations of chunk c0 (8
      // items of 4 columns), fetched one chunk ahead so their DRAM latency
      // hides behind the previous chunk's work
      constexpr int NS = EPI == kEpiSwigluBwd ? 8 : 1;
      uint2 zs[NS], gs[NS], zn[NS], gn[NS];
      auto fetch_saved = [&](int c, uint2* z, uint2* g) {
        const int hh = args.out_ld / 2;
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          const int item = et + 128 * i;
          const int col = item >> 5;
          z[i] = g[i] = make_uint2(0u, 0u);
          if (c + col < rows) {
            const uint16_t* sp =
                args.saved + (size_t)(row0 + c + col) * args.out_ld + col0 + (item & 31) * 4;
            z[i] = __ldg(reinterpret_cast<const uint2*>(sp));
            g[i] = __ldg(reinterpret_cast<const uint2*>(sp + hh));
          }
        }
      };
      if (EPI == kEpiSwigluBwd) fetch_saved(0, zn, gn);
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += C::CHUNK) {
        if (EPI == kEpiSwigluBwd) {
#pragma unroll
          for (int i = 0; i < NS; ++i) {
            zs[i] = zn[i];
            gs[i] = gn[i];
          }
          if (c0 + C::CHUNK < N) fetch_saved(c0 + C::CHUNK, zn, gn);
        }
        float v[32];
        tmem_ld_32(tacc + (uint32_t)c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) staging[i * 128 + q * 32 + lane] = v[i];
        tc_fence_before_sync();
        named_bar_sync(1, 128);
        if (GLU) {
          // 32 token rows x 16 groups of 4 hidden units; a at lane j, g at lane 64 + j
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int item = et + 128 * i;
            const int col = item >> 4;
            const int jq = item & 15;
            if (c0 + col < rows) {
              const float4 a = *reinterpret_cast<const float4*>(staging + col * 128 + jq * 4);
              const float4 g = *reinterpret_cast<const float4*>(staging + col * 128 + 64 + jq * 4);
              uint2 o;
              o.x = pack_bf16x2(silu_mul(a.x, g.x), silu_mul(a.y, g.y));
              o.y = pack_bf16x2(silu_mul(a.z, g.z), silu_mul(a.w, g.w));
              const size_t row = (size_t)(row0 + c0 + col);
              *reinterpret_cast<uint2*>(args.out + row * args.out_ld + col0 + jq * 4) = o;
              if (EPI == kEpiGluSave) {
                uint16_t* sv = args.save + row * 2 * args.out_ld + col0 + jq * 4;
                *reinterpret_cast<uint2*>(sv) =
                    make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
                *reinterpret_cast<uint2*>(sv + args.out_ld) =
                    make_uint2(pack_bf16x2(g.x, g.y), pack_bf16x2(g.z, g.w));
              }
            }
          }
        } else {
          // 32 token rows x 32 groups of 4 output columns
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int item = et + 128 * i;
            const int col = item >> 5;
            const int jq = item & 31;
            if (c0 + col < rows) {
              const float4 a = *reinterpret_cast<const float4*>(staging + col * 128 + jq * 4);
              const size_t row = (size_t)(row0 + c0 + col);
              if (EPI == kEpiSwigluBwd) {
                // a = dH; with the saved pre-activations z (gate) and g (up):
                // dZ = dH * g * SiLU'(z), dG = dH * SiLU(z)
                const int hh = args.out_ld / 2;
                const uint2 zb = zs[EPI == kEpiSwigluBwd ? i : 0];
                const uint2 gb = gs[EPI == kEpiSwigluBwd ? i : 0];
                const float dh[4] = {a.x, a.y, a.z, a.w};
                const float z[4] = {__uint_as_float(zb.x << 16), __uint_as_float(zb.x & 0xFFFF0000u),
                                    __uint_as_float(zb.y << 16), __uint_as_float(zb.y & 0xFFFF0000u)};
                const float g[4] = {__uint_as_float(gb.x << 16), __uint_as_float(gb.x & 0xFFFF0000u),
                                    __uint_as_float(gb.y << 16), __uint_as_float(gb.y & 0xFFFF0000u)};
                float dz[4], dg[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const float sg = __fdividef(1.0f, 1.0f + __expf(-z[u]));
                  dz[u] = dh[u] * g[u] * sg * (1.0f + z[u] * (1.0f - sg));
                  dg[u] = dh[u] * z[u] * sg;
                }
                *reinterpret_cast<uint2*>(args.out + row * args.out_ld + col0 + jq * 4) =
                    make_uint2(pack_bf16x2(dz[0], dz[1]), pack_bf16x2(dz[2], dz[3]));
                *reinterpret_cast<uint2*>(args.out + row * args.out_ld + hh + col0 + jq * 4) =
                    make_uint2(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]));
              } else {
                uint2 o;
                o.x = pack_bf16x2(a.x, a.y);
                o.y = pack_bf16x2(a.z, a.w);
                *reinterpret_cast<uint2*>(args.out + row * args.out_ld + col0 + jq * 4) = o;
              }
            }
          }
        }
        named_bar_sync(1, 128);  // staging is rewritten by the next chunk
      }
      // accumulator b may be overwritten once both CTAs' epilogues are done
      if (et == 0) mbar_arrive_cluster(smem_map_rank(smem_u32(&tempty[b]), 0));
    }
  }

  __syncthreads();
  cluster_sync_all();  // the pair's MMAs have completed; no remote arrival is pending
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, 2 * C::ACC_COLS);
  }
}

// ------------------------------------------------------------------ host ---

static PFN_cuTensorMapEncodeTiled_v12000 pair_tensor_map_encoder() {
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

// Row-major bf16 matrix [rows, cols], box of 64 columns x box_rows, 128-byte swizzle.
static bool pair_encode_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows,
                           uint32_t box_rows) {
  auto enc = pair_tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Grid of the pair kernel: two CTAs per co-resident cluster, at most one CTA per SM.
template <int EPI, int STAGES, bool AMN>
static int pair_grid(cudaError_t* err) {
  constexpr bool GLU = EPI == kEpiGlu || EPI == kEpiGluSave;
  using C = PairCfg<GLU, STAGES>;
  auto kern = pair_gemm_kernel<EPI, STAGES, AMN>;
  static int cached[64] = {0};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (*err != cudaSuccess) return 0;
  const int sms = num_sms();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sms & ~1));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  *err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
  if (*err != cudaSuccess) return 0;
  if (clusters < 1) {
    *err = cudaErrorInvalidConfiguration;
    return 0;
  }
  int grid = 2 * clusters;
  if (grid > (sms & ~1)) grid = sms & ~1;
  if (dev >= 0 && dev < 64) cached[dev] = grid;
  return grid;
}

template <int EPI, int STAGES, bool AMN = false>
static cudaError_t run_pair_gemm(const CUtensorMap& a, const CUtensorMap& w0,
                                 const CUtensorMap& w1, const PairArgs& args, cudaStream_t st) {
  constexpr bool GLU = EPI == kEpiGlu || EPI == kEpiGluSave;
  using C = PairCfg<GLU, STAGES>;
  cudaError_t e = cudaSuccess;
  const int grid = pair_grid<EPI, STAGES, AMN>(&e);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
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
  return cudaLaunchKernelEx(&cfg, pair_gemm_kernel<EPI, STAGES, AMN>, a, w0, w1, args);
}

bool pair_ffn_supported(const moe_shape& s) { return s.dim % 256 == 0 && s.hidden % 128 == 0; }

cudaError_t launch_expert_ffn_pair(const moe_shape& s, const uint16_t* x_perm,
                                   const int32_t* offsets, const uint16_t* w1, const uint16_t* w3,
                                   const uint16_t* w2, uint16_t* h, uint16_t* y_perm,
                                   uint32_t* err, cudaStream_t st, uint16_t* save,
                                   const int32_t* counts, int rows_alloc) {
  if (s.T * s.top_k == 0) return cudaSuccess;
  const int R = rows_alloc > 0 ? rows_alloc : s.T * s.top_k;
  if (!pair_ffn_supported(s)) return cudaErrorInvalidValue;
  const int d = s.dim, hd = s.hidden, n = s.n_experts;
  CUtensorMap tm_x, tm_w1, tm_w3, tm_h, tm_w2;
  if (!pair_encode_2d(&tm_x, x_perm, d, R, 128) ||
      !pair_encode_2d(&tm_w1, w1, d, (uint64_t)n * hd, 64) ||
      !pair_encode_2d(&tm_w3, w3, d, (uint64_t)n * hd, 64) ||
      !pair_encode_2d(&tm_h, h, hd, R, 128) ||
      !pair_encode_2d(&tm_w2, w2, hd, (uint64_t)n * d, 128))
    return cudaErrorInvalidValue;
  const PairArgs a1{offsets, h, err, kWaitLimitNs, n, d / 64, hd / 128, hd, hd, R, save, nullptr,
                    0, 0, counts};
  cudaError_t e = save != nullptr ? run_pair_gemm<kEpiGluSave, 6>(tm_x, tm_w1, tm_w3, a1, st)
                                  : run_pair_gemm<kEpiGlu, 6>(tm_x, tm_w1, tm_w3, a1, st);
  if (e != cudaSuccess) return e;
  const PairArgs a2{offsets, y_perm, err, kWaitLimitNs, n, hd / 64, d / 256, d, d, R, nullptr,
                    nullptr, 0, 0, counts};
  return run_pair_gemm<kEpiPlain, 6>(tm_h, tm_w2, tm_w2, a2, st);
}

// out[r][j] = bf16(sum_k act[r][k] B[e][k][j]) over the grouped rows r of each
// expert e, the weights read in their stored layout: B[e] is rows [0, w_k_rows)
// of expert block e of w0 ([n, w_k_rows, M], row-major), followed, when
// K == 2 * w_k_rows, by the same rows of w1.  act [R, K]; M % 256 == 0,
// w_k_rows % 64 == 0; out rows of out_ld elements (columns j < M).  With
// `saved` ([R, 2M] pre-activations a | g) the epilogue is the SwiGLU
// backward: the accumulator is dH and out = [dA | dG] (out_ld = 2M).  With
// `counts` the groups are padded apart: expert e's rows are [offsets[e],
// offsets[e] + counts[e]) of the R rows of act / out.
cudaError_t launch_pair_rowgemm(const uint16_t* act, const int32_t* offsets,
                                const int32_t* counts, int R, int n, int M, int K,
                                const uint16_t* w0, const uint16_t* w1, int w_k_rows,
                                uint16_t* out, int out_ld, const uint16_t* saved, uint32_t* err,
                                cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  if (M % 256 != 0 || w_k_rows % 64 != 0 || w_k_rows <= 0) return cudaErrorInvalidValue;
  if (K != w_k_rows && !(K == 2 * w_k_rows && w1 != nullptr)) return cudaErrorInvalidValue;
  CUtensorMap tm_a, tm_w0, tm_w1;
  const uint64_t wrows = (uint64_t)n * w_k_rows;
  if (!pair_encode_2d(&tm_a, act, K, R, 128) || !pair_encode_2d(&tm_w0, w0, M, wrows, 64) ||
      !pair_encode_2d(&tm_w1, w1 != nullptr ? w1 : w0, M, wrows, 64))
    return cudaErrorInvalidValue;
  const PairArgs a{offsets, out, err, kWaitLimitNs, n, K / 64, M / 256, M, out_ld, R, nullptr,
                   saved, w_k_rows / 64, w_k_rows, counts};
  if (saved != nullptr) return run_pair_gemm<kEpiSwigluBwd, 6, true>(tm_a, tm_w0, tm_w1, a, st);
  return run_pair_gemm<kEpiPlain, 6, true>(tm_a, tm_w0, tm_w1, a, st);
}

}  // namespace moe
