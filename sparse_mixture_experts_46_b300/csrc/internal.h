// internal.h -- host-side declarations shared by the .cu files of the library:
// workspace layout and kernel launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kPermuteChunk = 256;       // assignments per permute block
constexpr int kStreamTokens = 32;        // token chunk (MMA N) of the weight stream
constexpr int kAutoStreamMaxT = 32;      // MOE_FFN_AUTO: weight stream when T <= this
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// Workspace control region (zeroed by moe_workspace_init): the error word in
// the first 4 KB, then the per-tile arrival counters of the stream-K weight
// stream (left zero by every completed call).
constexpr size_t kWsHeaderBytes = 4096;
constexpr size_t kWsControlBytes = 65536;
constexpr int kStreamKCounters = (int)((kWsControlBytes - kWsHeaderBytes) / 4);
constexpr int kStreamKMaxCtas = 256;  // partial slots are sized for this many CTAs

// Device workspace layout: one header page, then 256-byte aligned arrays.
struct WsLayout {
  size_t err;          // uint32 error word (header)
  size_t counters;     // int32 [kStreamKCounters] (control region)
  size_t partials;     // f32 [kStreamKMaxCtas][2][128][64] stream-K accumulator slices
  size_t ids;          // int32 [R]
  size_t gates;        // f32 [R]
  size_t counts;       // int32 [n]
  size_t offsets;      // int32 [n + 1]
  size_t chunk_hist;   // int32 [nchunks * n]
  size_t chunk_base;   // int32 [nchunks * n]
  size_t perm_src;     // int32 [R]
  size_t slot_row;     // int32 [R]
  size_t u;            // bf16 [T, dim] (RMSNorm output)
  size_t x_perm;       // bf16 [R, dim]
  size_t h;            // bf16 [R, hidden]
  size_t y_perm;       // bf16 [R, dim]
  size_t total;
  int nchunks;
};

bool shape_supported(const moe_shape* s);
WsLayout ws_layout(const moe_shape* s);

// Launchers: return cudaSuccess or the launch error.
// Router: ids/gates (and counts when non-null); with u_out, routes
// u = RMSNorm(x) and writes u.  err: error word of the bounded waits (null:
// the library's own word, reported by moe_check_error).
cudaError_t launch_router(const moe_shape& s, const uint16_t* x, const uint16_t* wg, int32_t* ids,
                          float* gates, int32_t* counts, uint16_t* u_out, float eps,
                          uint32_t* err, cudaStream_t st);
// Tensor-core routers (n <= 16; 32 < n <= 256 with n % 8 == 0 and K <= 8) and
// the RMSNorm kernel they are paired with.
bool router_tc_supported(const moe_shape& s);
bool router_wide_supported(const moe_shape& s);
cudaError_t launch_router_tc(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                             int32_t* ids, float* gates, int32_t* counts, uint32_t* err,
                             cudaStream_t st);
cudaError_t launch_router_wide(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                               int32_t* ids, float* gates, int32_t* counts, uint32_t* err,
                               cudaStream_t st);
cudaError_t launch_rmsnorm(const moe_shape& s, const uint16_t* x, float eps, uint16_t* u,
                           cudaStream_t st);
// Read (synchronously) and clear the library's router error word.
cudaError_t router_err_read_clear(uint32_t* word);
// Rows a grouping of R assignments over n experts can occupy when every
// group starts on a multiple of `pad` rows.
constexpr int permute_padded_rows(int R, int n, int pad) {
  return (R + n * (pad - 1) + pad - 1) / pad * pad;
}
// Expert grouping.  pad > 1: groups start on multiples of `pad` (offsets hold
// the padded starts, counts_out must be non-null); perm_src and x_perm then
// hold rows_alloc >= permute_padded_rows(R, n, pad) rows, the padding rows of
// x_perm are zeros.
cudaError_t launch_permute(const moe_shape& s, const uint16_t* x, const int32_t* ids,
                           int32_t* counts_out, int32_t* offsets, int32_t* chunk_hist,
                           int32_t* chunk_base, int32_t* perm_src, int32_t* slot_row,
                           uint16_t* x_perm, int nchunks, cudaStream_t st, int pad = 1,
                           int rows_alloc = 0);
// Routing of a small batch in one launch (T <= 32, n <= 8): router, top-K and
// gates, the stable grouping (offsets, perm_src, slot_row) and the gather of
// x_perm; no counts, no RMSNorm.
bool route_small_supported(const moe_shape& s);
cudaError_t launch_route_small(const moe_shape& s, const uint16_t* x, const uint16_t* wg,
                               int32_t* ids, float* gates, int32_t* offsets, int32_t* perm_src,
                               int32_t* slot_row, uint16_t* x_perm, cudaStream_t st);
cudaError_t launch_combine(const moe_shape& s, const uint16_t* y_perm, const int32_t* slot_row,
                           const float* gates, const uint16_t* residual, uint16_t* y,
                           cudaStream_t st);
// Grouped expert FFN; returns cudaErrorInvalidValue when a tensor map cannot
// be encoded.
// partials / counters: the workspace's stream-K regions (null: the weight
// stream uses whole-tile rounds).
cudaError_t launch_expert_ffn(const moe_shape& s, const uint16_t* x_perm, const int32_t* offsets,
                              const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                              uint16_t* h, uint16_t* y_perm, int path, uint32_t* err,
                              float* partials, int* counters, cudaStream_t st);
// CTA-pair variant (weights on the MMA M side, cta_group::2); requires
// pair_ffn_supported(s).
bool pair_ffn_supported(const moe_shape& s);
// save (nullable): [rows, 2 * hidden] receives the gate/up pre-activations
// a | g.  counts (nullable): padded groups, expert e's rows are
// [offsets[e], offsets[e] + counts[e]) of rows_alloc rows (0: R).
cudaError_t launch_expert_ffn_pair(const moe_shape& s, const uint16_t* x_perm,
                                   const int32_t* offsets, const uint16_t* w1, const uint16_t* w3,
                                   const uint16_t* w2, uint16_t* h, uint16_t* y_perm,
                                   uint32_t* err, cudaStream_t st, uint16_t* save = nullptr,
                                   const int32_t* counts = nullptr, int rows_alloc = 0);
// out[r][j] = bf16(sum_k act[r][k] B_e[k][j]) per expert group (CTA-pair GEMM),
// B_e = rows of w0's expert block (then of w1's when K = 2 w_k_rows) in their
// stored [k][j] layout; with `saved` ([R, 2M] pre-activations a | g) the SwiGLU
// backward: out = [dA | dG].  counts: as for launch_expert_ffn_pair (R rows).
cudaError_t launch_pair_rowgemm(const uint16_t* act, const int32_t* offsets,
                                const int32_t* counts, int R, int n, int M, int K,
                                const uint16_t* w0, const uint16_t* w1, int w_k_rows,
                                uint16_t* out, int out_ld, const uint16_t* saved, uint32_t* err,
                                cudaStream_t st);
// Backward pass building blocks (backward.cu, wgrad_gemm.cu).  The grouped
// buffers hold `rows` rows, expert e's group at [offsets[e], offsets[e] +
// counts[e]) with offsets[e] a multiple of 64 (padded grouping).
// Zero the padding rows [offsets[e] + counts[e], offsets[e+1]) of up to three
// grouped bf16 buffers (null entries skipped).
cudaError_t launch_zero_pad_rows(const int32_t* offsets, const int32_t* counts, int n, int rows,
                                 uint16_t* b0, int c0, uint16_t* b1, int c1, uint16_t* b2, int c2,
                                 cudaStream_t st);
cudaError_t launch_combine_bwd(const moe_shape& s, const uint16_t* dy, const uint16_t* y_perm,
                               const int32_t* slot_row, const float* gates, int rows,
                               uint16_t* dO, float* dg, cudaStream_t st);
cudaError_t launch_router_bwd(const moe_shape& s, const float* gates, const float* dg,
                              const int32_t* slot_row, int rows, float* dl, float* dl_perm,
                              cudaStream_t st);
cudaError_t launch_router_wgrad(const moe_shape& s, const uint16_t* x_perm, const float* dl_perm,
                                const int32_t* offsets, const int32_t* counts, int rows,
                                float* dwg, cudaStream_t st);
// wgT: [n, dim] scratch for the transposed router weight.
cudaError_t launch_input_grad(const moe_shape& s, const uint16_t* dx_perm, const int32_t* slot_row,
                              const int32_t* ids, const float* dl, const uint16_t* wg,
                              uint16_t* wgT, int rows, uint16_t* dx, cudaStream_t st);
// C_e = P_e^T Q_e over expert e's padded group of rows: p [rows, M], q [rows, N].
cudaError_t launch_wgrad(const uint16_t* p, const uint16_t* q, int M, int N, int rows,
                         const int32_t* offsets, int n, float* out0, float* out1, int m_split,
                         uint32_t* err, cudaStream_t st);

// Routing statistics (slot_counts [K * n], repeats [2]); zeroes both first.
cudaError_t launch_routing_stats(const moe_shape& s, const int32_t* ids, int32_t* slot_counts,
                                 int32_t* repeats, cudaStream_t st);
cudaError_t launch_wait_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t st);

int num_sms();

}  // namespace moe

namespace moe {

// Launch `kernel` on `st` with programmatic dependent launch enabled (see
// pdl_wait in device.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
