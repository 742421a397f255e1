// moe_api.cu -- the extern "C" entry points declared in include/moe.h:
// argument and shape validation, the workspace layout, and the launch order of
// the router, grouping, expert FFN and combine kernels on the caller's stream.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace moe {

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {0};
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64) cache[dev] = sms;
  return sms;
}

bool shape_supported(const moe_shape* s) {
  if (s == nullptr) return false;
  if (s->T < 0 || s->n_experts < 1 || s->n_experts > kMaxExperts) return false;
  if (s->top_k < 1 || s->top_k > s->n_experts) return false;
  // more than 32 experts: the wide router (n a multiple of 8, K <= 8)
  if (s->n_experts > 32 && (s->n_experts % 8 != 0 || s->top_k > 8)) return false;
  if (s->dim < 128 || s->dim % 128 != 0) return false;
  if (s->hidden < 128 || s->hidden % 128 != 0) return false;
  const int64_t R = (int64_t)s->T * s->top_k;
  const int64_t wide = s->dim > s->hidden ? s->dim : s->hidden;
  if (R * wide >= (int64_t(1) << 31)) return false;
  if ((int64_t)s->n_experts * s->hidden >= (int64_t(1) << 31)) return false;
  if ((int64_t)s->n_experts * s->dim >= (int64_t(1) << 31)) return false;
  return true;
}

static size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(const moe_shape* s) {
  WsLayout L{};
  const size_t T = (size_t)s->T, R = T * (size_t)s->top_k, n = (size_t)s->n_experts;
  L.nchunks = (int)((R + kPermuteChunk - 1) / kPermuteChunk);
  size_t off = 0;
  L.err = off;
  L.counters = kWsHeaderBytes;
  off += kWsControlBytes;  // control region: error word, stream-K counters
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L.ids = take(R * 4);
  L.gates = take(R * 4);
  L.counts = take(n * 4);
  L.offsets = take((n + 1) * 4);
  L.chunk_hist = take((size_t)L.nchunks * n * 4);
  L.chunk_base = take((size_t)L.nchunks * n * 4);
  L.perm_src = take(R * 4);
  L.slot_row = take(R * 4);
  L.u = take(T * (size_t)s->dim * 2);
  L.x_perm = take(R * (size_t)s->dim * 2);
  L.h = take(R * (size_t)s->hidden * 2);
  L.y_perm = take(R * (size_t)s->dim * 2);
  L.partials = take((size_t)kStreamKMaxCtas * 2 * 128 * 64 * 4);
  L.total = off;
  return L;
}

// Workspace of moe_layer_backward: the recomputed forward (with the gate/up
// pre-activations) and the activation gradients, all in the padded grouping.
struct BwdLayout {
  size_t err, ids, gates, counts, offsets, chunk_hist, chunk_base, perm_src, slot_row;
  size_t x_perm, h, ab, y_perm, dO, dab, dx_perm, dg, dl, dl_perm, wgT;
  size_t total;
  int nchunks, rows;  // rows: grouped rows, every expert's group padded to 64
};

static BwdLayout bwd_layout(const moe_shape* s) {
  BwdLayout L{};
  const size_t T = (size_t)s->T, R = T * (size_t)s->top_k, n = (size_t)s->n_experts;
  const size_t d = (size_t)s->dim, h = (size_t)s->hidden;
  L.nchunks = (int)((R + kPermuteChunk - 1) / kPermuteChunk);
  L.rows = permute_padded_rows((int)R, (int)n, 64);
  const size_t rp = (size_t)L.rows;
  size_t off = kWsControlBytes;
  L.err = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  L.ids = take(R * 4);
  L.gates = take(R * 4);
  L.counts = take(n * 4);
  L.offsets = take((n + 1) * 4);
  L.chunk_hist = take((size_t)L.nchunks * n * 4);
  L.chunk_base = take((size_t)L.nchunks * n * 4);
  L.perm_src = take(rp * 4);
  L.slot_row = take(R * 4);
  L.x_perm = take(rp * d * 2);
  L.h = take(rp * h * 2);
  L.ab = take(rp * 2 * h * 2);
  L.y_perm = take(rp * d * 2);
  L.dO = take(rp * d * 2);
  L.dab = take(rp * 2 * h * 2);
  L.dx_perm = take(rp * d * 2);
  L.dg = take(R * 4);
  L.dl = take(R * 4);
  L.dl_perm = take(rp * 4);
  L.wgT = take(n * d * 2);
  L.total = off;
  return L;
}

static bool backward_supported(const moe_shape* s) {
  if (!shape_supported(s) || s->dim % 256 != 0 || s->hidden % 256 != 0) return false;
  const int64_t R = (int64_t)s->T * s->top_k;
  const int64_t rows = R + 64 * (int64_t)s->n_experts;  // bound of the padded grouping
  return rows * 2 * s->hidden < (int64_t(1) << 31);
}

}  // namespace moe

using namespace moe;

namespace {

template <typename P>
bool aligned16(P* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

template <typename P>
bool ok_ptr(P* p) {
  return p != nullptr && aligned16(p);
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<uint8_t*>(ws) + off);
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_bytes(const moe_shape* shape) {
  if (!shape_supported(shape)) return 0;
  return ws_layout(shape).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ok_ptr(ws) || ws_bytes < kWsHeaderBytes) return MOE_ERR_INVALID_ARG;
  const size_t n = ws_bytes < kWsControlBytes ? ws_bytes : kWsControlBytes;
  return cuda_status(cudaMemsetAsync(ws, 0, n, static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_topk(const moe_shape* shape, const moe_bf16* x, const moe_bf16* w_gate,
                           int32_t* ids, float* gates, int32_t* counts, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(counts)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(ids) || !ok_ptr(gates)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router(*shape, x, w_gate, ids, gates, counts, nullptr, 0.0f, nullptr,
                                   static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute(const moe_shape* shape, const moe_bf16* x, const int32_t* ids,
                       int32_t* offsets, int32_t* perm_src, int32_t* slot_row, moe_bf16* x_perm,
                       void* ws, size_t ws_bytes, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(offsets) || !ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!ok_ptr(x) || !ok_ptr(ids) || !ok_ptr(perm_src) || !ok_ptr(slot_row) ||
                       !ok_ptr(x_perm)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(shape);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return cuda_status(launch_permute(*shape, x, ids, nullptr, offsets, at<int32_t>(ws, L.chunk_hist),
                                    at<int32_t>(ws, L.chunk_base), perm_src, slot_row, x_perm,
                                    L.nchunks, static_cast<cudaStream_t>(stream)));
}

moe_status moe_expert_ffn_grouped(const moe_shape* shape, const moe_bf16* x_perm,
                                  const int32_t* offsets, const moe_bf16* w1, const moe_bf16* w3,
                                  const moe_bf16* w2, moe_bf16* h, moe_bf16* y_perm, int32_t path,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (path < MOE_FFN_AUTO || path > MOE_FFN_PAIR_GEMM) return MOE_ERR_INVALID_ARG;
  if (path == MOE_FFN_PAIR_GEMM && !pair_ffn_supported(*shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!ok_ptr(x_perm) || !ok_ptr(offsets) || !ok_ptr(w1) || !ok_ptr(w3) ||
                       !ok_ptr(w2) || !ok_ptr(h) || !ok_ptr(y_perm)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(shape);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const cudaError_t e = launch_expert_ffn(*shape, x_perm, offsets, w1, w3, w2, h, y_perm, path,
                                          at<uint32_t>(ws, L.err), at<float>(ws, L.partials),
                                          at<int>(ws, L.counters),
                                          static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

moe_status moe_combine(const moe_shape* shape, const moe_bf16* y_perm, const int32_t* slot_row,
                       const float* gates, const moe_bf16* residual, moe_bf16* y, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (shape->T > 0 && (!ok_ptr(y_perm) || !ok_ptr(slot_row) || !ok_ptr(gates) || !ok_ptr(y)))
    return MOE_ERR_INVALID_ARG;
  if (residual != nullptr && !aligned16(residual)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(*shape, y_perm, slot_row, gates, residual, y,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_forward(const moe_shape* shape, const moe_layer_opts* opts,
                             const moe_bf16* x, const moe_bf16* w_gate, const moe_bf16* w1,
                             const moe_bf16* w3, const moe_bf16* w2, moe_bf16* y, int32_t* ids,
                             float* gates, void* ws, size_t ws_bytes, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  const int path = opts ? opts->ffn_path : MOE_FFN_AUTO;
  if (path < MOE_FFN_AUTO || path > MOE_FFN_PAIR_GEMM) return MOE_ERR_INVALID_ARG;
  if (path == MOE_FFN_PAIR_GEMM && !pair_ffn_supported(*shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const bool norm = opts && opts->use_rmsnorm;
  if (norm && !(opts->rmsnorm_eps > 0.0f)) return MOE_ERR_INVALID_ARG;
  const moe_bf16* residual = opts ? opts->residual : nullptr;
  if (residual != nullptr && !aligned16(residual)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w3) ||
                       !ok_ptr(w2) || !ok_ptr(y)))
    return MOE_ERR_INVALID_ARG;
  if ((ids != nullptr && !aligned16(ids)) || (gates != nullptr && !aligned16(gates)))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(shape);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (shape->T == 0) return MOE_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* d_ids = ids ? ids : at<int32_t>(ws, L.ids);
  float* d_gates = gates ? gates : at<float>(ws, L.gates);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  uint16_t* u = norm ? at<uint16_t>(ws, L.u) : nullptr;
  const uint16_t* src = norm ? u : x;

  cudaError_t e;
  if (!norm && route_small_supported(*shape)) {
    // decode-sized batch: routing, grouping and gather in one launch
    e = launch_route_small(*shape, x, w_gate, d_ids, d_gates, offsets,
                           at<int32_t>(ws, L.perm_src), at<int32_t>(ws, L.slot_row),
                           at<uint16_t>(ws, L.x_perm), st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    // the grouping recounts the assignments from the ids: the router writes no counts
    e = launch_router(*shape, x, w_gate, d_ids, d_gates, nullptr, u,
                      norm ? opts->rmsnorm_eps : 0.0f, at<uint32_t>(ws, L.err), st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_permute(*shape, src, d_ids, nullptr, offsets, at<int32_t>(ws, L.chunk_hist),
                       at<int32_t>(ws, L.chunk_base), at<int32_t>(ws, L.perm_src),
                       at<int32_t>(ws, L.slot_row), at<uint16_t>(ws, L.x_perm), L.nchunks, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = launch_expert_ffn(*shape, at<uint16_t>(ws, L.x_perm), offsets, w1, w3, w2,
                        at<uint16_t>(ws, L.h), at<uint16_t>(ws, L.y_perm), path,
                        at<uint32_t>(ws, L.err), at<float>(ws, L.partials),
                        at<int>(ws, L.counters), st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  e = launch_combine(*shape, at<uint16_t>(ws, L.y_perm), at<int32_t>(ws, L.slot_row), d_gates,
                     residual, y, st);
  return cuda_status(e);
}

moe_status moe_routing_stats(const moe_shape* shape, const int32_t* ids, int32_t* slot_counts,
                             int32_t* repeats, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(slot_counts) || !ok_ptr(repeats)) return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && !ok_ptr(ids)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_routing_stats(*shape, ids, slot_counts, repeats,
                                          static_cast<cudaStream_t>(stream)));
}

size_t moe_backward_workspace_bytes(const moe_shape* shape) {
  if (!backward_supported(shape)) return 0;
  return bwd_layout(shape).total;
}

moe_status moe_layer_backward(const moe_shape* shape, const moe_bf16* x, const moe_bf16* w_gate,
                              const moe_bf16* w1, const moe_bf16* w3, const moe_bf16* w2,
                              const moe_bf16* dy, moe_bf16* dx, float* dw_gate, float* dw1,
                              float* dw3, float* dw2, void* ws, size_t ws_bytes, void* stream) {
  if (shape == nullptr) return MOE_ERR_INVALID_ARG;
  if (!backward_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!ok_ptr(ws) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w3) || !ok_ptr(w2) ||
      !ok_ptr(dw_gate) || !ok_ptr(dw1) || !ok_ptr(dw3) || !ok_ptr(dw2))
    return MOE_ERR_INVALID_ARG;
  if (shape->T > 0 && (!ok_ptr(x) || !ok_ptr(dy) || !ok_ptr(dx))) return MOE_ERR_INVALID_ARG;
  const BwdLayout L = bwd_layout(shape);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const moe_shape& s = *shape;
  const int T = s.T, n = s.n_experts, d = s.dim, h = s.hidden;
  uint32_t* err = at<uint32_t>(ws, L.err);
  const int64_t nw = (int64_t)n * h * d;  // elements of one expert-weight tensor
  if (T == 0) {
    // no tokens: every weight gradient is zero
    cudaError_t e = cudaMemsetAsync(dw_gate, 0, sizeof(float) * (size_t)d * n, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw1, 0, sizeof(float) * (size_t)nw, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw3, 0, sizeof(float) * (size_t)nw, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, sizeof(float) * (size_t)nw, st);
    return cuda_status(e);
  }
  int32_t* ids = at<int32_t>(ws, L.ids);
  float* gates = at<float>(ws, L.gates);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* slot_row = at<int32_t>(ws, L.slot_row);
  const int rows = L.rows;
  uint16_t* x_perm = at<uint16_t>(ws, L.x_perm);
  uint16_t* hb = at<uint16_t>(ws, L.h);
  uint16_t* ab = at<uint16_t>(ws, L.ab);
  uint16_t* y_perm = at<uint16_t>(ws, L.y_perm);
  uint16_t* dO = at<uint16_t>(ws, L.dO);
  uint16_t* dab = at<uint16_t>(ws, L.dab);
  uint16_t* dx_perm = at<uint16_t>(ws, L.dx_perm);
  float* dg = at<float>(ws, L.dg);
  float* dl = at<float>(ws, L.dl);
  float* dl_perm = at<float>(ws, L.dl_perm);

#define MOE_TRY(call)                           \
  do {                                          \
    const cudaError_t e_ = (call);              \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)
  // forward, recomputed: routing, grouping (every expert's group starting on a
  // multiple of 64 rows), expert FFN keeping the pre-activations
  MOE_TRY(launch_router(s, x, w_gate, ids, gates, nullptr, nullptr, 0.0f, err, st));
  MOE_TRY(launch_permute(s, x, ids, counts, offsets, at<int32_t>(ws, L.chunk_hist),
                         at<int32_t>(ws, L.chunk_base), at<int32_t>(ws, L.perm_src), slot_row,
                         x_perm, L.nchunks, st, 64, rows));
  MOE_TRY(launch_expert_ffn_pair(s, x_perm, offsets, w1, w3, w2, hb, y_perm, err, st, ab, counts,
                                 rows));
  // gated combine and router
  MOE_TRY(launch_combine_bwd(s, dy, y_perm, slot_row, gates, rows, dO, dg, st));
  MOE_TRY(launch_router_bwd(s, gates, dg, slot_row, rows, dl, dl_perm, st));
  MOE_TRY(launch_router_wgrad(s, x_perm, dl_perm, offsets, counts, rows, dw_gate, st));
  // dH = dO W2 -> [dA | dG] (SwiGLU backward from the saved pre-activations);
  // the weights are read in their stored layout (reduction over their rows)
  MOE_TRY(launch_pair_rowgemm(dO, offsets, counts, rows, n, h, d, w2, nullptr, d, dab, 2 * h, ab,
                              err, st));
  // dX_perm = dA W1 + dG W3
  MOE_TRY(launch_pair_rowgemm(dab, offsets, counts, rows, n, d, 2 * h, w1, w3, h, dx_perm, d,
                              nullptr, err, st));
  MOE_TRY(launch_input_grad(s, dx_perm, slot_row, ids, dl, w_gate, at<uint16_t>(ws, L.wgT), rows,
                            dx, st));
  // weight gradients over each expert's padded group (x_perm's padding rows
  // are zero from the grouping; dO's, H's and [dA | dG]'s are zeroed here)
  MOE_TRY(launch_zero_pad_rows(offsets, counts, n, rows, dO, d, hb, h, dab, 2 * h, st));
  MOE_TRY(launch_wgrad(dO, hb, d, h, rows, offsets, n, dw2, dw2, d, err, st));
  MOE_TRY(launch_wgrad(dab, x_perm, 2 * h, d, rows, offsets, n, dw1, dw3, h, err, st));
#undef MOE_TRY
  return MOE_OK;
}

moe_status moe_check_error(void* ws, void* stream) {
  if (!ok_ptr(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0, router_word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (router_err_read_clear(&router_word) != cudaSuccess) return MOE_ERR_CUDA;
  if (router_word != 0 && word == 0) return MOE_ERR_TIMEOUT;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(ws, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_ERR_TIMEOUT;
  }
  return MOE_OK;
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, void* stream) {
  if (!ok_ptr(ws) || ws_bytes < 4096) return MOE_ERR_INVALID_ARG;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_selftest(static_cast<uint32_t*>(ws), limit_ns,
                                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
