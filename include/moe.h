/*
 * moe.h -- C ABI of the B300 (sm_103a) Mixtral sparse mixture-of-experts
 * layer: the forward and its steps, the backward (routing held fixed) and the
 * routing statistics.
 *
 * The layer ("Mixtral of Experts", section 2.1):
 *     y = sum_i G(x)_i * E_i(x),         G(x) = Softmax(TopK(x . W_g)),
 *     E_i(x) = W2_i (SiLU(W1_i x) * (W3_i x))      (SwiGLU expert),
 * with n = 8 experts and K = 2 in Mixtral (Table 1).  TopK keeps the K largest
 * logits and sets the rest to minus infinity, so each token only evaluates its
 * K selected experts.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every array argument is caller-owned DEVICE memory, row-major, and must be
 *   16-byte aligned.  The library allocates nothing and never synchronises the
 *   stream, except moe_check_error.  It keeps state between calls in two
 *   places only, both process-wide device objects: (1) the error word of
 *   moe_router_topk, which has no workspace -- an expired bounded wait of any
 *   moe_router_topk call, on any stream, is recorded there, and ANY
 *   moe_check_error call reports and clears it, whatever workspace it is
 *   given; (2) the fixed scratch of moe_permute_noalloc (see there).  Every
 *   other entry point keeps its state in the caller's workspace.
 * - bf16 arrays are raw bfloat16 bit patterns (moe_bf16).
 * - Shapes: x, y [T, dim]; w_gate [dim, n]; w1, w3 [n, hidden, dim];
 *   w2 [n, dim, hidden]; ids [T, K] int32; gates [T, K] float32;
 *   counts [n]; offsets [n + 1]; perm_src, slot_row [T*K];
 *   x_perm, y_perm [T*K, dim]; h [T*K, hidden].
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  All work is
 *   enqueued asynchronously on it, in order.
 * - Routing conventions: slot k of a token holds its k-th largest logit, ties
 *   broken towards the lower expert index, a NaN logit counting as -infinity;
 *   gates are the softmax of the K selected logits (float32).  The grouped ("permuted") row order is the
 *   stable sort of the flat assignments a = t*K + k by expert id: rows
 *   [offsets[e], offsets[e+1]) belong to expert e, tokens ascending.
 * - Supported shapes: T >= 0 (T = 0 is a no-op), 1 <= top_k <= n_experts <= 256,
 *   with n_experts a multiple of 8 and top_k <= 8 when n_experts > 32 (the
 *   fine-grained variant: e.g. the top 8 of 160 smaller experts); dim and
 *   hidden positive multiples of 128; T*top_k*max(dim, hidden) < 2^31.
 * - Errors: argument and shape checks return synchronously (nothing is
 *   enqueued); a failed launch returns MOE_ERR_CUDA.  Kernels never trap:
 *   a bounded device-side wait that expires records MOE_ERR_TIMEOUT in the
 *   workspace error word, which moe_check_error reports.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(MOE_BUILD) && defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16; /* bfloat16 bit pattern */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null or misaligned pointer, bad option */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* shape outside the supported set above */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < moe_workspace_bytes(shape) */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed */
  MOE_ERR_TIMEOUT = 5               /* a bounded device wait expired */
} moe_status;

/* Problem shape of one layer call. */
typedef struct {
  int32_t T;         /* tokens */
  int32_t dim;       /* model dimension (4096 in Table 1) */
  int32_t hidden;    /* expert hidden dimension (14336 in Table 1) */
  int32_t n_experts; /* n (8) */
  int32_t top_k;     /* K (2) */
} moe_shape;

/* Expert-FFN implementation choice (moe_layer_opts.ffn_path, and the `path`
 * argument of moe_expert_ffn_grouped). */
enum {
  MOE_FFN_AUTO = 0,          /* weight stream for T <= 32; otherwise the CTA-pair
                                GEMM when dim % 256 == 0, else the grouped GEMM */
  MOE_FFN_GROUPED_GEMM = 1,  /* tokens on the MMA M side, 128-row token tiles */
  MOE_FFN_WEIGHT_STREAM = 2, /* weights on the MMA M side, 32-token chunks */
  MOE_FFN_PAIR_GEMM = 3      /* weights on the M side of a two-SM (CTA pair) MMA,
                                token tiles of up to 256 rows; needs dim % 256 == 0
                                (MOE_ERR_UNSUPPORTED_SHAPE otherwise) */
};

/* Options of moe_layer_forward; pass NULL for the plain layer. */
typedef struct {
  int32_t use_rmsnorm;      /* 1: route and evaluate experts on RMSNorm(x) */
  float rmsnorm_eps;        /* RMSNorm epsilon (unit gain), e.g. 1e-5 */
  const moe_bf16* residual; /* [T, dim] added to the output in fp32; nullable */
  int32_t ffn_path;         /* MOE_FFN_* */
} moe_layer_opts;

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(moe_status status);

/* Bytes of device workspace needed by moe_permute, moe_expert_ffn_grouped and
 * moe_layer_forward for this shape (one size serves all three).  Returns 0 for
 * an unsupported shape. */
MOE_API size_t moe_workspace_bytes(const moe_shape* shape);

/* Prepare a workspace: zero its first 64 KB (the error word and the arrival
 * counters of the weight stream's split tiles, which every completed call
 * leaves at zero).  Call once after allocating a workspace, and again after
 * moe_check_error has reported MOE_ERR_TIMEOUT (an aborted call may leave
 * counters behind). */
MOE_API moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* Router: logits l = x . w_gate in fp32 from bf16 inputs, top-K selection and
 * the softmax of the selected logits ("Mixtral of Experts" section 2.1, the
 * gating definition G(x) = Softmax(TopK(x . W_g))).
 *   out ids [T, K], gates [T, K], counts [n] (assignments per expert; zeroed
 *   and filled by this call). */
MOE_API moe_status moe_router_topk(const moe_shape* shape, const moe_bf16* x,
                           const moe_bf16* w_gate, int32_t* ids, float* gates,
                           int32_t* counts, void* stream);

/* Grouping of the T*K assignments by expert (the per-expert token groups of
 * section 2.1, where different experts receive different numbers of tokens):
 *   out offsets [n + 1] (exclusive prefix sum of the per-expert counts),
 *   perm_src [T*K] (grouped row -> token), slot_row [T*K] (assignment t*K+k ->
 *   grouped row), x_perm [T*K, dim] (x_perm[r] = x[perm_src[r]], bit copy).
 *   ws: workspace of moe_workspace_bytes(shape) bytes (scratch).
 * The per-expert counts are recounted from ids rather than taken as an input:
 * a stable order needs the per-expert counts of every block of assignments,
 * which the grouping computes anyway, and their sums are the per-expert
 * counts. */
MOE_API moe_status moe_permute(const moe_shape* shape, const moe_bf16* x,
                       const int32_t* ids, int32_t* offsets, int32_t* perm_src,
                       int32_t* slot_row, moe_bf16* x_perm, void* ws,
                       size_t ws_bytes, void* stream);

/* Expert SwiGLU FFN over the grouped rows (section 2.1, the SwiGLU expert
 * E_i(x)): for every expert e and row r in [offsets[e], offsets[e+1]):
 *   h[r]      = bf16( SiLU(x_perm[r] W1_e^T) * (x_perm[r] W3_e^T) )   (fp32 acc.)
 *   y_perm[r] = bf16( h[r] W2_e^T )                                   (fp32 acc.)
 * offsets is read on the device (the host never sees the counts).
 * path: MOE_FFN_* (AUTO picks the weight stream for T <= 32).
 * ws: workspace of moe_workspace_bytes(shape) bytes; its error word records
 * expired waits (see moe_check_error). */
MOE_API moe_status moe_expert_ffn_grouped(const moe_shape* shape, const moe_bf16* x_perm,
                                  const int32_t* offsets, const moe_bf16* w1,
                                  const moe_bf16* w3, const moe_bf16* w2,
                                  moe_bf16* h, moe_bf16* y_perm, int32_t path,
                                  void* ws, size_t ws_bytes, void* stream);

/* Gated combine (section 2.1, the weighted sum over the selected experts):
 *   y[t] = bf16( sum_{k<K} gates[t,k] * y_perm[slot_row[t*K+k]]  (+ residual[t]) )
 * in fp32, k ascending (deterministic).  residual is nullable. */
MOE_API moe_status moe_combine(const moe_shape* shape, const moe_bf16* y_perm,
                       const int32_t* slot_row, const float* gates,
                       const moe_bf16* residual, moe_bf16* y, void* stream);

/* The whole layer: router -> grouping -> expert FFN -> combine, all on
 * `stream`, no host synchronisation.  A decode-sized batch (T <= 32 tokens,
 * n <= 8 experts, no RMSNorm) is routed, grouped and gathered by one kernel
 * launch; its logits are summed in another order than moe_router_topk's, so
 * gates may differ from that entry point's in the last bits (ids agree
 * wherever the selection is decided).  ids and gates are optional outputs
 * (nullable; kept in the workspace otherwise).  With opts->use_rmsnorm the
 * layer routes and evaluates RMSNorm(x) (bf16, unit gain) and the combine
 * adds opts->residual (pass x for the residual block x + MoE(RMSNorm(x))). */
MOE_API moe_status moe_layer_forward(const moe_shape* shape, const moe_layer_opts* opts,
                             const moe_bf16* x, const moe_bf16* w_gate,
                             const moe_bf16* w1, const moe_bf16* w3,
                             const moe_bf16* w2, moe_bf16* y, int32_t* ids,
                             float* gates, void* ws, size_t ws_bytes,
                             void* stream);

/* Backward pass of the layer (the gradient of section 2.1's
 * y = sum_k G(x)_k E_k(x) for an upstream gradient dy, with the routing held
 * fixed: TopK is piecewise constant, so W_g and x receive the gradient of the
 * softmax over the selected logits).  Recomputes the forward (router,
 * grouping, expert FFN keeping the gate/up pre-activations) in `ws`, then:
 *   dx [T, dim] bf16;  dw_gate [dim, n], dw1 / dw3 [n, hidden, dim],
 *   dw2 [n, dim, hidden] float32 (overwritten, not accumulated).
 * The expert-weight gradients are summed over the tokens routed to each
 * expert by tcgen05 GEMMs; every sum has a fixed order (deterministic).
 * Needs dim and hidden multiples of 256 (MOE_ERR_UNSUPPORTED_SHAPE otherwise)
 * and a workspace of moe_backward_workspace_bytes(shape) bytes, initialised
 * with moe_workspace_init.  No RMSNorm / residual option. */
MOE_API size_t moe_backward_workspace_bytes(const moe_shape* shape);
MOE_API moe_status moe_layer_backward(const moe_shape* shape, const moe_bf16* x,
                                      const moe_bf16* w_gate, const moe_bf16* w1,
                                      const moe_bf16* w3, const moe_bf16* w2,
                                      const moe_bf16* dy, moe_bf16* dx, float* dw_gate,
                                      float* dw1, float* dw3, float* dw2, void* ws,
                                      size_t ws_bytes, void* stream);

/* Routing statistics ("Mixtral of Experts" section 5, Routing analysis) of
 * the expert ids [T, K] produced by moe_router_topk or moe_layer_forward:
 *   slot_counts [K * n]  slot_counts[k*n + e] = tokens whose k-th choice is
 *                        expert e (Fig. 7 shares: sum over k divided by T*K;
 *                        Fig. 9: per k divided by T);
 *   repeats [2]          repeats[0] = pairs of consecutive tokens (t, t+1)
 *                        with the same first choice; repeats[1] = pairs whose
 *                        K chosen experts share at least one expert (Table 5,
 *                        "first choice only" and "first or second choice";
 *                        divide by T-1 for the rates).
 * Both outputs are zeroed and filled by this call (integer counts: exact and
 * independent of scheduling).  Ids outside [0, n) are not counted. */
MOE_API moe_status moe_routing_stats(const moe_shape* shape, const int32_t* ids,
                                     int32_t* slot_counts, int32_t* repeats, void* stream);

/* Synchronise `stream`, read and clear the workspace error word and the
 * process-wide error word of moe_router_topk (see the conventions above).
 * Returns MOE_ERR_TIMEOUT if any bounded device wait of a call using this
 * workspace, or of any moe_router_topk call, expired since the last check;
 * MOE_ERR_CUDA on a pending CUDA error; MOE_OK otherwise.  After
 * MOE_ERR_TIMEOUT, call moe_workspace_init on the workspace again. */
MOE_API moe_status moe_check_error(void* ws, void* stream);

/* Diagnostic of the bounded-wait machinery (no counterpart on the pages):
 * launches one block that waits, through the same bounded mbarrier wait the
 * GEMM kernels use, on a barrier nothing ever arrives at, with a limit of
 * `limit_ns` nanoseconds; the expiry is recorded in the workspace error word
 * exactly as a real expiry would be.  moe_check_error then returns
 * MOE_ERR_TIMEOUT.  No GPU fault is involved. */
MOE_API moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes,
                                     uint64_t limit_ns, void* stream);

/* moe_permute without a workspace (the paper has no counterpart: this is an
 * interface convenience, not a step of the method).  Same outputs, same
 * kernels and same argument rules as moe_permute, but the call takes no `ws`
 * and allocates nothing: its scratch (two [chunk][expert] count tables) lives
 * in a fixed 512 KiB device array inside this library, held on every GPU that
 * loads the library until the process exits.
 *
 * It is meant for callers that receive only their input and output buffers
 * from a host framework (a plugin or custom-operator interface without a
 * workspace argument) and may not call cudaMalloc themselves, because the
 * framework owns all device memory or forbids allocation during a step.
 *
 * Limit: ceil(T*K / 256) * n_experts <= 65536 (T*K <= 2,097,152 for n = 8);
 * larger shapes return MOE_ERR_WORKSPACE_TOO_SMALL and enqueue nothing.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.
 * All calls share the one array: calls that may overlap on the GPU (other
 * streams, other threads) race on it and must be serialised by the caller.
 * Each call overwrites the tables completely before reading them. */
MOE_API moe_status moe_permute_noalloc(const moe_shape* shape, const moe_bf16* x,
                                       const int32_t* ids, int32_t* offsets,
                                       int32_t* perm_src, int32_t* slot_row,
                                       moe_bf16* x_perm, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
