/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) MoE decode-layer library
 * (libmoe_decode.so).
 *
 * One low-batch decode step of a DeepSeek/GLM-style MoE layer, as the vLLM
 * specialized-decode executor pages describe it:
 *   [decode page] vllm.models.glm5next.nvidia.specialized_decode.runtime.decode
 *   [draft page]  vllm.models.glm5next.nvidia.specialized_decode.runtime.draft
 *
 * Conventions shared by every entry point
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays that
 *     the caller allocated on the current CUDA device.  The library never
 *     allocates, frees or synchronises (moe_device_status excepted), and keeps
 *     no pointer past return.  Weights are read, never written (the decode
 *     executor leaves the model's own weights untouched: [decode page] class
 *     SpecializedDecode).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is only enqueued; every call is stream-ordered.
 *   - Return value: MOE_OK or an error code below.  Argument errors are found
 *     on the host before anything is enqueued.  There is no CPU fallback:
 *     an unsupported shape returns MOE_ERR_UNSUPPORTED and the caller decides
 *     (the pages' executors likewise refuse unsupported configurations and
 *     leave the step to the stock forward).
 *   - bf16 = IEEE bfloat16 stored as uint16; fp8 = E4M3 (OCP "E4M3FN") codes
 *     stored as uint8; fp32 = IEEE float.
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad value  */
  MOE_ERR_UNSUPPORTED = 2,          /* shape outside the supported range        */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below the *_workspace_size     */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed     */
  MOE_ERR_DEVICE_TIMEOUT = 5,       /* a bounded device-side wait gave up       */
  MOE_ERR_SCRATCH_LIMIT = 6         /* the problem needs more than the library's
                                       static scratch (splitk_gemm_bf16_noalloc) */
};

/*
 * Layer dimensions and switches ([decode page] LayerStages._build_mega: the
 * routed-expert kernel is built from num_experts_per_tok, swiglu_limit,
 * routed_scaling_factor and the e8m0 switch; only sigmoid scoring with
 * n_group == 1 and norm_topk_prob is accepted, which is the only routing this
 * library implements).
 *   hidden        H, multiple of 128, <= 16384
 *   inter         I (moe_intermediate_size), multiple of 128, <= 8192
 *   shared_inter  I_s of the shared expert, multiple of 128 (0 = none)
 *   num_experts   E routed experts, 1 <= E <= 512
 *   top_k         k, 1 <= k <= min(E, 16)
 *   routed_scaling  multiplies the normalised top-k weights
 *   swiglu_limit  L in h = silu(min(g, L)) * clamp(u, -L, L); +inf disables it
 *   rms_eps       epsilon inside the RMSNorm square root
 *   e8m0          nonzero: activation block scales are rounded up to powers of
 *                 two (the weights' scales are then expected to be powers of
 *                 two as well; they are used as given either way)
 */
typedef struct moe_layer_dims {
  int hidden;
  int inter;
  int shared_inter;
  int num_experts;
  int top_k;
  float routed_scaling;
  float swiglu_limit;
  float rms_eps;
  int e8m0;
} moe_layer_dims;

/*
 * Weights of one MoE layer ([decode page] LayerStages._build_mega:
 * w13_weight, w13_weight_scale_inv, w2_weight, w2_weight_scale_inv, the
 * shared expert's gate_up_proj / down_proj with their weight_scale_inv, the
 * gate's bf16 weight and e_score_correction_bias).
 *   router_w  bf16 [E, H]
 *   sel_bias  fp32 [E] or NULL: added to the sigmoid scores for selection only
 *   w13       fp8 [E, 2I, H]: rows [0, I) gate, rows [I, 2I) up
 *   w13_s     fp32 [E, 2I/128, H/128]: scale of each 128x128 block (w = code * s)
 *   w2        fp8 [E, H, I];  w2_s fp32 [E, H/128, I/128]
 *   sw13, sw13_s, sw2, sw2_s: the shared expert alike, without the E dimension
 *             (NULL when shared_inter == 0)
 *   norm_gain bf16 [H]: gain of the RMSNorm at the layer boundary
 * All weight pointers must be 16-byte aligned.
 */
typedef struct moe_layer_weights {
  const void *router_w;
  const float *sel_bias;
  const uint8_t *w13;
  const float *w13_s;
  const uint8_t *w2;
  const float *w2_s;
  const uint8_t *sw13;
  const float *sw13_s;
  const uint8_t *sw2;
  const float *sw2_s;
  const void *norm_gain;
} moe_layer_weights;

/* Bytes of device workspace moe_decode_layer needs for up to max_tokens
 * tokens (1 <= max_tokens <= 4096, max_tokens * top_k <= 4096). */
int moe_decode_workspace_size(const moe_layer_dims *dims, int max_tokens, size_t *bytes);

/* Zero a workspace (moe_decode_layer's or splitk_gemm_bf16's) once before its
 * first use.  Calls leave their counters at zero for the next call, so this
 * is needed only once per buffer, and again after a call returned an error
 * (a launch that failed part-way can leave a counter set). */
int moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/*
 * One decode step of the MoE layer plus the layer boundary, for M tokens:
 *   logits = x . router_w^T (fp32); s = sigmoid(logits); sel = s + sel_bias;
 *   ids = top-k of sel (descending; ties to the lower id);
 *   w = s[ids] / sum(s[ids]) * routed_scaling;
 *   route order: stable counting sort of r = t*k + j by expert;
 *   per routed expert and for the shared expert (weight 1), on FP8 activations
 *   quantised per token per 128-column group (scale = amax/448):
 *     [g; u] = x . w13^T, h = silu(min(g, L)) * clamp(u, -L, L),
 *     h quantised likewise, y = h . w2^T;
 *   m = sum_j w_j * y_(t,j) + y_shared;  r' = m + residual;
 *   residual_out = bf16(r');  out = bf16(r' * rsqrt(mean(r'^2) + eps) * gain).
 * ([decode page] LayerStages._mega_moe / _router; [draft page]
 * SpecializedDraft.reduced_norm: the boundary returns the normalised sum and
 * the updated residual.)
 *
 *   x, residual      bf16 [M, H] inputs (may not alias the outputs)
 *   out, residual_out  bf16 [M, H] outputs
 *   topk_ids         int32 [M, k] or NULL; topk_w fp32 [M, k] or NULL
 *   sorted_routes    int32 [M*k] or NULL: expanded route indices grouped by
 *                    expert (ascending), ascending within an expert
 *   expert_offsets   int32 [E+1] or NULL: start of each expert's routes
 *   workspace        from moe_decode_workspace_size(dims, max_tokens >= M),
 *                    zeroed once by moe_workspace_init; one workspace must not
 *                    be used by two calls that may run concurrently
 * M == 0 is a no-op.  Launches three kernels (router + top-k + route order;
 * the expert kernel; finalize + residual + RMSNorm), four when the
 * tensor-core expert kernel serves an MoE layer (the routed tokens' x codes
 * are first gathered in route order); moe_decode_layer_plan reports which.
 * The expert kernel is the warp-MMA kernel for narrow steps and the tcgen05
 * kernel where an expert's tokens can make a real contraction (a dense layer
 * from 4 tokens, an MoE layer from 16 tokens); both compute the same results
 * up to fp32 summation order and the SwiGLU's exponential.
 *
 * Dense layers ([decode page] LayerStages._build_dense: a dense FP8 MLP run as
 * GEMVs): num_experts = 0, top_k = 0, inter = 0 and the MLP's weights in the
 * shared-expert slot (sw13 [2 I_s, H], sw2 [H, I_s], I_s <= 32768); router_w,
 * w13 and w2 are not read and may be NULL.  Then m = y_shared and the same
 * boundary follows; topk_ids / topk_w / sorted_routes are empty and
 * expert_offsets[0] = 0.
 */
int moe_decode_layer(const moe_layer_dims *dims, const moe_layer_weights *w, int M,
                     const void *x, const void *residual, void *out, void *residual_out,
                     int32_t *topk_ids, float *topk_w, int32_t *sorted_routes,
                     int32_t *expert_offsets, void *workspace, size_t ws_bytes,
                     void *stream);

/* moe_decode_layer that also records four CUDA events (cudaEvent_t passed as
 * void*) on `stream`: events[0] before the router kernel, [1] before the
 * expert phase (the gather of routed rows, when it runs, and the expert
 * kernel), [2] before the boundary kernel, [3] after it, so that a caller can
 * time each phase.  The events are created by the caller. */
int moe_decode_layer_traced(const moe_layer_dims *dims, const moe_layer_weights *w, int M,
                            const void *x, const void *residual, void *out, void *residual_out,
                            int32_t *topk_ids, float *topk_w, int32_t *sorted_routes,
                            int32_t *expert_offsets, void *workspace, size_t ws_bytes,
                            void *stream, void *const *events);

/*
 * Tensor parallelism over each expert's intermediate dimension ([decode page]
 * LayerStages leaves the MoE sublayer "TP-partial"; [draft page] module
 * docstring: the boundaries fuse the all-reduce with the residual add and the
 * RMSNorm).  Rank g of G holds, of every routed expert and of the shared
 * expert, the gate rows [g I/G, (g+1) I/G) and the same up rows of w13, and the
 * same columns of w2, with their block scales (I/G and I_s/G multiples of 128,
 * so that no 128 x 128 scale block and no h quantisation group straddles two
 * ranks).  A rank's shard is therefore an MoE layer with inter = I/G and
 * shared_inter = I_s/G (router weight and bias replicated), and:
 *
 * moe_decode_layer_partial: moe_decode_layer on a rank's shard up to the
 *   weighted finalize: m_out (fp32 [M, H]) = sum_j w_j * y_(t,j) + y_shared,
 *   this rank's share of m; the ranks' m_out sum to the whole layer's m.  No
 *   residual, gain or bf16 outputs (norm_gain may be NULL).  Same workspace
 *   and routing outputs as moe_decode_layer; launches its kernels alike (the
 *   boundary kernel writes m_out instead of normalising).
 *
 * moe_tp_boundary: the layer boundary over G partial sums in this GPU's
 *   memory (gathered by the caller, e.g. an all-gather or peer copies):
 *   m = sum_{g < G} partials[g] (in rank order, fp32), r' = m + residual,
 *   residual_out = bf16(r'), out = bf16(bf16(r') * rsqrt(mean(bf16(r')^2) +
 *   eps) * gain).  partials fp32 [G, M, H]; the rest as rmsnorm_residual.
 */
int moe_decode_layer_partial(const moe_layer_dims *dims, const moe_layer_weights *w, int M,
                             const void *x, float *m_out, int32_t *topk_ids, float *topk_w,
                             int32_t *sorted_routes, int32_t *expert_offsets, void *workspace,
                             size_t ws_bytes, void *stream);
int moe_tp_boundary(const float *partials, int G, const void *residual, const void *gain, int M, int H,
                    float eps, void *out, void *residual_out, void *stream);

/* Bytes of workspace splitk_gemm_bf16 needs for this shape and split_k. */
int splitk_gemm_workspace_size(int M, int N, int K, int split_k, size_t *bytes);

/*
 * Split-K BF16 projection ([draft page] module docstring: the draft's BF16
 * projections such as eh_proj run a split-K GEMM above two tokens;
 * SpecializedDraft.run.  [decode page] LayerStages._router passes its split
 * count to the router's split-K GEMM explicitly):
 *   C[M, N] = alpha * A[M, K] . W[N, K]^T, fp32 accumulation.
 *   A bf16 [M, K]; W bf16 [N, K]; C bf16 [M, N] (c_fp32 == 0) or fp32 [M, N].
 *   1 <= M <= 256, N % 16 == 0, K % 128 == 0; A, W 16-byte aligned.
 *   split_k  0: the library divides the K dimension over the whole GPU
 *            (stream-K: every SM streams an equal share of W);
 *            S > 0: every (token chunk, 64-row tile) of C is cut into exactly
 *            S K-segments of K/(128 S) k-blocks each (rounded), one CTA a
 *            segment; 1 <= S <= K/128 (MOE_ERR_UNSUPPORTED above, a negative
 *            value is MOE_ERR_INVALID_ARG).
 * Partial sums are reduced in segment order, so results are deterministic for
 * a given split; different splits may differ in the last bits.
 */
int splitk_gemm_bf16(const void *A, const void *W, void *C, int c_fp32, int M, int N, int K,
                     int split_k, float alpha, void *ws, size_t ws_bytes, void *stream);

/*
 * splitk_gemm_bf16 without a caller-provided workspace, for callers that
 * cannot allocate device memory at the point where they run the projection
 * (for example a plugin whose enqueue function must not call cudaMalloc, or a
 * runtime that hands out only a fixed pool it owns).  No counterpart on the
 * source pages: this is an interface convenience of this library.
 *
 * Same arguments and result as splitk_gemm_bf16 (the same plan, hence the
 * same bits), minus ws / ws_bytes.  The
 * partial sums and tile counters live in one static device array of
 * MOE_NOALLOC_SCRATCH_BYTES (8 MiB) in the library, which every GPU that
 * loads the library holds until the process exits.  Nothing is allocated or
 * freed.  The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any work
 * whose ordering depends on it.  Every call shares the array: calls that may
 * overlap on the GPU (different streams, or different host threads without
 * ordering) race and corrupt each other's results; serialise them on one
 * stream.  A shape whose split needs more scratch than the limit returns
 * MOE_ERR_SCRATCH_LIMIT before anything is enqueued.  The tile counters are
 * cleared (cudaMemsetAsync on the array, no allocation) at every call.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int splitk_gemm_bf16_noalloc(const void *A, const void *W, void *C, int c_fp32, int M, int N, int K,
                             int split_k, float alpha, void *stream);

/* Test hook: fill the whole static scratch of splitk_gemm_bf16_noalloc on the
 * current device with `byte` (stream-ordered), so that a test can check that
 * a call clears the counters it uses whatever an earlier call left there. */
int moe_debug_fill_noalloc_scratch(int byte, void *stream);

/*
 * Layer boundary: optional weighted top-k finalize, residual add, RMSNorm
 * ([draft page] SpecializedDraft.reduced_norm; [decode page] _mega_moe hands
 * the routed rows over unfinalized, in expanded order, for this step):
 *   m[t] = (x ? x[t] : 0) + (rows ? sum_j route_w[t, j] * rows[t*k + j] : 0)
 *          + (shared ? shared[t] : 0)
 *   r' = m + residual;  residual_out = bf16(r');
 *   out = bf16(bf16(r') * rsqrt(mean(bf16(r')^2) + eps) * gain)
 *   x bf16 [M, H] or NULL; residual, gain bf16; rows fp32 [M*k, H] or NULL;
 *   route_w fp32 [M, k] (needed with rows); shared fp32 [M, H] or NULL;
 *   out, residual_out bf16 [M, H].  H % 128 == 0, H <= 16384.
 */
int rmsnorm_residual(const void *x, const void *residual, const void *gain, int M, int H,
                     float eps, const float *rows, const float *route_w, int k,
                     const float *shared, void *out, void *residual_out, void *stream);

/* The MTP layer's input projection ([draft page] vllm.models.glm5next.nvidia
 * .specialized_decode.runtime.draft, SpecializedDraft.run: the input tokens'
 * embeddings and the previous hidden state, each RMS-normalised with its own
 * gain, concatenated, then eh_proj):
 *   A[t] = [ bf16(e * rsqrt(mean(e^2) + eps) * enorm) | bf16(h * rsqrt(mean(h^2) + eps) * hnorm) ],
 *          e = embed[input_ids[t]], h = hidden[t]   (the embedding half first);
 *   out = A . eh_proj_w^T   (split-K BF16 GEMM, fp32 sums rounded once to bf16).
 *
 *   input_ids   int32 [M] device; ids outside [0, vocab) give a zero embedding
 *               half and MOE_ERR_INVALID_ARG in the workspace status word
 *               (moe_device_status), never a read outside the table
 *   embed       bf16 [vocab, H];  hidden bf16 [M, H];  enorm, hnorm bf16 [H]
 *   eh_proj_w   bf16 [H, 2H] row-major;  out bf16 [M, H]
 *   workspace   mtp_eh_front_workspace_size(M, H) bytes, zeroed once by
 *               moe_workspace_init; holds A (readable by the caller after the
 *               call, at byte offset 256, bf16 [M, 2H]) and the split-K sums
 * Limits: 1 <= M <= 256, H % 128 == 0, H <= 16384, vocab >= 1; 16-byte aligned
 * pointers.  Argument errors return before anything is enqueued.  Calls that
 * share a workspace must be stream-ordered.
 * Two kernels: the norm kernel, then the projection, launched with
 * programmatic dependent launch so that it prefetches its first weight tiles
 * into L2 while the norm kernel runs (eh_proj_w must not be written by the
 * kernel enqueued just before the call). */
int mtp_eh_front_workspace_size(int M, int H, size_t *bytes);
int mtp_eh_front(const int32_t *input_ids, const void *embed, int vocab, const void *hidden,
                 const void *enorm, const void *hnorm, float eps, const void *eh_proj_w, int M, int H,
                 void *out, void *ws, size_t ws_bytes, void *stream);

/* Expert kernels (moe_decode_layer_plan, moe_set_expert_path). */
enum moe_expert_path {
  MOE_PATH_AUTO = 0,      /* the library's choice by layer kind and token count */
  MOE_PATH_WARP_MMA = 1,  /* warp-level FP8 MMAs on 8/16/32-token passes       */
  MOE_PATH_TCGEN05 = 2    /* tcgen05 FP8 MMAs, tensor-memory accumulators,
                             passes of up to 64 tokens                          */
};

/* The expert kernel a moe_decode_layer call of M tokens runs (*path, never
 * MOE_PATH_AUTO for M > 0) and the number of kernels it launches
 * (*launches).  Host only. */
int moe_decode_layer_plan(const moe_layer_dims *dims, int M, int *path, int *launches);

/* Tuning and test hook: force the expert kernel of every later
 * moe_decode_layer call in the process (MOE_PATH_AUTO restores the library's
 * choice).  Process-wide; not meant to change while calls are being made
 * from other host threads. */
int moe_set_expert_path(int path);

/* Read and clear the device status word of a moe_decode_layer workspace:
 * MOE_OK, or MOE_ERR_DEVICE_TIMEOUT when a bounded wait inside the expert
 * kernel gave up.  Synchronises `stream`; meant for tests and diagnostics. */
int moe_device_status(void *ws, void *stream);

/* Test hook: nonzero `fault` makes the next moe_decode_layer calls on this
 * workspace withhold one expert's ready signal, so that the waits on it run
 * out (about 0.2 s) and report MOE_ERR_DEVICE_TIMEOUT.  Nothing faults. */
int moe_debug_set_fault(void *ws, int fault, void *stream);

/* Text of a status code. */
const char *moe_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_H */
