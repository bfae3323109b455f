/*
 * si_moe.h - decode-time Mixture-of-Experts FFN stage for GB300 (sm_103a).
 *
 * A C ABI over hand-written CUDA kernels. Plain pointers and sizes only.
 *
 * The calls follow the statement of the problem on three sparkinfer
 * pull-request pages:
 *   [R] "perf(qwen3.6): fused router GEMV+top-k + folded residual-norm (decode)"
 *       (PR #273), Summary items 1 and 2;
 *   [S] "perf(qwen3.6): fuse decode kernel launches - shared-expert + GDN
 *       conv/L2-norm" (PR #239), Summary item 1;
 *   [Q] "Q4_K shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN
 *       stage" (PR #359), Summary.
 *
 * Conventions for every call below.
 *  - Pointers named x, w_*, *_out, workspace are DEVICE pointers owned by the
 *    caller; layer descriptors and handles are host memory. Matrices are
 *    row-major with the reduction dimension contiguous. Quantised matrices are
 *    rows of standard blocks: Q4_K 144 bytes per 256 weights, Q8_0 34 bytes per
 *    32, Q8_1 36 bytes per 32; every row must start on a 16-byte boundary
 *    (true for the sizes accepted below) and every base pointer must be
 *    16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls only enqueue work: they never allocate device memory, never
 *    synchronise (except si_workspace_status) and are valid inside CUDA
 *    stream capture.
 *  - Arguments are checked on the host first; on failure the call returns
 *    SI_ERR_INVALID_ARG, SI_ERR_UNSUPPORTED or SI_ERR_WORKSPACE and enqueues
 *    nothing. A failed launch returns SI_ERR_CUDA. Errors found on the device
 *    (corrupted completion handshake, a bounded wait that ran out) are written
 *    to the status word at the start of the workspace; read it with
 *    si_workspace_status. No call throws.
 *  - Workspaces: size them with the matching *_workspace_bytes query, align to
 *    256 bytes and fill with zeros once before first use (cudaMemset). Their
 *    completion counters return to zero at the end of every run, so a
 *    workspace can be replayed from a CUDA graph with no reset node. Two calls
 *    that may run at the same time must not share a workspace.
 *  - Consecutive kernels of this library use programmatic dependent launch:
 *    each kernel may start while its predecessor in the stream is still
 *    running, and reads, before waiting for that predecessor, only inputs
 *    produced by work that precedes the predecessor. A caller's kernel placed
 *    between two calls behaves as an ordinary stream dependency.
 */
#ifndef SI_MOE_H
#define SI_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SI_OK = 0,
  SI_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  SI_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape / dtype combination) */
  SI_ERR_WORKSPACE = 3,     /* workspace null, too small or misaligned */
  SI_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  SI_ERR_HANDSHAKE = 5,     /* device: completion counter inconsistent (workspace not zeroed?) */
  SI_ERR_TIMEOUT = 6        /* device: a bounded wait ran out */
} si_status;

/* Element / block types; numbering follows GGML's type ids ([Q] names Q4_K as
 * type 12 in its routed-down dispatch). */
typedef enum {
  SI_F32 = 0,
  SI_F16 = 1,
  SI_Q8_0 = 8,
  SI_Q8_1 = 9,
  SI_Q4_K = 12,
  SI_Q5_K = 13,
  SI_BF16 = 30
} si_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char *si_status_string(int status);

/* Library ABI version: (major << 16) | minor. */
int si_version(void);

/* Bytes of one row of `k` elements of `type` (0 if k is not a multiple of the
 * type's block size). */
size_t si_row_bytes(si_dtype type, int64_t k);

/*
 * si_quantize_q8_1 - activation quantisation ("FNQ Q8_1", "quant_h Q8_1", [Q]).
 *
 * For each block of 32 values: amax = max|x|, d = amax / 127 (fp32, IEEE
 * division), q_i = round-half-away-from-zero(x_i / d) clamped to [-127, 127]
 * (all 0 when amax = 0), stored d16 = fp16(d), s16 = fp16(d * sum_i q_i).
 * Output block: {fp16 d16, fp16 s16, int8 q[32]} = 36 bytes.
 *   x       device, n values of x_type (SI_F32 or SI_BF16)
 *   n       number of values, > 0 and a multiple of 32
 *   y_q8_1  device, n/32 * 36 bytes
 */
si_status si_quantize_q8_1(const void *x, si_dtype x_type, int64_t n, void *y_q8_1,
                           void *stream);

/*
 * si_moe_router_topk - fused router GEMV + top-k + softmax ([R] item 1).
 *
 * logits[t][e] = sum_h w_router[e][h] * x[t][h] (fp32 accumulate, split along h
 * over thread blocks, partial sums reduced in a fixed order: deterministic);
 * the last block to finish (a wrapping completion counter in the workspace)
 * selects, per token, the top_k experts ordered by logit descending with ties
 * to the lower expert index, and writes w[t][r] = exp(l_r - l_0) /
 * sum_j exp(l_j - l_0) over the selected logits, in rank order.
 *   x          device [n_tokens][hidden], x_type SI_BF16 or SI_F32
 *   w_router   device [n_experts][hidden], w_type SI_BF16 or SI_F32
 *   hidden     multiple of 256, <= 16384
 *   n_experts  8..256; top_k 1..8 (top_k <= n_experts); n_tokens >= 1
 *   topk_ids   device int32 [n_tokens][top_k]; topk_w device fp32 [n_tokens][top_k]
 *   logits_out device fp32 [n_tokens][n_experts], or NULL
 *   workspace  si_moe_router_workspace_bytes(n_experts, hidden, n_tokens) bytes
 * NaN logits are outside the contract (selection among NaNs is unspecified).
 */
size_t si_moe_router_workspace_bytes(int n_experts, int hidden, int n_tokens);
si_status si_moe_router_topk(const void *x, si_dtype x_type, const void *w_router,
                             si_dtype w_type, int hidden, int n_experts, int top_k,
                             int n_tokens, int32_t *topk_ids, float *topk_w,
                             float *logits_out, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * si_moe_router_topk_noalloc - si_moe_router_topk without a caller workspace.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory when they route a token - for example a
 * serving loop that forbids cudaMalloc/cudaFree after start-up (both can
 * synchronise the whole device and stall other streams), or a plug-in running
 * inside a host whose allocator owns all device memory. Same arguments and
 * results as si_moe_router_topk, minus the workspace. It allocates nothing:
 * its scratch is a fixed array compiled into the library (133,376 bytes on
 * every GPU that loads it, held until the process exits).
 *   - Limit: n_tokens * n_experts <= 16384 (e.g. 64 tokens of 256 experts,
 *     2048 tokens of 8); every such shape fits the array. Larger calls return
 *     SI_ERR_UNSUPPORTED and enqueue nothing.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - All calls share the one array: calls that may overlap on the GPU (two
 *     streams, two threads) race and must be serialised by the caller. Each
 *     call clears the completion counters before its kernel (an asynchronous
 *     memset on `stream`).
 *   - Device-side errors of these calls (a completion count that does not add
 *     up, e.g. from two calls that overlapped: ids -1 and weights 0) are kept
 *     in the array's status word, the first one only, until
 *     si_moe_router_noalloc_status reads them.
 */
si_status si_moe_router_topk_noalloc(const void *x, si_dtype x_type, const void *w_router,
                                     si_dtype w_type, int hidden, int n_experts, int top_k,
                                     int n_tokens, int32_t *topk_ids, float *topk_w,
                                     float *logits_out, void *stream);

/* Synchronises `stream`, then reads the status word of the no-alloc router's
 * built-in scratch on the current device (SI_OK if no call recorded a
 * device-side error since the last read) and clears it. Like the router
 * call, it allocates nothing. */
si_status si_moe_router_noalloc_status(void *stream, int *status_out);

/* One MoE FFN layer: shapes, formats and device weight pointers. */
typedef struct si_moe_layer {
  int hidden;                 /* H, multiple of 256 (2048 in the studied models) */
  int n_experts;              /* E, 8..256 */
  int top_k;                  /* k, 1..8 */
  int inter;                  /* I, routed expert width, multiple of 256 */
  si_dtype expert_type;       /* SI_Q4_K or SI_BF16 (gate and up; down too unless down_type) */
  const void *w_gate;         /* [E][I] rows of H */
  const void *w_up;           /* [E][I] rows of H */
  const void *w_down;         /* [E][H] rows of I */
  int shared_inter;           /* I_s, multiple of 256, or 0 for no shared expert */
  si_dtype shared_type;       /* SI_Q8_0, SI_Q4_K or SI_BF16 (SI_BF16 iff expert_type is) */
  const void *ws_gate;        /* [I_s] rows of H */
  const void *ws_up;          /* [I_s] rows of H */
  const void *ws_down;        /* [H] rows of I_s */
  const void *w_shared_sigmoid; /* bf16 [H]: shared output is scaled by sigmoid(w . x) */
  /* used by si_moe_layer_decode and the stack only: */
  const void *w_router;       /* [E][H] of router_type */
  si_dtype router_type;       /* SI_BF16 or SI_F32 */
  const void *w_norm;         /* bf16 [H], RMSNorm weight */
  float eps;                  /* RMSNorm epsilon */
  /* Format of w_down when it differs from expert_type; 0 (SI_F32, never an
   * expert format) = expert_type. With Q4_K gate/up, SI_Q5_K is accepted: the
   * format the routed down ships in before the load-time requant ([Q] Summary,
   * bullet 2); such layers run as four kernels per layer. */
  si_dtype down_type;
} si_moe_layer;

/*
 * si_moe_ffn_decode - routed experts and shared expert for one token
 * ([S] item 1, [Q] Summary).
 *
 * For rank r = 0..k-1 with expert e = topk_ids[r]: g = G_e x, u = U_e x,
 * h = silu(g) * u (silu(z) = z / (1 + exp(-z))), y_r = D_e h;
 * routed = sum_r topk_w[r] * y_r (fp32, rank order) stored as bf16.
 * Shared: shared = sigmoid(w_shared_sigmoid . x) * D_s(silu(G_s x) * (U_s x)),
 * stored as bf16. With quantised weights the activations x and h enter the
 * GEMVs as Q8_1 blocks and every 32-block dot is an exact int32 sum of int8
 * products, scaled in fp32; with bf16 weights the GEMVs are fp32 dot products
 * of bf16 weights and fp32 activations.
 *   x          device bf16 [H]
 *   x_q8_1     device Q8_1 [H/32] blocks of x, or NULL (then quantised inside)
 *   topk_ids   device int32 [k]; topk_w device fp32 [k]
 *   routed_out device bf16 [H]; shared_out device bf16 [H] (ignored if no shared)
 *   n_tokens   must be 1 (several tokens: si_moe_ffn_batched)
 */
size_t si_moe_ffn_workspace_bytes(const si_moe_layer *L, int n_tokens);
si_status si_moe_ffn_decode(const si_moe_layer *L, int n_tokens, const void *x,
                            const void *x_q8_1, const int32_t *topk_ids, const float *topk_w,
                            void *routed_out, void *shared_out, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Expert-parallel partitions of si_moe_ffn_decode (the routed expert weights
 * read per token are what partitions: "Q4_K shared-expert FFN kernels +
 * Q8_0/Q5_K->Q4_K requant of the MoE FFN stage", Summary). A partition owns
 * the experts [e0, e1); every partition computes, for one token,
 *   slot_y[r][:] = y_r = D_e h_e (fp32 [H], the down GEMV of slot r's expert
 *                  e, as si_moe_ffn_decode forms it) if e lies in [e0, e1),
 *                  and 0 (all bits zero) otherwise,
 * and the shared expert in full (shared_out, replicated). Summing the
 * partitions' slot_y as 32-bit integers (each slot is non-zero in exactly one
 * partition) reproduces the single-partition values bit for bit, and
 * si_moe_combine_slots then forms routed exactly as si_moe_ffn_decode does.
 *   e0, e1     0 <= e0 <= e1 <= E; Q4_K routed experts only (SI_ERR_UNSUPPORTED otherwise)
 *   slot_y     device fp32 [k][H]; shared_out device bf16 [H] (if the layer has a shared expert)
 *   workspace  si_moe_ffn_workspace_bytes(L, 1) bytes
 * Experts outside [e0, e1) are neither read nor computed.
 *
 * si_moe_combine_slots: routed[j] = bf16(sum_r topk_w[r] * slot_y[r][j]),
 * the fp32 fma chain in rank order (k <= 8), on device buffers.
 */
si_status si_moe_ffn_decode_ep(const si_moe_layer *L, int e0, int e1, const void *x,
                               const void *x_q8_1, const int32_t *topk_ids, float *slot_y,
                               void *shared_out, void *workspace, size_t workspace_bytes,
                               void *stream);
si_status si_moe_combine_slots(const float *slot_y, const float *topk_w, int k, int hidden,
                               void *routed_out, void *stream);

/*
 * si_moe_ffn_batched - routed experts for n_tokens tokens with per-token
 * routing (not on the pages, which measure batch 1; the per-token arithmetic
 * is si_moe_ffn_decode's).
 *
 * The (token, rank) pairs are grouped by expert so that each selected
 * expert's rows are read once for all of its tokens; routed[t] =
 * sum_r topk_w[t][r] * y_{t,r} in rank order, stored as bf16.
 *   mode       SI_FFN_AUTO (0): SI_FFN_INT8, the faster mode at every supported
 *                               batch on GB300 (with 128 experts a batch of
 *                               64 tokens gives each selected expert ~4 tokens:
 *                               not dense enough to pay for dequantising the
 *                               weights for the tensor cores);
 *              SI_FFN_INT8 (1): Q8_1 activations, exact int32 block dots, as
 *                               si_moe_ffn_decode (n_tokens = 1 gives its bits);
 *              SI_FFN_TENSOR (2): tcgen05 tensor cores, fp16 operands: weights
 *                               dequantised (w = d*sc*q - dmin*m in fp32, then
 *                               fp16), x converted to fp16, h = silu(g)*u in
 *                               fp32 rounded to fp16; fp32 accumulation
 *   x          device bf16 [n_tokens][H]
 *   topk_ids   device int32 [n_tokens][k]; topk_w device fp32 [n_tokens][k]
 *   routed_out device bf16 [n_tokens][H]
 * Supported: Q4_K experts, no shared expert, 1 <= n_tokens, n_tokens * k <= 1024,
 * H <= 8192 (n_tokens = 0 returns SI_ERR_INVALID_ARG and enqueues nothing).
 */
enum { SI_FFN_AUTO = 0, SI_FFN_INT8 = 1, SI_FFN_TENSOR = 2 };
size_t si_moe_ffn_batched_workspace_bytes(const si_moe_layer *L, int n_tokens);
si_status si_moe_ffn_batched(const si_moe_layer *L, int n_tokens, int mode, const void *x,
                             const int32_t *topk_ids, const float *topk_w, void *routed_out,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * si_requant_q4_k - load-time requant of a weight matrix to Q4_K ([Q]
 * Summary bullets 1 and 2: the shared expert ships as Q8_0, the routed down
 * projection as Q5_K; both are requantised to Q4_K once, at model load).
 * Each row's weights are dequantised to fp32 and quantised with the library's
 * Q4_K quantiser, every step one IEEE fp32 operation: per 32-wide sub-block
 * lo = min w (if negative, else +0), hi = max w (if positive, else +0),
 * s = (hi - lo)/15, m' = -lo; d = fp16(max s / 63), dmin = fp16(max m' / 63);
 * sc = rint(s/d), m = rint(m'/dmin) in [0, 63]; q = rint((w + dmin*m)/(d*sc))
 * in [0, 15]; 0 wherever a divisor is 0; GGUF K-quant bytes.
 *   src       device, rows x si_row_bytes(src_type, cols) bytes, rows contiguous
 *   src_type  SI_Q8_0 or SI_Q5_K (176 bytes per 256 weights: fp16 d, fp16 dmin,
 *             12 scale bytes as Q4_K, 32 bytes of fifth bits, 128 code bytes)
 *   rows      >= 0; 0 returns SI_OK and enqueues nothing
 *   cols      weights per row, a multiple of 256
 *   dst       device, rows x (cols / 256 * 144) bytes
 * Not in place (src and dst must not overlap). Enqueues one kernel.
 */
si_status si_requant_q4_k(const void *src, si_dtype src_type, int64_t rows, int64_t cols,
                          void *dst, void *stream);

/*
 * si_add_rmsnorm3 - residual fold into the post-MoE RMSNorm ([R] item 2).
 *
 * Per row: t = bf16(a + b); sum = bf16(t + c) (c == NULL: sum = t);
 * y = bf16(sum * rsqrt(mean(sum^2) + eps) * w_norm), fp32 arithmetic.
 * Bit-identical to a separate residual add followed by the 2-input norm.
 *   a, b, c       device bf16 [n_rows][n]
 *   w_norm        device bf16 [n]
 *   n             multiple of 256, <= 16384; n_rows >= 1
 *   sum_out       device bf16 [n_rows][n] (the new residual stream)
 *   norm_out      device bf16 [n_rows][n]
 *   norm_q8_1_out device Q8_1 [n_rows][n/32] blocks of norm_out, or NULL
 * Outputs may not alias inputs.
 */
si_status si_add_rmsnorm3(const void *a, const void *b, const void *c, const void *w_norm,
                          int n, int n_rows, float eps, void *sum_out, void *norm_out,
                          void *norm_q8_1_out, void *stream);

/*
 * si_moe_layer_decode - one whole layer for one token: router + top-k,
 * routed and shared experts, residual fold (the calls above, enqueued back to
 * back with programmatic dependent launch).
 *   x          device bf16 [H]: FFN input (the previous norm's output)
 *   residual   device bf16 [H]: residual stream (may equal x)
 *   sum_out    device bf16 [H]: new residual; norm_out device bf16 [H]
 *   topk_ids, topk_w, routed_out, shared_out: optional device outputs (NULL to skip)
 */
size_t si_moe_layer_workspace_bytes(const si_moe_layer *L);
si_status si_moe_layer_decode(const si_moe_layer *L, const void *x, const void *residual,
                              void *sum_out, void *norm_out, int32_t *topk_ids,
                              float *topk_w, void *routed_out, void *shared_out,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Layer stack captured as one CUDA graph: n_tokens tokens, each through
 * n_layers layers in order; layer l takes (norm_out, sum_out) of layer l-1 as
 * (x, residual); layer 0 takes (x_in[t], x_in[t]). Tokens run one after the
 * other.
 *   n_layers, n_tokens  >= 1 (0 returns SI_ERR_INVALID_ARG)
 *   x_in     device bf16 [n_tokens][H]; y_out device bf16 [n_tokens][H] (last norm)
 *   sum_out  device bf16 [n_tokens][H] (last residual) or NULL
 *   ids_out  device int32 [n_tokens][n_layers][k] or NULL
 *   workspace si_moe_stack_workspace_bytes(layers, n_layers) bytes, zeroed once
 * The graph captures the pointers: buffers must outlive it. `stream` is used
 * for capture only (it must not be capturing already); launch on any stream.
 */
typedef struct si_graph si_graph;
size_t si_moe_stack_workspace_bytes(const si_moe_layer *layers, int n_layers);
si_status si_moe_stack_graph_create(const si_moe_layer *layers, int n_layers, int n_tokens,
                                    const void *x_in, void *y_out, void *sum_out,
                                    int32_t *ids_out, void *workspace, size_t workspace_bytes,
                                    void *stream, si_graph **graph_out);
/*
 * The same with the execution path chosen by the caller:
 *   SI_STACK_AUTO        as si_moe_stack_graph_create: the persistent kernel
 *                        whenever it supports the layers, else per layer;
 *   SI_STACK_PER_LAYER   four kernels per layer and token (router + top-k,
 *                        gate/up, down, add + RMSNorm), chained with
 *                        programmatic dependent launch;
 *   SI_STACK_PERSISTENT  one cooperative kernel, one block per SM, for the
 *                        whole stack ("perf(qwen3.6): fuse decode kernel
 *                        launches", Summary: decode is launch bound); returns
 *                        SI_ERR_UNSUPPORTED unless every layer has a bf16
 *                        router and either Q4_K routed experts (gate and up;
 *                        down Q4_K or Q5_K) with a Q4_K, Q8_0 or no shared
 *                        expert, or bf16
 *                        routed experts with a bf16 or no shared expert (one
 *                        format for all layers); all layers share one shape
 *                        with H a multiple of 2048 (<= 4096), E even (<= 256),
 *                        top_k <= 8, n_layers <= 128; one block per SM covers
 *                        every gate/up unit of 32 rows; and the block's shared
 *                        memory fits (bf16 down rows: J x top_k x inter x 2 B).
 *                        Its workspace also carries the epoch of its exchange
 *                        tags, which advances with every replay.
 * Both paths give bit-identical results. si_graph_is_persistent returns 1 for
 * a graph holding the persistent kernel, 0 for the per-layer path, -1 for NULL.
 */
enum { SI_STACK_AUTO = 0, SI_STACK_PER_LAYER = 1, SI_STACK_PERSISTENT = 2 };
si_status si_moe_stack_graph_create_mode(const si_moe_layer *layers, int n_layers, int n_tokens,
                                         const void *x_in, void *y_out, void *sum_out,
                                         int32_t *ids_out, void *workspace,
                                         size_t workspace_bytes, int mode, void *stream,
                                         si_graph **graph_out);
int si_graph_is_persistent(const si_graph *graph);
si_status si_graph_launch(si_graph *graph, void *stream);
void si_graph_destroy(si_graph *graph);

/*
 * si_moe_layer_decode_batched - one whole layer for n_tokens tokens, each
 * routed on its own (not on the pages, which measure batch 1; the per-token
 * arithmetic is si_moe_layer_decode's): router + top-k of every token, the
 * routed experts grouped by expert (si_moe_ffn_batched, `mode` as there), and
 * sum = bf16(routed + residual), norm = RMSNorm(sum) of every row.
 *   x          device bf16 [T][H]: FFN input; residual device bf16 [T][H] (may equal x)
 *   sum_out, norm_out device bf16 [T][H]
 *   topk_ids, topk_w, routed_out: optional device outputs int32 [T][k],
 *              fp32 [T][k], bf16 [T][H] (NULL to skip)
 *   workspace  si_moe_layer_batched_workspace_bytes(L, T) bytes, zeroed once
 * Supported: the layers si_moe_ffn_batched takes (Q4_K experts, no shared
 * expert) with a bf16 or fp32 router. In SI_FFN_INT8 / SI_FFN_AUTO mode
 * every token's results equal si_moe_layer_decode's on that token alone.
 */
size_t si_moe_layer_batched_workspace_bytes(const si_moe_layer *L, int n_tokens);
si_status si_moe_layer_decode_batched(const si_moe_layer *L, int n_tokens, int mode, const void *x,
                                      const void *residual, void *sum_out, void *norm_out,
                                      int32_t *topk_ids, float *topk_w, void *routed_out,
                                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Batched layer stack captured as one CUDA graph: n_tokens tokens go through
 * n_layers layers together (si_moe_layer_decode_batched per layer); layer l
 * takes (norm_out, sum_out) of layer l-1 as (x, residual), layer 0 takes
 * (x_in, x_in).
 *   x_in  device bf16 [T][H]; y_out device bf16 [T][H] (last norm);
 *   sum_out device bf16 [T][H] (last residual) or NULL;
 *   ids_out device int32 [n_layers][T][k] or NULL
 *   workspace si_moe_stack_batched_workspace_bytes(layers, n_layers, T) bytes, zeroed once
 * The graph captures the pointers; `stream` is used for capture only.
 * With one token and mode SI_FFN_AUTO the graph holds the persistent stack
 * kernel when it takes the layers (si_graph_is_persistent returns 1): the
 * same bits, one launch for the whole stack.
 */
size_t si_moe_stack_batched_workspace_bytes(const si_moe_layer *layers, int n_layers, int n_tokens);
si_status si_moe_stack_graph_create_batched(const si_moe_layer *layers, int n_layers, int n_tokens,
                                            int mode, const void *x_in, void *y_out, void *sum_out,
                                            int32_t *ids_out, void *workspace, size_t workspace_bytes,
                                            void *stream, si_graph **graph_out);

/* Synchronises `stream`, then reads the device status word of a workspace
 * used by any call above (SI_OK if no device-side error was recorded) and
 * clears it. */
si_status si_workspace_status(const void *workspace, void *stream, int *status_out);

/* ---- test-only exports (not on the hot path) ---------------------------- */

/* Exact int32 sum_i q_w,i * q_a,i for every (row, 32-block) of a Q4_K matrix
 * [rows][k] against Q8_1 activations [k/32]; out int32 [rows][k/32]. */
si_status si_test_q4k_block_dots(const void *w, int rows, int k, const void *a_q8_1,
                                 int32_t *out, void *stream);

/* Exact int32 sums sum_i q_w,i * q_a,i of every (vector, row, 32-block), taken
 * by the integer helper that each GEMV of the library uses ("Q4_K
 * shared-expert FFN kernels + Q8_0/Q5_K->Q4_K requant of the MoE FFN stage",
 * Summary: int8 dot products of Q8_1 activations with the weight codes):
 *   SI_TEST_DOTS_Q4K_SB          whole Q4_K super-blocks (gate/up GEMVs)
 *   SI_TEST_DOTS_Q4K_HALF        Q4_K halves of 128 weights (down GEMVs, and
 *                                the persistent stack's down step)
 *   SI_TEST_DOTS_Q5K_HALF        Q5_K halves (the Q5_K routed down)
 *   SI_TEST_DOTS_Q4K_SB_TOKENS   whole super-blocks, code words loaded once for
 *                                every vector (batched gate/up), n_vec <= 8
 *   SI_TEST_DOTS_Q4K_HALF_TOKENS halves, the same (batched down), n_vec <= 8
 *   w      device, rows x (k/256) super-blocks (144 bytes Q4_K, 176 Q5_K)
 *   k      multiple of 256, <= 16384; rows 1..65535
 *   a_q8_1 device, n_vec vectors of k/32 Q8_1 blocks (36 bytes), back to back
 *   out    device int32 [n_vec][rows][k/32] */
enum {
  SI_TEST_DOTS_Q4K_SB = 0,
  SI_TEST_DOTS_Q4K_HALF = 1,
  SI_TEST_DOTS_Q5K_HALF = 2,
  SI_TEST_DOTS_Q4K_SB_TOKENS = 3,
  SI_TEST_DOTS_Q4K_HALF_TOKENS = 4
};
si_status si_test_block_dots(int kind, const void *w, int rows, int k, const void *a_q8_1,
                             int n_vec, int32_t *out, void *stream);

/* Only the gate/up kernel of si_moe_ffn_decode (same arguments; h is left in
 * the workspace). For timing that kernel in isolation. */
si_status si_moe_ffn_gateup(const si_moe_layer *L, int n_tokens, const void *x,
                            const void *x_q8_1, const int32_t *topk_ids, void *workspace,
                            size_t workspace_bytes, void *stream);

/* A kernel whose mbarrier wait can never complete: it gives up after
 * budget_ns (<= 2 s) and writes SI_ERR_TIMEOUT to the workspace status word,
 * as every bounded wait of the library does. For testing that path. */
si_status si_test_wait_timeout(uint64_t budget_ns, void *workspace, void *stream);

/* The tagged-slot poll of the persistent stack kernel on a slot that never
 * receives the awaited tag: it gives up after budget_ns (<= 2 s) and writes
 * SI_ERR_TIMEOUT to the status word. workspace: 512 bytes, zero-filled (the
 * slot is the 16 bytes after the 256-byte status header). */
si_status si_test_poll_timeout(uint64_t budget_ns, void *workspace, void *stream);

/* D = A * B^T for one 128 x n x k block on the tensor cores (A fp16 [128][k],
 * B fp16 [n][k] row-major; n in {16..64} step 16, k in {16..256} step 16;
 * D fp32 [128][n]); workspace: 256 bytes, status word. */
si_status si_test_umma_f16(const void *a, const void *b, int n, int k, float *out,
                           void *workspace, void *stream);

/* The unfused chain the fold replaced: t = bf16(a + b) by one kernel, then the
 * 2-input norm of (t, c) by a second. Same outputs as si_add_rmsnorm3. */
si_status si_test_unfused_add_rmsnorm(const void *a, const void *b, const void *c,
                                      const void *w_norm, int n, int n_rows, float eps,
                                      void *t_scratch, void *sum_out, void *norm_out,
                                      void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SI_MOE_H */
