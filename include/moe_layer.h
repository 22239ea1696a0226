/*
 * moe_layer.h -- C ABI of a single-GPU Mixture-of-Experts FFN layer forward
 * pass over a prefill token batch, for NVIDIA GB300 (sm_103a).
 *
 * The layer (gated routing + expert computation, "Memory-Compute
 * Disaggregation for Large-Model Inference: AFD Architecture Analysis and
 * Performance Validation", section 3, Data-Flow Closed Loop step 3):
 *   1. router logits l = x W_r^T (+ bias), top-k experts per token, gate weights
 *   2. per-expert token histogram and a permutation grouping rows by expert
 *   3. grouped GEMM over each expert's W_gate / W_up with fused SwiGLU
 *   4. grouped down projection W_down, each row scaled by its gate weight
 *   5. combine back to token order (plus the always-on shared expert)
 * The grouped GEMMs take hidden states as the left operand and the layer's
 * expert weights as the right operand ("ASAP: A DiSaggregated and
 * Asynchronous Inference System for MoE Prefill", section 3.4.2), and read
 * every expert's weights from its own allocation through a per-expert
 * pointer list, with no merge copy ("DWDP: Distributed Weight Data
 * Parallelism for High-Performance LLM Inference on NVL72", section 4.2).
 *
 * Conventions for every call
 *   - Pointers named x, w_*, out, ... are DEVICE pointers into memory the
 *     caller owns (the library never frees them).  Arrays "of device
 *     pointers" are HOST arrays.  All matrices are row-major and dense.
 *   - bf16 matrices and every buffer read by TMA must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream): they enqueue kernels and return.  None synchronises
 *     or copies device->host, except moe_get_device_error and
 *     moe_weights_create / moe_weights_destroy.
 *   - Arguments are validated on the host BEFORE anything is enqueued; a
 *     failed check returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *     MOE_ERR_WORKSPACE with nothing launched, and moe_last_error_message()
 *     describes it.  No C++ exception crosses this boundary.
 *   - Device-side checks (an expert id outside [0,E), a row index outside
 *     [0,T*k), a bounded wait that expired) never trap: they set bits of a
 *     sticky status word at the start of the caller's workspace, skip the
 *     offending access and let the kernel finish.  moe_get_device_error()
 *     reads and clears that word.
 *   - Workspace: caller-allocated device memory of at least
 *     moe_workspace_size() bytes, 256-byte aligned, initialised once with
 *     moe_workspace_init().  Calls on one workspace must not overlap in time
 *     (use one stream per workspace).
 *   - The current CUDA device must be the one holding every pointer.
 */
#ifndef MOE_LAYER_H_
#define MOE_LAYER_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 2

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null / misaligned pointer, bad size or enum */
  MOE_ERR_UNSUPPORTED = 2,    /* valid but outside what the kernels handle */
  MOE_ERR_WORKSPACE = 3,      /* workspace too small or misaligned */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE_TIMEOUT = 5, /* a kernel's bounded wait expired */
  MOE_ERR_BOUNDS = 6          /* a kernel met an out-of-range index */
} moe_status_t;

typedef enum moe_score {
  MOE_SCORE_SOFTMAX = 0,      /* w = softmax over the selected logits (renormalize=1) */
  MOE_SCORE_SIGMOID = 1       /* w = sigmoid(l) / sum over the selection (renormalize=1) */
} moe_score_t;

typedef enum moe_dtype {
  MOE_DTYPE_BF16 = 0,         /* bf16 weights, bf16 x_perm / h, fp32 accumulation */
  MOE_DTYPE_FP8_E4M3 = 1,     /* e4m3 weights with 128x128 fp32 block scales;
                                 e4m3 activations with 1x128 fp32 group scales */
  MOE_DTYPE_NVFP4 = 2         /* NVFP4 weights and activations: E2M1 values, one
                                 e4m3 scale per 16 elements along K, an fp32 tensor
                                 scale per matrix (weights) or per layer (static
                                 activation scales); block-scaled fp4 tensor cores.
                                 Runs through moe_forward / moe_forward_stack only. */
} moe_dtype_t;

typedef enum moe_op {
  MOE_OP_ROUTE = 0,
  MOE_OP_PERMUTE = 1,
  MOE_OP_GROUPED_FFN = 2,
  MOE_OP_COMBINE = 3,
  MOE_OP_FORWARD = 4
} moe_op_t;

/* Layer shape and routing rule.
 *   T          tokens (>= 0; 0 makes every call a no-op); T*k < 2^31
 *   H          hidden size, multiple of 128 (of 256 for NVFP4), >= 128
 *   E          routed experts, 1..256
 *   k          experts per token, 1..min(E, 16)
 *   I          routed expert intermediate size, multiple of 128 (256 for NVFP4)
 *   I_shared   shared expert intermediate size, 0 (none) or multiple of 128
 *              (256 for NVFP4)
 *   score      moe_score_t
 *   renormalize 1: normalise the k selected weights to sum 1; 0: softmax over
 *              all E (softmax) or the raw sigmoid (sigmoid)
 *   route_scale multiplies every gate weight (e.g. 2.5), finite and > 0
 *   wtype      moe_dtype_t of the expert weights */
typedef struct moe_config {
  int64_t T;
  int32_t H;
  int32_t E;
  int32_t k;
  int32_t I;
  int32_t I_shared;
  int32_t score;
  int32_t renormalize;
  float route_scale;
  int32_t wtype;
} moe_config_t;

/* Per-expert weight pointer list (DWDP section 4.2: a list of separately
 * allocated weight buffers instead of one contiguous tensor).  Every pointer
 * is a device pointer, 16-byte aligned; the arrays themselves are host arrays
 * of length E.
 *   gate[e], up[e]  [I, H]      down[e] [H, I]        (bf16, or e4m3 bytes)
 *   *_scales[e]     fp8 only: fp32 block scales, gate/up [I/128, H/128],
 *                   down [H/128, I/128]; NULL arrays for bf16
 *   shared_*        the shared expert ([I_shared, H] / [H, I_shared]) and its
 *                   scales; NULL when I_shared == 0
 * NVFP4 (MOE_DTYPE_NVFP4), as written by moe_quantize_weight_nvfp4:
 *   gate[e]         the expert's stacked gate/up matrix, E2M1 codes [2I, H/2]
 *                   bytes (two values per byte, the even element in the low
 *                   nibble), rows interleaved in 128-row blocks [gate 128 | up 128];
 *                   up[] and the *_scales arrays are unused (may be NULL)
 *   down[e]         E2M1 codes [H, I/2]
 *   gate_sf[e], down_sf[e]   their e4m3 block scales in the MMA scale layout
 *                   (see moe_quantize_weight_nvfp4), 16-byte aligned
 *   gate_tscale[e], down_tscale[e]   device pointers to the fp32 tensor scales
 *   shared_gate / shared_down / shared_gate_sf / shared_down_sf /
 *   shared_gate_tscale / shared_down_tscale   the shared expert's, alike
 *   input_scale     static fp32 tensor scale g_x of the expert inputs, > 0
 *   hidden_scale    static fp32 tensor scale g_h of the intermediate h, > 0
 *   (NVFP4 checkpoints carry such static activation scales; every activation
 *   block scale is computed at run time from them.) */
typedef struct moe_weight_list {
  const void* const* gate;
  const void* const* up;
  const void* const* down;
  const float* const* gate_scales;
  const float* const* up_scales;
  const float* const* down_scales;
  const void* shared_gate;
  const void* shared_up;
  const void* shared_down;
  const float* shared_gate_scales;
  const float* shared_up_scales;
  const float* shared_down_scales;
  const void* const* gate_sf;
  const void* const* down_sf;
  const float* const* gate_tscale;
  const float* const* down_tscale;
  const void* shared_gate_sf;
  const void* shared_down_sf;
  const float* shared_gate_tscale;
  const float* shared_down_tscale;
  float input_scale;
  float hidden_scale;
} moe_weight_list_t;

typedef struct moe_weights* moe_weights_t;

/* Builds the device-side expert table: one TMA tensor descriptor per expert
 * matrix plus pointer arrays, in one small device allocation owned by the
 * returned handle.  The weights themselves are neither copied nor owned and
 * must stay valid while the handle is used.  Synchronous (one host->device
 * copy).  Errors: MOE_ERR_INVALID_ARG (null/misaligned pointer, bad config),
 * MOE_ERR_CUDA. */
MOE_API moe_status_t moe_weights_create(const moe_config_t* cfg, const moe_weight_list_t* weights,
                                moe_weights_t* out);
/* Frees the handle's device table (synchronises the device first).  NULL is a no-op. */
MOE_API void moe_weights_destroy(moe_weights_t weights);

/* Bytes of workspace that `op` needs for `cfg` (always a multiple of 256). */
MOE_API moe_status_t moe_workspace_size(const moe_config_t* cfg, int32_t op, size_t* bytes);

/* Zeroes the workspace's status header (asynchronous).  Call once after allocating. */
MOE_API moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 1 -- routing (AFD write-up section 3, "gated routing"; ASAP section
 * 5.1, 8 of 256 experts per token).
 *   x          bf16 [T, H]
 *   w_router   bf16 [E, H]
 *   logit_bias fp32 [E] added to every token's logits, or NULL
 *   topk_ids   int32 [T, k] out: selected experts in descending logit order,
 *              exact ties to the lower index
 *   topk_w     fp32 [T, k] out: gate weights (see moe_config_t)
 *   logits_out fp32 [T, E] out, or NULL: the fp32 logits used for selection
 * Logits accumulate in fp32 on the tensor cores. */
MOE_API moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* logit_bias, int32_t* topk_ids, float* topk_w,
                       float* logits_out, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Step 2 -- histogram and permutation (ASAP table 2: per-expert token counts
 * of the dispatch metadata).  Deterministic: rows of expert e are
 * [expert_offsets[e], expert_offsets[e+1]) in ascending token order.
 *   topk_ids        int32 [T, k] in (each row k distinct ids in [0, E); an id
 *                   outside [0, E) sets status bit 0 and a repeated id within
 *                   a row sets bit 3, and the outputs are then incomplete)
 *   topk_w          fp32 [T, k] in, or NULL
 *   x               bf16 [T, H] in, or NULL when x_perm is NULL
 *   expert_counts   int32 [E] out
 *   expert_offsets  int32 [E+1] out, exclusive prefix sum, [E] = T*k
 *   perm_token      int32 [T*k] out: row -> token
 *   inv_row         int32 [T, k] out: (token, slot) -> row
 *   row_weight      fp32 [T*k] out, or NULL: topk_w in row order (needs topk_w)
 *   x_perm          [T*k, H] out, or NULL: x[perm_token[r]]; bf16, or e4m3 codes
 *                   for MOE_DTYPE_FP8_E4M3 (each token quantised once in 1x128
 *                   groups: s = amax/448, q = rn_satfinite(x/s), in fp32)
 *   x_perm_scales   fp32 [T*k, H/128] out for fp8, else NULL */
MOE_API moe_status_t moe_permute(const moe_config_t* cfg, const int32_t* topk_ids, const float* topk_w,
                         const void* x, int32_t* expert_counts, int32_t* expert_offsets,
                         int32_t* perm_token, int32_t* inv_row, float* row_weight,
                         void* x_perm, float* x_perm_scales, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* moe_permute without a workspace: the same histogram and permutation, with
 * the same outputs, for callers that cannot allocate device memory -- code
 * recording a CUDA graph, runtimes whose memory is planned once at start-up,
 * plugins that are handed only their input and output tensors.  The pages
 * have no counterpart of this call; it is a property of this library.
 * Scratch: a fixed device array inside the library (about 2 MB, held by every
 * GPU that loads the library until exit), enough for E * ceil(T/64) <= 262144
 * (e.g. T <= 65536 at E = 256); larger layers get MOE_ERR_UNSUPPORTED and must
 * use moe_permute.  Every call made outside a stream capture looks up the
 * array's device address in the current CUDA context (cudaGetSymbolAddress, a
 * cheap lookup); a call made while its stream is being captured reuses the
 * address of the last such lookup in the same context, so make one call in
 * each context before any capture starts (a first call during capture returns
 * MOE_ERR_INVALID_ARG).  Calls allocate nothing.  All calls share the array: calls that run
 * concurrently on the GPU race and must be ordered (one stream, or events).
 *   device_status  optional device word (4-byte aligned) that receives the
 *                  status bits (as moe_get_device_error reports them); NULL
 *                  discards them.
 * Every other argument is as for moe_permute. */
MOE_API moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const int32_t* topk_ids,
                                         const float* topk_w, const void* x,
                                         int32_t* expert_counts, int32_t* expert_offsets,
                                         int32_t* perm_token, int32_t* inv_row, float* row_weight,
                                         void* x_perm, float* x_perm_scales,
                                         uint32_t* device_status, moe_stream_t stream);

/* Steps 3+4 -- grouped expert FFN (ASAP section 3.4.2 grouped matrix
 * multiplication; DWDP section 4.2 pointer-list weights):
 *   y_perm[r] = row_weight[r] * W_down[e] (silu(W_gate[e] x_perm[r]) * (W_up[e] x_perm[r]))
 * for r in expert e's segment, and, when x_shared != NULL and I_shared > 0,
 *   shared_out[t] = W_sd (silu(W_sg x_shared[t]) * (W_su x_shared[t])).
 *   x_perm          [T*k, H] bf16 (or e4m3 + x_perm_scales [T*k, H/128])
 *   expert_offsets  int32 [E+1] (device), as written by moe_permute
 *   row_weight      fp32 [T*k] or NULL (all ones)
 *   x_shared        [T, H] bf16 (or e4m3 + x_shared_scales [T, H/128]) or NULL
 *   y_perm          fp32 [T*k, H] out;  shared_out fp32 [T, H] out or NULL
 * The intermediate h is rounded to bf16 (e4m3 + 1x128 scales for fp8); the
 * expert outputs stay fp32 so that each token's rows are rounded only once,
 * after the combine has summed them. */
MOE_API moe_status_t moe_grouped_ffn(const moe_config_t* cfg, moe_weights_t weights, const void* x_perm,
                             const float* x_perm_scales, const int32_t* expert_offsets,
                             const float* row_weight, const void* x_shared,
                             const float* x_shared_scales, void* y_perm, void* shared_out,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* NVFP4 layers (MOE_DTYPE_NVFP4, the DeepSeek-R1 NVFP4 expert weights of
 * "DWDP: Distributed Weight Data Parallelism for High-Performance LLM
 * Inference on NVL72", section A4) run the two middle steps through the next
 * two calls: their permuted rows are NVFP4 codes in expert segments padded to
 * whole 128-row blocks.  moe_route and moe_combine are the same calls as for
 * bf16 layers, and the four calls give the bits of moe_forward.
 *
 * Row counts of the NVFP4 step buffers: *padded_rows (T*k + 127*E, rounded up
 * to 128: room for every expert's padded segment) and *padded_tokens (T
 * rounded up to 128: the token-order copy for the shared expert).  Either
 * pointer may be NULL. */
MOE_API moe_status_t moe_nvfp4_rows(const moe_config_t* cfg, int64_t* padded_rows,
                                    int64_t* padded_tokens);

/* Step 2 for NVFP4 layers -- histogram and permutation as moe_permute, with
 * every token quantised once with the layer's static input scale g_x (held by
 * `weights`) and its codes written to its k rows.
 *   weights         the layer's NVFP4 weights (moe_weights_create)
 *   expert_counts, expert_offsets, perm_token, inv_row, row_weight: as
 *                   moe_permute (unpadded row order)
 *   pad_offsets     int32 [E+1] out: expert e's rows are x_perm rows
 *                   [pad_offsets[e], pad_offsets[e] + counts[e]); the segment
 *                   ends at pad_offsets[e+1], a multiple of 128
 *   x_perm          uint8 [padded_rows, H/2] out: E2M1 codes, two per byte
 *                   (element 2i in the low nibble of byte i); 16-byte aligned
 *   x_perm_sf       uint8 [padded_rows * H/16] out: the e4m3 block scales in
 *                   the MMA scale layout (512-byte atoms of 128 rows x 4
 *                   16-element blocks); padding rows get scale 0
 *   x_tok, x_tok_sf the same for the tokens in token order ([padded_tokens,
 *                   H/2] and [padded_tokens * H/16]): the shared expert's
 *                   input; NULL skips it
 * Workspace: moe_workspace_size(cfg, MOE_OP_PERMUTE). */
MOE_API moe_status_t moe_permute_nvfp4(const moe_config_t* cfg, moe_weights_t weights,
                                       const int32_t* topk_ids, const float* topk_w,
                                       const void* x, int32_t* expert_counts,
                                       int32_t* expert_offsets, int32_t* pad_offsets,
                                       int32_t* perm_token, int32_t* inv_row, float* row_weight,
                                       uint8_t* x_perm, uint8_t* x_perm_sf, uint8_t* x_tok,
                                       uint8_t* x_tok_sf, void* ws, size_t ws_bytes,
                                       moe_stream_t stream);

/* Steps 3+4 for NVFP4 layers -- the grouped expert FFN on the outputs of
 * moe_permute_nvfp4: h = silu(x W_gate^T) * (x W_up^T) quantised to NVFP4 with
 * the layer's static g_h, then y = row_weight * (h W_down^T).
 *   y_perm      fp32 [T*k, H] out, unpadded row order (as moe_grouped_ffn)
 *   shared_out  fp32 [T, H] out, or NULL (skips the shared expert; needs
 *               x_tok / x_tok_sf otherwise)
 *   row_weight  fp32 [T*k] or NULL (all ones)
 * The expert rows are produced as fp16 with a power-of-two scale per 32
 * columns, as in moe_forward, and widened exactly to fp32.
 * Workspace: moe_workspace_size(cfg, MOE_OP_GROUPED_FFN). */
MOE_API moe_status_t moe_grouped_ffn_nvfp4(const moe_config_t* cfg, moe_weights_t weights,
                                           const uint8_t* x_perm, const uint8_t* x_perm_sf,
                                           const int32_t* expert_offsets,
                                           const int32_t* pad_offsets, const float* row_weight,
                                           const uint8_t* x_tok, const uint8_t* x_tok_sf,
                                           float* y_perm, float* shared_out, void* ws,
                                           size_t ws_bytes, moe_stream_t stream);

/* Step 5 -- combine: out[t] = sum_j y_perm[inv_row[t, j]] (+ shared_out[t]),
 * summed in fp32 in slot order j = 0..k-1, then the shared row, rounded to bf16.
 *   y_perm fp32 [T*k, H], inv_row int32 [T, k], shared_out fp32 [T, H] or NULL,
 *   out bf16 [T, H] (must not alias y_perm). */
MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const void* y_perm, const int32_t* inv_row,
                         const void* shared_out, void* out, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* Steps 1-5 in one call, all intermediates in the workspace.
 *   x bf16 [T, H], w_router bf16 [E, H], logit_bias fp32 [E] or NULL,
 *   out bf16 [T, H];  topk_ids_out int32 [T, k] / topk_w_out fp32 [T, k]
 *   optional copies of the routing decision (NULL to skip). */
MOE_API moe_status_t moe_forward(const moe_config_t* cfg, moe_weights_t weights, const void* x,
                         const void* w_router, const float* logit_bias, void* out,
                         int32_t* topk_ids_out, float* topk_w_out, void* ws, size_t ws_bytes,
                         moe_stream_t stream);

/* moe_forward with options.  flags:
 *   MOE_FORWARD_FUSED_DISPATCH  bf16 layers: the grouped gate/up GEMM reads each
 *     expert's rows straight from x by token index (TMA row gathers, four rows
 *     per copy) instead of from a permuted copy of x, so the permutation step
 *     writes only its index maps -- the fused dispatch + expert GEMM of "Memory-
 *     Compute Disaggregation for Large-Model Inference: AFD Architecture
 *     Analysis and Performance Validation", section 5 (operator fusion).  Same
 *     results; on GB300 the row gathers are slower than one permuted copy plus
 *     tile loads, so it is off by default.  Ignored for fp8 and NVFP4 layers.
 * Unknown flag bits give MOE_ERR_INVALID_ARG. */
#define MOE_FORWARD_FUSED_DISPATCH 0x1u
MOE_API moe_status_t moe_forward_ex(const moe_config_t* cfg, moe_weights_t weights, const void* x,
                                    const void* w_router, const float* logit_bias, void* out,
                                    int32_t* topk_ids_out, float* topk_w_out, uint32_t flags,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---- Layer stacks: one layer-oblivious descriptor table for L layers ----
 * The layer-oblivious MoE kernel of "ASAP: A DiSaggregated and Asynchronous
 * Inference System for MoE Prefill", section 3.4.2 (Bubble-Free Kernel
 * Dispatching): the kernels can reach the weights of every layer, the
 * per-layer addresses are precomputed in a device table, and the layer index
 * is a device-side argument read when the kernels run.  A launch sequence
 * recorded once (for instance a CUDA graph of moe_forward_stack) then serves
 * any layer: the caller writes the index into device memory and replays, with
 * no host work between layers.
 *
 * moe_stack_create
 *   cfg         shape shared by every layer (T is the batch of later calls)
 *   num_layers  L >= 1
 *   layers      host array [L] of weight lists (as for moe_weights_create)
 *   w_router    host array [L] of device pointers, bf16 [E, H] each
 *   logit_bias  host array [L] of device pointers (fp32 [E] each, entries may be
 *               NULL), or NULL for no bias in any layer
 *   out         receives the handle; the library allocates one device table
 *               (no weight copy).  The weights must outlive the handle.
 * Errors: as moe_weights_create, for any layer. */
typedef struct moe_stack* moe_stack_t;
MOE_API moe_status_t moe_stack_create(const moe_config_t* cfg, int32_t num_layers,
                                      const moe_weight_list_t* layers,
                                      const void* const* w_router,
                                      const float* const* logit_bias, moe_stack_t* out);
/* Frees the stack's device table (synchronises the device first).  NULL is a no-op. */
MOE_API void moe_stack_destroy(moe_stack_t stack);

/* moe_forward on layer *layer of the stack.  layer: device pointer to one
 * int32, read by the kernels when they run (not when this call returns), so it
 * may be written between the replays of a recorded graph.  An index outside
 * [0, L) sets MOE_ERR_BOUNDS in the status word and runs layer 0.  Other
 * arguments as moe_forward (workspace op MOE_OP_FORWARD).  No host
 * synchronisation, allocation or device->host copy: capturable in a CUDA graph. */
MOE_API moe_status_t moe_forward_stack(const moe_config_t* cfg, moe_stack_t stack,
                                       const int32_t* layer, const void* x, void* out,
                                       int32_t* topk_ids_out, float* topk_w_out, void* ws,
                                       size_t ws_bytes, moe_stream_t stream);

/* fp8 weight preparation: 128x128 block quantisation of an fp32 [N, K] matrix
 * (N, K multiples of 128): scales[N/128, K/128] = amax/448 (1 for an all-zero
 * block), q = e4m3 rn_satfinite(w/s), computed in fp32.  Asynchronous. */
MOE_API moe_status_t moe_quantize_weight_fp8(const float* w, int64_t N, int64_t K, uint8_t* q,
                                     float* scales, moe_stream_t stream);

/* fp8 activation quantisation of a bf16 [M, K] matrix (K multiple of 128) in
 * 1x128 groups: scales[M, K/128], codes q[M, K], same rule as above. */
MOE_API moe_status_t moe_quantize_act_fp8(const void* x, int64_t M, int64_t K, uint8_t* q, float* scales,
                                  moe_stream_t stream);

/* NVFP4 weight preparation (MoE weights in NVFP4: "DWDP: Distributed Weight
 * Data Parallelism for High-Performance LLM Inference on NVL72", section A4,
 * experimental setup).  w: bf16 [N, K]; w2: NULL, or a second bf16 [N, K]
 * matrix stacked with w (an expert's up projection next to its gate), in
 * which case the output has 2N rows interleaved in 128-row blocks
 * [w rows 128b..128b+127 | w2 rows 128b..128b+127].  Computed in fp32:
 *   g = amax / (6 * 448) over the whole (stacked) matrix (1 if all zero),
 *   per 16 consecutive elements of a row: s = e4m3_rn_satfinite(amax_b / (6 g)),
 *   q = E2M1 round-to-nearest-even, saturating at 6, of x / (s g)  (q = 0 if s g = 0).
 *   codes       [rows, K/2] bytes, element 2i in the low nibble of byte i
 *   sf          rows * K/16 bytes: the e4m3 codes of s in the MMA scale layout:
 *               512-byte atoms of 128 rows x 4 blocks; the scale of (row r,
 *               block b) is byte ((r/128) * (K/64) + b/4) * 512 + (r%32) * 16
 *               + ((r%128)/32) * 4 + b%4
 *   tensor_scale  device fp32, receives g
 * N a multiple of 128, K of 64.  Asynchronous; tensor_scale is
 * used as scratch until the call's last kernel has run. */
MOE_API moe_status_t moe_quantize_weight_nvfp4(const void* w, const void* w2, int64_t N, int64_t K,
                                               uint8_t* codes, uint8_t* sf, float* tensor_scale,
                                               moe_stream_t stream);

/* NVFP4 activation quantisation with a static tensor scale g (> 0) of a bf16
 * [M, K] matrix (K a multiple of 16), the same block rule: codes [M, K/2],
 * sf [M, K/16] e4m3 scale codes, row-major. */
MOE_API moe_status_t moe_quantize_act_nvfp4(const void* x, int64_t M, int64_t K, float g,
                                            uint8_t* codes, uint8_t* sf, moe_stream_t stream);

/* Waits for `stream`, reads the workspace's sticky device status word, clears
 * it and maps it to MOE_OK / MOE_ERR_BOUNDS / MOE_ERR_DEVICE_TIMEOUT.
 * *device_bits (optional) receives the raw word: bit 0 an index outside its
 * range, bit 1 a bounded wait that expired (MOE_ERR_DEVICE_TIMEOUT), bit 2 a
 * token with fewer than k selectable (non-NaN) logits, bit 3 a token whose k
 * expert ids are not distinct (bits 0, 2 and 3 give MOE_ERR_BOUNDS). */
MOE_API moe_status_t moe_get_device_error(void* ws, moe_stream_t stream, int32_t* device_bits);

/* Failure-path test hook (the pages have no counterpart).  Sets, for the
 * calling thread, how many of its next bf16 grouped GEMM1 launches (inside
 * moe_grouped_ffn, moe_forward or moe_forward_stack) stall on purpose: in such
 * a launch the MMA issuer of the first CTA pair waits, before its first tile,
 * on a barrier that nothing signals.  Like every wait in the kernels, that one
 * gives up after its limit (2 s): it sets the timeout bit of the workspace
 * status word and the pair abandons its remaining tiles, drains the loads it
 * issued, frees its tensor memory and exits; every other pair finishes.  The
 * call's outputs are then incomplete and moe_get_device_error returns
 * MOE_ERR_DEVICE_TIMEOUT; the next call on the same workspace runs normally.
 * For tests of failure detection and recovery only; 0 (the default) disables
 * it.  count < 0 gives MOE_ERR_INVALID_ARG. */
MOE_API moe_status_t moe_test_stall_gemm1(int32_t count);

/* Kernel tracing.  While a trace is set on the calling thread, every call
 * records one of the caller's CUDA events on its stream before each kernel it
 * launches (kernel_ids[i] = the moe_kernel_t that follows events[i]) and one
 * after the last (kernel_ids[i] = -1), so consecutive events bracket each
 * kernel.  A nonzero kernel_mask restricts the events to the kernels whose bit
 * (1 << moe_kernel_t) is set and drops the trailing one; e.g. the GEMM1 and
 * GEMM2 bits bracket GEMM1 alone.  Recording stops silently when `capacity`
 * is reached; `count` is advanced by the library.  The events must be created
 * by the caller (cudaEventCreate) on the current device.  NULL clears the
 * trace. */
typedef enum moe_kernel {
  MOE_K_ROUTER = 0,
  MOE_K_HIST = 1,
  MOE_K_SCAN = 2,
  MOE_K_SCATTER = 3,
  MOE_K_PLAN = 4,
  MOE_K_GEMM1 = 5,   /* grouped gate/up GEMM + SwiGLU */
  MOE_K_GEMM2 = 6,   /* grouped down GEMM x gate weight */
  MOE_K_COMBINE = 7,
  MOE_K_QUANT = 8,
  MOE_K_COUNT = 9
} moe_kernel_t;

typedef struct moe_trace {
  void** events;        /* cudaEvent_t[capacity] */
  int32_t* kernel_ids;  /* int32[capacity], written by the library */
  int32_t capacity;
  int32_t count;
  uint32_t kernel_mask; /* 0: every kernel; else only the kernels whose bit is set */
} moe_trace_t;

MOE_API moe_status_t moe_set_trace(moe_trace_t* trace);

MOE_API const char* moe_status_string(moe_status_t status);
/* Text of the last host-side failure on the calling thread ("" if none). */
MOE_API const char* moe_last_error_message(void);
MOE_API int32_t moe_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_LAYER_H_ */
