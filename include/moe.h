/*
 * moe.h - C ABI of libmoe.so: the sparse top-k Mixture-of-Experts FFN layer
 * forward on one GB300 (sm_103a).
 *
 * The layer, for each token row x (d_model values):
 *   r = x W_r^T (+ logit_bias)                  router scores, one per expert
 *   TopK = the k experts with the largest r + sel_bias
 *   g = softmax over the kept scores            (or: softmax over all N
 *                                                scores, kept ones renormalised)
 *   y = sum_{i in TopK} g_i E_i(x) + sum_{shared s} E_s(x)
 *   E(x) = W_down ( SiLU(W_gate x) * (W_up x) )  (SwiGLU expert, no biases)
 * Sources: "Mixture of experts and speculative decoding", sections
 * "Following one token through an MoE layer" and "Opening the hood: the MoE
 * layer precisely"; "Mixture of Experts and Guided Decoding", the sparse
 * top-k example; "MoE inference: the call centre with 256 specialists and 8
 * taking each call", section "The bare mechanism" (SwiGLU experts, shared
 * experts, bias-adjusted routing).
 *
 * Conventions for every entry point below:
 *  - Pointers marked [device] are device pointers owned by the caller. The
 *    library never allocates, frees or synchronises device memory except
 *    where a function says it synchronises (moe_stream_status,
 *    moe_profile_collect).
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and returns before it runs.
 *  - Row-major layouts. Weights follow the linear-layer convention [out][in]:
 *    w_router [N][d_model]; w_gate, w_up [N+n_shared][d_ff][d_model];
 *    w_down [N+n_shared][d_model][d_ff]; shared experts are stored after
 *    the N routed experts in the same arrays.
 *  - Element type of x, the weights, x_perm, y_perm and y is cfg->dtype
 *    (fp32, or bf16 stored as its 16-bit pattern). Router scores, gate
 *    weights, biases and statistics are always fp32; indices are int32.
 *  - Every device pointer must be 16-byte aligned, and a workspace 256-byte
 *    aligned; otherwise MOE_ERR_MISALIGNED and nothing is launched.
 *  - Host-side argument errors return a negative status and launch nothing.
 *    Errors found on the device while the work runs (an expert index out of
 *    range, a wait that timed out) are recorded in a status word at the
 *    start of the workspace and read back by moe_stream_status().
 *  - T = 0 is valid: nothing is launched except zeroing the outputs that
 *    are sums (counts, prob_sum).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

/* Status codes. */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)  /* NULL pointer, bad shape or bad enum      */
#define MOE_ERR_UNSUPPORTED (-2)  /* valid but not built: see moe_check_config */
#define MOE_ERR_MISALIGNED (-3)   /* a pointer is not 16-byte (ws: 256) aligned */
#define MOE_ERR_WORKSPACE (-4)    /* ws_bytes smaller than the *_workspace_size */
#define MOE_ERR_CUDA (-5)         /* a CUDA call failed; see moe_last_cuda_error */
#define MOE_ERR_TIMEOUT (-6)      /* a bounded device wait ran out              */
#define MOE_ERR_DEVICE_CHECK (-7) /* a device-side input check failed          */

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  /* g = softmax over the k kept scores ("Mixture of experts and speculative
   * decoding", step 3 and the layer equation). */
  MOE_GATE_TOPK_SOFTMAX = 0,
  /* g = softmax over all N scores, kept probabilities divided by their sum
   * (same page, step 3's alternative; "MoE inference ...", "The bare
   * mechanism"). Equal to the above up to rounding. */
  MOE_GATE_ALL_SOFTMAX_RENORM = 1
} moe_gate_mode;

typedef struct moe_config {
  int32_t T;         /* tokens in this call, >= 0                             */
  int32_t d_model;   /* >= 8, multiple of 8                                   */
  int32_t n_experts; /* N routed experts, 1..256                              */
  int32_t top_k;     /* k, 1..min(N, 8)                                       */
  int32_t n_shared;  /* shared (always-run) experts, 0..4; use d_ff too       */
  int32_t d_ff;      /* expert hidden width, >= 8, multiple of 8              */
  int32_t dtype;     /* moe_dtype                                             */
  int32_t gate_mode; /* moe_gate_mode                                         */
  int32_t capacity;  /* expert capacity C, >= 0; 0 = no cap. With C > 0 each
                      * routed expert runs at most the first C of its (token,
                      * slot) pairs in ascending token order; the others are
                      * dropped and add nothing to y, or rerouted (overflow)
                      * ("Mixture of experts and speculative decoding",
                      * "Keeping the experts busy": the extras are dropped or
                      * rerouted). Routing, counts and the balance statistics
                      * are those before the cap; shared experts are never
                      * capped.                                              */
  int32_t tiles;     /* moe_tiles: how the bf16 and E4M3 expert GEMMs cut
                      * their work. 0 (MOE_TILES_AUTO) lets the library
                      * choose; a named tiling changes only speed, never the
                      * rounding of a result. NVFP4 always runs 1-CTA tiles. */
  int32_t gather;    /* moe_gather: where moe_layer_forward gathers each
                      * expert's token rows (bf16). 0 (MOE_GATHER_AUTO) lets
                      * the library choose; the result is the same bits
                      * either way. */
  int32_t overflow;  /* moe_overflow: what the layers do with the pairs over
                      * an expert's capacity (only with capacity > 0) */
} moe_config;

/* The pairs over an expert's capacity (moe_config.overflow). "Mixture of
 * experts and speculative decoding", "Keeping the experts busy": the extras
 * are dropped or rerouted. */
typedef enum {
  /* dropped: they add nothing to y (the capacity cut of moe_config.capacity) */
  MOE_OVERFLOW_DROP = 0,
  /* rerouted in rounds to the token's next-best expert with room, as
   * moe_reroute computes; a pair that finds none is dropped */
  MOE_OVERFLOW_REROUTE = 1
} moe_overflow;

/* Where the layer's row gather runs (moe_config.gather). */
typedef enum {
  MOE_GATHER_AUTO = 0,
  /* a kernel of its own copies the routed token rows into x_perm, which the
   * gate/up GEMM reads ("batched kernels" in place of the per-expert loop of
   * "Mixture of experts and speculative decoding", "A toy MoE layer in
   * PyTorch") */
  MOE_GATHER_KERNEL = 1,
  /* the gate/up GEMM reads the token rows of x itself through the
   * permutation (no x_perm): only with weight-stationary CTA pairs
   * (MOE_TILES_WEIGHT_PAIR, bf16); otherwise the kernel above runs */
  MOE_GATHER_FUSED = 2
} moe_gather;

/* Tilings of the grouped expert GEMMs (moe_config.tiles). Every tiling
 * computes the same sums in the same order per output element. */
typedef enum {
  MOE_TILES_AUTO = 0,
  /* 128 token rows x 256 accumulator columns on one SM, or, for T <= 64,
   * weight rows x token columns on one SM; either may split K when there
   * are few tiles. */
  MOE_TILES_CTA = 1,
  /* 256 token rows x 256 columns on a pair of SMs (tcgen05 cta_group::2):
   * suits segments of many hundreds of rows, each ending in a partial
   * 256-row tile. */
  MOE_TILES_PAIR = 2,
  /* 256 weight rows (output features) x up to 256 token rows on a pair of
   * SMs: a segment's token tiles are cut to multiples of 16 rows, so
   * segments of a few hundred rows waste little. */
  MOE_TILES_WEIGHT_PAIR = 3
} moe_tiles;

/* Library version (major*10000 + minor*100 + patch). */
MOE_API int moe_version(void);

/* Text for a status code. Never NULL. */
MOE_API const char* moe_status_string(int status);

/* The cudaError_t of the most recent MOE_ERR_CUDA on the calling thread. */
MOE_API int moe_last_cuda_error(void);

/* Host-only validation of a configuration against the limits above; touches
 * no GPU. MOE_OK, MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED. */
MOE_API int moe_check_config(const moe_config* cfg);

/* Workspace bytes each entry point needs (0 if cfg is invalid). The
 * workspace is caller-owned device memory, 256-byte aligned; its contents
 * need not be initialised and are clobbered. */
MOE_API size_t moe_router_workspace_size(const moe_config* cfg);
MOE_API size_t moe_permute_workspace_size(const moe_config* cfg);
MOE_API size_t moe_grouped_workspace_size(const moe_config* cfg);
MOE_API size_t moe_workspace_size(const moe_config* cfg); /* moe_layer_forward */
MOE_API size_t moe_reroute_workspace_size(const moe_config* cfg);

/*
 * Router scores, top-k selection, gate weights and the per-expert
 * statistics of the balance loss, for T tokens.
 * ("Mixture of experts and speculative decoding", steps 1-3 and section
 * "Keeping the experts busy"; "MoE inference ...", "The bare mechanism".)
 *
 *  x          [device] [T][d_model] cfg->dtype. Ignored when logits_in is set.
 *  w_router   [device] [N][d_model] cfg->dtype. Ignored when logits_in is set.
 *  logit_bias [device] [N] fp32 or NULL: added to every token's scores
 *             (it moves selection, gate weights and P alike).
 *  sel_bias   [device] [N] fp32 or NULL: added only to the key the top-k is
 *             chosen on, key = fp32(r + sel_bias); never enters g or P.
 *  logits_in  [device] [T][N] fp32 or NULL: when set, these are the scores
 *             r verbatim (no GEMM; logit_bias must then be NULL).
 *  logits_out [device] [T][N] fp32 or NULL: receives r.
 *  topk_idx   [device] [T][k] int32 out: experts by descending key, equal
 *             keys ordered by lower index. A NaN key ranks below every
 *             number (as -inf), so the indices stay valid and distinct
 *             whatever the scores hold.
 *  topk_w     [device] [T][k] fp32 out: gate weights (cfg->gate_mode).
 *  counts     [device] [N] int32 out: tokens routed to each expert.
 *  prob_sum   [device] [N] fp32 out: sum over tokens of softmax(r) over all
 *             N experts (P_i = prob_sum_i / T). Summed in a fixed order, so
 *             repeated calls give identical bits.
 *  ws         [device] moe_router_workspace_size(cfg) bytes.
 */
MOE_API int moe_router_topk(const moe_config* cfg, const void* x, const void* w_router,
                    const float* logit_bias, const float* sel_bias,
                    const float* logits_in, float* logits_out,
                    int32_t* topk_idx, float* topk_w, int32_t* counts,
                    float* prob_sum, void* ws, size_t ws_bytes,
                    moe_stream_t stream);

/*
 * moe_router_topk for callers that cannot allocate: no workspace argument,
 * and the library allocates nothing. The pages have no counterpart; this
 * is an interface for callers whose device memory is all assigned in
 * advance (a runtime's memory planner, or a plugin slot that passes an
 * operator only its inputs and outputs), so they can neither call
 * cudaMalloc nor hand over the scratch moe_router_topk takes.
 * Arguments and results are those of moe_router_topk without ws/ws_bytes.
 * The scratch (a status word and per-block probability sums and counts) lives in
 * a fixed 1 MiB array of the library's own device memory on every GPU that
 * loads the library, held until the process exits:
 *  - a call needs 256 + 8 * B * N bytes of it, B = ceil(T / 64), or
 *    max(ceil(T / 64), min(T, 608)) when N <= 32 (for N = 8: T <= 1048320;
 *    N = 32: T <= 262080; N = 256: T <= 32704); a larger call returns
 *    MOE_ERR_WORKSPACE, launching nothing;
 *  - the first call made with a CUDA context current looks up the array's
 *    device address in that context; make that first call before any stream
 *    capture. The lookup is keyed on the context's process-unique id, so a
 *    context made after cudaDeviceReset, or a second context on the same
 *    device, gets its own lookup on its first call;
 *  - all calls share the array: calls whose work overlaps on the GPU race
 *    on it and give undefined results; order them on one stream;
 *  - errors found on the device while the router runs (a bounded wait of the
 *    tensor-core router, N > 32, that ran out: MOE_ERR_TIMEOUT) are recorded
 *    in the array's status word, which the call clears first; read it with
 *    moe_router_topk_noalloc_status after the call;
 *  - MOE_ERR_CUDA here leaves the CUDA error to cudaGetLastError.
 */
MOE_API int moe_router_topk_noalloc(const moe_config* cfg, const void* x,
                    const void* w_router, const float* logit_bias,
                    const float* sel_bias, const float* logits_in,
                    float* logits_out, int32_t* topk_idx, float* topk_w,
                    int32_t* counts, float* prob_sum, moe_stream_t stream);

/* Synchronises `stream`, then returns the device-side status that the last
 * moe_router_topk_noalloc call in the current context recorded in the
 * library's array (MOE_OK or MOE_ERR_TIMEOUT), or MOE_ERR_CUDA if a CUDA call
 * failed. Like the array, it is shared by every call: read it after the call
 * whose status is wanted and before the next one is enqueued. Allocates
 * nothing. */
MOE_API int moe_router_topk_noalloc_status(moe_stream_t stream);

/*
 * Groups the T*k (token, slot) pairs by expert and gathers their token rows.
 * Pair p = t*k + slot. Rows are expert-major; inside one expert, ascending
 * pair id (a token cannot pick an expert twice, so ascending token). This
 * is the batched form of the per-expert dispatch loop of the pages' toy
 * layers ("Mixture of experts and speculative decoding", "A toy MoE layer
 * in PyTorch"; "Mixture of Experts and Guided Decoding", sparse MoE code).
 * The result is unique, so it is bit-exact and deterministic.
 *
 *  x              [device] [T][d_model] cfg->dtype.
 *  topk_idx       [device] [T][k] int32, each in [0, N), or -1 for a pair
 *                 with no expert (one moe_reroute dropped): it gets no row
 *                 and inv_pos -1. Any other index out of range sets
 *                 MOE_ERR_DEVICE_CHECK in the workspace status; that pair is
 *                 then left out and the outputs are undefined.
 *  expert_offsets [device] [N+1] int32 out: exclusive prefix sum of the
 *                 per-expert rows, min(count, cfg->capacity) with a cap,
 *                 else count; expert_offsets[N] = rows kept (T*k uncapped).
 *  sorted_pair    [device] [T*k] int32 out: pair id stored at each row
 *                 (rows past expert_offsets[N] are left as they were).
 *  inv_pos        [device] [T*k] int32 out: row of each pair id, -1 for a
 *                 pair dropped by the capacity.
 *  x_perm         [device] [T*k][d_model] cfg->dtype out: x_perm[row] =
 *                 x[sorted_pair[row] / k], byte for byte, for the kept rows.
 *  ws             [device] moe_permute_workspace_size(cfg) bytes.
 */
MOE_API int moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                int32_t* expert_offsets, int32_t* sorted_pair,
                int32_t* inv_pos, void* x_perm, void* ws, size_t ws_bytes,
                moe_stream_t stream);

/*
 * Capacity overflow rerouted instead of dropped ("Mixture of experts and
 * speculative decoding", "Keeping the experts busy": the pairs over an
 * expert's capacity are dropped or rerouted; the page gives no order). With
 * C = cfg->capacity, pair p = t*k + slot:
 *  - round 0 is the capacity cut: each expert keeps the first C of its pairs
 *    in ascending pair order; the others are pending;
 *  - in each later round every pending pair, in slot order within its
 *    token, proposes the expert with the highest selection key
 *    fp32(logits + sel_bias) (equal keys: the lower index; NaN below every
 *    number) that has room left at the start of the round, that the token
 *    does not hold (its k routed experts and those it was rerouted to) and
 *    that no lower slot of the token proposed to in this round. A pair with
 *    no such expert is dropped. Each expert accepts the round's proposals
 *    in ascending pair id up to its room; the rest stay pending;
 *  - the rounds end when one has no proposal (at most N + 1 rounds).
 * The result is unique, so it is bit-exact and deterministic. A rerouted
 * pair keeps its slot's gate weight. capacity = 0 sets no cap
 * (assign = topk_idx).
 *
 *  logits   [device] [T][N] fp32: the router scores r (moe_router_topk's
 *           logits_out).
 *  sel_bias [device] [N] fp32 or NULL: as moe_router_topk.
 *  topk_idx [device] [T][k] int32: the router's choice. An index outside
 *           [0, N) sets MOE_ERR_DEVICE_CHECK and that pair is dropped.
 *  assign   [device] [T][k] int32 out: the expert each pair runs on, -1 for
 *           a dropped pair; moe_permute takes it in place of topk_idx.
 *  rounds   [device] int32 out, or NULL: the rounds after the cut.
 *  ws       [device] moe_reroute_workspace_size(cfg) bytes. Its status word
 *           records MOE_ERR_TIMEOUT if the kernel's bounded grid barrier
 *           ran out (outputs then undefined); read it with
 *           moe_stream_status.
 * One cooperative launch; its blocks wait on one another, so no other work
 * may hold the whole GPU while it runs.
 */
MOE_API int moe_reroute(const moe_config* cfg, const float* logits, const float* sel_bias,
                const int32_t* topk_idx, int32_t* assign, int32_t* rounds, void* ws,
                size_t ws_bytes, moe_stream_t stream);

/*
 * Every expert's SwiGLU FFN over its rows, for all experts in one pass:
 * routed expert e over x_perm rows [expert_offsets[e], expert_offsets[e+1]),
 * and each shared expert s over all T rows of x.
 *   y_perm[row] = w_row * W_down[e] ( SiLU(W_gate[e] a) * (W_up[e] a) )
 * where a is the row's input, w_row = topk_w[sorted_pair[row]] for routed
 * rows when topk_w is given, else 1. ("MoE inference ...", "The bare
 * mechanism": SwiGLU experts, shared experts; "Mixture of experts and
 * speculative decoding", layer equation.)
 * bf16: gate/up and down run on the tcgen05 tensor cores (bf16 operands,
 * fp32 accumulation), the SwiGLU hidden row is rounded to bf16 once.
 * fp32: CUDA-core fp32 throughout.
 *
 *  x_perm         [device] [T*k][d_model] cfg->dtype (from moe_permute).
 *  x              [device] [T][d_model] cfg->dtype: input of shared experts
 *                 (may be NULL when n_shared = 0).
 *  expert_offsets [device] [N+1] int32 (from moe_permute).
 *  sorted_pair    [device] [T*k] int32 (from moe_permute); may be NULL when
 *                 topk_w is NULL.
 *  topk_w         [device] [T][k] fp32 or NULL (then rows are unweighted).
 *  w_gate, w_up   [device] [N+n_shared][d_ff][d_model] cfg->dtype.
 *  w_down         [device] [N+n_shared][d_model][d_ff] cfg->dtype.
 *  y_perm         [device] [T*k + n_shared*T][d_model] cfg->dtype out:
 *                 routed rows first (x_perm order), then shared expert s at
 *                 rows T*k + s*T + t.
 *  ws             [device] moe_grouped_workspace_size(cfg) bytes (holds the
 *                 SwiGLU hidden rows).
 */
MOE_API int moe_grouped_swiglu(const moe_config* cfg, const void* x_perm,
                       const void* x, const int32_t* expert_offsets,
                       const int32_t* sorted_pair, const float* topk_w,
                       const void* w_gate, const void* w_up,
                       const void* w_down, void* y_perm, void* ws,
                       size_t ws_bytes, moe_stream_t stream);

/*
 * The gate-weighted sum back into token order, without atomics: each output
 * element is written once, summing in fp32 over slots 0..k-1 in order and
 * then the shared experts in order.
 *   y[t] = sum_slot w * y_perm[inv_pos[t*k+slot]] + sum_s y_perm[T*k+s*T+t]
 * with w = topk_w[t*k+slot] when topk_w is given, else 1 (rows already
 * weighted by moe_grouped_swiglu).
 * ("Mixture of experts and speculative decoding", step 4; "Mixture of
 * Experts and Guided Decoding", the three-expert gated sum.)
 *
 *  y_perm  [device] [T*k + n_shared*T][d_model] cfg->dtype.
 *  inv_pos [device] [T*k] int32 (from moe_permute). An entry outside
 *          [0, T*k) contributes zero.
 *  topk_w  [device] [T][k] fp32 or NULL.
 *  y       [device] [T][d_model] cfg->dtype out.
 */
MOE_API int moe_combine(const moe_config* cfg, const void* y_perm,
                const int32_t* inv_pos, const float* topk_w, void* y,
                moe_stream_t stream);

/*
 * The whole layer: moe_router_topk, moe_permute, moe_grouped_swiglu (rows
 * weighted by their gate) and moe_combine, enqueued back to back with no
 * host synchronisation.
 *
 *  x, w_router, logit_bias, sel_bias: as moe_router_topk.
 *  w_gate, w_up, w_down: as moe_grouped_swiglu.
 *  y        [device] [T][d_model] cfg->dtype out.
 *  topk_idx [device] [T][k] int32 out, or NULL.
 *  topk_w   [device] [T][k] fp32 out, or NULL.
 *  counts   [device] [N] int32 out, or NULL.
 *  prob_sum [device] [N] fp32 out, or NULL.
 *  ws       [device] moe_workspace_size(cfg) bytes.
 */
MOE_API int moe_layer_forward(const moe_config* cfg, const void* x,
                      const void* w_router, const float* logit_bias,
                      const float* sel_bias, const void* w_gate,
                      const void* w_up, const void* w_down, void* y,
                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                      float* prob_sum, void* ws, size_t ws_bytes,
                      moe_stream_t stream);

/*
 * FP8 experts. Deployed experts are stored, and tokens dispatched, in FP8
 * ("MoE inference: the call centre with 256 specialists and 8 taking each
 * call", "The maths that matters" and "DeepEP, EPLB and Wide-EP"). The
 * format is E4M3 (4 exponent bits, bias 7, 3 mantissa bits, largest finite
 * 448, no infinity) with one fp32 scale per row: s = fp32(amax / 448) and
 * codes q = E4M3(fp32(v * fp32(448 / amax))), rounded to nearest even and
 * saturated; a row of zeros has s = 0 and codes 0; a code stands for
 * decode(q) * s. The pages give no scaling rule; this is the library's.
 *
 * moe_quantize_fp8: rows x cols bf16 [device] -> q [rows][cols] uint8 and
 * scale [rows] fp32 [device]. cols a multiple of 8, pointers 16-byte
 * aligned. Quantize each weight tensor of moe_layer_forward_fp8 with it
 * (rows = output channels: E*d_ff for gate and up, E*d_model for down).
 */
MOE_API int moe_quantize_fp8(int64_t rows, int32_t cols, const void* src, uint8_t* q,
                    float* scale, moe_stream_t stream);

/*
 * moe_layer_forward with E4M3 experts: routing as moe_layer_forward (bf16 x
 * and W_r; cfg->dtype must be MOE_BF16), then every routed token row, x for
 * the shared experts, and each row of H are quantized as above, and both
 * expert projections run on the tensor cores in E4M3 (fp32 accumulation),
 * the row and channel scales applied in the GEMM epilogues. H is stored in
 * bf16 before its quantization; y is bf16.
 *
 *  wg_q, wu_q [device] [N+s][d_ff][d_model] uint8 codes;
 *  wg_scale, wu_scale [device] [N+s][d_ff] fp32 row scales;
 *  wd_q [device] [N+s][d_model][d_ff] uint8; wd_scale [N+s][d_model] fp32.
 *  Other arguments as moe_layer_forward; ws: moe_workspace_size_fp8(cfg).
 *  d_model and d_ff must be multiples of 16 (MOE_ERR_UNSUPPORTED otherwise).
 */
MOE_API size_t moe_workspace_size_fp8(const moe_config* cfg);
MOE_API int moe_layer_forward_fp8(const moe_config* cfg, const void* x, const void* w_router,
                    const float* logit_bias, const float* sel_bias,
                    const uint8_t* wg_q, const float* wg_scale,
                    const uint8_t* wu_q, const float* wu_scale,
                    const uint8_t* wd_q, const float* wd_scale, void* y,
                    int32_t* topk_idx, float* topk_w, int32_t* counts,
                    float* prob_sum, void* ws, size_t ws_bytes,
                    moe_stream_t stream);

/*
 * NVFP4 experts. The GB200 deployment keeps its experts in NVFP4 ("MoE
 * inference: the call centre with 256 specialists and 8 taking each call",
 * "The maths that matters" and "DeepEP, EPLB and Wide-EP"); the pages name
 * the format and no scaling rule. Format: E2M1 elements (magnitudes 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6) in blocks of 16 consecutive elements of a row, each
 * block with an unsigned E4M3 scale, and, as the library's rule, one fp32
 * scale per row. For a row with max |v| = amax > 0:
 *   row scale  s = fp32(amax / 2688)                        (2688 = 6 * 448)
 *   block      b = E4M3(fp32(bmax * fp32(448 / amax)))     (bmax: block max |v|)
 *   element    q = E2M1(fp32(v * fp32(fp32(2688 / amax) / e4m3(b))))
 * rounded to nearest even and saturated (448, 6), the sign kept when q
 * rounds to zero; a block whose scale is 0 has codes 0; a zero row has s = 0.
 * An element stands for e2m1(q) * e4m3(b) * s.
 *
 * Layout of a rows x cols NVFP4 matrix:
 *   q     [rows][cols / 2] uint8: two codes a byte, the lower column in the
 *         low nibble (sign in bit 3 of a nibble);
 *   sf    [rows][moe_nvfp4_scale_stride(cols)] uint8: E4M3 block scales,
 *         zero past cols / 16;
 *   scale [rows] fp32.
 *
 * moe_nvfp4_scale_stride: bytes of one row of block scales, cols / 16
 * rounded up to a multiple of 16 (0 for cols <= 0).
 * moe_quantize_nvfp4: rows x cols bf16 [device] -> q, sf, scale [device].
 * cols a multiple of 16; pointers 16-byte aligned. Quantize each weight
 * tensor of moe_layer_forward_nvfp4 with it (rows = output channels: E*d_ff
 * for gate and up, E*d_model for down). Returns MOE_ERR_INVALID_ARG for bad
 * sizes or null pointers, MOE_ERR_MISALIGNED for unaligned ones.
 */
MOE_API int32_t moe_nvfp4_scale_stride(int32_t cols);
MOE_API int moe_quantize_nvfp4(int64_t rows, int32_t cols, const void* src, uint8_t* q,
                    uint8_t* sf, float* scale, moe_stream_t stream);

/*
 * moe_layer_forward with NVFP4 experts: routing as moe_layer_forward (bf16
 * x and W_r; cfg->dtype must be MOE_BF16); every routed token row, x for the
 * shared experts and each row of H are quantized as above (H stored in bf16
 * first), and both expert projections run on the tensor cores as block-
 * scaled E2M1 products (tcgen05.mma kind::mxf4nvf4, the block scales applied
 * by the MMA, fp32 accumulation), the row scales applied in the GEMM
 * epilogues. y is bf16.
 *
 *  wg_q, wu_q [device] [N+s][d_ff][d_model/2]; wg_sf, wu_sf [N+s][d_ff][stride(d_model)];
 *  wg_scale, wu_scale [N+s][d_ff] fp32;
 *  wd_q [device] [N+s][d_model][d_ff/2]; wd_sf [N+s][d_model][stride(d_ff)];
 *  wd_scale [N+s][d_model] fp32.
 *  Other arguments as moe_layer_forward; ws: moe_workspace_size_nvfp4(cfg)
 *  bytes (0 when the shape is unsupported). d_model and d_ff must be
 *  multiples of 64 and at least 256 (MOE_ERR_UNSUPPORTED otherwise).
 */
MOE_API size_t moe_workspace_size_nvfp4(const moe_config* cfg);
MOE_API int moe_layer_forward_nvfp4(const moe_config* cfg, const void* x, const void* w_router,
                    const float* logit_bias, const float* sel_bias,
                    const uint8_t* wg_q, const uint8_t* wg_sf, const float* wg_scale,
                    const uint8_t* wu_q, const uint8_t* wu_sf, const float* wu_scale,
                    const uint8_t* wd_q, const uint8_t* wd_sf, const float* wd_scale,
                    void* y, int32_t* topk_idx, float* topk_w, int32_t* counts,
                    float* prob_sum, void* ws, size_t ws_bytes,
                    moe_stream_t stream);

/*
 * The load-balance statistics on the device: f_i = counts_i / (T*k),
 * P_i = prob_sum_i / T and aux = alpha * N * sum_i f_i P_i (one fixed-order
 * sum). ("Mixture of experts and speculative decoding", "Keeping the
 * experts busy"; "Mixture of Experts and Guided Decoding", auxiliary loss.)
 *
 *  counts   [device] [N] int32;  prob_sum [device] [N] fp32.
 *  f, P     [device] [N] fp32 out;  aux [device] [1] fp32 out.
 * With T = 0 all outputs are 0.
 */
MOE_API int moe_balance_stats(int32_t n_experts, int32_t T, int32_t top_k,
                      const int32_t* counts, const float* prob_sum,
                      float alpha, float* f, float* P, float* aux,
                      moe_stream_t stream);

/*
 * Backward of moe_layer_forward (bf16): the gradients of the scalar
 *   L = sum_{t,c} dy[t][c] * y[t][c] + aux_grad * aux,
 *   aux = alpha * N * sum_i f_i * P_i
 * (y the layer output, aux the balance loss of moe_balance_stats) with
 * respect to x, W_r, W_g, W_u and W_d ("Mixture of experts and speculative
 * decoding", the layer equation and "Keeping the experts busy"; "Mixture of
 * Experts and Guided Decoding", the auxiliary-loss formula). The top-k
 * choice, the capacity cut and the counts (so f) are hard decisions and are
 * held fixed: the gradient flows through the gate weights and through P.
 * The fp32 rounding of the scores only fixes the routing and counts as the
 * identity; logit_bias and sel_bias are constants.
 *
 * The forward is recomputed inside (router, permutation, both projections),
 * from the same inputs as the forward call. Rounding: H, the
 * pre-activations, dO = g * dy, da | db and each expert's input gradient
 * are bf16 intermediates; every sum accumulates in fp32.
 *
 *  x, w_router, logit_bias, sel_bias, w_gate, w_up, w_down: as
 *                 moe_layer_forward (bf16; cfg->dtype must be MOE_BF16).
 *  dy             [device] [T][d_model] bf16, dL/dy.
 *  alpha          the balance-loss coefficient (as moe_balance_stats).
 *  aux_grad       dL/daux (0 leaves the balance term out).
 *  dx             [device] [T][d_model] fp32 out.
 *  dw_router      [device] [N][d_model] fp32 out.
 *  dw_gate, dw_up [device] [N+s][d_ff][d_model] fp32 out.
 *  dw_down        [device] [N+s][d_model][d_ff] fp32 out. Experts that take
 *                 no token get zeros.
 *  ws             moe_workspace_size_backward(cfg) bytes.
 * d_ff must be a multiple of 64 (MOE_ERR_UNSUPPORTED otherwise; then
 * moe_workspace_size_backward returns 0). Every sum runs in a fixed order,
 * so two calls give the same bits.
 */
MOE_API size_t moe_workspace_size_backward(const moe_config* cfg);
MOE_API int moe_layer_backward(const moe_config* cfg, const void* x, const void* w_router,
                    const float* logit_bias, const float* sel_bias,
                    const void* w_gate, const void* w_up, const void* w_down,
                    const void* dy, float alpha, float aux_grad, float* dx,
                    float* dw_router, float* dw_gate, float* dw_up, float* dw_down,
                    void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronises `stream`, then returns the device-side status recorded in the
 * workspace `ws` by the last call that used it (MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE_CHECK), or MOE_ERR_CUDA if the stream reports an error. */
MOE_API int moe_stream_status(const void* ws, moe_stream_t stream);

/* Test hook for the failure path of the single-token decode kernel (the
 * one-launch layer that moe_layer_forward runs for T = 1; bf16, N <= 32).
 * That kernel has two grid-wide barriers, each a bounded wait: a CTA that
 * waits longer than the limit records MOE_ERR_TIMEOUT in the workspace
 * status word and returns, so a missing arrival ends the kernel with an
 * error that moe_stream_status reports instead of hanging the GPU. With
 * withhold != 0 the launches enqueued after this call wait for one arrival
 * more than the grid makes -- an arrival that never comes -- so every wait
 * runs out after limit_ns nanoseconds, the call's outputs are undefined and
 * its status is MOE_ERR_TIMEOUT. withhold = 0 with limit_ns = 0 restores
 * the defaults (no withheld arrival, a 2 s limit). The setting is
 * process-wide; no other kernel reads it. */
MOE_API void moe_set_decode_barrier_test(int32_t withhold, uint64_t limit_ns);

/* Kernel-level profiling. While enabled, each launch of the selected kernel
 * kinds is bracketed by CUDA events recorded on the launching stream (events
 * are created by the library, host-side). `mask` selects the kinds: bit i
 * for kind i (named by moe_profile_kernel_name(i)), -1 for all, 0 turns
 * profiling off. Events between launches cost the overlap of programmatic
 * dependent launch at that boundary, so select only the kernels to time.
 * moe_profile_collect synchronises on the last event, writes up to
 * `max_kernels` entries of per-kernel total milliseconds and launch counts
 * and clears the record; it returns the number of kernel kinds. */
MOE_API void moe_profile_enable(int mask);
MOE_API int moe_profile_collect(float* total_ms, int32_t* launches, int max_kernels);
MOE_API const char* moe_profile_kernel_name(int id);

/* Number of kernels this library has launched since it was loaded. */
MOE_API uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
