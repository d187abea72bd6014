/*
 * moe.h -- C ABI of libmoe.so, the GB300 (sm_103a) engine for one decode step
 * of a DeepSeek-style mixture-of-experts layer whose routed experts stay in
 * raw Q2_K (gate, up) and Q3_K (down) blocks.
 *
 * Sources (web pages of the "spark_model" crate, cited by page and item):
 *   [moe_v41]  spark_model/layers/moe_v41.rs -- module doc (the layer's math),
 *              struct MoeV41Cfg, struct MoeV41LayerWeights, struct Kernels,
 *              struct MoeV41 (buffers), fn shared_side, fn softplus,
 *              fn route_from_logits, fn bf16_bytes.
 *   [route]    spark_model/layers/moe_v41/device_route.rs -- module doc,
 *              fn header_words, fn arena_of, fn route_select_launch,
 *              fn slot_table_update, fn parse_header, fn route_device_m1,
 *              fn device_route_check.
 *   [step_seg] spark_model/layers/deepseek_v41_layer/step_seg.rs -- module
 *              doc (the step captured as CUDA graphs over layers).
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev or documented "device" are device pointers; the
 *    caller owns every buffer (the library allocates no device memory on the
 *    hot path). Host pointers are documented as such.
 *  - Calls only ENQUEUE work on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and return at once; nothing synchronises implicitly.
 *    Results are valid once the stream reaches the call.
 *  - Return 0 (MOE_OK) or a negative MOE_E* code; moe_last_error() then
 *    returns a message for the calling thread. Argument errors are detected
 *    on the host before anything is enqueued.
 *  - Calls that share a workspace must be ordered on one stream.
 *  - bf16 tensors are passed as raw 16-bit patterns (uint16_t storage).
 *
 * Shapes supported: dim and inter in {256, 512, 1024, 2048, 4096, 8192};
 * 1 <= topk <= 8; topk <= n_routed <= 1024; 1 <= m <= max_tokens <= 8;
 * m * dim <= 32768. Other shapes return MOE_EUNSUPPORTED (or MOE_EINVAL for
 * values that are wrong for any engine, e.g. topk = 0 or a non-multiple of 256).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* == cudaStream_t */

#define MOE_OK 0
#define MOE_EINVAL (-1)       /* an argument is invalid                       */
#define MOE_EUNSUPPORTED (-2) /* valid, but outside the shapes built here     */
#define MOE_ECUDA (-3)        /* a CUDA call failed (message has the error)   */
#define MOE_ECAPTURE (-4)     /* graph capture or instantiation failed        */

#define MOE_SLOT_TABLE_LAYERS 64 /* rows of the slot table ([route] slot table) */
#define MOE_MAX_TOPK 8
#define MOE_MAX_TOKENS 8
#define MOE_MAX_ROUTED 1024

/* Status bits in word 0 of each token's header row. */
#define MOE_HDR_MISS 1      /* a pick had slot -1: its pointers use slot 0 ([route] module doc) */
#define MOE_HDR_NONFINITE 2 /* a logit or key of the token was NaN or infinite                  */

/* Bits of the workspace status word (moe_read_status). */
#define MOE_WS_TIMEOUT 1   /* a bounded wait inside a kernel gave up           */
#define MOE_WS_PLAN 2      /* a plan exceeded a kernel's capacity; work skipped */
#define MOE_WS_TRIPLE 4    /* moe_slot_table_set met a triple outside the table */

/* Layer configuration ([moe_v41] struct MoeV41Cfg). norm_topk_prob is 0/1. */
typedef struct {
    int32_t dim, inter, n_routed, topk, norm_topk_prob, max_tokens;
    float gate_temp, route_scale, swiglu_limit;
} moe_cfg;

/* The expert arena: expert slot s holds gate (Q2_K [inter, dim]), up (Q2_K
 * [inter, dim]) and down (Q3_K [dim, inter]) blocks at base + s * slot_bytes
 * + {gate,up,down}_off ([route] fn arena_of). base and the three offsets
 * must be 16-byte aligned, slot_bytes a multiple of 16. Device memory. */
typedef struct {
    const void *base;
    uint64_t slot_bytes, gate_off, up_off, down_off;
} moe_arena;

/* Formats of the shared expert ([moe_v41] struct MoeV41LayerWeights: "bf16
 * or the GGUF's Q2_K (w1, w3) / Q3_K (w2) blocks on the routed experts'
 * kernels"). */
#define MOE_SHARED_BF16 0   /* w1, w3 bf16 [inter, dim]; w2 bf16 [dim, inter]   */
#define MOE_SHARED_KQUANT 1 /* w1, w3 Q2_K [inter, dim]; w2 Q3_K [dim, inter],
                               laid out as a routed expert's gate, up, down   */

/* One layer's resident weights ([moe_v41] struct MoeV41LayerWeights), all
 * device pointers: router_w bf16 [n_routed, dim] row-major; bias f32
 * [n_routed]; slot_row i32 [n_routed] (this layer's slot-table row, -1 = not
 * resident); sh_w1, sh_w3, sh_w2 the shared expert in format sh_format
 * (MOE_SHARED_*; all three NULL = no shared expert). 16-byte aligned. */
typedef struct {
    const void *router_w;
    const float *bias;
    const int32_t *slot_row;
    const void *sh_w1, *sh_w3, *sh_w2;
    int32_t sh_format;
} moe_layer;

/* Words (int32) of the route header for m tokens. Layout, k = topk:
 *   row t (t < m), 1 + 3k words ([route] fn header_words, module doc):
 *     [0] status bits (MOE_HDR_*); [1..k] picks in pick order;
 *     [k+1..2k] the weights' f32 bit patterns, pick order; [2k+1..3k] the
 *     slots of the token's picks in ascending expert id (-1 reported as 0)
 *   then the plan over all m tokens (distinct picked experts, ascending id):
 *     [m(1+3k)] ne; [+1 .. +1+m*k] pair_start[0..ne] (ne+1 used);
 *     [+2+m*k .. +1+2*m*k] plan_expert[0..ne-1]. */
int moe_header_words(const moe_cfg *cfg, int m);

/* Bytes of the device workspace for up to cfg->max_tokens tokens. */
int moe_workspace_bytes(const moe_cfg *cfg, size_t *bytes);

/* Zeroes a workspace (its counters must start at zero). Call once after
 * allocating it, on the stream that will use it, and again after a call whose
 * status has MOE_WS_TIMEOUT (a wait that gave up can leave counters mid-count). */
int moe_workspace_init(void *ws_dev, size_t bytes, moe_stream_t stream);

/* Router logits ([moe_v41] module doc: an f32-accumulated product of the bf16
 * input and the bf16 gate weight; struct Kernels router_gemv):
 *   logits[t, e] = sum_j x[t, j] * w[e, j], bf16 products exact in f32, f32
 *   accumulation in a fixed order that does not depend on m.
 * x_dev bf16 [m, dim]; w_dev bf16 [n_routed, dim]; logits_dev f32 [m, n_routed]. */
int moe_router_logits(const moe_cfg *cfg, const void *x_dev, const void *w_dev,
                      float *logits_dev, int m, moe_stream_t stream);

/* q8_1 quantisation of m bf16 rows ([moe_v41] module doc: the activation
 * quantised to q8_1; struct Kernels q8_rows): per 32 values d = amax / 127
 * (f32), q = round-half-away(x / d), stored as f16 d, f16 d * sum q, int8
 * q[32] (36 bytes). out_dev: m * dim / 32 blocks. */
int moe_quantize_q8_1(const moe_cfg *cfg, const void *x_dev, int m, void *out_dev,
                      moe_stream_t stream);

/* Device selection ([moe_v41] fn route_from_logits; [route] fn
 * route_select_launch, module doc): per token, scores s = the f32 chain
 * sqrt(ln_1p(exp(t))), t = l / temp, each step correctly rounded (t itself
 * in place of ln_1p(exp(t)) for t > 20; [moe_v41] fn softplus), picks = the top k of
 * s + bias with ties to the lower id, weights = picked scores divided by
 * (their f32 sum in pick order + 1e-20) when norm_topk_prob and k > 1, times
 * route_scale; then the plan, the plan weights and rows (pair-major:
 * experts ascending, tokens ascending within one), and the pointer table
 * ptrs[0..cap) gate, [cap..2cap) up, [2cap..3cap) down with cap = m * topk,
 * pointer = base + slot * slot_bytes + offset, slot -1 -> slot 0 and the
 * MOE_HDR_MISS bit. Scores, picks and weights are bit-identical to the
 * definition (each rounding of the score decided exactly).
 * logits_dev f32 [m, n_routed]; bias_dev f32 [n_routed]; slot_row_dev i32
 * [n_routed]; arena by value (host struct, device base); header_dev i32
 * [moe_header_words]; plan_w_dev f32 [m*topk]; plan_rows_dev i32 [m*topk];
 * ptrs_dev u64 [3*m*topk]. */
int moe_route_select(const moe_cfg *cfg, const float *logits_dev, const float *bias_dev,
                     const int32_t *slot_row_dev, const moe_arena *arena, int m,
                     int32_t *header_dev, float *plan_w_dev, int32_t *plan_rows_dev,
                     uint64_t *ptrs_dev, moe_stream_t stream);

/* The routing score of each logit ([moe_v41] fn softplus, fn
 * route_from_logits): t = f32(logits[i] / gate_temp); for t > 20
 * scores[i] = f32(sqrt(t)), else e = f32(e^t), p = f32(ln(1 + e)),
 * scores[i] = f32(sqrt(p)), each rounding to nearest as a correctly rounded
 * operation -- the score the router and the selection use. The roundings
 * are decided in float-float single precision, in double and then
 * double-double precision when that cannot decide them. logits_dev,
 * scores_dev f32 [count], count >= 0 (0: nothing is launched). */
int moe_route_scores(const moe_cfg *cfg, const float *logits_dev, int count, float *scores_dev,
                     moe_stream_t stream);

/* The routed experts of one call ([moe_v41] module doc: three K-quant GEMVs
 * per expert on the raw blocks, gate and up Q2_K, down Q3_K, q8_1 activation;
 * struct Kernels mmvq_q2k_experts / swiglu_q8 / mmvq_q3k_experts /
 * accumulate): for every plan expert p and each of its tokens t
 *   g, u = Q2_K(gate_p, up_p) . q8_1(x_t);  h = silu(min(g, L)) * clamp(u, -L, L)
 *   down = Q3_K(down_p) . q8_1(h);  acc_t = sum over t's plan, ascending id,
 *   of w * down (f32). Reads the plan from header_dev (moe_route_select).
 * acc_dev f32 [m, dim]; ws_dev: workspace (intermediates g, u, down stay there). */
int moe_expert_step(const moe_cfg *cfg, const void *x_dev, const uint64_t *ptrs_dev,
                    const float *plan_w_dev, const int32_t *plan_rows_dev,
                    const int32_t *header_dev, int m, float *acc_dev, void *ws_dev,
                    moe_stream_t stream);

/* Clamped SwiGLU and the q8_1 of its output ([moe_v41] struct Kernels
 * swiglu_q8): h[i] = silu(min(g, L)) * clamp(u, -L, L) in f32 (L <= 0: no
 * clamp); h_q8 as moe_quantize_q8_1. g_dev, u_dev, h_dev f32 [rows, inter];
 * hq8_dev rows * inter / 32 blocks (h_dev may be NULL). */
int moe_swiglu_q8(const moe_cfg *cfg, const float *g_dev, const float *u_dev, int rows,
                  float *h_dev, void *hq8_dev, moe_stream_t stream);

/* One whole MoE layer step for m tokens ([moe_v41] module doc and fn
 * shared_side; [route] module doc): router logits, selection, routed experts,
 * the shared expert (bf16: gs, us = W1 x, W3 x; hs = bf16(SwiGLU); sd = W2 hs;
 * K-quant: gs, us = Q2_K(W1, W3) . q8_1(x), hs = SwiGLU in f32, sd =
 * Q3_K(W2) . q8_1(hs), as a routed expert of weight 1 -- [moe_v41] struct
 * MoeV41 sh_q8),
 * acc = routed sum (ascending id) + sd added last, residual += acc,
 * x_next = bf16 round-to-nearest-even of residual ([moe_v41] fn bf16_bytes).
 * Launched as three kernels chained with programmatic dependent launch.
 * x_dev bf16 [m, dim]; residual_dev f32 [m, dim] (in/out); x_next_dev bf16
 * [m, dim] (may equal x_dev); header_dev i32 [moe_header_words]; acc, the
 * plan, pointers and intermediates are left in ws_dev (moe_ws_view). */
int moe_layer_step(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                   const void *x_dev, float *residual_dev, void *x_next_dev,
                   int32_t *header_dev, int m, void *ws_dev, moe_stream_t stream);

/* moe_layer_step without a caller workspace and without any device
 * allocation. The pages have no counterpart of this call: it exists for
 * callers that cannot allocate device memory (a plain C host program linking
 * only this library, with no device allocator of its own; a serving loop that
 * must not allocate once it runs, since cudaMalloc and cudaFree can
 * synchronise the device and can fail under memory pressure).
 * The workspace is a 4 MiB array in the library's device memory, one per
 * device. The first call on a device (with that device current) looks it up
 * with cudaGetSymbolAddress and zeroes it; make that first call before any
 * stream capture (a first call on a capturing stream returns
 * MOE_EUNSUPPORTED). The looked-up address is kept for the life of the
 * process: do not use this call across cudaDeviceReset of that device.
 * Every call clears the array's control words and counters on `stream`
 * first, then runs the same kernels as moe_layer_step.
 * Arguments as moe_layer_step; status_host: NULL, or a host word that
 * receives the workspace status (MOE_WS_*) of this call once `stream`
 * reaches the end of the call (pinned memory keeps the copy asynchronous).
 * The array is shared by every call on the device: calls that overlap in
 * time (other streams, other host threads) race on it and must be
 * serialised by the caller. Errors: MOE_EUNSUPPORTED when the configuration
 * needs more than 4 MiB of workspace (moe_workspace_bytes); MOE_EINVAL for
 * bad arguments; MOE_ECUDA when the look-up or a launch fails. */
int moe_layer_step_static(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                          const void *x_dev, float *residual_dev, void *x_next_dev,
                          int32_t *header_dev, int m, uint32_t *status_host, moe_stream_t stream);

/* Same step with HOST buffers: copies x (bf16 [m, dim], host) and residual
 * (f32 [m, dim], host) in, runs moe_layer_step, copies residual, x_next and
 * the header back to host buffers, all on `stream` (pinned host memory makes
 * the copies asynchronous). io_dev: device scratch of
 * moe_host_io_bytes(cfg, m) bytes. */
int moe_host_io_bytes(const moe_cfg *cfg, int m, size_t *bytes);
int moe_layer_step_host(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                        const void *x_host, float *residual_host, void *x_next_host,
                        int32_t *header_host, int m, void *io_dev, void *ws_dev,
                        moe_stream_t stream);

/* Where the intermediates of the last call live inside a workspace (device
 * pointers into ws_dev), for inspection. */
typedef struct {
    float *logits;      /* [m, n_routed]                                   */
    float *plan_w;      /* [m*topk]                                        */
    int32_t *plan_rows; /* [m*topk]                                        */
    uint64_t *ptrs;     /* [3*m*topk]                                      */
    float *g, *u;       /* [m*topk, inter] per plan pair                   */
    float *gs, *us;     /* [m, inter] shared expert                        */
    float *down;        /* [m*topk, dim] per plan pair                     */
    float *sd;          /* [m, dim] shared expert output                   */
    float *acc;         /* [m, dim] routed sum + shared                    */
    uint32_t *status;   /* one word, MOE_WS_* bits                         */
} moe_ws_view;
int moe_workspace_view(const moe_cfg *cfg, void *ws_dev, moe_ws_view *view);

/* Reads the workspace status word (MOE_WS_* bits) to a host variable; this
 * synchronises `stream`. */
int moe_read_status(void *ws_dev, uint32_t *status_host, moe_stream_t stream);

/* Sets the bound, in nanoseconds, on every wait inside the kernels (a wait
 * on a shared-memory barrier, on another CTA's count, or on the selection's
 * plan) for the calls enqueued after it; a graph keeps the bound it was
 * captured with. 0 restores the default of 2 s. Process-wide. When a wait
 * runs out, the kernel records MOE_WS_TIMEOUT in the workspace status and
 * returns instead of waiting on (page step_seg.rs has no counterpart: a
 * device wait there is unbounded). */
int moe_set_wait_limit_ns(uint64_t ns);

/* Failure-handling check, not a step of the layer: launches the two expert
 * kernels of a layer step as moe_layer_step does, but with no router kernel
 * before them, so the gate/up producers' bounded wait for the selection's
 * plan-ready word can only end by running out. header_dev must hold an empty
 * plan (zeros: ne = 0), so that no expert is read. After the stream reaches
 * it, the workspace status has MOE_WS_TIMEOUT and the workspace must be
 * initialised again (moe_workspace_init). x_dev bf16 [m, dim]. */
int moe_expert_step_unreleased(const moe_cfg *cfg, const void *x_dev, const int32_t *header_dev, int m,
                               void *ws_dev, moe_stream_t stream);

/* Slot-table update ([route] fn slot_table_update, struct Kernels
 * slot_table_set): for each of n (layer, expert, slot) int32 triples,
 * table[layer * n_routed + expert] = slot. The triples are applied in
 * parallel, so the caller must pass at most one triple per (layer, expert)
 * (moe_dedupe_triples gives the last-write-wins set). A triple outside
 * [0, 64) x [0, n_routed) is skipped and sets MOE_WS_TRIPLE in
 * *status_dev (may be NULL). table_dev i32 [64, n_routed]; triples_dev i32
 * [n, 3]. */
int moe_slot_table_set(int32_t *table_dev, int n_routed, const int32_t *triples_dev, int n,
                       uint32_t *status_dev, moe_stream_t stream);

/* Host helper: keeps only the last triple of each (layer, expert) key, in
 * place, preserving the order of first appearance of the kept keys; *n_out
 * = the count kept. Host pointer. */
int moe_dedupe_triples(int32_t *triples_host, int n, int *n_out);

/* Host helper ([route] fn parse_header): token t's status word, picks and
 * weights out of a header copied to the host. Fails (MOE_EINVAL) when a pick
 * lies outside 0..n_routed-1. picks_host i32 [topk], weights_host f32 [topk]. */
int moe_parse_header(const moe_cfg *cfg, const int32_t *header_host, int m, int t,
                     int32_t *status_host, int32_t *picks_host, float *weights_host);

/* Options of moe_graph_create. */
#define MOE_GRAPH_SNAPSHOTS 1       /* copy each layer's input (x and residual) to snapshot memory
                                       before the layer, inside the graph ([step_seg] module doc:
                                       a snapshot a layer, ~75 KB there), so the step can be rerun
                                       from a layer (moe_graph_rerun_from, moe_graph_step_cached) */
#define MOE_GRAPH_EAGER_FALLBACK 2  /* if capture or instantiation fails, the object runs the layers
                                       eagerly instead ([step_seg] fn close_or_disable: graph mode off) */
#define MOE_GRAPH_TEST_FAIL_CAPTURE 4 /* failure-handling check: treat the capture as failed (no capture
                                       is attempted), to exercise MOE_GRAPH_EAGER_FALLBACK */

/* A whole-step CUDA graph ([step_seg] module doc: the step captured once and
 * replayed, one read-back of the headers per launch): n_layers layer steps
 * chained, layer l reading x from x_a (l even) or x_b (l odd) and writing the
 * other, except that the last layer writes x_a, so each launch continues from
 * the previous launch's output; residual_dev carries between layers; layer
 * l's header lands at headers_dev + l * moe_header_words(cfg, m). layers is a
 * host array of n_layers structs (copied; their device pointers are baked
 * in); every buffer must outlive the graph. snap_dev: moe_graph_snapshot_bytes
 * of device memory with MOE_GRAPH_SNAPSHOTS, else may be NULL. flags:
 * MOE_GRAPH_*. Without MOE_GRAPH_EAGER_FALLBACK a failed capture returns
 * MOE_ECAPTURE and no object. */
int moe_graph_snapshot_bytes(const moe_cfg *cfg, int m, int n_layers, size_t *bytes);
int moe_graph_create(const moe_cfg *cfg, const moe_layer *layers, int n_layers,
                     const moe_arena *arena, int m, void *x_a_dev, void *x_b_dev,
                     float *residual_dev, int32_t *headers_dev, void *ws_dev, void *snap_dev,
                     unsigned flags, void **graph);
/* *eager = 1 when the object runs its layers eagerly (capture failed). */
int moe_graph_is_eager(void *graph, int *eager);
/* Restores layer `layer`'s snapshot into that layer's input buffers and runs
 * layers layer .. n_layers - 1 eagerly on `stream` (snapshots refreshed on
 * the way). Needs MOE_GRAPH_SNAPSHOTS. */
int moe_graph_rerun_from(void *graph, int layer, moe_stream_t stream);
int moe_graph_launch(void *graph, moe_stream_t stream);
int moe_graph_destroy(void *graph);

/* One graph launch with HOST buffers: copies x (bf16 [m, dim]) and residual
 * (f32 [m, dim]) from host memory into the graph's x_a / residual buffers,
 * launches the graph, and copies the output x (x_a), the residual and every
 * layer's header back to host memory, all on `stream` (pinned host memory
 * makes the copies asynchronous). headers_host: n_layers * moe_header_words. */
int moe_graph_launch_host(void *graph, const void *x_host, const float *residual_host, void *x_out_host,
                          float *residual_out_host, int32_t *headers_host, moe_stream_t stream);

/* Measurement entry point: the same layer step as moe_layer_step, but the
 * three kernels run back to back without overlap, bracketed by CUDA events on
 * `stream`; synchronises `stream` and writes the durations in milliseconds to
 * ms_host[0] (router + selection), ms_host[1] (gate/up GEMVs incl. the shared
 * W1/W3 rows), ms_host[2] (down GEMVs incl. shared W2, accumulate, residual). */
int moe_layer_step_profiled(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                            const void *x_dev, float *residual_dev, void *x_next_dev, int32_t *header_dev,
                            int m, void *ws_dev, moe_stream_t stream, float *ms_host);

/* Dense GEMM on the tensor cores (tcgen05.mma, f32 accumulator in tensor
 * memory, operands by TMA): d[n * ldd + r] = sum_k a[r, k] * b[n, k], a bf16
 * [M, K] and b bf16 [N, K] row-major (bf16 products exact, f32 sums) --
 * the contraction of the router and of the bf16 shared expert when many
 * tokens run at once ([moe_v41] struct Kernels gemm / gemm_f32out). K a
 * positive multiple of 64, ldd >= M, a and b 16-byte aligned with row
 * strides K * 2 a multiple of 16. Device pointers. */
int moe_gemm_bf16(const void *a_dev, const void *b_dev, float *d_dev, int M, int N, int K, int ldd,
                  moe_stream_t stream);

/* The batched (prefill) arm: one MoE layer step for m tokens at once
 * ([moe_v41] struct Kernels gather, scatter_add, sum_rows, quant_d2s6 /
 * quant_d4, mmq_q2k_*, mmq_q3k_*, gemm; struct MoeV41 a_rows, a_q8: an
 * expert group's gathered rows and their q8_1 activations). The arithmetic
 * is moe_layer_step's; the routed experts run as GEMMs over each expert's
 * group of tokens, on tensor cores:
 *   logits = router GEMM; scores, picks and weights as the decode selection;
 *   pairs (token, pick) grouped by expert in ascending id, tokens ascending;
 *   per expert g, u = Q2_K(gate, up) . q8_1(x) over its group, h = SwiGLU,
 *   q8_1(h), down = Q3_K(down) . q8_1(h), each times the pair's weight;
 *   the bf16 shared expert as dense GEMMs; acc = the pairs in ascending
 *   expert id then sd; residual += acc; x_next = bf16(residual).
 * The GEMM operands are the dequantised weights and the dequantised q8_1
 * activations rounded to fp16 (the products then differ from the exact
 * dequantise-then-dot by about 2^-12 relative per operand); accumulation
 * f32. Shapes: dim a multiple of 1024, inter of 2048 (the row strides of
 * the Q2_K / Q3_K blocks must be multiples of 16 bytes for TMA), the shared
 * expert bf16 or absent, 0 <= m <= 65536 (cfg->max_tokens is not used).
 * arena_slots: slots in the arena (the tensor maps cover that many). x_dev
 * bf16 [m, dim], 16-byte aligned (a TMA operand; otherwise MOE_EINVAL before
 * any launch); residual_dev f32 [m, dim] (in/out); x_next_dev bf16 [m, dim]
 * (16- and 8-byte alignment of these take the wider accesses); picks_dev i32 [m, topk], weights_dev f32 [m, topk] (pick
 * order); ws_dev: moe_prefill_workspace_bytes bytes (no initialisation
 * needed). Errors: MOE_EUNSUPPORTED for the shapes above; a picked expert
 * whose slot is -1 uses slot 0 and sets MOE_WS_PLAN (moe_prefill_status). */
int moe_prefill_workspace_bytes(const moe_cfg *cfg, int m, size_t *bytes);
int moe_prefill_step(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena, int64_t arena_slots,
                     const void *x_dev, float *residual_dev, void *x_next_dev, int32_t *picks_dev,
                     float *weights_dev, int m, void *ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Measurement entry point: moe_prefill_step with CUDA events between its
 * stages on `stream`; synchronises `stream` and writes milliseconds to
 * ms_host[0..8]: router GEMM; scores, top-k and grouping; q8_1 of x and the
 * gathers; gate GEMM; up GEMM; SwiGLU + q8_1(h); down GEMM; shared expert
 * (three GEMMs and its SwiGLU); finish. */
int moe_prefill_step_profiled(const moe_cfg *cfg, const moe_layer *layer, const moe_arena *arena,
                              int64_t arena_slots, const void *x_dev, float *residual_dev, void *x_next_dev,
                              int32_t *picks_dev, float *weights_dev, int m, void *ws_dev, size_t ws_bytes,
                              moe_stream_t stream, float *ms_host);

/* The status word (MOE_WS_* bits) of the last moe_prefill_step on ws_dev;
 * synchronises `stream`. */
int moe_prefill_status(const moe_cfg *cfg, int m, void *ws_dev, uint32_t *status_host, moe_stream_t stream);

/* Expert residency ([moe_v41] module doc: the ExpertLru gathers the picked
 * experts' raw slices into device-visible slots, misses read from the
 * source; [route] module doc and fn slot_table_update: the host touches the
 * picks, fetches the misses and uploads the slot changes to the device
 * table). A cache owns n_slots slots of the arena for layers 0 .. n_layers-1
 * of the slot table at slot_table_dev ([64][n_routed], row l for layer l; NULL
 * keeps the table on the host only), least recently used out first, and
 * fetches a missing expert with fetch(user, layer, expert, slot address,
 * slot_bytes, stream) -- which must enqueue the copy of the expert's slot
 * image on `stream` and return 0. Creating the cache marks every entry of its
 * rows not resident (-1). */
typedef int (*moe_expert_fetch_fn)(void *user, int layer, int expert, void *slot_dev, uint64_t slot_bytes,
                                   moe_stream_t stream);
int moe_cache_create(int n_layers, int n_routed, int n_slots, const moe_arena *arena, int32_t *slot_table_dev,
                     moe_expert_fetch_fn fetch, void *user, void **cache);
int moe_cache_destroy(void *cache);
/* Makes the experts (host array of n ids of one layer; repeats allowed)
 * resident: hits become most recently used, misses take the least recently
 * used slots (their previous experts marked -1) and are fetched; the changed
 * table rows are uploaded on `stream`. *n_fetched (may be NULL) = misses.
 * MOE_EUNSUPPORTED when more distinct experts are asked at once than slots. */
int moe_cache_ensure(void *cache, int layer, const int32_t *experts_host, int n, int *n_fetched,
                     moe_stream_t stream);
/* The slot of (layer, expert), -1 when not resident. */
int moe_cache_slot_of(void *cache, int layer, int expert, int32_t *slot);
int moe_cache_stats(void *cache, uint64_t *hits, uint64_t *misses, uint64_t *evictions);

/* An expert source over host memory: images_host[layer * n_routed + expert]
 * = host address of that expert's slot image (image_bytes; pinned memory
 * keeps the copies asynchronous). moe_fetch_host_images is its fetch
 * function (pass the source as `user`). */
int moe_host_source_create(const void *const *images_host, int n_layers, int n_routed, uint64_t image_bytes,
                           void **source);
int moe_host_source_destroy(void *source);
int moe_fetch_host_images(void *source, int layer, int expert, void *slot_dev, uint64_t slot_bytes,
                          moe_stream_t stream);

/* One launch of a graph with snapshots whose layers take their experts from
 * a cache (layer l using row l of the cache's table): launch, read the
 * headers; at the first layer whose header has MOE_HDR_MISS, make that
 * layer's picks resident, restore its snapshot and run the rest eagerly,
 * layer by layer, a layer with a miss fetched and rerun from its snapshot
 * ([step_seg] module doc and fn step_seg: restore, the layer's ffn eagerly,
 * eager to the end). On return (the stream synchronised) the graph's buffers
 * hold the result and headers_host (host, n_layers header rows) the final
 * headers; *layers_rerun (may be NULL) = layers run again. */
int moe_graph_step_cached(void *graph, void *cache, int32_t *headers_host, int *layers_rerun,
                          moe_stream_t stream);

/* Last error message of the calling thread ("" if none). */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
