/*
 * mk.h -- C ABI of the GB300 persistent verify-step megakernel.
 *
 * One call runs ONE speculative-verify decode step of a mixture-of-experts
 * transformer for a block of T = k+1 tokens (the last accepted token followed by
 * k drafts), fused into a single persistent kernel launch.
 *
 * What the call computes comes from two pages:
 *  - "Why one GB300 doesn't beat 4x RTX PRO 6000 at single-stream decode"
 *    (al-engr), section "The decomposition": tokens/s = tokens per verify step x
 *    verify steps/s, with tokens per step = accepted drafts + 1; section "Where the
 *    11.2 ms goes": the step is a stack of 43 MoE layers with 384 experts, decode
 *    attention, dense projections, a router top-k, an lm_head and one accept
 *    (rejection) kernel per step, spread over ~1,300 small kernels that this
 *    library replaces with one launch.
 *  - "DeepSeek-V4.1-Flash breaks 1,000 tokens per second for one user" (ezolabs),
 *    sections "How we got here" and "Serving stack": drafted tokens are checked
 *    together in blocks (block verification), 5-token draft blocks; the plugin
 *    keeps one persistent block per SM and refuses configurations it cannot run
 *    ("no silent fallback", section "What NVIDIA shipped").
 * The per-layer equations (pre-norm GQA attention with rotate-half RoPE over a
 * paged KV cache, sigmoid router with selection-only bias and top-K weights
 * normalised to 1, SwiGLU routed experts plus one shared expert) are the plain
 * reading of the workload the pages describe; the same reading drives the fp64
 * oracle in oracle/.
 *
 * Conventions for every entry point
 *  - All tensors are row-major and owned by the caller; the library never copies
 *    or frees them.  "dev" pointers are CUDA device memory on the current device,
 *    "host" pointers are host memory.  The library owns only its workspace
 *    (allocated in mk_create, freed in mk_destroy).
 *  - Calls taking a stream are asynchronous on that stream (a cudaStream_t passed
 *    as void*, NULL = legacy default stream).  Errors that the host can see are
 *    returned at once and nothing is launched; errors found on the device (a bad
 *    position or page-table entry, a wait that ran past its time limit) are
 *    recorded in a device status word that mk_get_status reads.  After a device
 *    error every later step exits at once until mk_reset is called.
 *  - A state is not thread-safe and allows one step in flight at a time.
 *  - There is no fallback path: unsupported shapes, dtypes or devices return
 *    MK_ERR_UNSUPPORTED.
 */
#ifndef MK_H
#define MK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MK_OK = 0,
    MK_ERR_INVALID = -1,      /* bad argument (null pointer, T out of range, ...)      */
    MK_ERR_UNSUPPORTED = -2,  /* shape/dtype/device this build does not run           */
    MK_ERR_NOMEM = -3,        /* workspace allocation failed                           */
    MK_ERR_TIMEOUT = -4,      /* a device-side wait ran past timeout_ms                */
    MK_ERR_CUDA = -5,         /* a CUDA runtime call failed                            */
    MK_ERR_BAD_STATE = -6,    /* call not valid in the current state                   */
    MK_ERR_BAD_INPUT = -7,    /* device-side input check failed (positions, page table)*/
    MK_ERR_RANGE = -8         /* a value left the kernel's number range: an f16 GEMV    */
                              /* input beyond 65504 (or NaN), or a partial sum of       */
                              /* magnitude >= 2^31 for the 2^-32 fixed-point sums       */
} mk_status;

/* storage types of weights and of the KV cache */
enum {
    MK_DT_F32 = 0,           /* float32                                                 */
    MK_DT_BF16 = 1,          /* bfloat16                                                */
    MK_DT_FP8E4M3_B128 = 2,  /* FP8 E4M3 codes + float32 scale per 1x128 input block:   */
                             /* W[n][k] = fp8(q[n][k]) * scale[k/128][n]                */
    MK_DT_FP8E4M3 = 4,       /* FP8 E4M3 codes times one float32 scale per tensor: the  */
                             /* KV cache (kv_dtype) with a K and a V scale per layer    */
    MK_DT_MXFP4_B32 = 3      /* MXFP4 (OCP Microscaling Formats v1.0): FP4 E2M1 codes,  */
                             /* two per byte (element 2j in the low nibble of byte j),  */
                             /* and one E8M0 scale byte per 1x32 input block:           */
                             /* W[n][k] = e2m1(q[n][k]) * 2^(scale[k/32][n] - 127).     */
                             /* Routed experts only (expert_dtype).                     */
};

#define MK_DESC_VERSION 3

/* Model description.  Limits of this build: T <= 8; hidden, expert_inter and
 * n_q_heads*head_dim multiples of 128 and <= 4096; page_size 64;
 * (n_q_heads/n_kv_heads)*T <= 64; n_experts a multiple of 4 and <= 512;
 * top_k <= 8; n_shared 0 or 1.  bf16 / FP8 weights need a bf16 KV cache and
 * head_dim 128.  F32 weights need an F32 router, head_dim 64,
 * (n_q_heads/n_kv_heads)*T <= 16 and hidden, n_q_heads*head_dim,
 * expert_inter <= 2048.  MXFP4 routed experts need bf16 or FP8 weights
 * elsewhere and hidden, expert_inter multiples of 256.
 * Passage for MXFP4 experts: ezolabs "DeepSeek-V4.1-Flash breaks 1,000 tokens
 * per second for one user", section "Appendix: method", Serving stack
 * ("MXFP4 expert weights"); al-engr, section "Where the 11.2 ms goes", kernel
 * table (the fp8 x fp4 expert GEMM). */
typedef struct {
    int version;              /* MK_DESC_VERSION                                      */
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim;
    float rope_base, rms_eps;
    int n_experts, top_k, n_shared, expert_inter;
    int vocab;                /* 0: no embedding / LM head (mk_layer_forward only)    */
    int page_size;            /* KV positions per page                                */
    int max_T;                /* largest verify block that will be passed (<= 8)      */
    int max_pages_per_stream; /* page-table row length; bounds positions              */
    int weight_dtype;         /* MK_DT_* of attention and expert matrices             */
    int router_dtype;         /* MK_DT_F32 or MK_DT_BF16                              */
    int kv_dtype;             /* MK_DT_F32, MK_DT_BF16 or MK_DT_FP8E4M3               */
    int timeout_ms;           /* limit of every device-side wait; 0 means 1000 ms     */
    int expert_dtype;         /* MK_DT_* of the routed experts (w1, w3, w2): equal to */
                              /* weight_dtype, or MK_DT_MXFP4_B32                     */
    int lm_head_dtype;        /* MK_DT_BF16, or MK_DT_FP8E4M3_B128 with bf16 / FP8    */
                              /* weights elsewhere                                    */
} mk_model_desc;

/* One layer's weights (dev pointers).  Shapes, with d = head_dim, H = hidden,
 * E = n_experts, I = expert_inter, NQKV = (n_q_heads + 2*n_kv_heads)*d:
 *   attn_norm, moe_norm  float32 [H]
 *   w_qkv   [NQKV][H]  rows: n_q_heads q heads, then n_kv_heads k heads, then v heads
 *   w_o     [H][n_q_heads*d]
 *   w_router [E][H] in router_dtype;  router_bias float32 [E] (selection only)
 *   w1, w3  [E][I][H];  w2 [E][H][I]        routed experts (gate, up, down)
 *   ws1, ws3 [I][H];    ws2 [H][I]          shared expert (NULL when n_shared = 0)
 * FP8 matrices carry a float32 scale array laid out [in/128][out] (for the
 * expert stacks [E][in/128][out]); it is ignored for other dtypes.  MXFP4
 * routed experts store their codes as bytes [E][rows][cols/2] and their E8M0
 * scales as bytes [E][cols/32][rows] (w1_scale, w3_scale, w2_scale). */
typedef struct {
    const float *attn_norm;
    const void *w_qkv;  const float *w_qkv_scale;
    const void *w_o;    const float *w_o_scale;
    const float *moe_norm;
    const void *w_router;
    const float *router_bias;
    const void *w1;     const void *w1_scale;
    const void *w3;     const void *w3_scale;
    const void *w2;     const void *w2_scale;
    const void *ws1;    const float *ws1_scale;
    const void *ws3;    const float *ws3_scale;
    const void *ws2;    const float *ws2_scale;
} mk_layer_weights;

/* The LM head is bf16 or, with lm_head_dtype MK_DT_FP8E4M3_B128, FP8 E4M3
 * codes [vocab][H] with float32 scales lm_head_scale [H/128][vocab].  Passage:
 * al-engr, section "Where the 11.2 ms goes" (the lm_head's bf16 weight reads)
 * and section "Credits" (an FP8 draft head). */
typedef struct {
    const void *embed;               /* bf16 [vocab][H] (dev; NULL if vocab == 0)     */
    const float *final_norm;         /* float32 [H]                                   */
    const void *lm_head;             /* [vocab][H] in lm_head_dtype                   */
    const mk_layer_weights *layers;  /* HOST array of n_layers entries                */
    const float *lm_head_scale;      /* FP8 LM head only: float32 [H/128][vocab]      */
} mk_weights;

/* Paged KV cache.  Layer l keeps k_pool[l], v_pool[l] (dev), each
 * [n_pages][n_kv_heads][page_size][head_dim] in kv_dtype; entries are stored
 * already rotated.  page_table (dev int32 [n_streams][max_pages_per_stream])
 * maps logical page j of a stream (positions j*P .. j*P+P-1) to a physical
 * page.  A step with positions p_t = ctx + t reads positions < ctx and writes
 * K/V of its T tokens at positions ctx..ctx+T-1; the caller then advances ctx
 * by accepted + 1 (rejected slots are overwritten by the next step).
 * An FP8 cache (kv_dtype MK_DT_FP8E4M3) holds E4M3 codes: an entry's value is
 * code * k_scale[l] (keys) or code * v_scale[l] (values), and the step stores
 * its new entries as the nearest code (ties to even, saturating at 448) of
 * value / scale.  Passage: ezolabs, section "Appendix: method", Serving stack
 * ("an fp8 (e4m3) KV cache"). */
typedef struct {
    void *const *k_pool;             /* HOST array [n_layers] of dev pointers         */
    void *const *v_pool;
    const int32_t *page_table;       /* dev                                           */
    int n_pages;                     /* physical pages in each pool                   */
    const float *k_scale;            /* HOST [n_layers] (FP8 cache only; NULL = 1.0)  */
    const float *v_scale;            /* HOST [n_layers] (FP8 cache only; NULL = 1.0)  */
} mk_kv_cache;

typedef struct {
    uint64_t steps;                  /* completed verify steps since create/reset     */
    uint64_t accepted_sum;           /* sum of accepted draft counts                   */
    uint64_t distinct_experts_sum;   /* routed experts streamed, summed over layers    */
    int32_t last_accepted;
    int32_t last_distinct_experts;   /* summed over the layers of the last step        */
    int32_t fused;                   /* 1: the persistent fused kernel ran             */
    int32_t grid_ctas;               /* persistent CTAs (one per SM)                   */
    int32_t launches_per_step;       /* kernel launches per step (1)                   */
    int32_t barriers_per_step;       /* grid-wide barriers per step                    */
} mk_stats;

typedef struct mk_state mk_state;

/* Validate the description, check the device (compute capability 10.3, all
 * persistent CTAs co-resident), build TMA descriptors for every weight matrix,
 * precompute the RoPE table (fp64 on the host, stored fp32) and allocate the
 * workspace.  Weights must stay valid until mk_destroy.  On success *out owns
 * the state.  Errors: MK_ERR_INVALID, MK_ERR_UNSUPPORTED, MK_ERR_NOMEM, MK_ERR_CUDA.
 * Passage: ezolabs "DeepSeek-V4.1-Flash breaks 1,000 tokens per second for one
 * user", section "What NVIDIA shipped, and why B300 was refused": the megakernel
 * keeps one persistent block per SM and refuses an SM count it was not built
 * for rather than falling back; here a device other than CC 10.3, or a grid
 * that cannot be fully co-resident, returns MK_ERR_UNSUPPORTED. */
mk_status mk_create(const mk_model_desc *desc, const mk_weights *weights, mk_state **out);

/* One verify step for one stream.
 *   draft_tokens  dev int32 [T]: d_0 (last accepted token) then the k drafts
 *   positions     dev int32 [T]: must be ctx, ctx+1, ..., ctx+T-1
 *   kv            cache (its page table row 0 is used)
 *   out_logits    dev float32 [T][vocab]
 *   out_accepted  dev int32 [1]: n = longest prefix of drafts with d_i = argmax_{i-1}
 *   out_argmax    dev int32 [T] or NULL
 * Requires vocab > 0 and 1 <= T <= max_T.  Device-side errors
 * (MK_ERR_BAD_INPUT, MK_ERR_TIMEOUT, MK_ERR_RANGE) land in the status word.
 * Passages: al-engr "Why one GB300 doesn't beat 4x RTX PRO 6000 at
 * single-stream decode", section "The decomposition" (tokens per verify step =
 * accepted drafts + 1, so the step reports the accepted-prefix count n and the
 * argmax a_n that becomes the next d_0), and section "Where the 11.2 ms goes"
 * (the per-step work -- 43 MoE layers, decode attention, dense projections,
 * router top-k, lm_head and the rejection kernel -- that this one launch
 * replaces); ezolabs, section "How we got here" (drafted tokens are verified
 * together in one block). */
mk_status mk_decode_step(mk_state *st, const int32_t *draft_tokens, int T,
                         const int32_t *positions, const mk_kv_cache *kv,
                         float *out_logits, int32_t *out_accepted, int32_t *out_argmax,
                         void *stream);

/* mk_decode_step with verification by sampling at temperature t (top-p 1)
 * instead of by argmax.  The drafts are taken as greedy proposals (a point
 * mass on each draft), for which speculative sampling accepts draft d_i with
 * probability p_{i-1}(d_i), p_i = softmax(logits_i / t):
 *   uniforms      dev float32 [T], each in [0, 1): draft i is accepted while
 *                 every earlier one was and uniforms[i-1] < p_{i-1}(d_i)
 *                 (i = 1..T-1); uniforms[T-1] draws the emitted token
 *   out_accepted  dev int32 [1]: n, the accepted drafts
 *   out_token     dev int32 [1]: the token emitted after d_1..d_n, drawn by
 *                 inverse CDF in token-id order from p_n without d_{n+1} (renormalised)
 *                 after a rejection, or from p_{T-1} when every draft was accepted
 *   out_logits    as mk_decode_step (before the temperature)
 * The probabilities are formed in float32 (maxima and sums of exp over the
 * vocabulary slices, combined in a fixed order).  temperature must lie in
 * [1e-3, 1e3] (else MK_ERR_INVALID).  The emitted tokens are distributed as
 * sampling the model one token at a time.
 * Passage: ezolabs, section "Appendix: method", Decode speed (temperature 1.0,
 * top-p 1.0); section "How we got here" (block verification). */
mk_status mk_decode_step_sample(mk_state *st, const int32_t *draft_tokens, int T,
                                const int32_t *positions, const mk_kv_cache *kv, float temperature,
                                const float *uniforms, float *out_logits, int32_t *out_accepted,
                                int32_t *out_token, void *stream);

/* One verify step for each of n_streams independent streams (the concurrency
 * workload): stream s has its own block of T tokens, positions ctx_s .. ctx_s+T-1
 * and page-table row s of kv.
 *   draft_tokens  dev int32 [n_streams][T]
 *   positions     dev int32 [n_streams][T]
 *   out_logits    dev float32 [n_streams][T][vocab]
 *   out_accepted  dev int32 [n_streams]
 *   out_argmax    dev int32 [n_streams][T] or NULL
 * Each stream's results are bit for bit those of mk_decode_step on that stream
 * alone.  This build runs the streams one after another on `stream` (one launch
 * per stream, each streaming the weights once); each counts as one step in
 * mk_get_stats.  Requires vocab > 0, 1 <= T <= max_T, n_streams >= 1 and a page
 * table with at least n_streams rows.
 * Passage: ezolabs, section "Speed", table "Gain by number of streams" (the
 * megakernel measured at 1 to 16 concurrent streams). */
mk_status mk_decode_batch(mk_state *st, int n_streams, const int32_t *draft_tokens, int T,
                          const int32_t *positions, const mk_kv_cache *kv, float *out_logits,
                          int32_t *out_accepted, int32_t *out_argmax, void *stream);

/* The same step through HOST buffers: copies the tokens and positions in, runs
 * the step, copies the results out and synchronizes the stream.  out_logits and
 * out_argmax may be NULL.  Returns the device status of the step.
 * Passage: as mk_decode_step; this is the end-to-end form a serving loop calls
 * (al-engr, section "The decomposition": tokens/s counts whole verify steps). */
mk_status mk_decode_step_host(mk_state *st, const int32_t *h_tokens, int T,
                              const int32_t *h_positions, const mk_kv_cache *kv,
                              float *h_logits, int32_t *h_accepted, int32_t *h_argmax,
                              void *stream);

/* One decoder layer on a given hidden state (no embedding, LM head or accept).
 *   hidden_in, hidden_out  dev float32 [T][H] (may not alias)
 *   out_topk_idx           dev int32 [T][top_k] or NULL (selected experts, key order)
 *   out_topk_w             dev float32 [T][top_k] or NULL (their weights)
 * K/V of the T tokens are written into layer `layer` of the cache.
 * Passage: al-engr, section "Where the 11.2 ms goes", kernel table (per layer:
 * q/kv norm, RoPE and KV insert, decode attention, dense projections, router
 * top-k, MoE experts); section "Tier 2: the fusion program" (one persistent
 * kernel per decoder layer). */
mk_status mk_layer_forward(mk_state *st, int layer, const float *hidden_in, int T,
                           const int32_t *positions, const mk_kv_cache *kv,
                           float *hidden_out, int32_t *out_topk_idx, float *out_topk_w,
                           void *stream);

/* mk_layer_forward without a state and without any device allocation.
 *
 * For callers that cannot call cudaMalloc: a runtime without a device
 * allocator, a host application that owns all device memory, or code that must
 * not allocate once serving has started (allocation can block, fragment the
 * pool or fail under memory pressure).  The pages have no counterpart: it is
 * an integration entry point.
 *
 * Runs one decoder layer with the weights lw, exactly as mk_layer_forward does
 * (same kernel, same results), for a model described by desc (n_layers is
 * ignored).  The KV pools, page table and positions are the caller's as in
 * mk_layer_forward.  ctx must equal positions[0]: the host stages the RoPE
 * rows of positions ctx .. ctx+T-1 only, and the kernel refuses a launch whose
 * positions[0] differs (MK_ERR_BAD_INPUT in out_status, before any stage runs).
 * All other state -- the model block, TMA descriptors, RoPE rows, control block
 * and accumulators -- lives in one file-scope device array of 24 MiB that every
 * device which loads this library holds until the process exits.  A model whose
 * working set does not fit returns MK_ERR_UNSUPPORTED (a layer of hidden 4096,
 * 32/4 heads of 128, 384 experts of width 512 takes about 23 MiB).  out_status
 * (dev int32 [1], may be NULL) receives the device status (MK_OK,
 * MK_ERR_BAD_INPUT, MK_ERR_TIMEOUT or MK_ERR_RANGE) in stream order.
 *
 * The first call on a device does that device's set-up (finding the array's
 * device address, the kernel's shared-memory attribute); make it with the
 * device current.  Each call stages its tables into the array with
 * stream-ordered copies from host memory, so it must not be made while
 * `stream` is being captured into a CUDA graph: it returns MK_ERR_UNSUPPORTED
 * then.  Every call reuses the same array, so calls that may overlap on the
 * device (different streams without ordering, several host threads) race and
 * give wrong results: serialise them.  Each call clears the control block it
 * needs; nothing else must start at zero.  No call allocates device or host
 * memory.  It takes no KV scales, so a model with an FP8 KV cache
 * (kv_dtype MK_DT_FP8E4M3) returns MK_ERR_UNSUPPORTED. */
mk_status mk_layer_forward_noalloc(const mk_model_desc *desc, const mk_layer_weights *lw,
                                   void *k_pool, void *v_pool, const int32_t *page_table,
                                   int n_pages, const float *hidden_in, int T, int ctx,
                                   const int32_t *positions, float *hidden_out,
                                   int32_t *out_topk_idx, float *out_topk_w,
                                   int32_t *out_status, void *stream);

/* Record, on every later mk_decode_step, each layer's selected experts into
 * idx_trace (dev int32 [n_layers][T][top_k], key order) and their normalised
 * weights into w_trace (dev float32 [n_layers][T][top_k]); either may be NULL,
 * both NULL turns tracing off.  The buffers must stay valid while tracing is
 * on.  Used to check routing layer by layer against a reference.
 * Passage: al-engr, section "Where the 11.2 ms goes" (the router top-k runs
 * once per layer); the router's selection and weights are the quantities the
 * per-layer check compares. */
mk_status mk_set_routing_trace(mk_state *st, int32_t *idx_trace, float *w_trace);

/* Timeline of later launches: for every CTA c and grid barrier b < capacity,
 * times[(c*capacity + b)*2] is the %globaltimer value (ns) when the CTA arrived
 * and times[... + 1] when it left the barrier (dev uint64 [grid][capacity][2],
 * grid = mk_stats.grid_ctas).  NULL turns it off.  Stage s of a step runs
 * between barriers s-1 and s, so this splits the single launch into stages.
 * events (dev uint64 [grid][1024][2], or NULL) receives (event id, time) pairs
 * at points inside the stages: id = stage*16 + k, k = 0 inputs staged, 1 first
 * weight tile arrived, 2 last tile reduced, 3 routing started, 5 stage code
 * entered, 6 activation fragments built, 7 first tile wait begins (attention:
 * 0 queries ready, 1 pages done, 2 group barrier passed, 3 merge done).
 * Passage: al-engr, section "Where the 11.2 ms goes" (a per-kernel time budget
 * of one step); with one launch per step the budget has to come from inside
 * the kernel. */
mk_status mk_set_stage_trace(mk_state *st, uint64_t *times, int capacity, uint64_t *events);

/* Test hook for the failure path: on every later launch, CTA 0 does not arrive
 * at grid barrier `barrier` (1-based, in launch order; 0 turns the hook off).
 * The other CTAs' waits then run out after timeout_ms, the launch ends with
 * MK_ERR_TIMEOUT in the device status and every CTA returns; nothing traps or
 * hangs.  mk_reset (with the hook off) restores a working state.
 * Passage: ezolabs, section "The safety layer" (a watchdog restarts an engine
 * whose megakernel stalls); here every device wait is bounded instead and a
 * stall becomes a status. */
mk_status mk_debug_skip_barrier(mk_state *st, int barrier);

/* Synchronize the last stream used and return the device status of the last
 * step (MK_OK, MK_ERR_TIMEOUT, MK_ERR_BAD_INPUT or MK_ERR_RANGE).
 * Passage: ezolabs, section "The safety layer" (stalls and divergence are
 * detected and reported instead of passing silently). */
mk_status mk_get_status(mk_state *st);

/* Synchronize and copy the counters.
 * Passage: ezolabs, section "What NVIDIA shipped" (callers on the old interface
 * silently ran the unfused path; `fused` and `launches_per_step` let a caller
 * check that the fused kernel ran) and al-engr, section "The decomposition"
 * (accepted_sum / steps + 1 is the tokens-per-step factor). */
mk_status mk_get_stats(mk_state *st, mk_stats *out);

/* Clear the device status, barrier epochs and counters (synchronous).
 * Passage: ezolabs, section "The safety layer" (recovery after a stall). */
mk_status mk_reset(mk_state *st);

/* Free the workspace.  Safe on NULL. */
void mk_destroy(mk_state *st);

/* Static text for a status code. */
const char *mk_status_string(mk_status s);

/* Text of the last host-side error of this state (a buffer inside the state);
 * with st == NULL, the reason the calling thread's last mk_create failed. */
const char *mk_last_error(const mk_state *st);

#ifdef __cplusplus
}
#endif
#endif /* MK_H */
