/*
 * moe.h -- C ABI of the top-k gated Mixture-of-Experts FFN layer, forward pass,
 * for one NVIDIA GB300 GPU (sm_103a).
 *
 * The layer (sources: "Qwen2-MoE代码解析：MoE架构原理、工程实现与部署避坑指南",
 * jsqmd.com, sections 3.1, 3.3, 3.4; the Qwen2-MoE module article, mlqm.cn,
 * sections 2.2 and 3.2; the MoE sparse-activation article, wmrh.cn, section 2.2):
 *
 *   l      = x Wg^T (+ gate_bias)                      router scores      [T, E]
 *   p      = softmax(l)                                                   [T, E]
 *   ids    = top-k of l, largest first, ties to the lower expert index    [T, K]
 *   w      = p[ids] / sum_j p[ids_j]                   renormalised       [T, K]
 *   group slots s = t*K + j by expert, stable in s; keep the first
 *   `capacity` slots of each expert (capacity <= 0: keep all)
 *   y_s    = W2[e] GELU(W1[e] x_t (+ b1[e])) (+ b2[e]) for kept slot s of expert e
 *   out[t] = sum_j w[t,j] * y_{t*K+j}   (dropped slots add nothing)
 *   aux    = E * sum_i (count_i / (T*K)) * (sum_t p[t,i] / T)
 *
 * Conventions for every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller, dense and
 *     row-major, 16-byte aligned, unless a call says otherwise.  Weights are
 *     read-only.  The library keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on it: they enqueue kernels and return.  They never
 *     allocate device memory and never synchronise, except moe_get_device_error.
 *   - `ws` is a caller-owned device workspace of at least moe_workspace_size()
 *     bytes, 256-byte aligned.  Calls that overlap on the GPU must not share one.
 *   - Return value: MOE_OK (0) or a negative moe_status.  Arguments are checked
 *     on the host before any launch; on error nothing is enqueued, except for
 *     MOE_ERR_CUDA (a launch failed; outputs are undefined).
 *   - Element types follow desc->dtype: MOE_BF16 -> x, Wg, W1, W2, x_perm,
 *     h_perm, y_perm and out are bf16; MOE_F32 -> all of them are fp32.
 *     Router logits, routing weights, biases and the loss are always fp32;
 *     indices and counts are int32.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID = -1,      /* bad argument: null pointer, shape, alignment */
  MOE_ERR_UNSUPPORTED = -2,  /* valid layer the library does not implement   */
  MOE_ERR_WORKSPACE = -3,    /* ws is NULL or smaller than moe_workspace_size */
  MOE_ERR_CUDA = -4,         /* a CUDA runtime / driver call failed          */
  MOE_ERR_TIMEOUT = -5,      /* a kernel gave up a bounded wait (device flag) */
  MOE_ERR_DEVICE = -6        /* a kernel's own bounds check fired (device flag) */
} moe_status;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* desc->flags bits */
#define MOE_FLAG_HOST_IO    (1u << 0) /* moe_layer_forward: x and out are host pointers */
#define MOE_FLAG_SIMT_FFN   (1u << 1) /* bf16: CUDA-core expert FFN instead of tensor cores (testing) */
#define MOE_FLAG_NO_DECODE  (1u << 2) /* never take the small-batch weight-streaming FFN */
#define MOE_FLAG_SIMT_ROUTER (1u << 3) /* bf16: CUDA-core router instead of tensor cores (testing) */
#define MOE_FLAG_GEMM_SINGLE (1u << 4) /* bf16: 128x256 single-SM expert GEMM tiles */
#define MOE_FLAG_GEMM_PAIR   (1u << 5) /* bf16: 256x256 tiles on SM pairs (cta_group::2) */
#define MOE_FLAG_SWIGLU      (1u << 6) /* experts are W2 (SiLU(W1 x) * W3 x); see moe_expert_ffn */
/* Testing only: with MOE_FLAG_GEMM_SINGLE, every CTA of the first expert
 * product withholds its first operand load, so the MMA's bounded wait runs
 * out (about 2 s): the kernel records MOE_ERR_TIMEOUT in the workspace error
 * word, drains the loads it issued, frees its tensor memory and returns;
 * outputs are undefined.  It exercises the timeout path without a fault. */
#define MOE_FLAG_TEST_WAIT_TIMEOUT (1u << 7)
/* bf16 with SM pairs: every block of an expert's token rows runs with the
 * rows on the MMA's M side (padded to 256), instead of the default where an
 * expert's last, short block runs swapped (rows on the N side, padded to
 * 16).  Same results; for comparing the two (testing). */
#define MOE_FLAG_GEMM_ROWS   (1u << 8)
/* Run the two expert products as two launches.  By default one persistent
 * launch runs both.  On SM pairs a tile of the second product starts as
 * soon as the first product has written every hidden column of its 256-row
 * block, so the second product's tiles fill the first one's tail; in the
 * weight-streaming kernel of decode-sized batches the second product's
 * weights stream right behind the first's through the same ring, and its
 * activation rows load once every CTA of the expert has stored its share.
 * Same results; for comparing the two (testing). */
#define MOE_FLAG_FFN_SPLIT   (1u << 9)
/* drop_tokens = False (the Qwen2-MoE walkthrough, jsqmd.com, section 3.4:
 * tokens over an expert's capacity go to the next-best expert instead of
 * being dropped).  With a capacity, moe_layer_forward keeps the slots the
 * capacity keeps and moves each other slot, in slot order, to the
 * best-scored expert its token does not use yet that still has room (see
 * moe_reroute); a moved slot keeps its routing weight.  `count` and the loss
 * stay those of the routing's own choices; `dropped` counts the slots left
 * without an expert.  No effect without a capacity. */
#define MOE_FLAG_REROUTE     (1u << 10)
/* bf16, K <= 2, SM-pair expert GEMMs: moe_layer_forward folds the weighted
 * combine into the second expert product's epilogue (each output row adds
 * w * y, with y rounded to bf16 as stored, to an fp32 copy of out in the
 * workspace with vector reductions; two additions onto zero give the same
 * sum in either order, so the result is deterministic), then converts it to
 * out.  y_perm is not written.  Ignored where it does not apply.  For
 * comparing the two (the MoE sparse-activation article, wmrh.cn, section
 * 4.3, on the dispatcher's memory traffic). */
#define MOE_FLAG_FUSED_COMBINE (1u << 11)
/* bf16 batches of at most 16 tokens: moe_layer_forward runs the layer as
 * its separate steps (router, dispatch, weight-streaming expert products,
 * combine: four launches) instead of the default one-launch decode layer,
 * in which one grid with every CTA resident computes the gate scores,
 * routes and places every token in each CTA, spreads the used experts'
 * weight rows evenly over the CTAs and combines, with counters in the
 * workspace between the steps.  Same results, bit for bit; for comparing
 * the two (testing). */
#define MOE_FLAG_DECODE_SPLIT  (1u << 12)
/* bf16 layers on the SM-pair expert GEMMs, without MOE_FLAG_REROUTE:
 * moe_layer_forward runs no gather of x rows; the first expert product
 * copies each kept row's token row from x itself (slot s = src[r] of kept
 * row r is token s / K; Qwen2-MoE walkthrough, jsqmd.com, section 3.1 item
 * 3, grouping without a host-side sort), so x_perm is never written.  Same
 * results, bit for bit.  Ignored where it does not apply. */
#define MOE_FLAG_GATHER_GEMM   (1u << 13)

/*
 * Layer description.  Field names follow the Qwen2MoEConfig fields of the
 * Qwen2-MoE module article (mlqm.cn), section 2.2: E = num_experts,
 * K = num_experts_per_tok, capacity = expert_capacity.
 * Limits: T >= 0; 1 <= K <= 8; K <= E <= 256; H, F >= 8 and multiples of 8;
 * T * K < 2^31.
 * temperature: the router softmax is taken of l / temperature (the MoE
 * sparse-activation article, wmrh.cn, section 5.2: 1.0 by default, 2.0
 * flattens, 0.5 sharpens).  It changes the routing weights and the
 * load-balancing probabilities, not which experts are chosen.  <= 0 means 1;
 * NaN or infinity is MOE_ERR_INVALID.
 */
typedef struct moe_desc {
  int64_t T;         /* tokens (batch * sequence, flattened)                 */
  int32_t H;         /* hidden size                                          */
  int32_t E;         /* number of experts                                    */
  int32_t K;         /* experts chosen per token (top-k)                     */
  int32_t F;         /* expert FFN width                                     */
  int32_t capacity;  /* slots kept per expert; <= 0 means no limit           */
  int32_t dtype;     /* moe_dtype                                            */
  uint32_t flags;    /* MOE_FLAG_*                                           */
  float temperature; /* router softmax temperature; <= 0 means 1             */
} moe_desc;

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(int status);

/* ceil(T / E) * K, the expert_capacity of the Qwen2-MoE module article
 * (mlqm.cn), section 2.2.  Returns -1 if E <= 0 or K <= 0. */
int64_t moe_capacity_default(int64_t T, int32_t E, int32_t K);

/* Rows of the permuted buffers (x_perm, h_perm, y_perm) needed for `desc`:
 * min(T*K, E*capacity) with a capacity, else T*K.  -1 if desc is invalid. */
int64_t moe_max_rows(const moe_desc* desc);

/* Bytes of device workspace every call below needs for `desc` (the same value
 * for all of them).  It holds routing results, dispatch tables, the permuted
 * activations and a device error word.  Returns MOE_ERR_INVALID for a bad desc. */
int moe_workspace_size(const moe_desc* desc, size_t* bytes);

/*
 * Router: gate linear, softmax, top-k, renormalisation (jsqmd.com section 3.1:
 * `gate` is nn.Linear(hidden, num_experts, bias=False), then F.softmax,
 * torch.topk and the division by the sum of the k weights; mlqm.cn section 3.2
 * steps 1-2).
 *   x         [T, H]  dtype
 *   Wg        [E, H]  dtype (nn.Linear [out, in] layout)
 *   gate_bias [E] fp32 or NULL (added to the scores; the pages' gate has none)
 *   logits    [T, E] fp32 out, or NULL: the scores l, fp32-accumulated (before
 *             the temperature is applied)
 *   ids       [T, K] int32 out: chosen experts, largest score first, equal
 *             scores ordered by ascending expert index
 *   w         [T, K] fp32 out: p[ids] / sum_j p[ids_j]  (sum to 1), with
 *             p = softmax(l / temperature)
 *   psum      [E] fp32 out, or NULL: sum over tokens of p[t, e], summed in a
 *             fixed order (deterministic)
 */
int moe_router_topk(const moe_desc* desc, const void* x, const void* Wg,
                    const float* gate_bias, float* logits, int32_t* ids,
                    float* w, float* psum, void* ws, size_t ws_bytes,
                    void* stream);

/*
 * Dispatch: group the T*K slots by expert (jsqmd.com section 3.1 item 3:
 * scatter + argsort by expert id) with the capacity rule of jsqmd.com section
 * 3.4 (tokens over an expert's capacity are dropped).  Slot s = t*K + j.
 * Within an expert, slots keep ascending s order, so with a capacity the
 * earliest tokens are kept.
 *   ids     [T, K] int32 in (each value in [0, E), or -1 for a slot with no
 *           expert, which is dropped; a token's other ids distinct)
 *   x       [T, H] dtype in, or NULL to skip the gather
 *   count   [E]    int32 out: slots routed to each expert, before dropping
 *   offs    [E+1]  int32 out: first permuted row of each expert; offs[E] = rows
 *   src     [moe_max_rows] int32 out: slot held by permuted row r (r < offs[E])
 *   pos     [T*K]  int32 out: permuted row of slot s, or -1 if dropped
 *   x_perm  [moe_max_rows, H] dtype out (if x != NULL): x_perm[r] = x[src[r] / K]
 *   dropped [1]    int32 out, or NULL: number of dropped slots
 * Out-of-range ids make the kernel set MOE_ERR_DEVICE in the workspace error
 * word (read it with moe_get_device_error); such slots are dropped.
 */
int moe_dispatch(const moe_desc* desc, const int32_t* ids, const void* x,
                 int32_t* count, int32_t* offs, int32_t* src, int32_t* pos,
                 void* x_perm, int32_t* dropped, void* ws, size_t ws_bytes,
                 void* stream);

/*
 * moe_dispatch without a workspace, for callers that cannot allocate device
 * memory where they route tokens: code running inside an allocator or memory-
 * pool callback, runtimes that reserve all device memory up front, plugin hosts
 * that forbid allocation on their execution path.  The pages have no
 * counterpart; this is a library convenience.
 *   Same arguments and results as moe_dispatch, minus ws/ws_bytes, plus
 *   device_error [1] int32 (device, or NULL): cleared by the call, then set to
 *   a nonzero code if an id is out of range (such slots are dropped).
 * The per-block histograms live in a 64 KiB array in device memory owned by
 * the library (held by every GPU that loads it until the process exits).  The
 * layer must fit it: E * blocks <= 8192, where for S = T*K slots
 * blocks = ceil(S / b), b = max(2048, ceil(S / 64)) rounded up to a multiple
 * of 256 (so at most 64 blocks: E <= 128 always fits, E = 256 up to
 * S = 65536); larger layers get MOE_ERR_UNSUPPORTED.  The call allocates
 * nothing.  Each call outside stream capture looks up the array's address on
 * the current device; a call during capture reuses the last one, so make the
 * first call on each device before any stream capture (and one more after a
 * device reset).  All calls on a device share the array: calls that overlap
 * on the GPU race and must be serialised by the caller.
 */
int moe_dispatch_noalloc(const moe_desc* desc, const int32_t* ids, const void* x,
                         int32_t* count, int32_t* offs, int32_t* src, int32_t* pos,
                         void* x_perm, int32_t* dropped, int32_t* device_error,
                         void* stream);

/*
 * Move the slots a capacity-limited dispatch dropped (drop_tokens = False;
 * the Qwen2-MoE walkthrough, jsqmd.com, section 3.4: tokens over capacity are
 * routed to the next-best expert instead of being dropped).  The slots the
 * capacity kept stay.  The others are taken one at a time in slot order
 * s = t*K + j; each goes to the expert with the highest score logits[t, e]
 * (equal scores: the lower index) that token t uses neither among its K
 * choices nor as the target of an earlier move, and that still has room
 * (capacity minus the slots it holds so far); if none has, the slot is
 * dropped.  The result equals that one-at-a-time walk exactly.
 *   logits  [T, E] fp32 in: the router's scores (moe_router_topk's logits)
 *   ids     [T, K] int32 in: the routing
 *   pos     [T*K]  int32 in: moe_dispatch's pos for ids with desc->capacity
 *                  (pos < 0: over capacity)
 *   offs    [E+1]  int32 in: moe_dispatch's offs for the same call
 *   ids_out [T, K] int32 out: each slot's expert after the moves, -1 if dropped
 *   dropped [1]    int32 out, or NULL: slots left without an expert
 * Dispatching ids_out again (moe_dispatch accepts -1 as "no expert") groups
 * the moved routing; no expert exceeds the capacity any more.  One block does
 * the walk: meant for capacities that drop a minority of the slots.
 */
int moe_reroute(const moe_desc* desc, const float* logits, const int32_t* ids, const int32_t* pos,
                const int32_t* offs, int32_t* ids_out, int32_t* dropped, void* ws, size_t ws_bytes,
                void* stream);

/*
 * Expert FFN over the permuted rows: for each expert e and each row r in
 * [offs[e], offs[e+1]):
 *   h_perm[r] = GELU(W1[e] x_perm[r] + b1[e])       (GELU erf form)
 *   y_perm[r] = W2[e] h_perm[r] + b2[e]
 * (mlqm.cn section 2.2: every expert is Linear - GELU - Linear).  On the bf16
 * path the products are accumulated in fp32 and h and y are rounded to bf16.
 *   x_perm [rows, H] dtype in; offs [E+1] int32 in (device; read on device only)
 *   W1 [E, F, H] dtype; W2 [E, H, F] dtype (nn.Linear [out, in] layout)
 *   b1 [E, F] fp32 or NULL; b2 [E, H] fp32 or NULL
 * With MOE_FLAG_SWIGLU the experts have three matrices W1, W2, W3 (the
 * Qwen2-MoE walkthrough, jsqmd.com, section 4.6), read as
 *   h_perm[r] = SiLU(W1[e] x + b1[e][:F]) * (W3[e] x + b1[e][F:])
 * and the W1 argument holds W1 and W3 stacked per expert: [E, 2F, H] (rows
 * 0..F-1 = W1, rows F..2F-1 = W3); b1 is then [E, 2F].
 *   h_perm [moe_max_rows, F] dtype out (intermediate, kept for inspection)
 *   y_perm [moe_max_rows, H] dtype out
 * bf16 with K-major operands runs on the tcgen05 tensor cores, either as
 * 128x256 tiles per SM or as 256x256 tiles per SM pair (chosen from the shape
 * unless a MOE_FLAG_GEMM_* flag forces one); fp32 runs on CUDA cores; T <= 16
 * runs a weight-streaming kernel (unless MOE_FLAG_NO_DECODE).
 */
int moe_expert_ffn(const moe_desc* desc, const void* x_perm, const int32_t* offs,
                   const void* W1, const float* b1, const void* W2, const float* b2,
                   void* h_perm, void* y_perm, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * Combine: out[t] = sum_{j=0..K-1} w[t,j] * y_perm[pos[t*K+j]], summed in fp32
 * in the order j = 0..K-1, then stored in dtype; slots with pos < 0 add
 * nothing (jsqmd.com section 3.1 item 2; wmrh.cn section 2.2).  No residual.
 *   y_perm [rows, H] dtype; pos [T*K] int32; w [T, K] fp32; out [T, H] dtype
 */
int moe_combine(const moe_desc* desc, const void* y_perm, const int32_t* pos,
                const float* w, void* out, void* stream);

/*
 * Load-balancing loss (jsqmd.com section 3.3):
 *   loss = E * sum_i f_i * P_i,  P_i = psum[i] / T,  f_i = count[i] / (T*K).
 * The raw value is returned; the caller scales it by router_aux_loss_coef.
 *   psum [E] fp32; count [E] int32; loss [1] fp32 out (device)
 */
int moe_aux_loss(const moe_desc* desc, const float* psum, const int32_t* count,
                 float* loss, void* stream);

/*
 * The whole layer: router -> dispatch -> expert FFN -> combine (+ aux loss),
 * enqueued on one stream with no host synchronisation (mlqm.cn section 3.2).
 *   x [T, H], out [T, H] dtype: device pointers, or host pointers if
 *     desc->flags has MOE_FLAG_HOST_IO (then the call copies x in and out
 *     through the workspace; pinned host memory is fastest, and `out` is
 *     valid once `stream` has been synchronised).  With host pointers, no
 *     capacity and T >= 2048, the batch runs as two halves of tokens whose
 *     copies overlap the other half's layer (the second half's output is
 *     combined and copied back in two parts, the copy of the first part
 *     overlapping the combine of the second): the copies go on two internal
 *     streams (created on the first such call of each host thread on each
 *     device, kept until the process exits) joined to `stream` by events,
 *     the outputs are the same bits, and count and the loss are the whole
 *     batch's.
 *   aux [1] fp32 out or NULL; count [E] int32 out or NULL; dropped [1] int32
 *     out or NULL (device pointers)
 */
int moe_layer_forward(const moe_desc* desc, const void* x, const void* Wg,
                      const float* gate_bias, const void* W1, const float* b1,
                      const void* W2, const float* b2, void* out, float* aux,
                      int32_t* count, int32_t* dropped, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * How many kernels one moe_layer_forward with this description launches
 * (no counterpart on the pages; it lets a caller or a benchmark account for
 * the launches it issues).  Depends on the shape only: the path taken
 * (one-block or multi-block dispatch, router variant) is chosen from it.
 * Returns the count (>= 1), or a negative MOE_ERR_* for an invalid desc.
 */
int moe_layer_launches(const moe_desc* desc);

/*
 * Which expert-FFN kernel moe_expert_ffn and moe_layer_forward run for this
 * description (no counterpart on the pages; it lets a caller or a benchmark
 * account for the launches and attribute time).  Depends on the shape and
 * flags only.  Returns one of MOE_FFN_*, or a negative MOE_ERR_* for an
 * invalid desc.
 */
#define MOE_FFN_STREAM    0 /* weight streaming for decode-sized batches, both products in 1 launch */
#define MOE_FFN_SIMT      1 /* CUDA cores (f32, or forced): 2 launches */
#define MOE_FFN_TC_SINGLE 2 /* tensor cores, 128x256 tiles per SM: 2 launches */
#define MOE_FFN_TC_PAIRS  3 /* tensor cores on SM pairs, one launch per product: 2 launches */
#define MOE_FFN_TC_FUSED  4 /* tensor cores on SM pairs, both products in 1 launch */
#define MOE_FFN_STREAM_SPLIT 5 /* weight streaming, one launch per product: 2 launches */
int moe_ffn_kernel(const moe_desc* desc);

/*
 * Whether moe_layer_forward runs this description as the one-launch decode
 * layer (see MOE_FLAG_DECODE_SPLIT): 1 if it does (two launches: its
 * counters zeroed, then the layer), 0 if it runs the separate steps, or a
 * negative MOE_ERR_* for an invalid desc.  No counterpart on the pages; it
 * lets a benchmark attribute the time.  Depends on the shape and flags only.
 */
int moe_layer_decode_fused(const moe_desc* desc);

/*
 * Stage timing for moe_layer_forward on the calling host thread (no
 * counterpart on the pages; a tracing aid in the spirit of the profiler runs
 * they describe).  `events` holds 6 cudaEvent_t created by the caller; each
 * later moe_layer_forward on this thread records them on its stream at the
 * stage boundaries: [0] start, [1] router done, [2] dispatch done, [3] first
 * expert product done, [4] second product done, [5] combine done.
 * events = NULL or n = 0 switches it off.  MOE_ERR_INVALID if n < 6 or an
 * event is NULL.
 */
int moe_profile_events(void* const* events, int n);

/*
 * Read and clear the workspace's device error word.  Synchronises `stream`.
 * *code receives MOE_OK, MOE_ERR_TIMEOUT (a tensor-core kernel gave up a
 * bounded wait) or MOE_ERR_DEVICE (an index check fired).  Returns MOE_OK or
 * MOE_ERR_CUDA.
 */
int moe_get_device_error(void* ws, int32_t* code, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
