/*
 * moe.h — C ABI of the single-GPU MoE FFN layer forward (B300, sm_103a).
 *
 * The layer, as the pages define it:
 *   router logits  l = x·W_g                       [Lesson 10 "专家并行 EP", §1]
 *   scores         Softmax(TopK(l, K)), or sigmoid  [Lesson 10 §1]
 *                  (optionally a selection-only per-expert bias  [Chương 10 "Song song MoE", §4],
 *                   and a group limit: a unit's K experts lie in at most M groups  [Lesson 10 §5])
 *   capacity       C = CF·K·T/E, picks past C are dropped            [Lesson 10 §4]
 *   dispatch       pack the units per expert                          [Lesson 10 §3, step 1]
 *   expert FFN     per-expert grouped GEMM                            [Lesson 10 §3, step 2]
 *   combine        y = Σ_{i∈TopK} s_i(x)·FFN_i(x), back in token order [Lesson 10 §1, §3 steps 3-4]
 *   aux loss       L_aux = α·E·Σ_i f_i·P_i                             [Lesson 10 §4]
 *   heads          x split into H heads, each routed independently     ["Multi-Head LatentMoE 与
 *                                                                       Head 并行", 摘要 and 评论 §1]
 * The expert is a SwiGLU FFN without biases: FFN_e(x) = W2_e·(silu(W1_e·x) ⊙ W3_e·x).
 *
 * Conventions shared by every call
 *  - Ownership: the caller owns every buffer. All data pointers are DEVICE pointers (cudaMalloc'd
 *    or torch tensors) unless a comment says otherwise. The library allocates no device memory
 *    and frees none; scratch lives in the caller's workspace `ws` (size from
 *    moe_workspace_size, 256-byte aligned, zeroed once by moe_workspace_init).
 *  - Asynchrony: every compute call only enqueues kernels on `stream` and returns; it never
 *    synchronises. moe_get_status is the one call that waits for the stream.
 *  - Errors: invalid arguments are reported synchronously (MOE_ERR_INVALID_ARG /
 *    MOE_ERR_UNSUPPORTED) and then nothing is enqueued. Faults the kernels detect in the data
 *    (an expert index out of range, inconsistent offsets, a wait that timed out) set bits in a
 *    status word inside `ws`; moe_get_status reports them. A kernel launch failure returns
 *    MOE_ERR_CUDA.
 *  - Layouts are row-major. A "unit" is a token (n_heads == 1) or a head sub-token: with H heads,
 *    x[T][h] is read as T' = T·H units of width h' = h/H, unit t·H+j = x[t][j·h' .. (j+1)·h').
 *    GEMM operands are K-major: W_gate/W_up [E][d_ff][h'], W_down [E][h'][d_ff]. The router weight
 *    keeps the pages' x·W_g orientation: W_g [h'][E].
 *  - dtype MOE_BF16: x, W_g, W_gate, W_up, W_down, x_packed, y_packed and y are bf16 (uint16
 *    storage); accumulation is fp32. dtype MOE_F32: all of those are fp32. Biases, logits, gates
 *    and the aux loss are fp32 in both.
 *  - Thread safety: the library keeps no per-call state; concurrent calls need separate workspaces.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

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

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* a config field or pointer is invalid; nothing was enqueued     */
  MOE_ERR_UNSUPPORTED = 2,   /* valid for the method but not for this library (e.g. E > 256)   */
  MOE_ERR_WORKSPACE = 3,     /* ws is NULL or not 256-byte aligned                             */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed                     */
  MOE_ERR_DEVICE_STATUS = 5, /* a kernel found bad data (index/offsets out of range)            */
  MOE_ERR_TIMEOUT = 6        /* a kernel wait gave up after its time limit                      */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* Softmax: TopK ranks the logits, gates = softmax over the K picked logits.
 * Sigmoid: TopK ranks σ(l) + select_bias (formed in fp64), gates = σ(l_i) / Σ_picked σ(l_j). */
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;

typedef struct {
  int64_t T;               /* tokens (>= 0)                                                      */
  double capacity_factor;  /* CF; <= 0 or +inf = no drop                                         */
  int32_t h;               /* token width, all heads                                             */
  int32_t E;               /* experts, 1..256                                                    */
  int32_t K;               /* experts per unit, 1..min(E, 8)                                     */
  int32_t d_ff;            /* expert hidden width                                                */
  int32_t n_heads;         /* H >= 1; H > 1 routes T·H sub-tokens of width h/H                  */
  int32_t n_groups;        /* expert groups for the group limit (1 = off), E % n_groups == 0     */
  int32_t topk_groups;     /* groups a unit may use (1..n_groups)                                */
  float aux_alpha;         /* α of the aux loss (0.01 in the pages' HAI-LLM config)              */
  int32_t score;           /* moe_score_t                                                        */
  int32_t dtype;           /* moe_dtype_t                                                        */
} moe_config_t;

/* Weights of one layer (device pointers). logit_bias / select_bias may be NULL. */
typedef struct {
  const void* w_router;    /* W_g [h'][E]                                                        */
  const float* logit_bias; /* [E] added to the logits (affects selection, gates and P_i)         */
  const float* select_bias;/* [E] sigmoid scoring only: added to σ(l) for selection alone        */
  const void* w_gate;      /* W1 [E][d_ff][h']                                                   */
  const void* w_up;        /* W3 [E][d_ff][h']                                                   */
  const void* w_down;      /* W2 [E][h'][d_ff]                                                   */
} moe_weights_t;

/* Optional outputs of moe_forward (device pointers; each may be NULL). */
typedef struct {
  int32_t* topk_idx;       /* [T'][K] picked experts, descending key, ties to the lower index    */
  float* topk_gate;        /* [T'][K] gates                                                      */
  float* logits;           /* [T'][E] fp32 router logits (logit bias included)                   */
  int32_t* counts;         /* [E] pre-drop picks per expert                                      */
  int32_t* offsets;        /* [E+1] exclusive scan of kept rows per expert                       */
  int32_t* slot_of;        /* [T'][K] packed row of pick (t,k), -1 if dropped                    */
  float* aux;              /* [1] aux loss                                                       */
} moe_outputs_t;

/* Bytes of workspace the calls need for this config (host only; no GPU call). Returns 0 for an
 * invalid config. One workspace serves every call below for the same config. */
MOE_API size_t moe_workspace_size(const moe_config_t* cfg);

/* Zero the workspace's status header. Call once after allocating `ws`. Enqueued on `stream`. */
MOE_API moe_status_t moe_workspace_init(const moe_config_t* cfg, void* ws, moe_stream_t stream);

/* Capacity C = ceil(CF·K·T'/E) evaluated in fp64 in that order, or -1 for no drop;
 * -2 for an invalid config. [Lesson 10 §4] Host only. */
MOE_API int64_t moe_capacity(const moe_config_t* cfg);

/* Router + scoring + group limit + Top-K + gates (+ aux statistics).   [Lesson 10 §1, §4, §5]
 *  x [T][h] (dtype), w_router [h'][E] (dtype), logit_bias/select_bias [E] fp32 or NULL.
 *  Out: topk_idx [T'][K] int32, topk_gate [T'][K] fp32; logits_out [T'][E] fp32 or NULL;
 *  aux_out [1] fp32 or NULL (uses the pre-drop counts of these picks). */
MOE_API moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* logit_bias, const float* select_bias, int32_t* topk_idx,
                       float* topk_gate, float* logits_out, float* aux_out, void* ws,
                       moe_stream_t stream);

/* The same routing from given fp32 logits [T'][E] (no router GEMM): the logit bias, if any, is
 * added in fp32 before selection.                                       [Lesson 10 §1, §4, §5] */
MOE_API moe_status_t moe_route_logits(const moe_config_t* cfg, const float* logits, const float* logit_bias,
                              const float* select_bias, int32_t* topk_idx, float* topk_gate,
                              float* aux_out, void* ws, moe_stream_t stream);

/* Capacity drop + pack.                                                 [Lesson 10 §3 step 1, §4]
 *  topk_idx [T'][K] (each unit's K picks distinct, in [0,E)).
 *  Out: counts [E] pre-drop picks (or NULL); offsets [E+1] kept rows per expert, exclusive scan;
 *  slot_of [T'][K] packed row or -1 (dropped); row_token [T'·K] source unit of each packed row,
 *  -1 past offsets[E]; x_packed [T'·K][h'] rows of x in packed order (rows past offsets[E] are
 *  left untouched). Within an expert, rows are in unit order; pick (t,k) is dropped when t is at
 *  or past place C of its expert's queue. */
MOE_API moe_status_t moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                          int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* row_token,
                          void* x_packed, void* ws, moe_stream_t stream);

/* Dispatch of one shard of a batch split by tokens over several processes (a data-parallel layer
 * whose capacity and drop order are those of the whole batch).          [Lesson 10 §3 step 1, §4]
 * The shard holds cfg->T of the batch's T_global tokens; earlier shards hold the batch's earlier
 * tokens. queue_base [E] (device, int32): picks of each expert on all earlier shards — the exclusive
 * scan over shards of their pre-drop counts, the one exchange step (an all-gather of E int32 per
 * shard). The capacity is the whole batch's, C = ceil(CF·K·T'_global/E); a pick of this shard at
 * place p in its expert's local queue is kept iff queue_base[e] + p < C. Outputs as moe_dispatch,
 * local to the shard (counts are this shard's pre-drop counts; offsets scan this shard's kept
 * rows). queue_base = 0 and T_global = T is moe_dispatch. */
MOE_API moe_status_t moe_dispatch_sharded(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                                          const int32_t* queue_base, int64_t T_global, int32_t* counts,
                                          int32_t* offsets, int32_t* slot_of, int32_t* row_token, void* x_packed,
                                          void* ws, moe_stream_t stream);

/* Per-expert SwiGLU FFN over the packed rows (grouped GEMMs).           [Lesson 10 §3 step 2]
 *  x_packed [T'·K][h'], offsets [E+1] (device; offsets[0] == 0, non-decreasing,
 *  offsets[E] <= T'·K), w_gate/w_up [E][d_ff][h'], w_down [E][h'][d_ff].
 *  Out: y_packed [T'·K][h'] rows [offsets[e], offsets[e+1]) = FFN_e of the same rows of x_packed;
 *  rows past offsets[E] untouched. bf16: the hidden activation is rounded to bf16 once. */
MOE_API moe_status_t moe_expert_ffn(const moe_config_t* cfg, const void* x_packed, const int32_t* offsets,
                            const void* w_gate, const void* w_up, const void* w_down,
                            void* y_packed, void* ws, moe_stream_t stream);

/* Gate-weighted combine back to unit order.                             [Lesson 10 §1, §3 step 4]
 *  y[u] = Σ_k topk_gate[u][k]·y_packed[slot_of[u][k]] over k with slot_of >= 0, in k order,
 *  fp32 accumulation; y [T][h] (dtype; a unit with every pick dropped gets 0). */
MOE_API moe_status_t moe_combine(const moe_config_t* cfg, const void* y_packed, const int32_t* slot_of,
                         const float* topk_gate, void* y, void* ws, moe_stream_t stream);

/* The whole layer: route → dispatch → expert FFN → combine (+ aux). x [T][h] → y [T][h].
 * `out` may be NULL or have NULL members; intermediates live in `ws`.
 * With K == 1 (bf16, 16-byte aligned y) the combine is folded into the down GEMM: each kept row
 * writes g·Y straight into y, with moe_combine's arithmetic, so y has the same bits as
 * route → dispatch → expert_ffn → combine; y_packed is then not written (moe_forward_train still
 * writes it). moe_set_expert_gemm can fold it for K >= 2 as well, or not at all. */
MOE_API moe_status_t moe_forward(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                         const moe_outputs_t* out, void* ws, moe_stream_t stream);

/* ---- hash gate ------------------------------------------------------------------------------
 * HAI-LLM offers a HashGate beside its GShard and Switch gates, top_k == 1 only
 *   ["HAI-LLM MoE：一键实现大模型的混合专家并行训练", §"HAI-LLM 上的使用"]; the page says no more.
 * Here a hash gate has no learned router: unit u goes to expert fmix32(token_ids[u]) mod E, with
 * fmix32 MurmurHash3's 32-bit finalizer (xor-shift 16, ·0x85ebca6b, xor-shift 13, ·0xc2b2ae35,
 * xor-shift 16) of the id's 32-bit pattern, and gate 1. Capacity and drops are as for any gate; with
 * no routing probabilities there is no aux loss (0). cfg.K must be 1 (else MOE_ERR_UNSUPPORTED);
 * score, groups and aux_alpha are not used. token_ids: [T'] int32 device array, one id per unit
 * (with H heads, one per sub-token). */
MOE_API moe_status_t moe_route_hash(const moe_config_t* cfg, const int32_t* token_ids, int32_t* topk_idx,
                                    float* topk_gate, void* ws, moe_stream_t stream);

/* The whole layer with the hash gate: moe_forward with the routing above. w->w_router, logit_bias
 * and select_bias are not used (may be NULL). out->logits is not written; out->aux gets 0. */
MOE_API moe_status_t moe_forward_hash(const moe_config_t* cfg, const void* x, const int32_t* token_ids,
                                      const moe_weights_t* w, void* y, const moe_outputs_t* out, void* ws,
                                      moe_stream_t stream);

/* moe_forward with a CUDA event recorded on `stream` at each boundary between its stages, for
 * timing them (instrumentation; the pages have no counterpart). events: 6 caller-created cudaEvent_t
 * (as void*), recorded before the routing, after the routing, after the scan (counts, offsets, aux
 * loss), after the pack, after the expert GEMMs and after the combine (recorded right after the
 * GEMMs where the combine is folded into the down GEMM). The kernels are the same as
 * moe_forward's, but neighbouring stages no longer overlap their launch (programmatic dependent
 * launch is off), so the sum of the stage times can exceed a moe_forward call's time.
 * MOE_ERR_INVALID_ARG if events or one of them is NULL. */
MOE_API moe_status_t moe_forward_profiled(const moe_config_t* cfg, const void* x, const moe_weights_t* w, void* y,
                                          const moe_outputs_t* out, void* ws, void* const* events,
                                          moe_stream_t stream);

/* ---- training: forward that keeps what the backward needs, and the backward ----------------
 * The pages train this layer ([HAI] §"HAI-LLM 上的使用"; [Lesson 10 §4] adds L_aux to the training
 * loss) but give no backward formulas. The backward here is the gradient of
 *     L = <dy, y> + d_aux·L_aux
 * with the routing held fixed: the Top-K picks, the group limit, the counts f_i and the capacity
 * drops are piecewise constant and get no gradient; gradients flow through the gates, the expert
 * FFNs, the probabilities P_i of L_aux and the router GEMM. The selection-only bias has none.
 * Supported: dtype MOE_BF16 with h' and d_ff multiples of 64 (else MOE_ERR_UNSUPPORTED). */

/* Bytes of the G | U buffer moe_forward_train fills: T'·K rows of 2·d_ff bf16 (host only). */
MOE_API size_t moe_saved_gu_size(const moe_config_t* cfg);

/* moe_forward, and also the SwiGLU inputs G = X_e·W1_eᵀ and U = X_e·W3_eᵀ of every kept packed
 * row, bf16, into gu [T'·K][2·d_ff] (G in columns [0, d_ff), U in [d_ff, 2·d_ff)).
 * `out` is required, with topk_idx, topk_gate, logits and slot_of non-NULL when T' > 0 (the
 * backward reads them); gu must be 16-byte aligned. Keep `ws`, `out` and `gu` unchanged until
 * moe_backward has run: the backward also reads the forward's packed rows, hidden activations
 * and expert outputs from `ws`. */
MOE_API moe_status_t moe_forward_train(const moe_config_t* cfg, const void* x, const moe_weights_t* w,
                                       void* y, const moe_outputs_t* out, void* gu, void* ws,
                                       moe_stream_t stream);

/* Gradients (device pointers). dlogits and dgate may be NULL (then they stay in `bws`). */
typedef struct {
  void* dx;                /* [T][h] bf16: dL/dx                                                  */
  float* dw_router;        /* [h'][E] fp32: dL/dW_g                                               */
  float* dw_gate;          /* [E][d_ff][h'] fp32: dL/dW1                                           */
  float* dw_up;            /* [E][d_ff][h'] fp32: dL/dW3                                           */
  float* dw_down;          /* [E][h'][d_ff] fp32: dL/dW2                                           */
  float* dlogits;          /* [T'][E] fp32: dL/dl (l the router logits, logit bias included)       */
  float* dgate;            /* [T'][K] fp32: dL/d gate (0 for dropped picks)                        */
} moe_grads_t;

/* Bytes of backward scratch `bws` for this config (host only; 256-byte aligned when allocated). */
MOE_API size_t moe_backward_workspace_size(const moe_config_t* cfg);

/* Backward of the moe_forward_train call that filled `ws`, `out` and `gu` for this x and w.
 *  dy [T][h] bf16: dL/dy. d_aux: weight of L_aux in L (host float).
 *  Out: every member of `grads` except dlogits/dgate is required (dx only when T' > 0); dw_* are
 *  overwritten (not accumulated). x, dy, gu, dx, the expert weights and dw_* must be 16-byte
 *  aligned; bws 256-byte aligned. Deterministic: the same inputs give the same bits. Errors as
 *  for moe_forward; kernel faults set the status word of `ws`. */
MOE_API moe_status_t moe_backward(const moe_config_t* cfg, const void* x, const moe_weights_t* w,
                                  const void* dy, float d_aux, const moe_outputs_t* out, const void* gu,
                                  void* ws, const moe_grads_t* grads, void* bws, moe_stream_t stream);

/* Wait for `stream`, read and clear the status word in `ws`: MOE_OK, MOE_ERR_DEVICE_STATUS or
 * MOE_ERR_TIMEOUT (or MOE_ERR_CUDA if the wait itself failed). */
MOE_API moe_status_t moe_get_status(void* ws, moe_stream_t stream);

/* Static text of a status code. */
MOE_API const char* moe_status_string(moe_status_t s);

/* Kernels this library has launched in this process (monotonic counter; host only). */
MOE_API uint64_t moe_launch_count(void);

/* MOE_ABI_VERSION of the loaded library. */
MOE_API int32_t moe_abi_version(void);

/* Choices of the tensor-core expert GEMMs, process-wide, for tests and tuning (the pages have no
 * counterpart). Each is 1 (on), 0 (off) or -1 (automatic).
 *  pair_tiles: CTA-pair 256-row tiles instead of single-CTA 128-row tiles; automatic: when the
 *    packed rows average at least 256 per expert.
 *  transposed_tails: pair-tile tails of up to 224 rows run transposed; automatic: when the
 *    reduction has at least 16 k-blocks of 64.
 *  fold_combine: moe_forward folds the combine into the down GEMM (bf16, 16-byte aligned y);
 *    automatic: when K == 1, where each unit's one kept row writes g·Y straight into y. With K >= 2
 *    the last row of each unit sums it (arrival counters per 32 columns), which costs the down GEMM
 *    more than the separate combine launch on the measured layers.
 * Takes effect at the next launch; y has the same bits either way. MOE_ERR_INVALID_ARG for other
 * values. Host only. */
MOE_API moe_status_t moe_set_expert_gemm(int32_t pair_tiles, int32_t transposed_tails, int32_t fold_combine);

/* Dispatch for callers that cannot allocate device memory. (The pages have no counterpart of this
 * call; it exists for how the library is deployed, not for the method.)
 * Some callers cannot call cudaMalloc: a plugin inside a host framework that owns all device
 * memory and hands the plugin only its input and output buffers, or a serving process whose
 * device memory is fixed at start-up and that allows no allocation afterwards. Such a caller
 * cannot size and keep a workspace, so this call takes no `ws`: its scratch (per-chunk
 * histograms and queue bases, per-expert totals and offsets) is a fixed 1 MiB array inside the
 * library, which every GPU that loads the library holds until the process exits.
 *  - Same inputs, outputs and results as moe_dispatch (bit for bit).
 *  - Limit: 8·ceil(T'/256)·E bytes + about 8·E bytes must fit in 1 MiB (with E = 256, up to
 *    about 130,000 units); larger problems return MOE_ERR_UNSUPPORTED and enqueue nothing.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *    that device current) and keeps it; make that first call before any stream capture. Under
 *    CUDA's lazy module loading (the default that PyTorch sets) that first lookup is also when the
 *    device reserves the 1 MiB: a caller whose device memory is fixed at start-up should make one
 *    call (any size, e.g. T = 0) at start-up, while memory is still free.
 *  - The kept address belongs to the device's context: after cudaDeviceReset (or any teardown of
 *    the primary context) the library must be reloaded before this call is used again.
 *  - It allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *  - All calls on a device share the array, which keeps the last call's contents; each call
 *    rewrites every part it reads before reading it, and the one counter in it (zero when the
 *    library loads) is back at zero when a call's kernels finish, so nothing needs clearing.
 *    Calls that overlap on the GPU (e.g. on two streams) race and give wrong results: serialise
 *    them.
 *  - Bad indices (out of range or repeated within a unit) give that unit slot -1 for every pick,
 *    as in moe_dispatch, but are not reported: there is no workspace status word here. */
MOE_API moe_status_t moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                                          const int32_t* topk_idx, int32_t* counts,
                                          int32_t* offsets, int32_t* slot_of, int32_t* row_token,
                                          void* x_packed, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
