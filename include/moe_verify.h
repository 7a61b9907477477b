/*
 * moe_verify.h -- C ABI of the MoE verification-pass library (libmoe_verify.so)
 *
 * The library computes the MoE layer of a speculative-decoding verification
 * pass on one GB300 GPU (sm_103a):
 *
 *   1. router scores s = W_g h and top-k selection            (moe_route_topk)
 *      ("Making Every Verified Token Count: Adaptive Verification for MoE
 *      Speculative Decoding", Sec. 2.2, eq. (4) and the sentence after it:
 *      the selected scores are normalised by softmax or sigmoid);
 *   2. the union of the experts the n tokens select, with a grouping of the
 *      n*k (token, slot) pairs by expert                        (moe_union_plan)
 *      (same page, eq. (5); "Less Experts, Faster Decoding: Cost-Aware
 *      Speculative Decoding for Mixture-of-Experts", eq. (1); "The Limits of
 *      Speculation: Bounding Speculative Decoding in Mixture-of-Experts",
 *      App. A.4.1, eqs. (A1)-(A2));
 *   3. each selected expert's SwiGLU FFN on the tokens routed to it, combined
 *      with the router weights, by one of two engines
 *      ("Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
 *      Kernel Bandwidth and the Best Draft Length", abstract and Fig. 3):
 *        - deduplicating: every union expert's weights are read from HBM
 *          once per pass (union bytes U*b)                    (moe_verify_dedup)
 *        - per-slot: an expert's weights are read once per (token, slot)
 *          that names it (requested bytes n*k*b)            (moe_verify_perslot)
 *   4. optionally, a verification-time expert budget (MoE-Spec, as "The
 *      Limits of Speculation", Sec. 2.4 describes it): the plan keeps at
 *      most B routed experts, those of largest summed gate weight, and the
 *      dropped slots leave the output
 *                         (moe_union_plan_budgeted, moe_route_plan_budgeted)
 *
 * Conventions shared by every call
 *   - Pointers named "device" are CUDA device pointers that the caller
 *     allocates and owns; the library allocates and frees nothing.
 *   - Every launching call is asynchronous on `stream` and never synchronises
 *     the host, so a whole pass can be captured in a CUDA graph.  The one
 *     exception is moe_last_error(), which synchronises `stream`.
 *   - Arguments are checked on the host before anything is enqueued; a bad
 *     argument returns a non-OK status and enqueues nothing.  With n == 0 a
 *     call reads and writes nothing, so its array pointers may be NULL
 *     (moe_union_plan still writes U = 0 and offs[0] = 0).
 *   - Device arrays must start on a 16-byte boundary.
 *   - Outputs are fully overwritten.  No C++ exception crosses this ABI.
 *   - Layout of a layer (row-major everywhere):
 *       h          [n][d]           act_dtype
 *       router_w   [N][d]           act_dtype           (W_g; row = expert)
 *       w13        [N][2I][d]       w_dtype  (rows 0..I-1 gate W1, I..2I-1 up W3)
 *       w2         [N][d][I]        w_dtype  (down projection)
 *       s13        [N][2I/128][d/128] float (E4M3 only: block scales)
 *       s2         [N][d/128][I/128]  float (E4M3 only)
 *       sh_*       the shared expert, same shapes without the leading N
 *       y          [n][d]           act_dtype
 *     An E4M3 weight is q * s where q is the OCP FP8 E4M3 value of the byte
 *     and s the fp32 scale of its 128 x 128 block.
 *   - Packed weights: moe_verify_dedup and moe_verify_perslot read w13, w2,
 *     sh_w13 and sh_w2 in the tile layout that moe_pack_expert_weights
 *     writes once, when the model is loaded (moe_packed_bytes gives the
 *     sizes: those of the row-major arrays, plus for E4M3 the block scales,
 *     which the packed tiles carry; identical to the row-major arrays for
 *     F32).
 *   - Limits (else MOE_ERR_UNSUPPORTED): N <= 256, 1 <= k <= min(N, 32),
 *     0 <= n <= n_max <= 64, n_shared 0 or 1, d % 8 == 0; F32 weights go with
 *     F32 activations and need I % 4 == 0; BF16 and E4M3 weights go with BF16
 *     activations; BF16 needs d % 64 == 0 and I % 64 == 0, E4M3 needs
 *     d % 128 == 0, I % 128 == 0, d <= 8192 and I <= 8192.
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle (cudaStream_t); 0 is the legacy default stream. */
typedef void *moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, size out of range, bad enum   */
  MOE_ERR_UNSUPPORTED = 2, /* a size this build does not handle           */
  MOE_ERR_ALIGNMENT = 3,   /* a device array not on a 16-byte boundary    */
  MOE_ERR_WORKSPACE = 4,   /* workspace smaller than moe_workspace_bytes() */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed        */
  MOE_ERR_TIMEOUT = 6,     /* a device-side wait hit its time limit       */
  MOE_ERR_DEVICE_INPUT = 7 /* an expert id, a tree or a plan read on the
                              device was malformed (see each call)        */
} moe_status;

typedef enum {
  MOE_F32 = 0,      /* IEEE binary32                                     */
  MOE_BF16 = 1,     /* bfloat16                                          */
  MOE_E4M3_B128 = 2 /* OCP FP8 E4M3 with one fp32 scale per 128x128 block */
} moe_dtype;

typedef enum {
  MOE_GATE_SOFTMAX = 0,        /* softmax over all N scores; keep the k selected  */
  MOE_GATE_SOFTMAX_RENORM = 1, /* softmax over the k selected scores              */
  MOE_GATE_SIGMOID_RENORM = 2  /* sigmoid of the k selected scores / their sum    */
} moe_gate;

typedef struct {
  int32_t d;               /* hidden size                                 */
  int32_t n_experts;       /* routed experts N                            */
  int32_t top_k;           /* experts per token k                         */
  int32_t inter;           /* SwiGLU intermediate size I                  */
  int32_t n_shared;        /* 0 or 1 shared expert, applied with weight 1 */
  int32_t n_max;           /* largest n any call with this desc will pass */
  int32_t act_dtype;       /* MOE_F32 or MOE_BF16 (h, router_w, y)        */
  int32_t w_dtype;         /* moe_dtype of the expert weights             */
  int32_t gate;            /* moe_gate                                    */
  int32_t wait_timeout_us; /* limit of every device-side wait; 0 = 1 s    */
} moe_layer_desc;

/* The experts as moe_pack_expert_weights wrote them (E4M3: with their
 * block scales). */
typedef struct {
  const void *w13;    /* device, N packed W13 matrices              */
  const void *w2;     /* device, N packed W2 matrices               */
  const void *sh_w13; /* device, the shared expert's packed W13; NULL if none */
  const void *sh_w2;  /* device, the shared expert's packed W2      */
} moe_expert_weights;

/* The union plan (all device arrays, owned by the caller). */
typedef struct {
  int32_t *hist;        /* [N]     slots that name each expert                */
  int32_t *uniq;        /* [N]     the U distinct experts, ascending; the
                                   entries from U on are left unspecified     */
  int32_t *n_uniq;      /* [1]     U                                          */
  int32_t *offs;        /* [N+1]   group u of perm is offs[u] .. offs[u+1]-1;
                                   offs[U] = n*k; later entries unspecified   */
  int32_t *perm;        /* [n_max*k] slot indices t*k+j grouped by expert in
                                   uniq order, ascending inside a group       */
  int64_t *union_bytes; /* [1]     (U + n_shared) * (expert weight bytes +
                                   expert scale bytes)                        */
} moe_plan;

/* Bytes of the caller-owned workspace that moe_verify_dedup and
 * moe_verify_perslot need for this desc (sized for desc->n_max).  Returns 0
 * for an invalid desc. */
size_t moe_workspace_bytes(const moe_layer_desc *desc);

/* Bytes of one expert: its three matrices (*weight_bytes = 3*d*I*element
 * size) and, for E4M3, its fp32 block scales (*scale_bytes).  Either
 * pointer may be NULL. */
moe_status moe_expert_bytes(const moe_layer_desc *desc, int64_t *weight_bytes,
                            int64_t *scale_bytes);

/* Bytes of one expert's packed W13 and W2 (either pointer may be NULL). */
moe_status moe_packed_bytes(const moe_layer_desc *desc, int64_t *w13_bytes,
                            int64_t *w2_bytes);

/* Repacks n_matrices experts' W13 and W2 (device, row-major as in the layout
 * above) into the tile layout the expert engines stream (device, caller
 * allocated, n_matrices times moe_packed_bytes, not in place).  BF16 and
 * E4M3: each expert matrix becomes a sequence of tiles of 64 rows x 512
 * bytes (the last tile of a row block narrower when a row is not a multiple
 * of 512 bytes); a W13 tile holds gate rows 32b..32b+31 followed by up rows
 * I+32b..I+32b+31; tiles of a row block follow each other in K order, row
 * blocks follow each other, so that one pipeline stage is one contiguous
 * bulk copy.  Inside a tile, BF16: [128-byte column q][8-row group m][row r]
 * [16-byte chunk], where chunk j of row 8m+r (bytes 128q+16j..+15 of K) is
 * stored at position j XOR r (the tensor cores' 128-byte swizzled K-major
 * layout); E4M3: the 16-byte pieces are ordered [64-byte column chunk]
 * [16-row tile][row half][lane] (lane = 4 g + c takes row 16 t + 8 h + g,
 * bytes 64 w + 16 c of the chunk).  E4M3: every tile is followed by its 8 block
 * scales from s13 / s2 (device, [n_matrices][rows/128][cols/128] float as in
 * the layout above; NULL for other weight types): the scales of the tile's
 * four 128-column blocks for the 128-row block of its first 32 rows, then
 * of its last 32 rows (0 past the last column block).  F32: a plain copy.
 * Call once per layer (N routed experts) and once for the shared expert
 * (n_matrices = 1). */
moe_status moe_pack_expert_weights(const moe_layer_desc *desc, const void *w13,
                                   const void *w2, const float *s13,
                                   const float *s2, int32_t n_matrices,
                                   void *w13_packed, void *w2_packed,
                                   moe_stream_t stream);

/* Router scores and top-k ("Making Every Verified Token Count", Sec. 2.2,
 * eq. (4)).  For each of the n tokens: logits[t][e] = sum_i router_w[e][i] *
 * h[t][i] accumulated in fp32; ids[t][0..k) = the k experts with the largest
 * logits, largest first, equal logits ordered by lower id; w[t][j] = the
 * gate weight of ids[t][j] (desc->gate).
 *   router_w  device [N][d] act_dtype;   h  device [n][d] act_dtype
 *   ids       device [n][k] int32 (out); w  device [n][k] float (out)
 *   logits    device [n][N] float (out; required: the scores are staged
 *             there between the two kernels)
 * n may be 0 (nothing is enqueued). */
moe_status moe_route_topk(const moe_layer_desc *desc, const void *router_w,
                          const void *h, int32_t n, int32_t *ids, float *w,
                          float *logits, moe_stream_t stream);

/* The top-k and gate stage of moe_route_topk on given fp32 logits
 * (device [n][N]).  Its ids equal a full sort of each row by (logit
 * descending, id ascending), bit for bit. */
moe_status moe_topk_from_logits(const moe_layer_desc *desc,
                                const float *logits, int32_t n, int32_t *ids,
                                float *w, moe_stream_t stream);

/* The expert union of the routed ids (device [n][k] int32) and the grouping
 * of the n*k slots by expert, written to `plan` (see moe_plan).  An id
 * outside [0, N) is left out of the plan and makes moe_last_error() report
 * MOE_ERR_DEVICE_INPUT when `error_word` is not NULL.
 *   error_word  device int32 that receives the first device-side error, or
 *               NULL; the workspace of moe_verify_* starts with such a word. */
moe_status moe_union_plan(const moe_layer_desc *desc, const int32_t *ids,
                          int32_t n, const moe_plan *plan, int32_t *error_word,
                          moe_stream_t stream);

/* moe_route_topk followed by moe_union_plan, in one kernel launch: the
 * router CTAs write the scores; the last CTA to finish each group of 8
 * tokens selects their top-k and gates, and the last of those builds the
 * plan.  Same outputs, bit for bit.
 *   workspace  a workspace initialised by moe_workspace_init (only its
 *              256-byte header is used: the error word, and ticket counters
 *              the kernel leaves at zero); ws_bytes >= 256.  Calls sharing a
 *              workspace must not overlap on the GPU.
 * n may be 0: the plan becomes empty (U = 0). */
moe_status moe_route_plan(const moe_layer_desc *desc, const void *router_w,
                          const void *h, int32_t n, int32_t *ids, float *w,
                          float *logits, const moe_plan *plan, void *workspace,
                          size_t ws_bytes, moe_stream_t stream);

/* Verification-time expert budget (MoE-Spec, as its abstract is listed on
 * "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
 * Bandwidth and the Best Draft Length"; "The Limits of Speculation",
 * Sec. 2.4: each layer loads at most a fixed number of experts, the most
 * useful ones, and skips the rarely used rest).  moe_union_plan, except
 * that at most `budget` routed experts enter the plan:
 *   - an expert's contribution is the sum of the weights w of the slots
 *     that name it, added in double in ascending slot order;
 *   - when more than `budget` experts are used, the kept ones are the first
 *     `budget` by (contribution descending, id ascending); otherwise all;
 *   - `plan` is the plan of the kept slots only (a dropped expert has
 *     hist 0, is not in uniq, and its slots are not in perm; offs[U] is the
 *     number of kept slots; union_bytes counts the kept experts + shared);
 *   - w_kept[p] = w[p] for a kept slot and 0 for a dropped slot (or an
 *     invalid id).  Passing w_kept as the weights of moe_verify_dedup gives
 *     the budgeted layer output: dropped terms are left out, the kept
 *     weights are not renormalised, the shared expert is always applied.
 *   w             device [n][k] float, the gate weights of ids
 *   budget        >= 0 (0 keeps no routed expert); else MOE_ERR_INVALID_ARG
 *   w_kept        device [n][k] float (out); may not alias w
 *   routed_union  device int32 (out): U before the cap, or NULL
 * The output is lossy whenever the cap drops an expert. */
moe_status moe_union_plan_budgeted(const moe_layer_desc *desc,
                                   const int32_t *ids, const float *w,
                                   int32_t n, int32_t budget,
                                   const moe_plan *plan, float *w_kept,
                                   int32_t *routed_union, int32_t *error_word,
                                   moe_stream_t stream);

/* moe_route_plan with the budgeted plan of moe_union_plan_budgeted: one
 * launch routes, gates, caps the union at `budget` experts and writes
 * w_kept (and routed_union unless NULL).  Same outputs, bit for bit, as
 * moe_route_topk followed by moe_union_plan_budgeted. */
moe_status moe_route_plan_budgeted(const moe_layer_desc *desc,
                                   const void *router_w, const void *h,
                                   int32_t n, int32_t budget, int32_t *ids,
                                   float *w, float *logits,
                                   const moe_plan *plan, float *w_kept,
                                   int32_t *routed_union, void *workspace,
                                   size_t ws_bytes, moe_stream_t stream);

/* The layer output with the deduplicating engine: every expert of the plan
 * (plus the shared expert) is applied once to all tokens routed to it, its
 * weights streamed from HBM once per pass, and
 *   y[t] = sum_j w[t][j] * FFN_{ids[t][j]}(h[t]) (+ FFN_shared(h[t])),
 * summed in the fixed order j = 0..k-1, then the shared expert.
 *   weights    the layer's experts (device pointers inside)
 *   h          device [n][d] act_dtype;   ids  device [n][k] int32
 *   w          device [n][k] float;       plan built by moe_union_plan from ids
 *              (or w_kept and the plan of moe_union_plan_budgeted; a slot
 *              of weight 0 is skipped in the sum)
 *   workspace  device, ws_bytes >= moe_workspace_bytes(desc)
 *   y          device [n][d] act_dtype (out)
 * The intermediate activations a = silu(g) * u are kept in fp32 (F32
 * weights) or bf16 (BF16 and E4M3 weights).  E4M3 weights are multiplied
 * on fp16 tensor cores (every E4M3 value is exact in fp16): each token's
 * hidden row, and each slot's row of a, reaches them scaled by the exact
 * power of two that puts its largest magnitude in [2^14, 2^15), and the
 * sums are scaled back in fp32.  So any finite bf16 hidden state is
 * accepted, and within a row every element above 2^-28 of the row's
 * largest keeps all its bits (smaller ones, whose terms cannot reach the
 * output tolerance, lose bits or become 0).  Sums beyond fp32's range
 * become inf, as in an fp32 accumulation.
 * With BF16 weights and n >= 25, an expert routed by more than 8 of the
 * tokens (or the shared expert) is computed on the 5th-generation tensor
 * cores (tcgen05, accumulators in tensor memory) with all of its tokens at
 * once; its fp32 sums are then added in another order than on the mma.sync
 * path, so its outputs may differ in the last bits from a pass of fewer
 * tokens or one that routes it fewer tokens.  A given call repeats bit for
 * bit.
 * The kernels check the plan before they use its indices: U outside [0, N],
 * a uniq entry outside [0, N), offs decreasing, negative or past n*k, or a
 * perm entry outside [0, n*k) makes moe_last_error() report
 * MOE_ERR_DEVICE_INPUT.  The bad entries are skipped, never followed (the
 * F32 kernels skip each malformed expert group, or all of them when U is
 * out of range; the BF16 and FP8 kernels skip every routed expert), and y
 * is then not the layer output. */
moe_status moe_verify_dedup(const moe_layer_desc *desc,
                            const moe_expert_weights *weights, const void *h,
                            int32_t n, const int32_t *ids, const float *w,
                            const moe_plan *plan, void *workspace,
                            size_t ws_bytes, void *y, moe_stream_t stream);

/* One whole verification pass of the layer: moe_route_plan (or
 * moe_route_plan_budgeted when budget >= 0), then moe_verify_dedup on its
 * plan (with w, or w_kept under a budget), enqueued together.  Outputs are
 * those of the separate calls, bit for bit.  Because the library knows that
 * the kernel ahead of the expert kernels is this pass's own plan kernel,
 * which writes nothing they read except the plan, the first expert kernel
 * starts on the shared expert (which needs no plan) while the routing is
 * still running; moe_verify_dedup alone cannot assume this and waits for
 * every earlier kernel in the stream.
 *   budget     -1 for no expert budget, else as moe_union_plan_budgeted
 *   ids, w, logits, plan          as moe_route_plan (outputs)
 *   w_kept, routed_union          as moe_union_plan_budgeted (budget >= 0;
 *                                 otherwise not used and may be NULL)
 *   workspace  as moe_verify_dedup (its header also serves the routing)
 * The plan kernel hands the plan to the first expert kernel through a flag
 * in the workspace header (with E4M3 weights it also writes the expert
 * kernels' scaled fp16 rows of h, counted in a second header word), which
 * the pass's last kernel clears; after a
 * call that failed (a non-OK status, or MOE_ERR_TIMEOUT from
 * moe_last_error), call moe_workspace_init before reusing the workspace.
 * n may be 0: the plan becomes empty and nothing else is enqueued. */
moe_status moe_verify_pass(const moe_layer_desc *desc,
                           const moe_expert_weights *weights,
                           const void *router_w, const void *h, int32_t n,
                           int32_t budget, int32_t *ids, float *w,
                           float *logits, const moe_plan *plan, float *w_kept,
                           int32_t *routed_union, void *workspace,
                           size_t ws_bytes, void *y, moe_stream_t stream);

/* The same output with the per-slot engine: each (token, slot) pair, and
 * each token's shared-expert slot, runs its expert's FFN for that one token,
 * reading the expert's weights once per pair.  No plan is needed. */
moe_status moe_verify_perslot(const moe_layer_desc *desc,
                              const moe_expert_weights *weights,
                              const void *h, int32_t n, const int32_t *ids,
                              const float *w, void *workspace, size_t ws_bytes,
                              void *y, moe_stream_t stream);

/* ---- pre-verification selection over a batch of draft trees ----
 *
 * Before the verification pass, these calls choose which draft-tree nodes
 * to verify.  Each tree has K = n_nodes nodes:
 *   parent  device [n_trees][K] int32: node 0 is the root (the token the
 *           target model already sampled), parent[0] = -1, and
 *           0 <= parent[v] < v for every other node (e.g. BFS numbering);
 *   q       device [n_trees][K] float: the draft model's probability of node
 *           v's token given its prefix (q of the root is not read: the root
 *           counts with factor 1).
 * A node's cumulative score is the product of q along its root path
 * ("Making Every Verified Token Count", Sec. 3.1, eq. (7)).  Both calls
 * decide in double, in the order the definitions give, so their outputs are
 * exact.  Ties go to the lower node index (or the smaller k).  A malformed
 * tree makes moe_last_error() report MOE_ERR_DEVICE_INPUT (through
 * error_word, when not NULL), and that tree's outputs are marked
 * (k_star 0 / selected -1 / union_size -1).  1 <= K <= 256; n_trees == 0
 * enqueues nothing. */

/* EVICT's utility-guided prefix ("Making Every Verified Token Count",
 * Sec. 3.2): T_k = the k nodes of largest score (an ancestor-closed subtree,
 * Sec. 3.2.1); E_hat[A(T_k)] = the sum of their scores (eq. (8)), added in
 * rank order; k* = argmax over k = 1..K of E_hat[A(T_k)] / C(k) (eqs. (9)-
 * (10)), with C(k) a profiled cost table (Sec. 3.2.3).
 *   cost      device [K] float: C(k) at cost[k-1], shared by all trees
 *   order     device [n_trees][K] int32 (out): nodes by rank; verify the
 *             first k_star of them
 *   exp_len   device [n_trees][K] double (out, or NULL): E_hat[A(T_k)]
 *   utility   device [n_trees][K] double (out, or NULL): E_hat / C(k)
 *   k_star    device [n_trees] int32 (out) */
moe_status moe_evict_select(const int32_t *parent, const float *q,
                            int32_t n_trees, int32_t n_nodes, const float *cost,
                            int32_t *order, double *exp_len, double *utility,
                            int32_t *k_star, int32_t *error_word,
                            moe_stream_t stream);

/* EcoSpec's cost-aware draft selection ("Less Experts, Faster Decoding:
 * Cost-Aware Speculative Decoding for Mixture-of-Experts", Sec. 4.2,
 * eqs. (7)-(9), and its appendix algorithm).  Start from the buffer B = B0,
 * then repeat gamma times (K times when gamma > K):
 *   - for every unselected node t, E_traj(t) is the union of the predicted
 *     (layer, expert) sets over t's root path;
 *   - its score is P(t) / (|E_traj(t) \ B| + eps);
 *   - select the node of largest score and add its E_traj to B.
 *   pred_ids    device [n_trees][K][n_layers][pred_k] int32: the experts
 *               predicted for each node at each layer (ids outside
 *               [0, n_experts) are ignored)
 *   eps         > 0
 *   buffer0     device [n_trees][n_layers][ceil(n_experts/32)] uint32
 *               bitsets (bit e%32 of word e/32) of B0, or NULL for empty
 *   selected    device [n_trees][min(gamma, K)] int32 (out), in pick order
 *   buffer_out  device, the final B in buffer0's layout (out, or NULL)
 *   union_size  device [n_trees] int32 (out): |B| at the end
 * MOE_ERR_UNSUPPORTED when (K + 1) * n_layers * ceil(n_experts/32) * 4
 * bytes exceed 200 KB (the bitsets live in shared memory). */
moe_status moe_ecospec_select(const int32_t *parent, const float *q,
                              const int32_t *pred_ids, int32_t n_trees,
                              int32_t n_nodes, int32_t n_layers,
                              int32_t n_experts, int32_t pred_k, int32_t gamma,
                              double eps, const uint32_t *buffer0,
                              int32_t *selected, uint32_t *buffer_out,
                              int32_t *union_size, int32_t *error_word,
                              moe_stream_t stream);

/* Zeroes the error word at the start of a fresh workspace (enqueued on
 * `stream`).  Call once after allocating a workspace; moe_last_error() clears
 * the word again after reading it. */
moe_status moe_workspace_init(void *workspace, size_t ws_bytes,
                              moe_stream_t stream);

/* moe_verify_dedup for callers that cannot provide a workspace.
 *
 * No counterpart on the pages: this exists for callers that may not allocate
 * device memory themselves, e.g. code whose device memory belongs to a
 * framework allocator it must not go around, or a latency-critical path that
 * must never call cudaMalloc (which can synchronise the device and may fail
 * where nothing can recover).  It computes the same output as
 * moe_verify_dedup with the same arguments, but its scratch (error word,
 * intermediate activations, per-slot outputs) is a fixed 16 MiB array inside
 * the library, held on every GPU that loads the library until the process
 * exits; the call itself allocates and frees nothing.
 *   - Limit: the scratch for n tokens must fit 16 MiB, i.e.
 *     256 + n*(k + n_shared)*(I*e + 4*d) bytes, plus for E4M3 weights
 *     n*(2*d + 4) + 4*n*(k + n_shared) bytes (each part rounded up to 256
 *     bytes; e = 4 for F32 weights, else 2); a larger call returns
 *     MOE_ERR_WORKSPACE and enqueues nothing (DeepSeek-V3 shapes: n <= 54).
 *   - Each call looks up the array's device address on the current device
 *     (a stale address is never used, e.g. after a device reset).  A call
 *     made while `stream` is being captured uses the address found by an
 *     earlier call on that device; make that earlier call before any stream
 *     capture (a first call during capture returns MOE_ERR_UNSUPPORTED).
 *   - Every call shares the array: calls whose execution may overlap on the
 *     GPU (other streams, other host threads) race; serialise them.
 *   - error_word: device int32 (4-byte aligned) that receives the call's
 *     device-side status (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_INPUT)
 *     once the call's work completes on `stream`.  It may be NULL, but then
 *     the device-side status is not reported anywhere, and on malformed
 *     input (an id or plan the kernels reject) y is unspecified. */
moe_status moe_verify_dedup_noalloc(const moe_layer_desc *desc,
                                    const moe_expert_weights *weights,
                                    const void *h, int32_t n,
                                    const int32_t *ids, const float *w,
                                    const moe_plan *plan, void *y,
                                    int32_t *error_word, moe_stream_t stream);

/* Synchronises `stream`, then returns (and clears) the first error that a
 * kernel recorded in the workspace's error word: MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE_INPUT; MOE_ERR_CUDA if the synchronisation itself failed. */
moe_status moe_last_error(void *workspace, moe_stream_t stream);

/* Self-test of the device-side bounded wait used by every kernel: launches
 * one CTA that waits on a barrier nothing ever arrives on, gives up after
 * limit_us microseconds (1 <= limit_us <= 1000000), records MOE_ERR_TIMEOUT
 * in *error_word (device int32) and returns, leaving the context usable. */
moe_status moe_selftest_bounded_wait(int32_t *error_word, int32_t limit_us,
                                     moe_stream_t stream);

/* A short English description of a status code (static storage). */
const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
