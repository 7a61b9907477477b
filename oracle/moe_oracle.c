/*
 * moe_oracle.c -- plain CPU oracle for the MoE layer of a speculative
 * verification pass.  TEST INFRASTRUCTURE ONLY: it is called by the tests,
 * by __graft_entry__.smoke() and by the cpu_baseline leg of bench.py, and by
 * nothing on the product path.  It shares no code, header, table or helper
 * with the CUDA library; neither side includes or links the other.
 *
 * Everything is a plain per-token loop in double precision, written from the
 * definitions on the pages, with no blocking, fusion or reordering:
 *
 *   router scores    s = W_g h, W_g in R^{N x d}
 *                    ("Making Every Verified Token Count", Sec. 2.2, eq. (4))
 *   top-k            indices of the k largest scores (same place); ties are
 *                    broken toward the lower expert id and ids are emitted in
 *                    descending score order (a reading: the pages are silent)
 *   gate             softmax or sigmoid of the selected scores "depending on
 *                    the architecture" (same place), three variants below
 *   expert union     E_verify = union over verified tokens of S(x_t)
 *                    ("Less Experts, Faster Decoding", eq. (1); "Making Every
 *                    Verified Token Count", eq. (5); "The Limits of
 *                    Speculation", App. A.4.1, eqs. (A1)-(A2))
 *   expert FFN       SwiGLU: a = silu(W1 h) * (W3 h), o = W2 a, with the gate
 *                    rows W1 stored before the up rows W3 (a reading)
 *   layer output     y = sum_j w_j o_j  (+ the shared expert with weight 1)
 *
 * The deduplicating and per-slot engines of "Speculative Decoding for MoE
 * Models: Expert Bytes, Kernel Bandwidth and the Best Draft Length"
 * (abstract; Fig. 3) are two schedules of this same sum; the oracle computes
 * the sum itself, once per (token, selected expert).
 *
 * Stored numbers are read from the very bytes the GPU receives:
 *   bf16  -> double is exact (the 16 bits are the top half of an IEEE float);
 *   e4m3  -> double is decoded from the OCP 8-bit floating point format
 *            definition (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *            bits; exponent field 0 is subnormal; S.1111.111 is NaN; no
 *            infinities), then multiplied by its fp32 128x128 block scale.
 *
 * Parity pins live in tests/test_oracle_pins.py; every function here has one.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element types of stored arrays */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };
/* gate variants */
enum { ORC_GATE_SOFTMAX = 0,        /* softmax over all experts, take the k  */
       ORC_GATE_SOFTMAX_RENORM = 1, /* softmax restricted to the k selected  */
       ORC_GATE_SIGMOID_RENORM = 2  /* sigmoid of the k, divided by its sum */
};

#define ORC_BLOCK 128 /* side of a square FP8 scale block */

/* ---------------------------------------------------------------- decoding */

double orc_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double orc_f32_to_double(uint32_t bits) {
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3: value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 *                       (-1)^s * 2^(-6)  * (m/8)     for e == 0,
 * and NaN for e == 15, m == 7.  No infinities; largest finite is 448. */
double orc_e4m3_to_double(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* One stored element, as a double.  For E4M3 the caller applies the scale. */
static double load_elem(const void *base, int type, size_t idx) {
  switch (type) {
  case ORC_F32: {
    uint32_t b;
    memcpy(&b, (const char *)base + 4 * idx, 4);
    return orc_f32_to_double(b);
  }
  case ORC_BF16: {
    uint16_t b;
    memcpy(&b, (const char *)base + 2 * idx, 2);
    return orc_bf16_to_double(b);
  }
  case ORC_E4M3:
    return orc_e4m3_to_double(((const uint8_t *)base)[idx]);
  }
  return NAN;
}

/* ------------------------------------------------------------------ layer */

typedef struct {
  int d;          /* hidden size                                   */
  int n_experts;  /* routed experts N                              */
  int top_k;      /* experts per token k                           */
  int inter;      /* SwiGLU intermediate size I                    */
  int n_shared;   /* shared experts always applied (0 or 1)        */
  int act_type;   /* ORC_F32 or ORC_BF16: h and W_g                */
  int w_type;     /* ORC_F32, ORC_BF16 or ORC_E4M3: expert weights */
  int gate;       /* ORC_GATE_*                                    */
  const void *wg;  /* [N][d]                                        */
  const void *w13; /* [N][2I][d]: rows 0..I-1 gate, rows I..2I-1 up */
  const void *w2;  /* [N][d][I]                                     */
  const float *s13; /* E4M3 only: [N][2I/128][d/128]                */
  const float *s2;  /* E4M3 only: [N][d/128][I/128]                 */
  const void *sh_w13; /* shared expert: [2I][d]                     */
  const void *sh_w2;  /* shared expert: [d][I]                      */
  const float *sh_s13;
  const float *sh_s2;
} orc_layer;

/* Weight element (row, col) of a [rows][cols] matrix at `base`, with its
 * block scale table `scale` ([rows/128][cols/128]) applied for E4M3. */
static double weight_at(const orc_layer *L, const void *base,
                        const float *scale, int rows, int cols, int row,
                        int col) {
  double v = load_elem(base, L->w_type, (size_t)row * cols + col);
  (void)rows;
  if (L->w_type == ORC_E4M3) {
    int scale_cols = cols / ORC_BLOCK;
    v *= (double)scale[(size_t)(row / ORC_BLOCK) * scale_cols + col / ORC_BLOCK];
  }
  return v;
}

static size_t elem_size(int type) {
  return type == ORC_F32 ? 4 : type == ORC_BF16 ? 2 : 1;
}

/* Router scores of one token: z[e] = sum_i W_g[e][i] h[i]
 * ("Making Every Verified Token Count", Sec. 2.2). */
void orc_router_scores(const orc_layer *L, const double *h, double *z) {
  for (int e = 0; e < L->n_experts; ++e) {
    double acc = 0.0;
    for (int i = 0; i < L->d; ++i)
      acc += load_elem(L->wg, L->act_type, (size_t)e * L->d + i) * h[i];
    z[e] = acc;
  }
}

/* Order used by TopK: larger score first; equal scores, lower id first. */
typedef struct {
  double z;
  int id;
} scored;

static int cmp_scored(const void *a, const void *b) {
  const scored *x = (const scored *)a, *y = (const scored *)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

/* TopK of eq. (4): the k experts with the largest scores, by a full sort of
 * all N scores. */
void orc_topk(const double *z, int n_experts, int k, int32_t *ids) {
  scored *s = (scored *)malloc(sizeof(scored) * (size_t)n_experts);
  for (int e = 0; e < n_experts; ++e) {
    s[e].z = z[e];
    s[e].id = e;
  }
  qsort(s, (size_t)n_experts, sizeof(scored), cmp_scored);
  for (int j = 0; j < k; ++j) ids[j] = s[j].id;
  free(s);
}

/* Gate weights of the selected experts (eq. (4) and the sentence after it:
 * the selected scores become weights through a softmax or a sigmoid, the
 * choice being the model's). */
void orc_gate(const double *z, int n_experts, const int32_t *ids, int k,
              int gate, double *w) {
  if (gate == ORC_GATE_SOFTMAX) {
    double zmax = z[0];
    for (int e = 1; e < n_experts; ++e)
      if (z[e] > zmax) zmax = z[e];
    double sum = 0.0;
    for (int e = 0; e < n_experts; ++e) sum += exp(z[e] - zmax);
    for (int j = 0; j < k; ++j) w[j] = exp(z[ids[j]] - zmax) / sum;
  } else if (gate == ORC_GATE_SOFTMAX_RENORM) {
    double zmax = z[ids[0]];
    for (int j = 1; j < k; ++j)
      if (z[ids[j]] > zmax) zmax = z[ids[j]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += exp(z[ids[j]] - zmax);
    for (int j = 0; j < k; ++j) w[j] = exp(z[ids[j]] - zmax) / sum;
  } else {
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
      w[j] = 1.0 / (1.0 + exp(-z[ids[j]]));
      sum += w[j];
    }
    for (int j = 0; j < k; ++j) w[j] /= sum;
  }
}

/* One expert's SwiGLU FFN on one token, accumulated into y with weight wt:
 *   g_i = W1[i] . h,  u_i = W3[i] . h,  a_i = g_i * sigmoid(g_i) * u_i,
 *   o_r = W2[r] . a,  y_r += wt * o_r. */
static void expert_ffn(const orc_layer *L, const void *w13, const float *s13,
                       const void *w2, const float *s2, const double *h,
                       double wt, double *a, double *y) {
  int d = L->d, I = L->inter;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < d; ++c) {
      g += weight_at(L, w13, s13, 2 * I, d, i, c) * h[c];
      u += weight_at(L, w13, s13, 2 * I, d, I + i, c) * h[c];
    }
    a[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int r = 0; r < d; ++r) {
    double o = 0.0;
    for (int i = 0; i < I; ++i) o += weight_at(L, w2, s2, d, I, r, i) * a[i];
    y[r] += wt * o;
  }
}

/* Pointers to expert e's matrices inside the expert-major arrays. */
static void expert_ptrs(const orc_layer *L, int e, const void **w13,
                        const float **s13, const void **w2, const float **s2) {
  size_t es = elem_size(L->w_type);
  size_t n13 = (size_t)2 * L->inter * L->d, n2 = (size_t)L->d * L->inter;
  *w13 = (const char *)L->w13 + (size_t)e * n13 * es;
  *w2 = (const char *)L->w2 + (size_t)e * n2 * es;
  *s13 = NULL;
  *s2 = NULL;
  if (L->w_type == ORC_E4M3) {
    *s13 = L->s13 + (size_t)e * (n13 / (ORC_BLOCK * ORC_BLOCK));
    *s2 = L->s2 + (size_t)e * (n2 / (ORC_BLOCK * ORC_BLOCK));
  }
}

/* Router scores, top-k and gate of token t. */
static void route_token(const orc_layer *L, const void *hs, int t, int32_t *ids,
                        double *w, double *z) {
  int d = L->d;
  double *h = (double *)malloc(sizeof(double) * (size_t)d);
  for (int c = 0; c < d; ++c)
    h[c] = load_elem(hs, L->act_type, (size_t)t * d + c);
  orc_router_scores(L, h, z);
  orc_topk(z, L->n_experts, L->top_k, ids);
  orc_gate(z, L->n_experts, ids, L->top_k, L->gate, w);
  free(h);
}

/* Router scores of token t and the gate of the given ids (a routing chosen
 * elsewhere, e.g. a GPU's on fp32 scores that differ from the oracle's top-k
 * only among scores closer than fp32 rounding): z = W_g h, w = gate(z, ids). */
static void gate_given_token(const orc_layer *L, const void *hs, int t,
                             const int32_t *ids, double *w, double *z) {
  int d = L->d;
  double *h = (double *)malloc(sizeof(double) * (size_t)d);
  for (int c = 0; c < d; ++c)
    h[c] = load_elem(hs, L->act_type, (size_t)t * d + c);
  orc_router_scores(L, h, z);
  orc_gate(z, L->n_experts, ids, L->top_k, L->gate, w);
  free(h);
}

/* The layer output of token t from its routed ids and weights:
 * y = sum over j of w[j] * FFN_{ids[j]}(h), in slot order, then the shared
 * expert with weight 1.  With `keep` (NULL = every expert), a slot whose
 * expert e has keep[e] == 0 is left out of the sum. */
static void ffn_token(const orc_layer *L, const void *hs, int t,
                      const int32_t *ids, const double *w, const uint8_t *keep,
                      double *y) {
  int d = L->d;
  double *h = (double *)malloc(sizeof(double) * (size_t)d);
  double *a = (double *)malloc(sizeof(double) * (size_t)L->inter);
  for (int c = 0; c < d; ++c)
    h[c] = load_elem(hs, L->act_type, (size_t)t * d + c);
  for (int r = 0; r < d; ++r) y[r] = 0.0;
  for (int j = 0; j < L->top_k; ++j) {
    if (keep && !keep[ids[j]]) continue;
    const void *w13, *w2;
    const float *s13, *s2;
    expert_ptrs(L, ids[j], &w13, &s13, &w2, &s2);
    expert_ffn(L, w13, s13, w2, s2, h, w[j], a, y);
  }
  for (int s = 0; s < L->n_shared; ++s)
    expert_ffn(L, L->sh_w13, L->sh_s13, L->sh_w2, L->sh_s2, h, 1.0, a, y);
  free(a);
  free(h);
}

/* What a worker does for each of its tokens. */
enum { DO_ROUTE_AND_FFN = 0, DO_ROUTE = 1, DO_FFN = 2, DO_GATE_AND_FFN = 3 };

typedef struct {
  const orc_layer *L;
  const void *hs;
  const int32_t *tokens;
  int n_tokens;
  int stride;
  int first;
  int mode;
  const uint8_t *keep;
  int32_t *ids;
  double *w, *z, *y;
} worker_arg;

static void *worker(void *p) {
  worker_arg *A = (worker_arg *)p;
  const orc_layer *L = A->L;
  for (int i = A->first; i < A->n_tokens; i += A->stride) {
    int t = A->tokens ? A->tokens[i] : i;
    int32_t *ids = A->ids + (size_t)i * L->top_k;
    double *w = A->w + (size_t)i * L->top_k;
    if (A->mode == DO_GATE_AND_FFN)
      gate_given_token(L, A->hs, t, ids, w, A->z + (size_t)i * L->n_experts);
    else if (A->mode != DO_FFN)
      route_token(L, A->hs, t, ids, w, A->z + (size_t)i * L->n_experts);
    if (A->mode != DO_ROUTE)
      ffn_token(L, A->hs, t, ids, w, A->keep, A->y + (size_t)i * L->d);
  }
  return NULL;
}

/* Runs `worker` over n_tokens tokens on n_threads host threads. */
static void run_workers(const orc_layer *L, const void *hs, const int32_t *tokens,
                        int n_tokens, int n_threads, int mode,
                        const uint8_t *keep, int32_t *ids, double *w,
                        double *z, double *y) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > n_tokens) n_threads = n_tokens > 0 ? n_tokens : 1;
  if (n_threads == 1) {
    worker_arg A = {L, hs, tokens, n_tokens, 1, 0, mode, keep, ids, w, z, y};
    worker(&A);
    return;
  }
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
  worker_arg *A = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)n_threads);
  for (int i = 0; i < n_threads; ++i) {
    worker_arg a = {L, hs, tokens, n_tokens, n_threads, i, mode, keep, ids, w, z, y};
    A[i] = a;
    pthread_create(&th[i], NULL, worker, &A[i]);
  }
  for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
  free(A);
  free(th);
}

/* The verification pass for the tokens listed in `tokens` (all n tokens in
 * order when `tokens` is NULL; then n_tokens = n).  Output row i belongs to
 * token tokens[i].  Tokens are independent, so the loop may be split across
 * n_threads host threads without changing any result. */
int orc_verify(const orc_layer *L, const void *hs, const int32_t *tokens,
               int n_tokens, int n_threads, int32_t *ids, double *w, double *z,
               double *y) {
  run_workers(L, hs, tokens, n_tokens, n_threads, DO_ROUTE_AND_FFN, NULL, ids,
              w, z, y);
  return 0;
}

/* orc_verify with the routing given: ids[i][0..k) are token tokens[i]'s
 * experts (in [0, N), distinct), read instead of the top-k; the router
 * scores, the gate of those ids and the layer output are computed as in
 * orc_verify. */
int orc_verify_routed(const orc_layer *L, const void *hs, const int32_t *tokens,
                      int n_tokens, int n_threads, const int32_t *ids,
                      double *w, double *z, double *y) {
  run_workers(L, hs, tokens, n_tokens, n_threads, DO_GATE_AND_FFN, NULL,
              (int32_t *)ids, w, z, y);
  return 0;
}

/* TopK and gate on given fp32 scores (the same ordering, on exactly the
 * numbers a GPU produced, widened to double without rounding). */
void orc_topk_from_scores(const float *scores, int n, int n_experts, int k,
                          int gate, int32_t *ids, double *w) {
  double *z = (double *)malloc(sizeof(double) * (size_t)n_experts);
  for (int t = 0; t < n; ++t) {
    for (int e = 0; e < n_experts; ++e)
      z[e] = (double)scores[(size_t)t * n_experts + e];
    orc_topk(z, n_experts, k, ids + (size_t)t * k);
    orc_gate(z, n_experts, ids + (size_t)t * k, k, gate, w + (size_t)t * k);
  }
  free(z);
}

/* ------------------------------------------------------------ union plan */

/* The union of the routed experts of all n tokens and the grouping of the
 * n*k (token, slot) pairs by expert ("Less Experts, Faster Decoding", eq. (1);
 * "Making Every Verified Token Count", eq. (5)).
 *   hist[e]   number of slots that name expert e
 *   uniq[u]   the distinct experts, ascending (u < U)
 *   offs[u]   first position of expert uniq[u]'s group in perm; offs[U] = n*k
 *   perm[p]   slot indices t*k+j, grouped by expert in uniq order, ascending
 *             slot index inside a group
 * Returns U. */
int orc_union_plan(const int32_t *ids, int n_slots, int n_experts,
                   int32_t *hist, int32_t *uniq, int32_t *offs,
                   int32_t *perm) {
  int U = 0;
  for (int e = 0; e < n_experts; ++e) hist[e] = 0;
  for (int p = 0; p < n_slots; ++p) hist[ids[p]] += 1;
  for (int e = 0; e < n_experts; ++e)
    if (hist[e] > 0) uniq[U++] = e;
  int pos = 0;
  for (int u = 0; u < U; ++u) {
    offs[u] = pos;
    for (int p = 0; p < n_slots; ++p)
      if (ids[p] == uniq[u]) perm[pos++] = p;
  }
  offs[U] = pos;
  return U;
}

/* Bytes of one expert: the three d x I matrices, plus, for E4M3, the fp32
 * block scales ("Less Experts, Faster Decoding", Fig. 1(c): one FP8 expert of
 * a 7168 x 2048 layer is 44.04 MB). */
void orc_expert_bytes(int d, int inter, int w_type, int64_t *weights,
                      int64_t *scales) {
  *weights = (int64_t)3 * d * inter * (int64_t)elem_size(w_type);
  *scales = 0;
  if (w_type == ORC_E4M3)
    *scales = (int64_t)4 * (((int64_t)2 * inter / ORC_BLOCK) * (d / ORC_BLOCK) +
                            ((int64_t)d / ORC_BLOCK) * (inter / ORC_BLOCK));
}

/* ---------------------------------------------------------- expert budget */

/* Verification-time expert budgeting, MoE-Spec: each layer loads at most a
 * fixed number of experts, the most useful ones for the pass, and skips the
 * many that few slots use (its abstract, in the list of
 * related papers on "Speculative Decoding for Mixture-of-Experts Models:
 * Expert Bytes, Kernel Bandwidth and the Best Draft Length"; "The Limits of
 * Speculation", Sec. 2.4: the per-layer expert budget is capped; "Making
 * Every Verified Token Count", Sec. 5: the active expert set is truncated,
 * so the output is lossy).
 * The pages give no formula; the readings taken here:
 *   contribution of expert e  = the sum of the gate weights of the slots
 *                               that name e, added in ascending slot order
 *                               in double;
 *   kept experts              = the first `budget` of the used experts in
 *                               the order (contribution descending, id
 *                               ascending), all of them when U <= budget;
 *   a dropped slot            = its term is left out of the layer output;
 *                               the other weights are not renormalised;
 *   the shared expert         = always applied, not counted in the budget.
 *   keep[e]   1 for a kept expert, else 0
 *   score[e]  the contribution (0 for an expert no slot names)
 * Returns the number of kept experts. */
typedef struct {
  double score;
  int id;
} scored_expert;

static int cmp_contribution(const void *a, const void *b) {
  const scored_expert *x = (const scored_expert *)a, *y = (const scored_expert *)b;
  if (x->score != y->score) return x->score < y->score ? 1 : -1;
  return x->id < y->id ? -1 : (x->id > y->id ? 1 : 0);
}

int orc_expert_budget(const int32_t *ids, const double *w, int n_slots,
                      int n_experts, int budget, uint8_t *keep, double *score) {
  int *used = (int *)calloc((size_t)n_experts, sizeof(int));
  for (int e = 0; e < n_experts; ++e) {
    score[e] = 0.0;
    keep[e] = 0;
  }
  for (int p = 0; p < n_slots; ++p) {
    score[ids[p]] += w[p];
    used[ids[p]] = 1;
  }
  scored_expert *order = (scored_expert *)malloc(sizeof(scored_expert) * (size_t)(n_experts + 1));
  int U = 0;
  for (int e = 0; e < n_experts; ++e)
    if (used[e]) {
      order[U].score = score[e];
      order[U].id = e;
      ++U;
    }
  qsort(order, (size_t)U, sizeof(scored_expert), cmp_contribution);
  int kept = U < budget ? U : budget;
  for (int r = 0; r < kept; ++r) keep[order[r].id] = 1;
  free(order);
  free(used);
  return kept;
}

/* The union plan of the kept slots only (same layout as orc_union_plan, the
 * dropped slots absent from hist, uniq, offs and perm), and the weights the
 * layer output uses: w_kept[p] = w[p] for a kept slot, 0 for a dropped one.
 * Returns the kept union size. */
int orc_budget_plan(const int32_t *ids, const double *w, int n_slots,
                    int n_experts, int budget, uint8_t *keep, double *score,
                    int32_t *hist, int32_t *uniq, int32_t *offs, int32_t *perm,
                    double *w_kept) {
  orc_expert_budget(ids, w, n_slots, n_experts, budget, keep, score);
  int U = 0;
  for (int e = 0; e < n_experts; ++e) hist[e] = 0;
  for (int p = 0; p < n_slots; ++p) {
    w_kept[p] = keep[ids[p]] ? w[p] : 0.0;
    if (keep[ids[p]]) hist[ids[p]] += 1;
  }
  for (int e = 0; e < n_experts; ++e)
    if (hist[e] > 0) uniq[U++] = e;
  int pos = 0;
  for (int u = 0; u < U; ++u) {
    offs[u] = pos;
    for (int p = 0; p < n_slots; ++p)
      if (uniq[u] == ids[p]) perm[pos++] = p; /* kept slots, ascending */
  }
  offs[U] = pos;
  return U;
}

/* The verification pass of n tokens under an expert budget: every token is
 * routed, the kept experts are chosen from all n*k slots (the routed ids and
 * their double gate weights), and each output sums its token's kept slots
 * only (plus the shared expert).  Outputs are written for the tokens listed
 * in `tokens` (all n in order when NULL; then n_tokens = n): y row i belongs
 * to token tokens[i]; ids, w, z hold all n tokens.  keep: [N] out.  Returns
 * the number of kept experts. */
int orc_verify_budget(const orc_layer *L, const void *hs, int n,
                      const int32_t *tokens, int n_tokens, int n_threads,
                      int budget, int32_t *ids, double *w, double *z,
                      double *y, uint8_t *keep) {
  run_workers(L, hs, NULL, n, n_threads, DO_ROUTE, NULL, ids, w, z, NULL);
  double *score = (double *)malloc(sizeof(double) * (size_t)L->n_experts);
  int kept = orc_expert_budget(ids, w, n * L->top_k, L->n_experts, budget, keep, score);
  free(score);
  if (!tokens) {
    run_workers(L, hs, NULL, n, n_threads, DO_FFN, keep, ids, w, z, y);
    return kept;
  }
  /* the listed tokens' routing, gathered in list order */
  int k = L->top_k;
  int32_t *ids_l = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_tokens * k + 1));
  double *w_l = (double *)malloc(sizeof(double) * (size_t)(n_tokens * k + 1));
  for (int i = 0; i < n_tokens; ++i)
    for (int j = 0; j < k; ++j) {
      ids_l[(size_t)i * k + j] = ids[(size_t)tokens[i] * k + j];
      w_l[(size_t)i * k + j] = w[(size_t)tokens[i] * k + j];
    }
  run_workers(L, hs, tokens, n_tokens, n_threads, DO_FFN, keep, ids_l, w_l, NULL, y);
  free(w_l);
  free(ids_l);
  return kept;
}

/* ----------------------------------------------- pre-verification selection */

/* Draft trees: K nodes, node 0 the root (the token the target model already
 * sampled), parent[0] = -1 and 0 <= parent[v] < v for every other node.
 * q[v] is the draft model's probability of node v's token given its prefix. */

/* Cumulative draft score of every node ("Making Every Verified Token Count",
 * Sec. 3.1, eq. (7)): the product of q over the path from the root to v,
 * multiplied in path order from the root.  The root's own factor is 1 (a
 * reading: it is the target's token and is always accepted). */
void orc_tree_scores(const int32_t *parent, const float *q, int K, double *score) {
  int32_t *path = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K + 1));
  for (int v = 0; v < K; ++v) {
    int len = 0;
    for (int u = v; u > 0; u = parent[u]) path[len++] = u;  /* v up to a child of the root */
    double s = 1.0;                                         /* the root */
    for (int i = len - 1; i >= 0; --i) s *= (double)q[path[i]];
    score[v] = s;
  }
  free(path);
}

typedef struct {
  double s;
  int v;
} scored_node;

/* larger score first; equal scores, lower node index first (a reading) */
static int cmp_node(const void *a, const void *b) {
  const scored_node *x = (const scored_node *)a, *y = (const scored_node *)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->v > y->v) - (x->v < y->v);
}

/* EVICT's utility-guided prefix ("Making Every Verified Token Count",
 * Sec. 3.2): T_k = the k nodes of largest score (Sec. 3.2.1);
 * E_hat[A(T_k)] = the sum of their scores (eq. (8)), added in rank order;
 * the utility of k is E_hat[A(T_k)] / C(k) (eq. (9) without the constant
 * C_AR); k* = the k in 1..K of largest utility (eq. (10)), the smallest k on
 * a tie (a reading).  cost[k-1] = C(k), widened to double.
 *   order[r]    node of rank r           exp_len[k-1]  E_hat[A(T_k)]
 *   utility[k-1]                         returns k* */
int orc_evict_select(const int32_t *parent, const float *q, int K, const float *cost,
                     int32_t *order, double *exp_len, double *utility) {
  double *score = (double *)malloc(sizeof(double) * (size_t)K);
  scored_node *sn = (scored_node *)malloc(sizeof(scored_node) * (size_t)K);
  orc_tree_scores(parent, q, K, score);
  for (int v = 0; v < K; ++v) {
    sn[v].s = score[v];
    sn[v].v = v;
  }
  qsort(sn, (size_t)K, sizeof(scored_node), cmp_node);
  double acc = 0.0;
  int best = 1;
  for (int k = 1; k <= K; ++k) {
    order[k - 1] = sn[k - 1].v;
    acc += sn[k - 1].s;
    exp_len[k - 1] = acc;
    utility[k - 1] = acc / (double)cost[k - 1];
    if (utility[k - 1] > utility[best - 1]) best = k;
  }
  free(sn);
  free(score);
  return best;
}

/* EcoSpec's cost-aware draft selection ("Less Experts, Faster Decoding",
 * Sec. 4.2, eqs. (7)-(9), and its appendix algorithm): starting from the
 * buffer B = B0, gamma times (all K nodes when gamma > K):
 *   for every unselected node t:  E_traj(t) = the union of the predicted
 *     expert sets over the path from the root to t (eq. (7));
 *     cost = |E_traj(t) \ B| (eq. (8));  score = P(t) / (cost + eps) (eq. (9)),
 *     P(t) the cumulative draft score of orc_tree_scores;
 *   select the node of largest score (lowest index on a tie: a reading) and
 *   add E_traj of it to B.
 * Expert sets are sets of (layer, expert) pairs: pred_ids[v][l][j], j < kp,
 * names the experts predicted for node v at layer l (ids outside [0, E) are
 * ignored).  buf0: [L][E] bytes, nonzero = in B0, or NULL for an empty B0.
 *   selected[i]  the i-th selected node     buf_out  [L][E], the final B
 * Returns |B| at the end. */
int orc_ecospec_select(const int32_t *parent, const float *q, const int32_t *pred_ids,
                       int K, int L, int E, int kp, int gamma, const uint8_t *buf0,
                       double eps, int32_t *selected, uint8_t *buf_out) {
  const size_t LE = (size_t)L * (size_t)E;
  double *P = (double *)malloc(sizeof(double) * (size_t)K);
  uint8_t *traj = (uint8_t *)calloc((size_t)K * LE, 1);
  uint8_t *taken = (uint8_t *)calloc((size_t)K, 1);
  orc_tree_scores(parent, q, K, P);
  /* eq. (7): walk every node's path and mark the predicted pairs */
  for (int v = 0; v < K; ++v) {
    uint8_t *tv = traj + (size_t)v * LE;
    for (int u = v;; u = parent[u]) {
      for (int l = 0; l < L; ++l)
        for (int j = 0; j < kp; ++j) {
          const int e = pred_ids[((size_t)u * L + l) * kp + j];
          if (e >= 0 && e < E) tv[(size_t)l * E + e] = 1;
        }
      if (u == 0) break;
    }
  }
  for (size_t i = 0; i < LE; ++i) buf_out[i] = buf0 ? (buf0[i] != 0) : 0;
  const int n_sel = gamma < K ? gamma : K;
  for (int it = 0; it < n_sel; ++it) {
    int best = -1;
    double best_score = 0.0;
    for (int v = 0; v < K; ++v) {
      if (taken[v]) continue;
      const uint8_t *tv = traj + (size_t)v * LE;
      int cost = 0;
      for (size_t i = 0; i < LE; ++i) cost += tv[i] && !buf_out[i];
      const double score = P[v] / ((double)cost + eps);
      if (best < 0 || score > best_score) {
        best = v;
        best_score = score;
      }
    }
    selected[it] = best;
    taken[best] = 1;
    const uint8_t *tb = traj + (size_t)best * LE;
    for (size_t i = 0; i < LE; ++i) buf_out[i] |= tb[i];
  }
  int count = 0;
  for (size_t i = 0; i < LE; ++i) count += buf_out[i];
  free(taken);
  free(traj);
  free(P);
  return count;
}
