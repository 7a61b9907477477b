// api.cu -- the C ABI (include/moe_verify.h): argument checks on the host,
// then the launches of one verification pass on the caller's stream.
// Nothing here allocates device memory or synchronises the host, except
// moe_last_error().
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "kernels.h"
#include "moe_common.cuh"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr int MAX_EXPERTS = 256;
constexpr int MAX_TOPK = 32;
constexpr int MAX_TOKENS = 64;
constexpr uint64_t DEFAULT_TIMEOUT_NS = 1000ull * 1000 * 1000;
// Passes of fewer tokens run the mma.sync instance alone, whose segments of
// 9-24 tokens take 2-3 passes over their weights: against it, the instance
// with tcgen05 CTAs measured 3-8% slower at n = 9-16 (dedup calls and passes,
// Qwen3- and OLMoE-shaped; 4-5% on 48-layer stacks), between -4% and +8% at
// n = 17-24 depending on the tree, and never slower from n = 32 (to 25% faster).
constexpr int WIDE_MIN_TOKENS = 25;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_desc(const moe_layer_desc *L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (L->d <= 0 || L->n_experts <= 0 || L->top_k <= 0 || L->inter <= 0 || L->n_max <= 0 ||
      L->n_shared < 0 || L->wait_timeout_us < 0)
    return MOE_ERR_INVALID_ARG;
  if (L->top_k > L->n_experts) return MOE_ERR_INVALID_ARG;
  if (L->act_dtype != MOE_F32 && L->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (L->w_dtype != MOE_F32 && L->w_dtype != MOE_BF16 && L->w_dtype != MOE_E4M3_B128)
    return MOE_ERR_INVALID_ARG;
  if (L->gate != MOE_GATE_SOFTMAX && L->gate != MOE_GATE_SOFTMAX_RENORM &&
      L->gate != MOE_GATE_SIGMOID_RENORM)
    return MOE_ERR_INVALID_ARG;
  if (L->n_experts > MAX_EXPERTS || L->top_k > MAX_TOPK || L->n_max > MAX_TOKENS ||
      L->n_shared > 1)
    return MOE_ERR_UNSUPPORTED;
  // fp32 weights go with fp32 activations; bf16/E4M3 weights with bf16 ones
  if ((L->w_dtype == MOE_F32) != (L->act_dtype == MOE_F32)) return MOE_ERR_UNSUPPORTED;
  if (L->d % 8) return MOE_ERR_UNSUPPORTED;
  switch (L->w_dtype) {
    case MOE_F32:
      if (L->inter % 4) return MOE_ERR_UNSUPPORTED;
      break;
    case MOE_BF16:
      // whole 128-byte columns of the swizzled tile layout in W13 and W2
      if (L->d % 64 || L->inter % 64) return MOE_ERR_UNSUPPORTED;
      break;
    default:
      if (L->d % 128 || L->inter % 128) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

size_t w_size(const moe_layer_desc &L) {
  return L.w_dtype == MOE_F32 ? 4 : L.w_dtype == MOE_BF16 ? 2 : 1;
}

void expert_bytes(const moe_layer_desc &L, int64_t *wb, int64_t *sb) {
  *wb = int64_t(3) * L.d * L.inter * int64_t(w_size(L));
  *sb = 0;
  if (L.w_dtype == MOE_E4M3_B128)
    *sb = int64_t(4) * ((int64_t(2) * L.inter / 128) * (L.d / 128) +
                        (int64_t(L.d) / 128) * (L.inter / 128));
}

uint64_t timeout_ns(const moe_layer_desc &L) {
  return L.wait_timeout_us > 0 ? uint64_t(L.wait_timeout_us) * 1000ull : DEFAULT_TIMEOUT_NS;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_weights(const moe_layer_desc &L, const moe_expert_weights *W) {
  if (!W || !W->w13 || !W->w2) return MOE_ERR_INVALID_ARG;
  if (!aligned16(W->w13) || !aligned16(W->w2)) return MOE_ERR_ALIGNMENT;
  if (L.n_shared) {
    if (!W->sh_w13 || !W->sh_w2) return MOE_ERR_INVALID_ARG;
    if (!aligned16(W->sh_w13) || !aligned16(W->sh_w2)) return MOE_ERR_ALIGNMENT;
  }
  return MOE_OK;
}

// Where the E4M3 engines' fp16 hidden rows live in a workspace.
ActScaleOut act_scale_out(const moe_layer_desc &L, void *workspace, bool counted) {
  const Workspace ws = workspace_layout(L);
  uint8_t *wsb = static_cast<uint8_t *>(workspace);
  ActScaleOut S;
  S.h16 = reinterpret_cast<__half *>(wsb + ws.h16);
  S.hshift = reinterpret_cast<int32_t *>(wsb + ws.hshift);
  S.acts = counted ? reinterpret_cast<unsigned int *>(wsb + WS_ACTS_OFFSET) : nullptr;
  return S;
}

// The expert FFN of one pass (both phases) and the combine, for either engine.
// early_shared: the caller has just enqueued this pass's plan kernel on
// `stream` (moe_verify_pass), so phase 1 may start the shared expert before
// that kernel ends; that kernel has also written the E4M3 engines' fp16
// hidden rows (counting them in the workspace header), which otherwise a
// kernel of their own writes here.
moe_status run_experts(const moe_layer_desc &L, const moe_expert_weights &W, const void *h, int n,
                       const int32_t *ids, const float *w, const moe_plan *plan, void *workspace,
                       void *y, cudaStream_t stream, bool early_shared = false) {
  const Workspace ws = workspace_layout(L);
  uint8_t *wsb = static_cast<uint8_t *>(workspace);
  int32_t *err = reinterpret_cast<int32_t *>(wsb);
  const int sms = sm_count();
  if (sms <= 0) return MOE_ERR_CUDA;
  uint32_t *ready = reinterpret_cast<uint32_t *>(wsb + WS_READY_OFFSET);

  SegTables T;
  memset(&T, 0, sizeof T);
  T.ids = ids;
  T.n = n;
  T.k = L.top_k;
  T.n_experts = L.n_experts;
  T.n_shared = L.n_shared;
  T.dedup = plan != nullptr;
  if (plan) {
    T.uniq = plan->uniq;
    T.offs = plan->offs;
    T.perm = plan->perm;
    T.n_uniq = plan->n_uniq;
  }
  cudaError_t e = cudaSuccess;
  if (L.w_dtype == MOE_F32) {
    F32Params P;
    P.T = T;
    P.w13 = static_cast<const float *>(W.w13);
    P.w2 = static_cast<const float *>(W.w2);
    P.sh_w13 = static_cast<const float *>(W.sh_w13);
    P.sh_w2 = static_cast<const float *>(W.sh_w2);
    P.d = L.d;
    P.inter = L.inter;
    P.h = static_cast<const float *>(h);
    P.inter_out = reinterpret_cast<float *>(wsb + ws.inter);
    P.yslot = reinterpret_cast<float *>(wsb + ws.yslot);
    P.err = err;
    e = launch_expert_f32(1, P, 2 * sms, stream);
    if (e == cudaSuccess) e = launch_expert_f32(2, P, 2 * sms, stream);
  } else {
    const bool fp8 = L.w_dtype == MOE_E4M3_B128;
    const void *act = h;  // bf16; E4M3: the fp16 rows of act_scale.cuh
    const ActScaleOut S = act_scale_out(L, workspace, early_shared);
    if (fp8) {
      act = S.h16;
      if (!early_shared) e = launch_act_scale(h, n, L.d, S, stream);
    }
    // One 8-token mma.sync tile per pass over a work item.  A BF16 segment of
    // more tokens in a pass of WIDE_MIN_TOKENS or more runs on tcgen05 CTAs,
    // all its tokens in one pass (P.wide); otherwise (and for E4M3, e.g. the
    // shared expert at n > 8) a segment takes one pass per 8 tokens.
    // Wider mma.sync tiles (2 or 4 per pass) fit in registers, but their
    // activation rows leave the ring 3 or 4 stages, and they measured slower
    // than the extra passes.
    const int n_tiles = 1;
    TcParams P;
    P.T = T;
    P.err = err;
    P.timeout_ns = timeout_ns(L);
    // Segments of more than 8 tokens on tcgen05 CTAs (BF16, deduplicating,
    // n >= WIDE_MIN_TOKENS).  Their B operands come through TMA tensor maps:
    // phase 1 all n hidden rows in one box, phase 2 boxes of 16, 32, 48 or
    // 64 rows of aperm.  A driver that cannot encode them leaves the pass to
    // the mma.sync CTAs alone (same outputs, up to the summation order).
    P.wide = (!fp8 && plan != nullptr && n >= WIDE_MIN_TOKENS) ? 1 : 0;
    P.aperm = wsb + ws.aperm;
    const int slots = n * (L.top_k + L.n_shared);
    CUtensorMap down_maps[4];
    if (P.wide) {
      cudaError_t me = encode_act_map(&P.act_map[0], h, n, L.d, (n + 15) & ~15);
      for (int j = 0; j < 4 && me == cudaSuccess; ++j)
        me = encode_act_map(&down_maps[j], P.aperm, slots, L.inter, 16 * (j + 1));
      if (me != cudaSuccess) P.wide = 0;
    }
    P.early_shared = early_shared && plan != nullptr && !P.wide;
    P.ready = P.early_shared ? ready : nullptr;
    int32_t *ashift = reinterpret_cast<int32_t *>(wsb + ws.ashift);
    P.hshift = S.hshift;
    P.ashift = ashift;
    P.acts = fp8 && P.early_shared ? S.acts : nullptr;
    P.inter = L.inter;
    const size_t es = w_size(L);
    // phase 1: gate/up over W13, K = d
    P.w = static_cast<const uint8_t *>(W.w13);
    P.w_sh = static_cast<const uint8_t *>(W.sh_w13);
    P.expert_stride = packed_matrix_bytes(2 * L.inter, int(L.d * es), fp8);
    P.rows_total = 2 * L.inter;
    P.kdim = L.d;
    P.row_blocks = L.inter / 32;
    P.act = act;
    P.out = wsb + ws.inter;
    if (e == cudaSuccess) e = launch_expert_tc(fp8, 1, n_tiles, P, sms, stream);
    // E4M3: each slot's row of a into fp16 range, in place
    if (fp8 && e == cudaSuccess)
      e = launch_a16_scale(wsb + ws.inter, slots, L.inter, ashift, sms, stream);
    // phase 2: down over W2, K = I
    P.w = static_cast<const uint8_t *>(W.w2);
    P.w_sh = static_cast<const uint8_t *>(W.sh_w2);
    P.expert_stride = packed_matrix_bytes(L.d, int(L.inter * es), fp8);
    P.rows_total = L.d;
    P.kdim = L.inter;
    P.row_blocks = L.d / 64;
    P.act = wsb + ws.inter;
    P.out = wsb + ws.yslot;
    if (P.wide)
      for (int j = 0; j < 4; ++j) P.act_map[j] = down_maps[j];
    if (e == cudaSuccess) e = launch_expert_tc(fp8, 2, n_tiles, P, sms, stream);
  }
  if (e == cudaSuccess)
    e = launch_combine(reinterpret_cast<const float *>(wsb + ws.yslot), w, n, L.top_k, L.d,
                       L.n_shared, L.act_dtype == MOE_BF16, y, early_shared ? ready : nullptr,
                       stream);
  return cuda_status(e);
}

moe_status check_verify_args(const moe_layer_desc *desc, const moe_expert_weights *weights,
                             const void *h, int32_t n, const int32_t *ids, const float *w,
                             void *workspace, size_t ws_bytes, void *y) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;  // nothing is read or written
  s = check_weights(*desc, weights);
  if (s != MOE_OK) return s;
  if (!h || !ids || !w || !workspace || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(ids) || !aligned16(w) || !aligned16(workspace) ||
      !aligned16(y))
    return MOE_ERR_ALIGNMENT;
  if (ws_bytes < workspace_layout(*desc).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// Waits on a barrier that nothing arrives on; the wait must give up.
__global__ void bounded_wait_selftest_kernel(int32_t *err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const bool done = mbar_wait_bounded(&bar, 0, limit_ns);
  if (!done && threadIdx.x == 0) record_error(err, MOE_ERR_TIMEOUT);
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_selftest_bounded_wait(int32_t *error_word, int32_t limit_us,
                                             moe_stream_t stream) {
  if (!error_word || limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      error_word, uint64_t(limit_us) * 1000ull);
  return cuda_status(cudaGetLastError());
}

MOE_API size_t moe_workspace_bytes(const moe_layer_desc *desc) {
  if (check_desc(desc) != MOE_OK) return 0;
  return workspace_layout(*desc).total;
}

MOE_API moe_status moe_expert_bytes(const moe_layer_desc *desc, int64_t *weight_bytes,
                                    int64_t *scale_bytes) {
  const moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  int64_t wb, sb;
  expert_bytes(*desc, &wb, &sb);
  if (weight_bytes) *weight_bytes = wb;
  if (scale_bytes) *scale_bytes = sb;
  return MOE_OK;
}

MOE_API moe_status moe_route_topk(const moe_layer_desc *desc, const void *router_w, const void *h,
                                  int32_t n, int32_t *ids, float *w, float *logits,
                                  moe_stream_t stream) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;  // nothing is read or written
  if (!router_w || !h || !ids || !w || !logits) return MOE_ERR_INVALID_ARG;
  if (!aligned16(router_w) || !aligned16(h) || !aligned16(ids) || !aligned16(w) ||
      !aligned16(logits))
    return MOE_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_router_scores(desc->act_dtype == MOE_BF16, router_w, h, n, desc->d,
                                       desc->n_experts, logits, st);
  if (e == cudaSuccess)
    e = launch_topk_gate(logits, n, desc->n_experts, desc->top_k, desc->gate, ids, w, st);
  return cuda_status(e);
}

MOE_API moe_status moe_topk_from_logits(const moe_layer_desc *desc, const float *logits,
                                        int32_t n, int32_t *ids, float *w, moe_stream_t stream) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;  // nothing is read or written
  if (!logits || !ids || !w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(ids) || !aligned16(w)) return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_topk_gate(logits, n, desc->n_experts, desc->top_k, desc->gate, ids, w,
                                      static_cast<cudaStream_t>(stream)));
}

namespace moe {
namespace {

moe_status check_plan(const moe_plan *plan) {
  if (!plan || !plan->hist || !plan->uniq || !plan->n_uniq || !plan->offs || !plan->perm ||
      !plan->union_bytes)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(plan->hist) || !aligned16(plan->uniq) || !aligned16(plan->offs) ||
      !aligned16(plan->perm))
    return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

// budget < 0: the plain plan (w, w_kept, routed_u unused).
moe_status union_plan(const moe_layer_desc *desc, const int32_t *ids, const float *w, int32_t n,
                      int32_t budget, const moe_plan *plan, float *w_kept, int32_t *routed_u,
                      int32_t *error_word, cudaStream_t st) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if ((s = check_plan(plan)) != MOE_OK) return s;
  if (n > 0 && (!ids || (budget >= 0 && (!w || !w_kept)))) return MOE_ERR_INVALID_ARG;
  if ((ids && !aligned16(ids)) || (w && !aligned16(w)) || (w_kept && !aligned16(w_kept)))
    return MOE_ERR_ALIGNMENT;
  int64_t wb, sb;
  expert_bytes(*desc, &wb, &sb);
  const int n_slots = n * desc->top_k;
  if (budget < 0)
    return cuda_status(launch_union_plan(ids, n_slots, desc->n_experts, desc->n_shared, wb + sb,
                                         plan->hist, plan->uniq, plan->n_uniq, plan->offs,
                                         plan->perm, plan->union_bytes, error_word, st));
  return cuda_status(launch_union_plan_budgeted(
      ids, w, n_slots, desc->n_experts, desc->n_shared, wb + sb, budget, plan->hist, plan->uniq,
      plan->n_uniq, plan->offs, plan->perm, plan->union_bytes, w_kept, routed_u, error_word, st));
}

// signal_ready: raise the plan-ready flag of the workspace once the plan is
// written, and for E4M3 weights write the expert kernels' fp16 rows into the
// workspace, counted in its header (moe_verify_pass only, whose workspace
// has been checked whole; its combine clears both words).
moe_status route_plan(const moe_layer_desc *desc, const void *router_w, const void *h, int32_t n,
                      int32_t budget, int32_t *ids, float *w, float *logits, const moe_plan *plan,
                      float *w_kept, int32_t *routed_u, void *workspace, size_t ws_bytes,
                      cudaStream_t st, bool signal_ready = false) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if ((s = check_plan(plan)) != MOE_OK) return s;
  if (!workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MOE_ERR_ALIGNMENT;
  if (ws_bytes < 256) return MOE_ERR_WORKSPACE;
  int64_t wb, sb;
  expert_bytes(*desc, &wb, &sb);
  uint8_t *wsb = static_cast<uint8_t *>(workspace);
  int32_t *err = reinterpret_cast<int32_t *>(wsb);
  if (n == 0)  // the empty plan: U = 0, offs[0] = 0
    return union_plan(desc, nullptr, nullptr, 0, budget, plan, nullptr, routed_u, err, st);
  if (!router_w || !h || !ids || !w || !logits || (budget >= 0 && !w_kept))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(router_w) || !aligned16(h) || !aligned16(ids) || !aligned16(w) ||
      !aligned16(logits) || (w_kept && !aligned16(w_kept)))
    return MOE_ERR_ALIGNMENT;
  ActScaleOut S = act_scale_out(*desc, workspace, true);
  if (!signal_ready || desc->w_dtype != MOE_E4M3_B128) S.acts = nullptr;
  return cuda_status(launch_route_plan(
      desc->act_dtype == MOE_BF16, router_w, h, n, desc->d, desc->n_experts, desc->top_k,
      desc->gate, desc->n_shared, wb + sb, logits, ids, w, plan->hist, plan->uniq, plan->n_uniq,
      plan->offs, plan->perm, plan->union_bytes, budget, w_kept, routed_u, err,
      reinterpret_cast<unsigned int *>(wsb + WS_TICKET_OFFSET),
      reinterpret_cast<unsigned int *>(wsb + WS_GROUP_TICKETS_OFFSET),
      signal_ready ? reinterpret_cast<unsigned int *>(wsb + WS_READY_OFFSET) : nullptr, S, st));
}

}  // namespace
}  // namespace moe

MOE_API moe_status moe_union_plan(const moe_layer_desc *desc, const int32_t *ids, int32_t n,
                                  const moe_plan *plan, int32_t *error_word,
                                  moe_stream_t stream) {
  return union_plan(desc, ids, nullptr, n, -1, plan, nullptr, nullptr, error_word,
                    static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_union_plan_budgeted(const moe_layer_desc *desc, const int32_t *ids,
                                           const float *w, int32_t n, int32_t budget,
                                           const moe_plan *plan, float *w_kept,
                                           int32_t *routed_union, int32_t *error_word,
                                           moe_stream_t stream) {
  if (budget < 0) return MOE_ERR_INVALID_ARG;
  return union_plan(desc, ids, w, n, budget, plan, w_kept, routed_union, error_word,
                    static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_route_plan(const moe_layer_desc *desc, const void *router_w, const void *h,
                                  int32_t n, int32_t *ids, float *w, float *logits,
                                  const moe_plan *plan, void *workspace, size_t ws_bytes,
                                  moe_stream_t stream) {
  return route_plan(desc, router_w, h, n, -1, ids, w, logits, plan, nullptr, nullptr, workspace,
                    ws_bytes, static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_route_plan_budgeted(const moe_layer_desc *desc, const void *router_w,
                                           const void *h, int32_t n, int32_t budget,
                                           int32_t *ids, float *w, float *logits,
                                           const moe_plan *plan, float *w_kept,
                                           int32_t *routed_union, void *workspace,
                                           size_t ws_bytes, moe_stream_t stream) {
  if (budget < 0) return MOE_ERR_INVALID_ARG;
  return route_plan(desc, router_w, h, n, budget, ids, w, logits, plan, w_kept, routed_union,
                    workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_evict_select(const int32_t *parent, const float *q, int32_t n_trees,
                                    int32_t n_nodes, const float *cost, int32_t *order,
                                    double *exp_len, double *utility, int32_t *k_star,
                                    int32_t *error_word, moe_stream_t stream) {
  if (n_trees < 0 || n_nodes < 1 || n_nodes > SEL_MAX_NODES) return MOE_ERR_INVALID_ARG;
  if (n_trees == 0) return MOE_OK;
  if (!parent || !q || !cost || !order || !k_star) return MOE_ERR_INVALID_ARG;
  if (!aligned16(parent) || !aligned16(q) || !aligned16(cost) || !aligned16(order) ||
      !aligned16(k_star) || (exp_len && !aligned16(exp_len)) ||
      (utility && !aligned16(utility)))
    return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_evict_select(parent, q, n_trees, n_nodes, cost, order, exp_len,
                                         utility, k_star, error_word,
                                         static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status moe_ecospec_select(const int32_t *parent, const float *q,
                                      const int32_t *pred_ids, int32_t n_trees, int32_t n_nodes,
                                      int32_t n_layers, int32_t n_experts, int32_t pred_k,
                                      int32_t gamma, double eps, const uint32_t *buffer0,
                                      int32_t *selected, uint32_t *buffer_out,
                                      int32_t *union_size, int32_t *error_word,
                                      moe_stream_t stream) {
  if (n_trees < 0 || n_nodes < 1 || n_nodes > SEL_MAX_NODES || n_layers < 1 || n_experts < 1 ||
      pred_k < 1 || gamma < 0 || !(eps > 0.0))
    return MOE_ERR_INVALID_ARG;
  if (ecospec_smem_bytes(n_nodes, n_layers, n_experts) > SEL_MAX_SMEM) return MOE_ERR_UNSUPPORTED;
  if (n_trees == 0) return MOE_OK;
  if (!parent || !q || !pred_ids || !union_size || (gamma > 0 && !selected))
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(parent) || !aligned16(q) || !aligned16(pred_ids) || !aligned16(union_size) ||
      (selected && !aligned16(selected)) || (buffer0 && !aligned16(buffer0)) ||
      (buffer_out && !aligned16(buffer_out)))
    return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_ecospec_select(parent, q, pred_ids, n_trees, n_nodes, n_layers,
                                           n_experts, pred_k, gamma, eps, buffer0, selected,
                                           buffer_out, union_size, error_word,
                                           static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status moe_verify_dedup(const moe_layer_desc *desc, const moe_expert_weights *weights,
                                    const void *h, int32_t n, const int32_t *ids, const float *w,
                                    const moe_plan *plan, void *workspace, size_t ws_bytes,
                                    void *y, moe_stream_t stream) {
  moe_status s = check_verify_args(desc, weights, h, n, ids, w, workspace, ws_bytes, y);
  if (s != MOE_OK) return s;
  if (!plan || !plan->uniq || !plan->offs || !plan->perm || !plan->n_uniq)
    return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  return run_experts(*desc, *weights, h, n, ids, w, plan, workspace, y,
                     static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_verify_pass(const moe_layer_desc *desc, const moe_expert_weights *weights,
                                   const void *router_w, const void *h, int32_t n,
                                   int32_t budget, int32_t *ids, float *w, float *logits,
                                   const moe_plan *plan, float *w_kept, int32_t *routed_union,
                                   void *workspace, size_t ws_bytes, void *y,
                                   moe_stream_t stream) {
  moe_status s = check_verify_args(desc, weights, h, n, n > 0 ? ids : nullptr,
                                   n > 0 ? w : nullptr, workspace, ws_bytes, y);
  if (s != MOE_OK) return s;
  if (budget < -1) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = route_plan(desc, router_w, h, n, budget, ids, w, logits, plan, w_kept, routed_union,
                 workspace, ws_bytes, st, /*signal_ready=*/true);
  if (s != MOE_OK || n == 0) return s;
  return run_experts(*desc, *weights, h, n, ids, budget >= 0 ? w_kept : w, plan, workspace, y,
                     st, true);
}

MOE_API moe_status moe_verify_perslot(const moe_layer_desc *desc,
                                      const moe_expert_weights *weights, const void *h, int32_t n,
                                      const int32_t *ids, const float *w, void *workspace,
                                      size_t ws_bytes, void *y, moe_stream_t stream) {
  moe_status s = check_verify_args(desc, weights, h, n, ids, w, workspace, ws_bytes, y);
  if (s != MOE_OK) return s;
  if (n == 0) return MOE_OK;
  return run_experts(*desc, *weights, h, n, ids, w, nullptr, workspace, y,
                     static_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Deduplicating pass without caller-provided scratch.
//
// For callers that cannot hand the library a workspace: code whose device
// memory is owned by a framework allocator it may not bypass, or a hot path
// that must never call cudaMalloc (which can synchronise the device and whose
// failure it could not handle there).  The scratch of such a call lives in
// this fixed, file-scope device array, which every GPU that loads the library
// keeps until the process exits.  All calls share it: it holds whatever the
// last call left, so calls whose execution overlaps on the GPU (e.g. on two
// streams, or from two threads) race and must be serialised by the caller.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[NOALLOC_MAX_DEVICES] = {nullptr};

// The array's device address on the current device (host code only holds a
// stand-in symbol, not a usable address).  Outside stream capture it is
// looked up on every call, so that an address that changed (after a device
// reset, the module is loaded again) is never used stale; during capture,
// where the lookup may not run, the address found by an earlier call is
// used, and without one the call returns MOE_ERR_UNSUPPORTED.
moe_status noalloc_scratch(cudaStream_t st, void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES)
    return MOE_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (cs == cudaStreamCaptureStatusNone) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  } else if (!g_noalloc_addr[dev]) {
    return MOE_ERR_UNSUPPORTED;
  }
  *out = g_noalloc_addr[dev];
  return MOE_OK;
}
}  // namespace

MOE_API moe_status moe_verify_dedup_noalloc(const moe_layer_desc *desc,
                                            const moe_expert_weights *weights, const void *h,
                                            int32_t n, const int32_t *ids, const float *w,
                                            const moe_plan *plan, void *y, int32_t *error_word,
                                            moe_stream_t stream) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n < 0 || n > desc->n_max) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  s = check_weights(*desc, weights);
  if (s != MOE_OK) return s;
  if (!h || !ids || !w || !y || !plan || !plan->uniq || !plan->offs || !plan->perm ||
      !plan->n_uniq)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(ids) || !aligned16(w) || !aligned16(y) ||
      (error_word && (reinterpret_cast<uintptr_t>(error_word) & 3u)))
    return MOE_ERR_ALIGNMENT;
  // the scratch this call needs, laid out for exactly n tokens
  moe_layer_desc L = *desc;
  L.n_max = n;
  if (workspace_layout(L).total > NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void *scratch = nullptr;
  s = noalloc_scratch(st, &scratch);
  if (s != MOE_OK) return s;
  // the error word must start at zero; the rest is fully written before it is read
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) return MOE_ERR_CUDA;
  s = run_experts(L, *weights, h, n, ids, w, plan, scratch, y, st);
  if (s != MOE_OK) return s;
  if (error_word &&
      cudaMemcpyAsync(error_word, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

MOE_API moe_status moe_packed_bytes(const moe_layer_desc *desc, int64_t *w13_bytes,
                                    int64_t *w2_bytes) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  const moe_layer_desc &L = *desc;
  const int es = int(w_size(L));
  const bool fp8 = L.w_dtype == MOE_E4M3_B128;
  const bool tiled = L.w_dtype != MOE_F32;
  if (w13_bytes)
    *w13_bytes = tiled ? packed_matrix_bytes(2 * L.inter, L.d * es, fp8)
                       : int64_t(2) * L.inter * L.d * es;
  if (w2_bytes)
    *w2_bytes = tiled ? packed_matrix_bytes(L.d, L.inter * es, fp8) : int64_t(L.d) * L.inter * es;
  return MOE_OK;
}

MOE_API moe_status moe_pack_expert_weights(const moe_layer_desc *desc, const void *w13,
                                           const void *w2, const float *s13, const float *s2,
                                           int32_t n_matrices, void *w13_packed, void *w2_packed,
                                           moe_stream_t stream) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (n_matrices < 0) return MOE_ERR_INVALID_ARG;
  if (n_matrices == 0) return MOE_OK;
  if (!w13 || !w2 || !w13_packed || !w2_packed) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w13) || !aligned16(w2) || !aligned16(w13_packed) || !aligned16(w2_packed))
    return MOE_ERR_ALIGNMENT;
  if (w13 == w13_packed || w2 == w2_packed) return MOE_ERR_INVALID_ARG;  // not in place
  const moe_layer_desc &L = *desc;
  const bool fp8 = L.w_dtype == MOE_E4M3_B128;
  if (fp8 && (!s13 || !s2)) return MOE_ERR_INVALID_ARG;
  if (fp8 && (!aligned16(s13) || !aligned16(s2))) return MOE_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t es = w_size(L);
  const size_t n13 = size_t(n_matrices) * 2 * L.inter * L.d * es;
  const size_t n2 = size_t(n_matrices) * L.d * L.inter * es;
  cudaError_t e;
  if (L.w_dtype == MOE_F32) {
    // the fp32 kernel reads the row-major layout itself
    e = cudaMemcpyAsync(w13_packed, w13, n13, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(w2_packed, w2, n2, cudaMemcpyDeviceToDevice, st);
  } else {
    e = launch_pack(w13, fp8 ? s13 : nullptr, w13_packed, n_matrices, 2 * L.inter, int(L.d * es),
                    L.inter, true, st);
    if (e == cudaSuccess)
      e = launch_pack(w2, fp8 ? s2 : nullptr, w2_packed, n_matrices, L.d, int(L.inter * es),
                      L.inter, false, st);
  }
  return cuda_status(e);
}

MOE_API moe_status moe_workspace_init(void *workspace, size_t ws_bytes, moe_stream_t stream) {
  if (!workspace || ws_bytes < 256) return MOE_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return MOE_ERR_ALIGNMENT;
  return cuda_status(cudaMemsetAsync(workspace, 0, 256, static_cast<cudaStream_t>(stream)));
}

MOE_API moe_status moe_last_error(void *workspace, moe_stream_t stream) {
  if (!workspace) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaMemset(workspace, 0, sizeof word) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(word);
}

MOE_API const char *moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or type combination";
    case MOE_ERR_ALIGNMENT: return "device array not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_INPUT: return "expert id out of range on the device";
  }
  return "unknown status";
}
