// kernels.h -- launchers of the library's kernels (internal; C++ linkage).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_common.cuh"

namespace moe {

// Launches `kern` with the programmatic stream serialization attribute, so
// that it may start while the kernel ahead of it in the stream is still
// running (the kernel itself calls pdl_wait() before it reads that kernel's
// results).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Parameters of one launch of the tensor-core expert kernel (expert_tc.cu).
struct TcParams {
  SegTables T;
  const uint8_t *w;       // routed experts' matrix (W13 or W2), expert-major
  const uint8_t *w_sh;    // the shared expert's matrix, or null
  int64_t expert_stride;  // bytes between consecutive experts in `w` (packed)
  int32_t rows_total;     // rows of one expert's matrix: 2I (phase 1) or d (phase 2)
  int32_t kdim;           // columns: d (phase 1) or I (phase 2)
  int32_t inter;          // I
  int32_t row_blocks;     // work items per segment: I/32 (phase 1) or d/64 (phase 2)
  const void *act;        // phase 1: hidden states [n][d] (bf16) by token; phase 2: a [slots][I]
  void *out;              // phase 1: a [slots][I]; phase 2: yslot [slots][d] fp32
  int32_t *err;           // workspace error word
  uint64_t timeout_ns;    // limit of every wait
  // 1 when the kernel ahead of phase 1 in the stream is the same pass's
  // plan kernel, which writes nothing phase 1 reads except the plan: phase 1
  // may then start the shared expert before that kernel ends
  int32_t early_shared;
  uint32_t *ready;  // early_shared: the plan kernel's plan-ready flag
  // E4M3 weights (fp16 MMA; act_scale.cuh): phase 1's `act` is the fp16
  // rows h16, token t scaled by 2^hshift[t], and it writes a in bf16; phase
  // 2's `act` is a in fp16, row `slot` scaled by 2^ashift[slot].  Each phase
  // scales its sums back.  With early_shared, the rows h16 come from the
  // plan kernel, which counts the 8-token blocks it has written in *acts.
  const int32_t *hshift;
  const int32_t *ashift;
  const uint32_t *acts;
  // BF16 deduplicating pass of 25 tokens or more, not in the early-start
  // mode: segments of more than 8 tokens run on tcgen05 CTAs (expert_tc.cu).
  // Their activations come in 2-D TMA boxes of 64 elements x 16 (j + 1) rows
  // through act_map[j] (128-byte swizzle): phase 1 the hidden states [n][d]
  // (one map, all tokens), phase 2 `aperm` [slots][I], which phase 1 writes
  // for these segments in plan order.
  int32_t wide;
  void *aperm;
  CUtensorMap act_map[4];
};

// A tensor map of `rows` rows of `kdim` bf16 elements at `act` (kdim % 64 ==
// 0), boxes of 64 elements x box_rows rows, 128-byte swizzle.
cudaError_t encode_act_map(CUtensorMap *map, const void *act, int rows, int kdim, int box_rows);

// Tensor-core expert FFN (BF16 weights, or E4M3 with fp32 block scales);
// n_tiles = 8-token MMA tiles per pass (1, 2 or 4).
cudaError_t launch_expert_tc(bool fp8, int phase, int n_tiles, const TcParams &P, int grid,
                             cudaStream_t stream);

// FP32 expert FFN on CUDA cores (same segment tables, same outputs).
struct F32Params {
  SegTables T;
  const float *w13, *w2;        // routed experts
  const float *sh_w13, *sh_w2;  // shared expert (or null)
  int32_t d, inter;
  const float *h;               // [n][d]
  float *inter_out;             // [slots][I]
  float *yslot;                 // [slots][d]
  int32_t *err;
};
cudaError_t launch_expert_f32(int phase, const F32Params &P, int grid, cudaStream_t stream);

// Repacks n_matrices expert matrices (rows x kbytes, row-major) into the
// tile layout of the tensor-core kernel (pack.cu); gate_up selects the W13
// row order (gate rows, then the matching up rows, per tile).  With E4M3
// block scales ([n_matrices][rows/128][kbytes/128]; else NULL) every tile is
// followed by its own.
cudaError_t launch_pack(const void *src, const float *scales, void *dst, int n_matrices, int rows,
                        int kbytes, int inter, bool gate_up, cudaStream_t stream);

// Where the E4M3 engines' fp16 hidden rows go (act_scale.cuh), in the workspace.
struct ActScaleOut {
  __half *h16;         // [n][d] fp16 rows, h[t] * 2^hshift[t]
  int32_t *hshift;     // [n]
  unsigned int *acts;  // launch_route_plan: blocks written so far (null: none)
};

// The E4M3 engines' fp16 rows of h [n][d] (bf16, d <= 8192), one CTA per token,
// launched as a programmatic dependent of the kernel ahead (it waits for
// that kernel before reading h).  (act_scale.cu)
cudaError_t launch_act_scale(const void *h, int n, int d, const ActScaleOut &S,
                             cudaStream_t stream);

// The E4M3 engines' fp16 rows of a [slots][I]: each bf16 row rewritten in
// place as fp16 times 2^ashift[slot], a warp per row, at most max_ctas CTAs;
// launched as a programmatic dependent of the gate/up kernel.  (act_scale.cu)
cudaError_t launch_a16_scale(void *a, int slots, int inter, int32_t *ashift, int max_ctas,
                             cudaStream_t stream);

// Router scores logits[t][e] = W_g[e] . h[t] (fp32 accumulation).
cudaError_t launch_router_scores(bool bf16, const void *router_w, const void *h, int n, int d,
                                 int n_experts, float *logits, cudaStream_t stream);

// Top-k (largest first, ties to the lower id) and gate weights per token.
cudaError_t launch_topk_gate(const float *logits, int n, int n_experts, int k, int gate,
                             int32_t *ids, float *w, cudaStream_t stream);

// Router scores + top-k + gate + union plan in one launch; `counter` is a
// zeroed device word and `group_counter` (n + 7) / 8 of them, all left
// zeroed by the kernel.  budget >= 0: the
// budgeted plan (w_kept written, routed_u if not NULL); budget < 0: none.
// `ready` (or null): set to 1 with release semantics once the plan is written.
// S.acts (or null): bf16 activations only; the launch also writes the E4M3
// engines' fp16 rows into S and counts each 8-token block in *S.acts (release).
cudaError_t launch_route_plan(bool bf16, const void *router_w, const void *h, int n, int d,
                              int n_experts, int k, int gate, int n_shared, int64_t expert_bytes,
                              float *logits, int32_t *ids, float *w, int32_t *hist, int32_t *uniq,
                              int32_t *n_uniq, int32_t *offs, int32_t *perm, int64_t *union_bytes,
                              int budget, float *w_kept, int32_t *routed_u, int32_t *err,
                              unsigned int *counter, unsigned int *group_counter,
                              unsigned int *ready, const ActScaleOut &S, cudaStream_t stream);

// Expert union and slot permutation (one CTA).
cudaError_t launch_union_plan(const int32_t *ids, int n_slots, int n_experts, int n_shared,
                              int64_t expert_bytes, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                              int32_t *offs, int32_t *perm, int64_t *union_bytes, int32_t *err,
                              cudaStream_t stream);

// The same under an expert budget (budget >= 0): see union_plan_block.
cudaError_t launch_union_plan_budgeted(const int32_t *ids, const float *w, int n_slots,
                                       int n_experts, int n_shared, int64_t expert_bytes,
                                       int budget, int32_t *hist, int32_t *uniq, int32_t *n_uniq,
                                       int32_t *offs, int32_t *perm, int64_t *union_bytes,
                                       float *w_kept, int32_t *routed_u, int32_t *err,
                                       cudaStream_t stream);

// Pre-verification selection over a batch of draft trees (select.cu), one
// CTA per tree of at most SEL_MAX_NODES nodes.
constexpr int SEL_MAX_NODES = 256;
constexpr size_t SEL_MAX_SMEM = 200 * 1024;  // EcoSpec bitsets: (K + 1) words x layers x E/32
cudaError_t launch_evict_select(const int32_t *parent, const float *q, int n_trees, int K,
                                const float *cost, int32_t *order, double *exp_len,
                                double *utility, int32_t *k_star, int32_t *err,
                                cudaStream_t stream);
size_t ecospec_smem_bytes(int K, int n_layers, int n_experts);
cudaError_t launch_ecospec_select(const int32_t *parent, const float *q, const int32_t *pred,
                                  int n_trees, int K, int n_layers, int n_experts, int kp,
                                  int gamma, double eps, const uint32_t *buf0,
                                  int32_t *selected, uint32_t *buf_out, int32_t *union_size,
                                  int32_t *err, cudaStream_t stream);

// y[t] = sum_j w[t][j] yslot[t*k+j] (+ yslot[n*k+t]) -> y (fp32 or bf16).
// `flags` (or null): moe_verify_pass's two header words, the plan-ready flag
// and the scaled-rows counter, cleared here.
cudaError_t launch_combine(const float *yslot, const float *w, int n, int k, int d, int n_shared,
                           bool out_bf16, void *y, uint32_t *flags, cudaStream_t stream);

}  // namespace moe
