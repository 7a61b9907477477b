// select.cu -- pre-verification selection over a batch of draft trees, one
// CTA per tree.  Every decision (an order, an arg-max) is taken in double,
// with the operations in the order the definitions give them, so the
// results equal a plain sequential evaluation bit for bit.
//
//   evict_select_kernel    "Making Every Verified Token Count", Sec. 3: node
//                          scores (eq. (7)), the top-k ranking (Sec. 3.2.1),
//                          the estimated accepted length of every prefix
//                          (eq. (8)) and the best prefix k* (eq. (10))
//   ecospec_select_kernel  "Less Experts, Faster Decoding", Sec. 4.2 and its
//                          appendix algorithm: gamma greedy picks by draft
//                          score over new experts (eqs. (7)-(9))
//
// Trees: K <= 256 nodes, node 0 the root, parent[0] = -1, 0 <= parent[v] < v.
#include "kernels.h"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int SEL_THREADS = 256;
constexpr int SEL_WARPS = SEL_THREADS / 32;

struct TreeSmem {
  double P[SEL_MAX_NODES];       // cumulative draft score
  int32_t parent[SEL_MAX_NODES];
  int32_t depth[SEL_MAX_NODES];  // -1 until P is known
  int32_t max_depth;
};

// Loads tree `parent`/`q` (thread v = node v), checks its shape and computes
// every node's cumulative score: P[root] = 1 (the target's own token) and
// P[v] = P[parent[v]] * q[v], so that P[v] is the product of q along the
// root path, multiplied in path order.  Level by level: in round r the nodes
// whose parent is known take their score (depth r).  Returns false, for the
// whole block, on a malformed tree.
__device__ bool tree_scores_block(TreeSmem &S, const int32_t *parent, const float *q, int K) {
  const int v = threadIdx.x;
  int par = -1;
  double qv = 1.0;
  bool bad = false;
  if (v == 0) S.max_depth = 0;
  if (v < K) {
    par = parent[v];
    qv = double(q[v]);
    bad = v == 0 ? par != -1 : (par < 0 || par >= v);
    S.parent[v] = par;
    S.depth[v] = v == 0 ? 0 : -1;
    if (v == 0) S.P[0] = 1.0;
  }
  if (__syncthreads_or(bad)) return false;
  for (int round = 1; round < K; ++round) {
    const bool go = v < K && S.depth[v] < 0 && S.depth[par] >= 0;
    __syncthreads();
    if (go) {
      S.P[v] = S.P[par] * qv;
      S.depth[v] = round;
      atomicMax(&S.max_depth, round);
    }
    if (!__syncthreads_or(v < K && S.depth[v] < 0)) break;
  }
  return true;
}

// Block arg-max of (key, index): the largest key, the smallest index among
// equal keys.  Threads without a candidate pass key 0; candidates pass
// cand_key(), which is at least 1, so the winner is always a candidate.
// Every thread gets the winning index.
// order_key of a candidate's value, lifted to 1 for the one NaN pattern
// whose key would be 0 (the order of every other value is unchanged).
__device__ __forceinline__ unsigned long long cand_key(double x) {
  const unsigned long long k = order_key(x);
  return k ? k : 1ull;
}

__device__ int block_argmax(unsigned long long key, int idx, unsigned long long *wkey,
                            int *widx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long ok = __shfl_xor_sync(0xffffffffu, key, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ok > key || (ok == key && oi < idx)) {
      key = ok;
      idx = oi;
    }
  }
  if (lane == 0) {
    wkey[warp] = key;
    widx[warp] = idx;
  }
  __syncthreads();
  unsigned long long bk = wkey[0];
  int bi = widx[0];
  for (int w = 1; w < SEL_WARPS; ++w)
    if (wkey[w] > bk || (wkey[w] == bk && widx[w] < bi)) {
      bk = wkey[w];
      bi = widx[w];
    }
  __syncthreads();  // wkey/widx may be reused
  return bi;
}

__global__ void __launch_bounds__(SEL_THREADS) evict_select_kernel(
    const int32_t *__restrict__ parent, const float *__restrict__ q, int K,
    const float *__restrict__ cost, int32_t *__restrict__ order, double *__restrict__ exp_len,
    double *__restrict__ utility, int32_t *__restrict__ k_star, int32_t *err) {
  __shared__ TreeSmem S;
  __shared__ unsigned long long skey[SEL_MAX_NODES];
  __shared__ int32_t srank_node[SEL_MAX_NODES];
  __shared__ double sE[SEL_MAX_NODES];
  __shared__ unsigned long long wkey[SEL_WARPS];
  __shared__ int widx[SEL_WARPS];
  const int t = blockIdx.x, v = threadIdx.x;
  const int64_t base = int64_t(t) * K;
  if (!tree_scores_block(S, parent + base, q + base, K)) {
    if (v == 0) {
      record_error(err, MOE_ERR_DEVICE_INPUT);
      k_star[t] = 0;
    }
    if (v < K) order[base + v] = -1;
    return;
  }
  // rank: nodes of larger score first, equal scores by lower index
  if (v < K) skey[v] = order_key(S.P[v]);
  __syncthreads();
  if (v < K) {
    const unsigned long long mine = skey[v];
    int r = 0;
    for (int u = 0; u < K; ++u) r += skey[u] > mine || (skey[u] == mine && u < v);
    srank_node[r] = v;
  }
  __syncthreads();
  // E_hat[A(T_k)]: the scores summed in rank order, one add after another
  if (v == 0) {
    double acc = 0.0;
    for (int r = 0; r < K; ++r) {
      acc += S.P[srank_node[r]];
      sE[r] = acc;
    }
  }
  __syncthreads();
  unsigned long long key = 0;
  if (v < K) {
    const double u_k = sE[v] / double(cost[v]);
    key = cand_key(u_k);
    order[base + v] = srank_node[v];
    if (exp_len) exp_len[base + v] = sE[v];
    if (utility) utility[base + v] = u_k;
  }
  const int best = block_argmax(key, v, wkey, widx);
  if (v == 0) k_star[t] = best + 1;
}

struct EcoParams {
  const int32_t *parent;    // [trees][K]
  const float *q;           // [trees][K]
  const int32_t *pred;      // [trees][K][L][kp]
  const uint32_t *buf0;     // [trees][L][wpl] or null
  int32_t *selected;        // [trees][n_sel]
  uint32_t *buf_out;        // [trees][L][wpl] or null
  int32_t *union_size;      // [trees]
  int32_t *err;
  double eps;
  int K, L, E, kp, wpl, n_sel;
};

__global__ void __launch_bounds__(SEL_THREADS) ecospec_select_kernel(const EcoParams p) {
  extern __shared__ __align__(16) uint32_t dyn[];
  __shared__ TreeSmem S;
  __shared__ int32_t taken[SEL_MAX_NODES];
  __shared__ unsigned long long wkey[SEL_WARPS];
  __shared__ int widx[SEL_WARPS];
  __shared__ int s_count;
  const int t = blockIdx.x, v = threadIdx.x, tid = threadIdx.x;
  const int K = p.K, W = p.L * p.wpl;
  uint32_t *traj = dyn;               // [K][W]: predicted, then path-union expert bits
  uint32_t *B = dyn + size_t(K) * W;  // [W]: the buffer
  const int64_t base = int64_t(t) * K;
  if (!tree_scores_block(S, p.parent + base, p.q + base, K)) {
    if (v == 0) {
      record_error(p.err, MOE_ERR_DEVICE_INPUT);
      p.union_size[t] = -1;
    }
    for (int i = v; i < p.n_sel; i += SEL_THREADS) p.selected[int64_t(t) * p.n_sel + i] = -1;
    return;
  }
  // bits of a layer's last word that name no expert
  const uint32_t tail_mask = (p.E & 31) ? ((1u << (p.E & 31)) - 1u) : 0xffffffffu;
  for (int i = tid; i < K * W; i += SEL_THREADS) traj[i] = 0u;
  for (int i = tid; i < W; i += SEL_THREADS) {
    uint32_t b = p.buf0 ? p.buf0[int64_t(t) * W + i] : 0u;
    if (i % p.wpl == p.wpl - 1) b &= tail_mask;
    B[i] = b;
  }
  if (tid == 0) s_count = 0;
  if (v < K) taken[v] = 0;
  __syncthreads();
  // predicted sets (eq. (4)): ids outside [0, E) are ignored
  const int per_node = p.L * p.kp;
  for (int i = tid; i < K * per_node; i += SEL_THREADS) {
    const int node = i / per_node, l = (i / p.kp) % p.L;
    const int e = p.pred[base * per_node + i];
    if (e >= 0 && e < p.E) atomicOr(&traj[node * W + l * p.wpl + (e >> 5)], 1u << (e & 31));
  }
  __syncthreads();
  // path unions (eq. (7)), one depth after another
  for (int d = 1; d <= S.max_depth; ++d) {
    for (int i = tid; i < K * W; i += SEL_THREADS) {
      const int node = i / W;
      if (S.depth[node] == d) traj[i] |= traj[S.parent[node] * W + (i - node * W)];
    }
    __syncthreads();
  }
  // greedy picks: score = P / (|E_traj \ B| + eps) (eqs. (8)-(9))
  for (int it = 0; it < p.n_sel; ++it) {
    unsigned long long key = 0;
    if (v < K && !taken[v]) {
      int c = 0;
      const uint32_t *tv = traj + v * W;
      for (int w = 0; w < W; ++w) c += __popc(tv[w] & ~B[w]);
      key = cand_key(S.P[v] / (double(c) + p.eps));
    }
    const int pick = block_argmax(key, v, wkey, widx);
    if (tid == 0) {
      p.selected[int64_t(t) * p.n_sel + it] = pick;
      taken[pick] = 1;
    }
    for (int w = tid; w < W; w += SEL_THREADS) B[w] |= traj[pick * W + w];
    __syncthreads();
  }
  int c = 0;
  for (int w = tid; w < W; w += SEL_THREADS) {
    c += __popc(B[w]);
    if (p.buf_out) p.buf_out[int64_t(t) * W + w] = B[w];
  }
  atomicAdd(&s_count, c);
  __syncthreads();
  if (tid == 0) p.union_size[t] = s_count;
}

}  // namespace

cudaError_t launch_evict_select(const int32_t *parent, const float *q, int n_trees, int K,
                                const float *cost, int32_t *order, double *exp_len,
                                double *utility, int32_t *k_star, int32_t *err,
                                cudaStream_t stream) {
  evict_select_kernel<<<n_trees, SEL_THREADS, 0, stream>>>(parent, q, K, cost, order, exp_len,
                                                          utility, k_star, err);
  return cudaGetLastError();
}

size_t ecospec_smem_bytes(int K, int n_layers, int n_experts) {
  const size_t W = size_t(n_layers) * size_t((n_experts + 31) / 32);
  return (size_t(K) * W + W) * 4;
}

cudaError_t launch_ecospec_select(const int32_t *parent, const float *q, const int32_t *pred,
                                  int n_trees, int K, int n_layers, int n_experts, int kp,
                                  int gamma, double eps, const uint32_t *buf0,
                                  int32_t *selected, uint32_t *buf_out, int32_t *union_size,
                                  int32_t *err, cudaStream_t stream) {
  EcoParams p{parent, q, pred, buf0, selected, buf_out, union_size, err, eps, K, n_layers,
              n_experts, kp, (n_experts + 31) / 32, gamma < K ? gamma : K};
  const size_t smem = ecospec_smem_bytes(K, n_layers, n_experts);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(ecospec_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
  }
  ecospec_select_kernel<<<n_trees, SEL_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
