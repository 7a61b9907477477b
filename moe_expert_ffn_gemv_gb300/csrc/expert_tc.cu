// expert_tc.cu -- the grouped expert FFN on tensor cores, for BF16 and
// FP8-E4M3 (128x128 block-scaled) expert weights.
//
// One kernel template serves both engines of "Speculative Decoding for
// Mixture-of-Experts Models: Expert Bytes, Kernel Bandwidth and the Best
// Draft Length" (abstract; Fig. 3):
//   deduplicating  a segment is one union expert with all m tokens routed to
//                  it, so each expert's weights cross HBM once per pass;
//   per-slot       a segment is one (token, slot) pair, so an expert's weights
//                  are requested once per pair that names it.
// and both halves of the SwiGLU FFN:
//   PHASE 1  a = silu(W1 x) * (W3 x)  over gate rows [32 rb, 32 rb + 32) and the
//            matching up rows, K = d; writes a[slot][I] (bf16);
//   PHASE 2  y_slot = W2 a           over rows [64 rb, 64 rb + 64) of W2, K = I;
//            writes yslot[slot][d] (fp32).
//
// Structure (one CTA per SM, persistent over work items (segment, row block,
// token group of 8 tokens)):
//   - the weights are stored pre-packed (pack.cu): the 64 rows x 512 bytes of
//     one pipeline stage form one contiguous tile, its 16-byte pieces in the
//     order the consumer threads read them, an E4M3 tile followed by its 8
//     block scales;
//   - two producer warps fill each slot of a 5-stage shared-memory ring,
//     both completing on the slot's mbarrier: warp 8 with one 1-D TMA bulk
//     copy (cp.async.bulk) of the tile and its scales, warp 10 with one bulk
//     copy per token of the K chunk of that token's activation row.  So the
//     consumers read nothing but shared memory: a global load issued by a
//     consumer returns behind the SM's stream of weight tiles, several
//     stages late, and stalls it.  A warp's issue time per copy is what
//     keeps it from running further ahead, hence one copy a stage for the
//     weight stream (no separate scale copy; the rows on their own warp);
//   - warps 0..7 consume: warp w owns 64 bytes of every row of a stage (a
//     K-split across warps) and runs mma.sync m16n8k16 with the weights as
//     the 16-row A operand (4 row tiles) and the segment's tokens as the
//     8-wide N operand (NT tiles).  Because a dot product does not depend on
//     the order of its terms, each thread's 16 contiguous weight bytes feed
//     the A fragment directly (no ldmatrix); the activations (B fragment) are
//     read with the same permutation of K.  E4M3: warp w owns bytes
//     [64 w, 64 w + 64), the tile's pieces are in the threads' order (lane-
//     contiguous 16-byte loads).  BF16 (tiles in the 128-byte swizzled layout
//     that tcgen05 also reads, pack.cu): warp w owns the chunks j = 2 c +
//     w % 2 (thread c) of the 128-byte column w / 2, so a wavefront of 8 lanes
//     (rows g, g + 1) covers 8 distinct bank groups.  The tokens' activation
//     rows are padded apart so that they hit distinct banks;
//   - E4M3 bytes become fp16 with cvt.rn.f16x2.e4m3x2 (exact); the block scale
//     multiplies the fp32 partial sum of each 64-column chunk, which lies in a
//     single 128x128 scale block.  The activations reach this fp16 MMA scaled
//     into fp16 range by exact powers of two (act_scale.cuh): phase 1 streams
//     the fp16 rows h16 = h * 2^hshift[t], its epilogue scales g and u back
//     and stores a in bf16; a kernel between the phases rewrites each slot's
//     row of a as fp16 times 2^ashift[slot], which phase 2 streams and its
//     epilogue scales back;
//   - after the last stage of an item each consumer warp drops its partial
//     sums into a reduction buffer (two for BF16, one for E4M3, whose ring
//     slots are larger) and goes on streaming; warp 9, the epilogue warp,
//     adds the 8 warps' partials in a fixed order (deterministic) and applies
//     silu(g)*u (phase 1) or stores the fp32 rows (phase 2).
// Every wait is bounded; on time-out the kernel records MOE_ERR_TIMEOUT in the
// workspace error word, keeps its barrier structure, lets its own copies land
// and returns.
#include "moe_common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int ROWS = PACK_ROWS;      // weight rows per stage (4 MMA row tiles)
constexpr int KBYTES = PACK_KBYTES;  // bytes of each row per stage
constexpr int STAGE_BYTES = ROWS * KBYTES;
constexpr int CONSUMERS = 8;                      // warps 0..7
constexpr int PRODUCER = CONSUMERS;                // warp 8: weight tiles
constexpr int EPILOGUE = CONSUMERS + 1;            // warp 9
constexpr int ACTS = CONSUMERS + 2;                // warp 10: activation rows
constexpr int THREADS = (CONSUMERS + 3) * 32;
constexpr uint64_t DRAIN_LIMIT_NS = 200ull * 1000 * 1000;
// Phase 2: stages past the first S that each CTA prefetches into L2 once its
// ring is full.  Phase 2's CTAs start as phase 1's finish, and phase 1's
// last CTAs end some 9 us after the median one: the prefetch puts the HBM
// bandwidth they leave idle to use (-4 us on the n = 8 pass).  Passes of
// fewer than 4 items a CTA leave no such idle time, and there the prefetch
// only delays the copies queued behind it, so it is skipped.
constexpr int PREFETCH_AHEAD = 8;

// Shared memory: a ring of S slots, each with one stage's weight tile (E4M3:
// with its 8 block scales behind it) and the activation rows of its tokens;
// the cross-warp reduction buffers (consumers hand an item's partial sums to
// the epilogue warp there); the barriers.
template <bool FP8, int NT>
constexpr int n_red_bufs() { return FP8 || NT >= 4 ? 1 : 2; }

template <int NT>
constexpr size_t red_bytes() { return size_t(CONSUMERS) * 4 * NT * 32 * 16; }

// One activation row of a stage: its K columns as 16-bit values, plus a pad
// of 16 bytes (4 banks) that sets consecutive rows apart, so that the
// consumers' 16-byte reads of two tokens' rows never meet in a bank (BF16:
// the chunks a warp reads in a row all have the parity of w % 2, and the pad
// flips it from one token to the next).
template <bool FP8>
constexpr int act_row_bytes() { return KBYTES / (FP8 ? 1 : 2) * 2 + 16; }

// where a slot's activation rows start: behind the largest tile
template <bool FP8>
constexpr int act_offset() { return STAGE_BYTES + (FP8 ? PACK_SCALE_BYTES : 0); }

template <bool FP8, int NT>
constexpr int slot_bytes() {
  return (act_offset<FP8>() + 8 * NT * act_row_bytes<FP8>() + 127) / 128 * 128;
}

template <bool FP8, int NT>
constexpr int n_stages() { return NT >= 2 ? 4 : 5; }

template <bool FP8, int NT>
constexpr size_t smem_bytes() {
  return size_t(n_stages<FP8, NT>()) * slot_bytes<FP8, NT>() +
         n_red_bufs<FP8, NT>() * red_bytes<NT>() +
         2 * (n_stages<FP8, NT>() + n_red_bufs<FP8, NT>()) * 8;
}

__device__ __forceinline__ float silu_times(float g, float u) {
  return g / (1.0f + __expf(-g)) * u;
}

// The plan (or, per-slot, the routed ids) copied to shared memory at kernel
// start, so that stepping from one work item to the next costs no global
// round trip.
constexpr int MAX_TOKENS = 64;
constexpr int MAX_SLOTS = MAX_TOKENS * 32;
constexpr int MAX_EXPERTS = 256;
// every slot of a pass: n*k routed, then the shared expert's n*k + t
constexpr int MAX_ALL_SLOTS = MAX_SLOTS + MAX_TOKENS;

// Deduplicating segments: the shared expert first (segment 0, all n tokens;
// it needs no plan), then the U routed experts in plan order.  Per-slot
// segments: the n*k routed slots, then the n shared-expert slots.
struct LocalTables {
  const int32_t *uniq;  // [U]      dedup
  const int32_t *offs;  // [U + 1]  dedup
  const int16_t *tab;   // [n*k]    dedup: perm; per-slot: ids (-1: out of range)
  const int *U;         // U, in shared memory (read once the plan is there)
  int n, k, n_experts, n_shared, dedup;

  __device__ int n_segments() const { return dedup ? *U + n_shared : n * k + n_shared * n; }
  // segments whose work items are known before the plan is read
  __device__ int plan_free_segments() const { return dedup ? n_shared : 0; }

  __device__ Seg segment(int u) const {
    Seg s;
    const int nk = n * k;
    if (dedup) {
      if (u < n_shared) {
        s.expert = -1;
        s.first = 0;
        s.m = n;
      } else {
        const int r = u - n_shared;
        s.expert = uniq[r];
        s.first = offs[r];
        s.m = offs[r + 1] - s.first;
      }
    } else {
      s.m = 1;
      s.first = u;
      if (u < nk) {
        const int e = tab[u];
        s.expert = (e >= 0 && e < n_experts) ? e : -2;
      } else {
        s.expert = -1;
      }
    }
    return s;
  }
  // slot index of the i-th token of segment s
  __device__ int slot(const Seg &s, int i) const {
    if (!dedup) return s.first;
    if (s.expert == -1) return n * k + i;
    return tab[s.first + i];
  }
  __device__ int token(int slot) const { return slot < n * k ? slot / k : slot - n * k; }
};

// Position in the (work item, K stage) sequence a CTA walks; the producer,
// activation, consumer and epilogue warps all walk the same sequence.  A
// work item is (segment, row block, token group of TOK tokens); items are
// numbered segment by segment, row block by row block, the token group
// innermost, and CTA b takes items b, b + gridDim.x, ...  A segment of more
// than TOK tokens (the shared expert at n > 8, a popular routed expert) thus
// spreads its groups over consecutive CTAs, which balances the CTAs' work
// and has them read the same tiles at about the same time (L2 hits after
// the first).
struct Cursor {
  int item, rb, grp, ks, groups;
  int u, seg_first, seg_items;  // segment, its first item, its items
  Seg sg;
};

__device__ __forceinline__ void cursor_start(Cursor &c) {
  c.item = blockIdx.x;
  c.u = -1;
  c.seg_first = 0;
  c.seg_items = 0;
}

// ensure() makes the plan's tables usable (it may wait for them) and
// returns false when the kernel must stop.
template <int TOK, typename Ensure>
__device__ __forceinline__ bool cursor_item(Cursor &c, const LocalTables &T, int row_blocks,
                                            Ensure &ensure, int32_t *err, bool report) {
  for (;;) {
    if (c.item < c.seg_first + c.seg_items) {
      const int j = c.item - c.seg_first;
      c.rb = j / c.groups;
      c.grp = j - c.rb * c.groups;
      c.ks = 0;
      return true;
    }
    c.seg_first += c.seg_items;
    c.u += 1;
    if (c.u >= T.plan_free_segments()) {
      if (!ensure()) return false;
      if (c.u >= T.n_segments()) return false;
    }
    c.sg = T.segment(c.u);
    if (c.sg.expert == -2) {
      if (report) record_error(err, MOE_ERR_DEVICE_INPUT);
      c.seg_items = 0;
      continue;
    }
    c.groups = (c.sg.m + TOK - 1) / TOK;
    c.seg_items = row_blocks * c.groups;
  }
}

template <int TOK, typename Ensure>
__device__ __forceinline__ bool cursor_next(Cursor &c, const LocalTables &T, int row_blocks,
                                            int kstages, Ensure &ensure, int32_t *err,
                                            bool report) {
  if (++c.ks < kstages) return true;
  c.item += gridDim.x;
  return cursor_item<TOK>(c, T, row_blocks, ensure, err, report);
}

template <bool FP8, int PHASE, int NT>
__global__ void __launch_bounds__(THREADS, 1) expert_tc_kernel(const TcParams P) {
  constexpr int S = n_stages<FP8, NT>();
  constexpr int SLOT = slot_bytes<FP8, NT>();
  constexpr int RB = n_red_bufs<FP8, NT>();
  constexpr int ES = FP8 ? 1 : 2;       // bytes per weight element
  constexpr int TOK = 8 * NT;           // tokens per pass over an item
  constexpr int BW = FP8 ? 8 : 4;       // B-fragment words per N tile and stage
  constexpr int ACT_ROW = act_row_bytes<FP8>();
  constexpr int ACT_OFF = act_offset<FP8>();  // a slot's activation rows
  constexpr int TRAILER = FP8 ? PACK_SCALE_BYTES : 0;  // scale bytes behind a tile
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  float4 *red = reinterpret_cast<float4 *>(smem + S * SLOT);   // [RB][red_bytes]
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * SLOT + RB * red_bytes<NT>());
  uint64_t *empty = full + S;
  uint64_t *rfull = empty + S;    // consumers -> epilogue warp (count CONSUMERS)
  uint64_t *rempty = rfull + RB;  // epilogue warp -> consumers (count 1)
  constexpr int RED_F4 = int(red_bytes<NT>() / 16);
  __shared__ volatile int s_abort;
  __shared__ int32_t s_uniq[MAX_EXPERTS];
  __shared__ int32_t s_offs[MAX_EXPERTS + 1];
  __shared__ int16_t s_tab[MAX_SLOTS];  // entries below 2048; -1 stands for any other
  __shared__ int32_t s_U;
  __shared__ uint64_t tables_bar;  // the plan is in shared memory (lazy phase 1)
  // E4M3: phase 1's token shifts (hshift), phase 2's slot shifts (ashift),
  // read by the epilogue warp
  __shared__ int32_t s_hshift[FP8 && PHASE == 1 ? MAX_TOKENS : 1];
  __shared__ int8_t s_ashift[FP8 && PHASE == 2 ? MAX_ALL_SLOTS : 1];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = P.T.n * P.T.k;
  // Launch order: the plan, phase 1, phase 2, the combine, each of the last
  // three launched as a programmatic dependent of the one before.
  //  - Phase 1 of the deduplicating engine with a shared expert, launched
  //    right behind its pass's plan kernel (early_shared; "lazy"): the
  //    shared expert's items need no plan, so the CTAs start on them at
  //    once.  When its walk leaves the shared segment, the weight warp
  //    waits (bounded) for the plan kernel's plan-ready flag, copies the
  //    plan through L2 to shared memory and signals tables_bar, on which
  //    the other warps wait (bounded).  Once the ring is full it also waits
  //    for the plan kernel to end (programmatic dependent launch) and only
  //    then triggers phase 2, so phase 2 still reads a complete plan, and
  //    phase 1 never ends before the plan kernel.
  //  - Otherwise phase 1 waits for the plan at once; phase 2 reads the plan
  //    (complete before phase 1 triggered it) at once.  Phase 2's weight
  //    warp streams its first S stages' tiles from the start, behind the
  //    end of phase 1; its activation warp waits for phase 1 to end before
  //    it copies phase 1's activations, which completes those stages.
  const bool lazy =
      PHASE == 1 && P.T.dedup && P.T.n_shared > 0 && P.early_shared && P.ready != nullptr;
  // Lazy E4M3 phase 1 reads the fp16 rows that the plan kernel, still
  // running, writes: the activation and epilogue warps wait (bounded) until
  // it has counted every 8-token block, each lane acquiring the count itself.
  const bool acts_flag = FP8 && PHASE == 1 && lazy && P.acts != nullptr;
  auto await_acts = [&]() -> bool {
    const uint32_t need = uint32_t((P.T.n + 7) / 8);
    bool seen = true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(P.acts) < need)
      if (globaltimer_ns() - t0 > P.timeout_ns) {
        seen = false;
        break;
      }
    return __all_sync(0xffffffffu, seen);
  };
  // the plan (or, per-slot, the ids) into shared memory, threads first,
  // first + step, ... (the early-start mode has its own loader, below)
  auto load_tables = [&](int first, int step) {
    auto rd = [](const int32_t *p) { return *p; };
    const int32_t *src = P.T.dedup ? P.T.perm : P.T.ids;
    const int lim = P.T.dedup ? nk : P.T.n_experts;
    for (int i = first; i < nk; i += step) {
      const int32_t v = rd(src + i);
      s_tab[i] = int16_t(v >= 0 && v < lim ? v : -1);
    }
    if (P.T.dedup)
      for (int i = first; i <= P.T.n_experts; i += step) {
        if (i < P.T.n_experts) s_uniq[i] = rd(P.T.uniq + i);
        s_offs[i] = rd(P.T.offs + i);
      }
    if (first == 0) s_U = P.T.dedup ? rd(P.T.n_uniq) : 0;
  };
  // A caller may hand moe_verify_dedup any plan: before its indices are
  // used, check that U is at most N, every uniq entry is an expert id, offs
  // starts at or above 0, never decreases and ends at or below n*k, and
  // every perm entry of the groups is a slot below n*k.  Returns this
  // thread's verdict on its share (every step-th entry from first); the
  // caller combines the verdicts and empties a bad plan (U = 0).
  auto plan_bad = [&](int first, int step) -> bool {
    if (!P.T.dedup) return false;
    const int U = s_U;
    if (U < 0 || U > P.T.n_experts) return true;
    if (s_offs[0] < 0 || s_offs[U] > nk) return true;
    bool bad = false;
    for (int r = first; r < U; r += step)
      bad |= s_uniq[r] < 0 || s_uniq[r] >= P.T.n_experts || s_offs[r] > s_offs[r + 1];
    for (int i = s_offs[0] + first; i < s_offs[U]; i += step) bad |= s_tab[i] < 0 || s_tab[i] >= nk;
    return bad;
  };
  if (!lazy) {
    if (PHASE == 1) pdl_wait();
    pdl_trigger();
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);  // the tile's and the activations' producers
      mbar_init(&empty[s], CONSUMERS);
    }
    for (int b = 0; b < RB; ++b) {
      mbar_init(&rfull[b], CONSUMERS);
      mbar_init(&rempty[b], 1);
    }
    mbar_init(&tables_bar, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (!lazy) load_tables(threadIdx.x, THREADS);
  __syncthreads();
  if (!lazy && __syncthreads_or(plan_bad(threadIdx.x, THREADS))) {
    if (threadIdx.x == 0) {
      s_U = 0;
      record_error(P.err, MOE_ERR_DEVICE_INPUT);
    }
    __syncthreads();
  }
  LocalTables T{s_uniq, s_offs, s_tab, &s_U, P.T.n, P.T.k, P.T.n_experts, P.T.n_shared,
                P.T.dedup};
  // The plan gate of the warps other than the producer: a bounded wait on
  // tables_bar the first time a walk needs the plan.
  bool have_tables = !lazy;
  auto await_tables = [&]() -> bool {
    if (have_tables) return true;
    if (!mbar_wait_bounded(&tables_bar, 0, P.timeout_ns)) {
      s_abort = 1;
      if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
      return false;
    }
    have_tables = true;
    return true;
  };

  const int kbytes = P.kdim * ES;
  const int kstages = (kbytes + KBYTES - 1) / KBYTES;
  // packed bytes of one row block: its tiles, each followed by its scales
  const int64_t rb_bytes = int64_t(ROWS) * kbytes + int64_t(kstages) * TRAILER;

  if (warp == EPILOGUE) {
    // -------------------------------------------------------------- epilogue
    // For each (item, token group), in the consumers' order: add the 8 warps'
    // K-partials in a fixed order, then silu(g)*u (phase 1) or the fp32 rows
    // (phase 2), and give the buffer back.
    bool aborted = false;
    uint32_t ep = 0;
    if constexpr (FP8 && PHASE == 1) {
      if (acts_flag && !await_acts()) {
        aborted = true;
        s_abort = 1;
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
      }
      for (int i = lane; i < P.T.n; i += 32) s_hshift[i] = aborted ? 0 : __ldcg(P.hshift + i);
      __syncwarp();
    }
    if constexpr (FP8 && PHASE == 2) {
      // the kernel ahead rewrote a and wrote the slot shifts
      pdl_wait();
      const int n_all = nk + P.T.n_shared * P.T.n;
      for (int i = lane; i < n_all; i += 32) s_ashift[i] = int8_t(__ldcg(P.ashift + i));
      __syncwarp();
    }
    Cursor cur;
    cursor_start(cur);
    bool have = cursor_item<TOK>(cur, T, P.row_blocks, await_tables, P.err, false);
    while (have) {
      const int b = ep % RB;
      const uint32_t round = ep / RB;
      if (!aborted && s_abort) aborted = true;
      if (!aborted && !mbar_wait_bounded(&rfull[b], round & 1, P.timeout_ns)) {
        aborted = true;
        s_abort = 1;
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
      }
      if (!aborted) {
        const float4 *rb_buf = red + b * RED_F4;
        const int m_left = cur.sg.m - cur.grp * TOK;
        constexpr int MT_OUT = PHASE == 1 ? 2 : 4;
        for (int q = lane; q < MT_OUT * NT * 32; q += 32) {
          const int ln = q & 31, nt = (q >> 5) % NT, mt = q / (32 * NT);
          if (nt * 8 >= m_left) continue;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f), w4 = v;
#pragma unroll
          for (int w = 0; w < CONSUMERS; ++w) {
            const float4 x = rb_buf[((w * 4 + mt) * NT + nt) * 32 + ln];
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
            if (PHASE == 1) {
              const float4 y = rb_buf[((w * 4 + mt + 2) * NT + nt) * 32 + ln];
              w4.x += y.x; w4.y += y.y; w4.z += y.z; w4.w += y.w;
            }
          }
          const int gg = ln >> 2, cc = ln & 3;
          const float vals[4] = {v.x, v.y, v.z, v.w};
          const float ups[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = mt * 16 + gg + (e >> 1) * 8;
            const int col = nt * 8 + 2 * cc + (e & 1);
            if (col >= m_left) continue;
            const int slot = T.slot(cur.sg, cur.grp * TOK + col);
            if (PHASE == 1) {
              float gv = vals[e], uv = ups[e];
              if (FP8) {
                // the rows were scaled by 2^hshift: scale the sums back
                const float back = pow2f(-s_hshift[T.token(slot)]);
                gv *= back;
                uv *= back;
              }
              const float a = silu_times(gv, uv);
              uint16_t *out =
                  static_cast<uint16_t *>(P.out) + int64_t(slot) * P.inter + cur.rb * 32 + row;
              *reinterpret_cast<__nv_bfloat16 *>(out) = __float2bfloat16_rn(a);
            } else {
              float *out = static_cast<float *>(P.out) + int64_t(slot) * P.rows_total +
                           cur.rb * ROWS + row;
              // E4M3: a reached the MMA scaled by 2^ashift[slot]
              *out = FP8 ? vals[e] * pow2f(-s_ashift[slot]) : vals[e];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rempty[b]);
      ++ep;
      cur.ks = kstages - 1;  // step to the next (item, token group)
      have = cursor_next<TOK>(cur, T, P.row_blocks, kstages, await_tables, P.err, false);
    }
    return;
  }

  if (warp == PRODUCER) {
    // ------------------------------------------------------------ producer
    // A segment of more than TOK tokens (the shared expert at n > TOK, a
    // popular routed expert) streams a row block's tiles once per group of
    // TOK tokens, consecutive work items.  A routed expert's groups before
    // the last load them at normal L2 priority, so that the evict-first
    // stream leaves them for the later groups; the shared expert's stay
    // evict-first (measured faster on DeepSeek-V3 stacks).
    const uint64_t policy = policy_evict_first();
    const uint64_t keep = policy_evict_normal();
    uint32_t it = 0;
    bool ok = true;
    // The plan gate of the producer (lazy phase 1): wait (bounded) for the
    // plan-ready flag, copy the plan to shared memory and signal the other
    // warps.  The wait for the plan kernel's end, and the trigger of phase 2,
    // come later (`joined`).
    bool plan_ready = !lazy;
    bool joined = !lazy;
    int since_plan = 0;  // stages issued since the plan arrived
    auto load_plan = [&]() -> bool {
      if (plan_ready) return true;
      // every lane acquires the flag itself, so that its own plan reads
      // below are ordered after the plan kernel's writes
      bool seen = true;
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(P.ready) == 0u)
        if (globaltimer_ns() - t0 > P.timeout_ns) {
          seen = false;
          break;
        }
      if (!__all_sync(0xffffffffu, seen)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        s_abort = 1;
        return false;
      }
      // The plan through L2 (its kernel wrote it just now), in as few round
      // trips as the warp can: U, then the n*k perm entries and the U uniq
      // and U + 1 offs entries (all the walk reads) as one index space, 8
      // loads in flight a lane before any store.  Loading every table entry
      // in lane-strided loops took 2.3-2.9 us here.
      const int U = __ldcg(P.T.n_uniq);
      const int Uc = U < 0 ? 0 : U > P.T.n_experts ? P.T.n_experts : U;
      const int total = nk + Uc + Uc + 1;
      for (int base = 0; base < total; base += 8 * 32) {
        int32_t v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = base + q * 32 + lane;
          const int32_t *src = i < nk        ? P.T.perm + i
                               : i < nk + Uc ? P.T.uniq + (i - nk)
                                             : P.T.offs + (i - nk - Uc);
          v[q] = i < total ? __ldcg(src) : 0;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = base + q * 32 + lane;
          if (i < nk) s_tab[i] = int16_t(v[q] >= 0 && v[q] < nk ? v[q] : -1);
          else if (i < nk + Uc) s_uniq[i - nk] = v[q];
          else if (i < total) s_offs[i - nk - Uc] = v[q];
        }
      }
      if (lane == 0) s_U = U;
      __syncwarp();
      if (__any_sync(0xffffffffu, plan_bad(lane, 32)) && lane == 0) {
        s_U = 0;
        record_error(P.err, MOE_ERR_DEVICE_INPUT);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&tables_bar);
      plan_ready = true;
      return true;
    };
    // Stage q's packed tile of (row block, K chunk) into slot s: contiguous,
    // ROWS * nb bytes of weights followed (E4M3) by the tile's block scales,
    // one bulk copy.  The copy issue time of this warp bounds how far ahead
    // of HBM it can run, hence a single copy a stage (the scales packed into
    // the tile, the activation rows left to their own warp).
    auto issue_tile = [&](const Cursor &q, int s) {
      const int nb = min(KBYTES, kbytes - q.ks * KBYTES);
      const uint32_t tile_bytes = uint32_t(ROWS * nb + TRAILER);
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], tile_bytes);
        const uint8_t *base =
            q.sg.expert >= 0 ? P.w + int64_t(q.sg.expert) * P.expert_stride : P.w_sh;
        bulk_g2s(ring + s * SLOT, base + q.rb * rb_bytes + int64_t(q.ks) * (ROWS * KBYTES + TRAILER),
                 tile_bytes, &full[s], q.sg.expert >= 0 && q.grp + 1 < q.groups ? keep : policy);
      }
      __syncwarp();
    };
    // The tiles of the next `stages` stages from q into L2 (one prefetch per
    // item: an item's tiles are contiguous).
    auto prefetch_stages = [&](Cursor q, int stages) {
      bool h = true;
      while (h && stages > 0) {
        const int n = min(stages, kstages - q.ks);
        const uint8_t *base =
            q.sg.expert >= 0 ? P.w + int64_t(q.sg.expert) * P.expert_stride : P.w_sh;
        const int64_t off = q.rb * rb_bytes + int64_t(q.ks) * (ROWS * KBYTES + TRAILER);
        const int64_t end = q.ks + n == kstages ? (q.rb + 1) * rb_bytes
                                                : off + int64_t(n) * (ROWS * KBYTES + TRAILER);
        if (lane == 0) prefetch_l2(base + off, uint64_t(end - off));
        stages -= n;
        q.ks += n - 1;
        h = cursor_next<TOK>(q, T, P.row_blocks, kstages, load_plan, P.err, false);
      }
    };
    Cursor cur;
    cursor_start(cur);
    bool have = cursor_item<TOK>(cur, T, P.row_blocks, load_plan, P.err, false);
    while (have) {
      const int s = it % S;
      const uint32_t round = it / S;
      if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, P.timeout_ns)) {
        ok = false;
        break;
      }
      if (s_abort) { ok = false; break; }
      issue_tile(cur, s);
      ++it;
      if (PHASE == 2 && PREFETCH_AHEAD > 0 && it == uint32_t(S) &&
          T.n_segments() * P.row_blocks >= 4 * int(gridDim.x)) {
        Cursor q = cur;
        if (cursor_next<TOK>(q, T, P.row_blocks, kstages, load_plan, P.err, false))
          prefetch_stages(q, PREFETCH_AHEAD);
      }
      if (plan_ready && !joined && ++since_plan >= S) {
        // the ring is full: wait for the plan kernel's end, then let phase 2 launch
        pdl_wait();
        pdl_trigger();
        joined = true;
      }
      have = cursor_next<TOK>(cur, T, P.row_blocks, kstages, load_plan, P.err, false);
    }
    // Phase 1 must not end before the plan kernel, whatever path led here.
    if (!joined) pdl_wait();
    if (!ok) {
      if (lane == 0) {
        record_error(P.err, MOE_ERR_TIMEOUT);
        s_abort = 1;
      }
    }
    // Let every copy this warp issued land before the CTA may exit.
    const uint32_t issued = it;
    const uint32_t first = issued > uint32_t(S) ? issued - S : 0;
    for (uint32_t j = first; j < issued; ++j)
      if (!mbar_wait_bounded(&full[j % S], (j / S) & 1, DRAIN_LIMIT_NS)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        break;
      }
    return;
  }

  if (warp == ACTS) {
    // ---------------------------------------------------- activation rows
    // For each stage, the K chunk of each of its tokens' activation rows,
    // one bulk copy per row into the slot, behind the slot's tile: the
    // consumers then read nothing but shared memory (a global load of
    // theirs would come back behind the SM's stream of weight tiles,
    // several stages late).  Phase 2 reads phase 1's activations, so it
    // waits for phase 1 to end first; its weight tiles stream meanwhile.
    if (PHASE == 2) pdl_wait();
    const uint64_t keep = policy_evict_normal();
    const uint8_t *act = static_cast<const uint8_t *>(P.act);
    uint32_t it = 0;
    bool ok = true;
    if (acts_flag) {
      // lazy E4M3 phase 1: the fp16 rows come from the plan kernel
      ok = await_acts();
      fence_proxy_async_global();
    }
    Cursor cur;
    cursor_start(cur);
    bool have = ok && cursor_item<TOK>(cur, T, P.row_blocks, await_tables, P.err, false);
    while (have) {
      const int s = it % S;
      const uint32_t round = it / S;
      if (round > 0 && !mbar_wait_bounded(&empty[s], (round - 1) & 1, P.timeout_ns)) {
        ok = false;
        break;
      }
      if (s_abort) break;
      const int k0 = cur.ks * KBYTES;
      const uint32_t row_bytes = uint32_t(min(KBYTES, kbytes - k0) / ES) * 2;
      const int m_rows = max(0, min(TOK, cur.sg.m - cur.grp * TOK));
      if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(m_rows) * row_bytes);
      __syncwarp();
      for (int j = lane; j < m_rows; j += 32) {
        const int sl = T.slot(cur.sg, cur.grp * TOK + j);
        const int row = PHASE == 1 ? T.token(sl) : sl;
        bulk_g2s(ring + s * SLOT + ACT_OFF + j * ACT_ROW,
                 act + (int64_t(row) * P.kdim + k0 / ES) * 2, row_bytes, &full[s], keep);
      }
      __syncwarp();
      ++it;
      have = cursor_next<TOK>(cur, T, P.row_blocks, kstages, await_tables, P.err, false);
    }
    if (!ok && lane == 0) {
      record_error(P.err, MOE_ERR_TIMEOUT);
      s_abort = 1;
    }
    // Let every copy this warp issued land before the CTA may exit.
    const uint32_t first = it > uint32_t(S) ? it - S : 0;
    for (uint32_t j = first; j < it; ++j)
      if (!mbar_wait_bounded(&full[j % S], (j / S) & 1, DRAIN_LIMIT_NS)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        break;
      }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g = lane >> 2, c = lane & 3;
  const int tid = threadIdx.x;
  uint32_t it = 0;
  uint32_t ep = 0;  // (item, token group)s handed to the epilogue warp
  bool aborted = false;

  float acc[4][NT][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[mt][nt][q] = 0.f;

  Cursor cur;
  cursor_start(cur);
  bool have = cursor_item<TOK>(cur, T, P.row_blocks, await_tables, P.err, tid == 0);

  while (have) {
    const int s = it % S;
    const uint32_t round = it / S;
    const int m_left = cur.sg.m - cur.grp * TOK;
    // (a BF16 K tail is whole 128-byte columns, an E4M3 one whole 64-byte chunks)
    const bool active = cur.ks * KBYTES + (FP8 ? warp * 64 : (warp >> 1) * 128) < kbytes;
    if (!aborted && s_abort) aborted = true;
    if (!aborted && !mbar_wait_bounded(&full[s], round & 1, P.timeout_ns)) {
      aborted = true;
      s_abort = 1;
      if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
    }
    if (!aborted && active) {
      const uint8_t *slot = ring + s * SLOT;
      // B fragments: this lane's token (row g of each N tile) at the warp's
      // columns of the stage, in the order of the thread's weight bytes
      uint32_t bfr[NT][BW];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // the K elements of this thread's weight bytes
        const int k_el = FP8 ? warp * 64 + 16 * c : (warp >> 1) * 64 + 8 * (2 * c + (warp & 1));
        const uint4 *src = reinterpret_cast<const uint4 *>(
            slot + ACT_OFF + (nt * 8 + g) * ACT_ROW + k_el * 2);
#pragma unroll
        for (int v = 0; v < BW / 4; ++v) {
          const uint4 x = src[v];
          bfr[nt][4 * v + 0] = x.x;
          bfr[nt][4 * v + 1] = x.y;
          bfr[nt][4 * v + 2] = x.z;
          bfr[nt][4 * v + 3] = x.w;
        }
      }
      // the block scales of the warp's 64 columns (one 128-column block),
      // behind the tile: the gate rows' and the up rows' (phase 1), or the
      // rows' (phase 2)
      float sc_a = 1.f, sc_b = 1.f;
      if constexpr (FP8) {
        const float *sc = reinterpret_cast<const float *>(slot + ROWS * min(KBYTES, kbytes - cur.ks * KBYTES));
        const int col = warp * 64 / 128;
        sc_a = sc[col];
        sc_b = PHASE == 1 ? sc[4 + col] : sc_a;
      }
      // this warp's 4 KB of the stage: [row tile mt][half h][lane][16 bytes];
      // all of it first, then the MMAs with the four row tiles' chains
      // interleaved (consecutive MMAs are independent)
      // E4M3: [warp][row tile][half][lane]; BF16: row 8 m + g (m = 2 mt + half)
      // of column w / 2 at chunk position (2 c + w % 2) ^ g, groups 64 pieces apart
      const uint4 *st =
          reinterpret_cast<const uint4 *>(slot) +
          (FP8 ? warp * 256 + lane : (warp >> 1) * 512 + g * 8 + ((2 * c + (warp & 1)) ^ g));
      constexpr int GROUP = FP8 ? 32 : 64;  // pieces between consecutive row halves
      uint32_t wl[4][4], wh[4][4];
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        const uint4 lo = st[(mt * 2 + 0) * GROUP];
        const uint4 hi = st[(mt * 2 + 1) * GROUP];
        wl[mt][0] = lo.x; wl[mt][1] = lo.y; wl[mt][2] = lo.z; wl[mt][3] = lo.w;
        wh[mt][0] = hi.x; wh[mt][1] = hi.y; wh[mt][2] = hi.z; wh[mt][3] = hi.w;
      }
      if (FP8) {
        float tmp[4][NT][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) tmp[mt][nt][q] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            uint32_t a[4];
            e4m3x4_to_f16x2x2(wl[mt][j], a[0], a[2]);
            e4m3x4_to_f16x2x2(wh[mt][j], a[1], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt * 8 < m_left)
                mma_16816<false>(tmp[mt][nt], a, bfr[nt][2 * j], bfr[nt][2 * j + 1]);
          }
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          const float scl = mt < 2 ? sc_a : sc_b;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mt][nt][q] = fmaf(scl, tmp[mt][nt][q], acc[mt][nt][q]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const uint32_t a[4] = {wl[mt][2 * j], wh[mt][2 * j], wl[mt][2 * j + 1],
                                   wh[mt][2 * j + 1]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              if (nt * 8 < m_left)
                mma_16816<true>(acc[mt][nt], a, bfr[nt][2 * j], bfr[nt][2 * j + 1]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++it;

    if (cur.ks == kstages - 1) {
      // hand this (item, token group)'s K-partials to the epilogue warp
      const int b = ep % RB;
      const uint32_t round = ep / RB;
      if (!aborted && s_abort) aborted = true;
      if (!aborted && round > 0 && !mbar_wait_bounded(&rempty[b], (round - 1) & 1, P.timeout_ns)) {
        aborted = true;
        s_abort = 1;
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
      }
      if (!aborted) {
        float4 *rb_buf = red + b * RED_F4;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            rb_buf[((warp * 4 + mt) * NT + nt) * 32 + lane] =
                make_float4(acc[mt][nt][0], acc[mt][nt][1], acc[mt][nt][2], acc[mt][nt][3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[b]);
      ++ep;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[mt][nt][q] = 0.f;
    }

    have = cursor_next<TOK>(cur, T, P.row_blocks, kstages, await_tables, P.err, tid == 0);
  }
}

template <bool FP8, int PHASE, int NT>
cudaError_t launch_one(const TcParams &P, int grid, cudaStream_t stream) {
  auto kern = expert_tc_kernel<FP8, PHASE, NT>;
  constexpr size_t smem = smem_bytes<FP8, NT>();
  // 227 KB per CTA, of which the static plan tables take under 6.5 KB
  // (E4M3 phase 2 adds its 2.1 KB table of slot exponents)
  static_assert(smem + 6656 + (FP8 && PHASE == 2 ? MAX_ALL_SLOTS : 0) <= 232448,
                "the ring does not fit in shared memory");
  // the shared-memory opt-in is set once per device (the first call), so
  // later calls, e.g. under stream capture, only launch
  static unsigned long long configured = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  return launch_dependent(kern, dim3(grid), dim3(THREADS), smem, stream, P);
}

template <bool FP8, int PHASE>
cudaError_t launch_nt(const TcParams &P, int nt, int grid, cudaStream_t stream) {
  if (nt != 1) return cudaErrorInvalidValue;  // only the 8-token tile is built
  return launch_one<FP8, PHASE, 1>(P, grid, stream);
}

}  // namespace

cudaError_t launch_expert_tc(bool fp8, int phase, int n_tiles, const TcParams &P, int grid,
                             cudaStream_t stream) {
  if (fp8) {
    return phase == 1 ? launch_nt<true, 1>(P, n_tiles, grid, stream)
                      : launch_nt<true, 2>(P, n_tiles, grid, stream);
  }
  return phase == 1 ? launch_nt<false, 1>(P, n_tiles, grid, stream)
                    : launch_nt<false, 2>(P, n_tiles, grid, stream);
}

}  // namespace moe
