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
#include <mutex>

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
  int wide_m;           // segments of more tokens go to the tcgen05 CTAs (wide_cta)

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
  int stride;                   // CTAs walking these items
  Seg sg;
};

// CTA `first` of `stride` (the CTAs that run this path; the others, if any,
// run the segments of more than T.wide_m tokens on tcgen05).
__device__ __forceinline__ void cursor_start(Cursor &c, int first, int stride) {
  c.item = first;
  c.stride = stride;
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
    if (c.sg.m > T.wide_m) {  // a tcgen05 CTA's
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
  c.item += c.stride;
  return cursor_item<TOK>(c, T, row_blocks, ensure, err, report);
}

// ------------------------------------------------------------- wide CTAs
//
// A segment of more than WIDE_M tokens (a popular routed expert in a
// correlated draft tree, identical tokens, a shared expert at n > 8) would
// stream its weights through the mma.sync path once per 8 tokens.  In the
// WIDE instance (which the host launches for BF16 deduplicating passes of
// 25 tokens or more) it runs instead on the 5th-generation tensor cores, on
// CTAs of its own (the first W of the grid), so that each weight row crosses
// the SM once per pass:
//   - a work item is (segment, row pair): 128 weight rows, the packed tiles
//     of row blocks 2p and 2p + 1, against all m <= 64 tokens of the segment;
//   - a stage is one 128-byte column of K: the two tiles' 8 KB columns (one
//     bulk copy each, warp 0) are the A operand as they are (the packed BF16
//     tiles are in the 128-byte swizzled K-major layout); B is one 2-D TMA
//     box of that column (warp 1, the tensor map swizzling it as the MMA
//     reads it): in phase 1 the hidden rows of all n tokens (the MMA runs
//     every token and the epilogue keeps the segment's: rows of h are
//     contiguous, the segment's tokens are not), in phase 2 the segment's
//     rows of aperm, where phase 1 wrote them in plan order;
//   - warp 8 allocates 128 tensor-memory columns (two accumulators of up to
//     64 columns) and one of its threads issues tcgen05.mma (M = 128, N = n
//     (phase 1) or m (phase 2) rounded up to 16, K = 16; four a stage),
//     committing each stage's slot back to the producers and each finished
//     item to the epilogue;
//   - warps 4-7 read the accumulator rows of their lane quarter with
//     tcgen05.ld.  Phase 1: the gate warp and the up warp of a tile put
//     their sums in shared memory and share out a = silu(g)*u of the
//     segment's tokens (a short loop over the m tokens, not one unrolled
//     over all n columns: under the bulk-copy traffic each cold stretch of
//     code costs about a microsecond to fetch), then write aperm in 16-byte
//     pieces.  Phase 2 writes the per-slot output rows, also transposed
//     through shared memory into 16-byte stores (each store instruction
//     costs ~0.1-0.3 us under that traffic; one 4-byte store a column and
//     lane held the first items up for 4-19 us).
// W is the split of the grid with the shortest modelled makespan, a wide
// item costing W_ITEM_COST_P1 (gate/up) or W_ITEM_COST_P2 (down) hundredths
// of a narrow one.  While both kinds
// stream, HBM is saturated and a tensor-memory CTA completes a 16 KB stage
// every ~0.42 us against ~0.7 us for a narrow CTA's 32 KB (its share of the
// memory system: a 5-slot ring measured the same); with the start offsets,
// the wide epilogue's tail and whole items per CTA, 3 measured best overall.
// Every wait is bounded; after a time-out the warps keep walking their items
// without waiting, so that all of them reach the final barrier, and the
// tensor memory is freed only after every issued MMA has completed.
constexpr int WIDE_M = 8;
constexpr int W_A_BYTES = 16384;  // 128 rows x 128 bytes of K
// Shared memory: the ring, then the epilogue's buffers, in what the narrow
// kernel's layout leaves below its barriers (less 1 KB for the alignment).
// A ring slot is the A operand and a B box of up to pad16(n) rows of 128
// bytes; as many slots as fit (at most W_MAX_STAGES) keep 110-180 KB of
// weights in flight, as the mma.sync CTAs do (160 KB).
constexpr int W_MAX_STAGES = 12;
// the modelled cost of a wide item, in hundredths of a narrow item's, for
// the gate/up and the down kernel: the best of 230-360 (gate/up) and
// 240-500 (down) on Qwen3- and OLMoE-shaped trees of 25-64 tokens.  A down
// cost of 360 against 300 took OLMoE rho = 0.9 n = 32 from 119.5 to
// 112.3 us and Qwen3 sigma = 1.0 n = 64 from 166.6 to 159.4 us (dedup
// calls), and left the others level.
constexpr int W_ITEM_COST_P1 = 300;
constexpr int W_ITEM_COST_P2 = 360;
constexpr int W_AVAIL =
    int(n_stages<false, 1>() * size_t(slot_bytes<false, 1>()) + n_red_bufs<false, 1>() * red_bytes<1>()) -
    1024;
// Epilogue buffers.  Phase 1, for each pair of warps (gate rows, up rows of
// one tile): the gate and the up sums [pad16(n) tokens][32 rows] fp32, the
// bf16 rows of a [m <= 64][32] and the segment's tokens [64] int16.
// Phase 2: each warp's output staging, 32 columns x 32 rows of fp32.
__host__ __device__ constexpr int wide_pair_bytes(int ncol) { return ncol * 32 * 4 * 2 + 64 * 32 * 2 + 128; }
__host__ __device__ constexpr int wide_epi_bytes(int phase, int ncol) {
  return phase == 1 ? 2 * wide_pair_bytes(ncol) : 4 * 32 * 32 * 4;
}
static_assert(W_AVAIL - wide_epi_bytes(1, 64) >= 4 * (W_A_BYTES + 64 * 128), "wide ring under 4 stages");
constexpr uint32_t W_TMEM_COLS = 128;
constexpr int W_PRODUCER = 0, W_BWARP = 1, W_EPI0 = 4, W_MMA = 8;

// Wide item sequence of one CTA: items numbered segment by segment (wide
// segments only), row pair innermost; CTA b of W takes items b, b + W, ...
struct WideCursor {
  int item, stride, u, first, count, p;
  Seg sg;
};

__device__ __forceinline__ bool wide_next(WideCursor &c, const LocalTables &T, int pairs) {
  while (c.item >= c.first + c.count) {
    c.first += c.count;
    c.u += 1;
    if (c.u >= T.n_segments()) return false;
    c.sg = T.segment(c.u);
    c.count = (c.sg.expert != -2 && c.sg.m > T.wide_m) ? pairs : 0;
  }
  c.p = c.item - c.first;
  return true;
}

template <int PHASE>
__device__ __forceinline__ void wide_cta(const TcParams &P, const LocalTables &T, uint8_t *dyn,
                                      int W, volatile int *abort_flag) {
  __shared__ uint64_t wfull[W_MAX_STAGES], wempty[W_MAX_STAGES], tfull[2], tempty[2], wdone;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 128-byte swizzled operands start on 1024-byte boundaries
  uint8_t *base = dyn + ((1024 - (smem_u32(dyn) & 1023)) & 1023);
  // slot = A + a B box of pad16(n) rows (phase 2's boxes, pad16(m), are no larger)
  const int ncol = (T.n + 15) & ~15;
  const int wslot = W_A_BYTES + ncol * 128;
  const int WS = min(W_MAX_STAGES, (W_AVAIL - wide_epi_bytes(PHASE, ncol)) / wslot);
  uint8_t *epi = base + WS * wslot;  // the epilogue's buffers
  const int kst = P.kdim / 64;  // 128-byte columns of K
  const int64_t rb_bytes = int64_t(ROWS) * P.kdim * 2;
  const int pairs = (P.row_blocks + 1) / 2;
  const uint64_t limit = P.timeout_ns;
  if (threadIdx.x == 0) {
    for (int s = 0; s < WS; ++s) {
      mbar_init(&wfull[s], 2);  // the A and B warps' arrivals, with their copies' bytes
      mbar_init(&wempty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(&wdone, 1);
    fence_barrier_init();
  }
  if (warp == W_MMA) tmem_alloc(&tmem_slot, W_TMEM_COLS);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  auto fail = [&]() {
    *abort_flag = 1;
    if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
  };
  WideCursor cur;
  cur.item = blockIdx.x;
  cur.stride = W;
  cur.u = -1;
  cur.first = 0;
  cur.count = 0;

  if (warp == W_PRODUCER) {
    // ------------------------------------------------ A: two tiles' columns
    const uint64_t policy = policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    while (ok && wide_next(cur, T, pairs)) {
      const uint8_t *ebase =
          cur.sg.expert >= 0 ? P.w + int64_t(cur.sg.expert) * P.expert_stride : P.w_sh;
      const int rb0 = 2 * cur.p;
      const bool two = rb0 + 1 < P.row_blocks;  // phase 2 may end on a single tile
      for (int q = 0; q < kst; ++q, ++it) {
        const int s = it % WS;
        const uint32_t round = it / WS;
        if (round > 0 && !mbar_wait_bounded(&wempty[s], (round - 1) & 1, limit)) {
          ok = false;
          break;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t *a = base + s * wslot;
          mbar_arrive_expect_tx(&wfull[s], two ? 16384u : 8192u);
          bulk_g2s(a, ebase + rb0 * rb_bytes + int64_t(q) * 8192, 8192, &wfull[s], policy);
          if (two)
            bulk_g2s(a + 8192, ebase + (rb0 + 1) * rb_bytes + int64_t(q) * 8192, 8192, &wfull[s],
                     policy);
        }
        __syncwarp();
      }
      cur.item += cur.stride;
    }
    if (!ok) fail();
    // let every copy this warp issued land before the CTA may exit
    const uint32_t first = it > uint32_t(WS) ? it - WS : 0;
    for (uint32_t j = first; j < it; ++j)
      if (!mbar_wait_bounded(&wfull[j % WS], (j / WS) & 1, DRAIN_LIMIT_NS)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        break;
      }
  } else if (warp == W_BWARP) {
    // ------------------------------- B: one TMA box of the column a stage
    // Phase 2 reads phase 1's aperm, so it waits for phase 1 first.  Row t of
    // a box lands at t * 128 from a 1024-byte boundary, where the map's
    // 128-byte swizzle puts its chunk j at position j ^ (t % 8).  Rows past
    // the segment's m (phase 2) belong to the next segment or arrive as
    // zeros: they only reach accumulator columns that nothing reads.
    if (PHASE == 2) pdl_wait();
    uint32_t it = 0;
    bool ok = true;
    const int nk = T.n * T.k;
    while (ok && wide_next(cur, T, pairs)) {
      const int nb = PHASE == 1 ? (T.n + 15) & ~15 : (cur.sg.m + 15) & ~15;  // rows of the box
      const void *map = &P.act_map[PHASE == 1 ? 0 : nb / 16 - 1];
      const int y0 = PHASE == 1 ? 0 : cur.sg.expert == -1 ? nk : cur.sg.first;
      for (int q = 0; q < kst; ++q, ++it) {
        const int s = it % WS;
        const uint32_t round = it / WS;
        if (round > 0 && !mbar_wait_bounded(&wempty[s], (round - 1) & 1, limit)) {
          ok = false;
          break;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t *b = base + s * wslot + W_A_BYTES;
          mbar_arrive_expect_tx(&wfull[s], uint32_t(nb) * 128);
          tma_load_2d(b, map, q * 64, y0, &wfull[s]);
        }
        __syncwarp();
      }
      cur.item += cur.stride;
    }
    if (!ok) fail();
    // let every copy this warp issued land before the CTA may exit
    const uint32_t first = it > uint32_t(WS) ? it - WS : 0;
    for (uint32_t j = first; j < it; ++j)
      if (!mbar_wait_bounded(&wfull[j % WS], (j / WS) & 1, DRAIN_LIMIT_NS)) {
        if (lane == 0) record_error(P.err, MOE_ERR_TIMEOUT);
        break;
      }
  } else if (warp == W_MMA) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t it = 0, ic = 0;
      bool ok = true, issued = false;
      while (ok && wide_next(cur, T, pairs)) {
        const uint32_t idesc =
            umma_idesc_bf16(128, PHASE == 1 ? (T.n + 15) & ~15 : (cur.sg.m + 15) & ~15);
        const int acc = ic & 1;
        const uint32_t tround = ic >> 1;
        if (tround > 0 && !mbar_wait_bounded(&tempty[acc], (tround - 1) & 1, limit)) {
          ok = false;
          break;
        }
        tmem_fence_after_sync();
        const uint32_t d = tmem + acc * 64;
        for (int q = 0; q < kst; ++q, ++it) {
          const int s = it % WS;
          const uint32_t round = it / WS;
          if (!mbar_wait_bounded(&wfull[s], round & 1, limit) || *abort_flag) {
            ok = false;
            break;
          }
          tmem_fence_after_sync();
          const uint32_t a = smem_u32(base + s * wslot), b = a + W_A_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(d, umma_desc_sw128(a + 32 * k), umma_desc_sw128(b + 32 * k), idesc,
                      q > 0 || k > 0);
          umma_commit(&wempty[s]);
          issued = true;
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        ++ic;
        cur.item += cur.stride;
      }
      // every MMA issued has completed before tensor memory is freed
      if (issued) {
        umma_commit(&wdone);
        if (!mbar_wait_bounded(&wdone, 0, DRAIN_LIMIT_NS)) record_error(P.err, MOE_ERR_TIMEOUT);
      }
      if (!ok) {
        *abort_flag = 1;
        record_error(P.err, MOE_ERR_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp >= W_EPI0 && warp < W_EPI0 + 4) {
    // ------------------------------------------------------------ epilogue
    const int qd = warp - W_EPI0;  // tensor-memory lane quarter
    const int nk = T.n * T.k;
    uint32_t ic = 0;
    bool ok = true;
    while (wide_next(cur, T, pairs)) {
      const int m = cur.sg.m;
      const int acc = ic & 1;
      const uint32_t tround = ic >> 1;
      if (ok && (*abort_flag || !mbar_wait_bounded(&tfull[acc], tround & 1, limit))) {
        ok = false;
        fail();
      }
      uint32_t v[64];
      if (ok) {
        tmem_fence_after_sync();
        tmem_ld_x64(tmem + (uint32_t(32 * qd) << 16) + uint32_t(acc * 64), v);
        tmem_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      }
      if (PHASE == 1) {
        // Accumulator column c is token c.  Quarters 0 and 1 hold the gate
        // and the up rows of tile 0, quarters 2 and 3 those of tile 1; each
        // pair meets in shared memory, where its two warps compute
        // a = silu(g) * u of the segment's tokens (alternate tokens, a lane
        // a row) and write them to aperm in 16-byte pieces.  The two pair
        // barriers are passed on every item, also after a time-out.
        const int pr = qd >> 1, up = qd & 1;
        float *gs = reinterpret_cast<float *>(epi + pr * wide_pair_bytes(ncol));  // [ncol][32]
        float *us = gs + ncol * 32;
        __nv_bfloat16 *ob = reinterpret_cast<__nv_bfloat16 *>(us + ncol * 32);  // [m][32]
        int16_t *tok = reinterpret_cast<int16_t *>(ob + 64 * 32);               // [m]
        if (ok) {
          float *dst = up ? us : gs;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < ncol) dst[c * 32 + lane] = __uint_as_float(v[c]);
          if (!up)
            for (int i = lane; i < m; i += 32) tok[i] = int16_t(T.token(T.slot(cur.sg, i)));
        }
        if (pr) named_sync<2>(64); else named_sync<1>(64);
        if (ok) {
#pragma unroll 2
          for (int i = up; i < m; i += 2) {
            const int c = tok[i];
            ob[i * 32 + lane] = __float2bfloat16_rn(silu_times(gs[c * 32 + lane], us[c * 32 + lane]));
          }
        }
        if (pr) named_sync<2>(64); else named_sync<1>(64);
        if (ok) {
          // row i of the block: columns 64p + 32 pr .. + 31 of aperm row y0 + i
          const int y0 = cur.sg.expert == -1 ? nk : cur.sg.first;
          __nv_bfloat16 *a0 = static_cast<__nv_bfloat16 *>(P.aperm) + 64 * cur.p + 32 * pr;
          for (int j = up * 32 + lane; j < 4 * m; j += 64) {
            const int i = j >> 2, piece = j & 3;
            *reinterpret_cast<uint4 *>(a0 + int64_t(y0 + i) * P.inter + piece * 8) =
                *reinterpret_cast<const uint4 *>(ob + i * 32 + piece * 8);
          }
        }
      } else if (ok) {
        // rows 128p + 32qd .. +31 of the per-slot outputs, 32 columns at a time
        // through this warp's 4 KB of the staging area
        const int row0 = 128 * cur.p + 32 * qd;
        float *st = reinterpret_cast<float *>(epi) + qd * 32 * 32;
        float *out = static_cast<float *>(P.out);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          if (half * 32 < m) {
#pragma unroll
            for (int c = 0; c < 32; ++c) st[c * 32 + lane] = __uint_as_float(v[half * 32 + c]);
            __syncwarp();
            const int c = half * 32 + lane;
            if (c < m && row0 < P.rows_total) {
              const uint4 *src = reinterpret_cast<const uint4 *>(st + lane * 32);
              uint4 *dst = reinterpret_cast<uint4 *>(out + int64_t(T.slot(cur.sg, c)) * P.rows_total + row0);
#pragma unroll
              for (int j = 0; j < 8; ++j) dst[j] = src[j];
            }
            __syncwarp();
          }
        }
      }
      ++ic;
      cur.item += cur.stride;
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == W_MMA) tmem_dealloc(tmem, W_TMEM_COLS);
}

template <bool FP8, int PHASE, int NT, bool WIDE>
__global__ void __launch_bounds__(THREADS, 1) expert_tc_kernel(const __grid_constant__ TcParams P) {
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
    const bool seen = await_flag(P.acts, need, P.timeout_ns);
    if (seen) (void)ld_acquire_gpu(P.acts);  // this lane's own acquire (the count only grows)
    return seen;
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
                P.T.dedup, (!FP8 && WIDE) ? WIDE_M : 0x7fffffff};
  // The WIDE instance (BF16 deduplicating passes the host picks, never the
  // early-start mode): the first W CTAs take the segments of more than
  // WIDE_M tokens on tcgen05; every CTA computes the same W from the plan.
  int W = 0;
  if constexpr (!FP8 && WIDE) {
    {
      __shared__ int s_wide_ctas;
      if (warp == 0) {
        // narrow items (row block x token group) and wide items (row pairs)
        int nb = 0, wi = 0;
        const int ns = T.n_segments();
        for (int u = lane; u < ns; u += 32) {
          const Seg sg = T.segment(u);
          if (sg.expert == -2 || sg.m <= 0) continue;
          if (sg.m > WIDE_M) {
            wi += (P.row_blocks + 1) / 2;
          } else {
            nb += ((sg.m + TOK - 1) / TOK) * P.row_blocks;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          nb += __shfl_xor_sync(0xffffffffu, nb, o);
          wi += __shfl_xor_sync(0xffffffffu, wi, o);
        }
        // W: the split of the grid with the shortest modelled makespan, a
        // wide item (two row blocks) costing W_ITEM_COST_P1/_P2 hundredths of a
        // narrow one (one row block, one token group); each lane tries every
        // 32nd W, the warp takes the best (ties to the smaller W)
        const int G = gridDim.x;
        int best_t = 0x7fffffff, best_w = 0;
        if (wi > 0 && nb == 0) {
          best_w = min(G, wi);
        } else if (wi > 0) {
          for (int w = 1 + lane; w < G && w <= wi; w += 32) {
            const int t = max((PHASE == 1 ? W_ITEM_COST_P1 : W_ITEM_COST_P2) * ((wi + w - 1) / w),
                              100 * ((nb + (G - w) - 1) / (G - w)));
            if (t < best_t) { best_t = t; best_w = w; }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const int ot = __shfl_xor_sync(0xffffffffu, best_t, o);
          const int ow = __shfl_xor_sync(0xffffffffu, best_w, o);
          if (ot < best_t || (ot == best_t && ow < best_w)) { best_t = ot; best_w = ow; }
        }
        if (lane == 0) s_wide_ctas = best_w;
      }
      __syncthreads();
      W = s_wide_ctas;
      if (int(blockIdx.x) < W) {
        wide_cta<PHASE>(P, T, smem, W, &s_abort);
        return;
      }
    }
  }
  const int n_first = int(blockIdx.x) - W, n_stride = int(gridDim.x) - W;
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
    cursor_start(cur, n_first, n_stride);
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
        float4 *rb_buf = red + b * RED_F4;
        const int m_left = cur.sg.m - cur.grp * TOK;
        constexpr int MT_OUT = PHASE == 1 ? 2 : 4;
        const int gg = lane >> 2, cc = lane & 3;
        // this lane's outputs: (row tile mt, N tile nt) = (j / NT, j % NT),
        // rows mt*16 + gg (+8), columns nt*8 + 2cc (+1); the 8 warps'
        // K-partials added in a fixed order
        float res[MT_OUT * NT][4];
#pragma unroll
        for (int j = 0; j < MT_OUT * NT; ++j) {
          const int nt = j % NT, mt = j / NT;
          if (nt * 8 >= m_left) continue;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f), w4 = v;
#pragma unroll
          for (int w = 0; w < CONSUMERS; ++w) {
            const float4 x = rb_buf[((w * 4 + mt) * NT + nt) * 32 + lane];
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
            if (PHASE == 1) {
              const float4 y = rb_buf[((w * 4 + mt + 2) * NT + nt) * 32 + lane];
              w4.x += y.x; w4.y += y.y; w4.z += y.z; w4.w += y.w;
            }
          }
          const float vals[4] = {v.x, v.y, v.z, v.w};
          const float ups[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (PHASE == 1) {
              // columns past the segment's tokens are left out (never stored)
              float gv = vals[e], uv = ups[e];
              const int col = nt * 8 + 2 * cc + (e & 1);
              res[j][e] = 0.f;
              if (col < m_left) {
                if (FP8) {
                  // the rows were scaled by 2^hshift: scale the sums back
                  const float back = pow2f(-s_hshift[T.token(T.slot(cur.sg, cur.grp * TOK + col))]);
                  gv *= back;
                  uv *= back;
                }
                res[j][e] = silu_times(gv, uv);
              }
            } else {
              res[j][e] = vals[e];
            }
          }
        }
        // Through the buffer just read: [column][row] fp32, CS floats a
        // column (a stride that puts the 32 lanes' writes in 32 banks), then
        // each column's rows leave as 16-byte pieces: one store instruction
        // in place of 8 (phase 1) or 16 (phase 2) of 2 or 4 bytes a lane,
        // each of which costs ~0.1-0.3 us under the bulk-copy traffic.
        constexpr int CS = PHASE == 1 ? 36 : 68;
        float *st = reinterpret_cast<float *>(rb_buf);
        __syncwarp();
#pragma unroll
        for (int j = 0; j < MT_OUT * NT; ++j) {
          const int nt = j % NT, mt = j / NT;
          if (nt * 8 >= m_left) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            st[(nt * 8 + 2 * cc + (e & 1)) * CS + mt * 16 + gg + (e >> 1) * 8] = res[j][e];
        }
        __syncwarp();
        const int mcols = min(m_left, TOK);
        if (PHASE == 1) {
          // a column: rows rb*32 .. +31 of a, 4 pieces of 8 bf16
          for (int q = lane; q < mcols * 4; q += 32) {
            const int col = q >> 2, piece = q & 3;
            const float4 lo = *reinterpret_cast<const float4 *>(st + col * CS + piece * 8);
            const float4 hi = *reinterpret_cast<const float4 *>(st + col * CS + piece * 8 + 4);
            const __nv_bfloat162 p0 = __floats2bfloat162_rn(lo.x, lo.y), p1 = __floats2bfloat162_rn(lo.z, lo.w);
            const __nv_bfloat162 p2 = __floats2bfloat162_rn(hi.x, hi.y), p3 = __floats2bfloat162_rn(hi.z, hi.w);
            uint4 o;
            o.x = *reinterpret_cast<const uint32_t *>(&p0);
            o.y = *reinterpret_cast<const uint32_t *>(&p1);
            o.z = *reinterpret_cast<const uint32_t *>(&p2);
            o.w = *reinterpret_cast<const uint32_t *>(&p3);
            const int slot = T.slot(cur.sg, cur.grp * TOK + col);
            *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(P.out) + int64_t(slot) * P.inter +
                                       cur.rb * 32 + piece * 8) = o;
          }
        } else {
          // a column: rows rb*64 .. +63 of the slot's output, 16 pieces of 4
          for (int q = lane; q < mcols * 16; q += 32) {
            const int col = q >> 4, piece = q & 15;
            float4 x = *reinterpret_cast<const float4 *>(st + col * CS + piece * 4);
            const int slot = T.slot(cur.sg, cur.grp * TOK + col);
            if (FP8) {
              // E4M3: a reached the MMA scaled by 2^ashift[slot]
              const float back = pow2f(-s_ashift[slot]);
              x.x *= back; x.y *= back; x.z *= back; x.w *= back;
            }
            *reinterpret_cast<float4 *>(static_cast<float *>(P.out) + int64_t(slot) * P.rows_total +
                                        cur.rb * ROWS + piece * 4) = x;
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
      // lane 0 waits for the flag; then every lane acquires it itself (it
      // stays raised until the pass's combine), so that its own plan reads
      // below are ordered after the plan kernel's writes
      const bool seen = await_flag(P.ready, 1u, P.timeout_ns);
      if (seen) (void)ld_acquire_gpu(P.ready);
      if (!seen) {
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
    cursor_start(cur, n_first, n_stride);
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
    cursor_start(cur, n_first, n_stride);
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
  cursor_start(cur, n_first, n_stride);
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

template <bool FP8, int PHASE, int NT, bool WIDE>
cudaError_t launch_one(const TcParams &P, int grid, cudaStream_t stream) {
  auto kern = expert_tc_kernel<FP8, PHASE, NT, WIDE>;
  constexpr size_t smem = smem_bytes<FP8, NT>();
  // 227 KB per CTA, of which the static plan tables take under 6.5 KB
  // (E4M3 phase 2 adds its 2.1 KB table of slot exponents)
  static_assert(smem + 6656 + (FP8 && PHASE == 2 ? MAX_ALL_SLOTS : 0) <= 232448,
                "the ring does not fit in shared memory");
  // the wide CTAs' layout (W_AVAIL) stays below the ring's barriers (set up by every CTA)
  static_assert(FP8 || size_t(W_AVAIL) + 1024 <= size_t(n_stages<FP8, NT>()) * slot_bytes<FP8, NT>() +
                                                  n_red_bufs<FP8, NT>() * red_bytes<NT>(),
                "the wide layout overlaps the ring's barriers");
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
  // the tcgen05 CTAs are compiled into a kernel of their own, so that passes
  // without them run the mma.sync code as it is
  if constexpr (!FP8)
    if (P.wide) return launch_one<FP8, PHASE, 1, true>(P, grid, stream);
  return launch_one<FP8, PHASE, 1, false>(P, grid, stream);
}

}  // namespace

cudaError_t encode_act_map(CUtensorMap *map, const void *act, int rows, int kdim, int box_rows) {
  // cuTensorMapEncodeTiled from the driver, found once through the runtime
  using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode fn = nullptr;
  static cudaError_t found = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    found = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q);
    if (found == cudaSuccess && (q != cudaDriverEntryPointSuccess || !p))
      found = cudaErrorNotSupported;
    fn = reinterpret_cast<Encode>(p);
  });
  if (found != cudaSuccess) return found;
  // [rows][kdim] bf16, row stride kdim * 2 bytes (kdim % 64 == 0); boxes of
  // 64 elements (128 bytes) x box_rows rows, swizzled 128 bytes as the MMA
  // reads B; rows past the end arrive as zeros
  const cuuint64_t dims[2] = {cuuint64_t(kdim), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(kdim) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(act), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

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
