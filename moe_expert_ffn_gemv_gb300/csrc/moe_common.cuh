// moe_common.cuh -- device helpers shared by the library's kernels:
// mbarrier and bulk-copy (TMA) wrappers in inline PTX, bounded waits, error
// recording and the workspace layout.  Internal to the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_verify.h"

namespace moe {

// Geometry of a packed weight tile (pack.cu) = one pipeline stage of the
// tensor-core expert kernel: 64 rows x 512 bytes, 8 consumer warps x 64 bytes.
// An E4M3 tile is followed by its block scales: 8 floats, the 4 128-column
// blocks of its first 32 rows, then those of its last 32 rows (W13: gate,
// then up rows; W2: one 128-row block, so the two halves are equal).
constexpr int PACK_ROWS = 64;
constexpr int PACK_KBYTES = 512;
constexpr int PACK_SCALE_BYTES = 32;

// Packed bytes of one expert matrix of `rows` rows and `kbytes` bytes a row.
inline int64_t packed_matrix_bytes(int rows, int kbytes, bool fp8) {
  const int64_t tiles = int64_t(rows / PACK_ROWS) * ((kbytes + PACK_KBYTES - 1) / PACK_KBYTES);
  return int64_t(rows) * kbytes + (fp8 ? tiles * PACK_SCALE_BYTES : 0);
}

// ------------------------------------------------------------------ status

// The first device-side error wins; later ones are dropped.
__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// An unsigned integer with the order of the double s (for s not NaN): the
// sign bit flipped for s >= 0, all bits flipped for s < 0, and -0 taken as
// +0 so that equal values give equal keys.  Every key of a non-NaN value is
// above 0.  Ranking on keys costs integer compares instead of fp64 ones.
__device__ __forceinline__ unsigned long long order_key(double s) {
  if (s == 0.0) s = 0.0;
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(s));
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream serialization attribute may start before the kernel ahead of it in
// the stream has finished: pdl_wait() returns once that kernel has completed
// and its memory is visible (at once when the launch had no such
// attribute), and pdl_trigger() lets the kernel behind this one start
// launching once every CTA of this one has triggered or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's earlier generic-proxy view of global memory (e.g.
// data another CTA published through a release / acquire pair) before its
// later async-proxy accesses (bulk copies).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Called by a whole warp: lane 0 polls the device word *p (acquire, with a
// short sleep between reads, so that many waiting warps do not crowd the
// L2 slice that holds it) until it reaches `target` or `limit_ns` passes.
// Returns, in every lane, whether it was reached.
__device__ __forceinline__ bool await_flag(const uint32_t *p, uint32_t target,
                                           uint64_t limit_ns) {
  int seen = 1;
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(p) < target) {
      if (globaltimer_ns() - t0 > limit_ns) {
        seen = 0;
        break;
      }
      __nanosleep(64);
    }
  }
  return __shfl_sync(0xffffffffu, seen, 0) != 0;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete, for at most
// `limit_ns` nanoseconds.  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return mbar_try_wait(bar, parity);
  }
}

// ------------------------------------------------------------- bulk copies

// L2 policy for data read exactly once (expert weights): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// For data read again soon (the next pass over the same weights): normal
// L2 priority, so the evict-first stream goes before it.
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One-dimensional TMA bulk copy global -> shared, completing `bytes` of
// transaction count on `bar`.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Two-dimensional TMA tensor copy global -> shared of the box at element
// coordinates (x, y) of the tensor map (x, the innermost, a multiple of 16
// bytes' worth of elements), completing its bytes on `bar`.  `map` is the
// generic address of a tensor map in kernel parameter space.
__device__ __forceinline__ void tma_load_2d(void *dst, const void *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Asks L2 to fetch [p, p + bytes) ahead of use, at normal priority (a hint;
// p and bytes multiples of 16).
__device__ __forceinline__ void prefetch_l2(const void *p, uint64_t bytes) {
  const char *c = static_cast<const char *>(p);
  while (bytes > 0) {
    const uint32_t n = uint32_t(bytes < (1u << 20) ? bytes : (1u << 20));
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(n) : "memory");
    c += n;
    bytes -= n;
  }
}

// ------------------------------------------------------------ tensor cores

// D += A * B for one m16n8k16 tile, f16 or bf16 inputs, fp32 accumulators.
// Not volatile: the compiler may interleave independent MMAs.
template <bool BF16>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ---- tcgen05 (5th-generation tensor cores; accumulators in tensor memory)
//
// Shared-memory operand descriptor of a K-major tile in the 128-byte swizzled
// layout: rows of 128 bytes, 8-row groups 1024 bytes apart (the stride
// field), 16-byte chunk j of row r stored at position j ^ (r % 8), groups
// starting on 1024-byte boundaries.  Fields: start address >> 4 (bits
// 0-13), leading offset (unused by this layout, 1), stride offset >> 4
// (bits 32-45), descriptor version 1 (bit 46), layout 2 = 128-byte swizzle
// (bits 61-63).  A K step of 16 bf16 elements (32 bytes) inside the 128-byte
// row advances the start address by 32.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr) {
  return uint64_t((smem_addr >> 4) & 0x3FFF) | (uint64_t(1) << 16) |
         (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and
// fp32 accumulators: D format (bits 4-5) 1 = f32, A format (7-9) and B
// format (10-12) 1 = bf16, N >> 3 (17-22), M >> 4 (24-28).
__device__ __forceinline__ uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
         (uint32_t(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate)));
}

// Arrives (once) on `bar` when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `cols` tensor-memory columns (a power of two >= 32),
// the base address written to *slot; then give up the right to allocate more.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Whole warp.
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols)
               : "memory");
}

// Whole warp: 64 consecutive 32-bit columns of the warp's 32 lanes (lane l
// of the warp gets row (taddr lane) + l), then waits for the load.
__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
        "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
        "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]),
        "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (tcgen05.mma operand reads, bulk copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier ID (1..15) over `threads` threads (a multiple of 32).
template <int ID>
__device__ __forceinline__ void named_sync(int threads) {
  asm volatile("bar.sync %0, %1;" ::"n"(ID), "r"(threads) : "memory");
}

// Four E4M3 bytes b0..b3 (b0 least significant) -> two f16x2 words:
// lo = (b0, b1), hi = (b2, b3), the lower byte in the lower half.  Exact:
// every E4M3 value is an fp16 value.  One cvt per pair, no repacking.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four_bytes, uint32_t &lo,
                                                  uint32_t &hi) {
  asm("{\n"
      ".reg .b16 l, h;\n"
      "mov.b32 {l, h}, %2;\n"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n"
      "}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(four_bytes));
}

// --------------------------------------------------- fp16 range of E4M3 MMA
//
// The E4M3 engines multiply on fp16 tensor cores (every E4M3 value is an
// fp16 value), so each activation row reaches them scaled by an exact power
// of two 2^shift that puts its largest magnitude m in [2^14, 2^15): no
// element overflows fp16, and every element above m * 2^-28 keeps all its
// bf16 bits.  The sums are scaled back by 2^-shift in fp32.  `bits` are the
// bits of m >= 0 as a float: shift = 14 - floor(log2 m), clamped to
// [-113, 126] so that both 2^shift and 2^-shift are normal floats (a row
// whose largest magnitude is below 2^-112 lands below 2^14, still exactly);
// 0 for m = 0, inf or NaN (they pass through unchanged).
__device__ __forceinline__ int fp16_range_shift(uint32_t bits) {
  const int e = int(bits >> 23);  // biased exponent of m
  if (bits == 0u || e >= 255) return 0;
  const int s = 141 - e;          // 14 - (e - 127)
  return s < -113 ? -113 : s > 126 ? 126 : s;
}

// 2^s as a float, for s in [-126, 127].
__device__ __forceinline__ float pow2f(int s) { return __int_as_float((s + 127) << 23); }

// --------------------------------------------------------------- workspace

// Layout of the caller's workspace (all offsets 256-byte aligned):
//   [0, 256)           header: int32 error word at byte 0, the fused
//                      route + plan kernel's ticket counters at byte 64
//                      and at bytes 128 .. 159 (one an 8-token group),
//                      moe_verify_pass's plan-ready flag at byte 72 and its
//                      scaled-rows counter at byte 76
//   inter              [n_max*(k+n_shared)][I] intermediate a = silu(g)*u
//                      (fp32 for F32 weights, bf16 for BF16; E4M3: bf16 as
//                      the gate/up kernel writes it, then fp16 in place, row
//                      `slot` scaled by 2^ashift[slot])
//   yslot              [n_max*(k+n_shared)][d] fp32 per-slot expert outputs
//   E4M3 weights only:
//   h16                [n_max][d] fp16: h[t] * 2^hshift[t]
//   hshift             [n_max] int32
//   ashift             [n_max*(k+n_shared)] int32
//   BF16 weights only:
//   aperm              [n_max*(k+n_shared)][I] bf16: a of the segments the
//                      tcgen05 CTAs run, in plan order (row offs[u] + i for
//                      slot perm[offs[u] + i]; the shared expert at n*k + t)
struct Workspace {
  size_t inter, yslot, h16, hshift, ashift, aperm, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr size_t WS_TICKET_OFFSET = 64;
// The fused route + plan kernel's ticket counters of the 8-token groups
// (n_max / 8 <= 8 of them), at bytes 128 .. 159; each is back at zero when
// the kernel ends.
constexpr size_t WS_GROUP_TICKETS_OFFSET = 128;
// The plan-ready flag of moe_verify_pass: raised by its plan kernel once the
// plan is written, read by its first expert kernel, cleared by its combine.
constexpr size_t WS_READY_OFFSET = 72;
// moe_verify_pass with E4M3 weights: the count of 8-token blocks whose
// scaled rows (h16, hshift) its plan kernel has written; read by the first
// expert kernel, cleared by the combine.
constexpr size_t WS_ACTS_OFFSET = 76;

inline Workspace workspace_layout(const moe_layer_desc &L) {
  const size_t slots = size_t(L.n_max) * size_t(L.top_k + L.n_shared);
  const size_t inter_es = L.w_dtype == MOE_F32 ? 4 : 2;
  const bool e4m3 = L.w_dtype == MOE_E4M3_B128;
  Workspace w;
  size_t off = 256;
  w.inter = off;
  off += align256(slots * size_t(L.inter) * inter_es);
  w.yslot = off;
  off += align256(slots * size_t(L.d) * 4);
  w.h16 = off;
  off += e4m3 ? align256(size_t(L.n_max) * size_t(L.d) * 2) : 0;
  w.hshift = off;
  off += e4m3 ? align256(size_t(L.n_max) * 4) : 0;
  w.ashift = off;
  off += e4m3 ? align256(slots * 4) : 0;
  w.aperm = off;
  off += L.w_dtype == MOE_BF16 ? align256(slots * size_t(L.inter) * 2) : 0;
  w.total = off;
  return w;
}

// Which slot rows a segment of expert work covers.
//   dedup:    segment u < U is expert uniq[u], slots perm[offs[u] .. offs[u+1]);
//             segment U (if a shared expert exists) is the shared expert on
//             slots n*k + t for every token t.
//   per-slot: segment s < n*k is expert ids[s] on slot s alone; segment
//             n*k + t is the shared expert on slot n*k + t alone.
struct SegTables {
  const int32_t *ids;     // [n*k]
  const int32_t *uniq;    // dedup only
  const int32_t *offs;    // dedup only
  const int32_t *perm;    // dedup only
  const int32_t *n_uniq;  // dedup only
  int32_t n, k, n_experts, n_shared;
  int32_t dedup;  // 1 = deduplicating engine, 0 = per-slot
};

struct Seg {
  int32_t expert;  // -1 = shared expert, -2 = invalid id (skip)
  int32_t m;       // tokens (slots) in the segment
  int32_t first;   // dedup: offset into perm; per-slot: the slot index
};

// U of a deduplicating plan, or 0 when it is out of [0, N] (the plan is
// then treated as empty; get_segment reports it).
__device__ __forceinline__ int32_t plan_U(const SegTables &T) {
  const int32_t U = __ldg(T.n_uniq);
  return (U >= 0 && U <= T.n_experts) ? U : 0;
}

__device__ __forceinline__ int32_t n_segments(const SegTables &T) {
  if (T.dedup) return plan_U(T) + T.n_shared;
  return T.n * T.k + T.n_shared * T.n;
}

__device__ __forceinline__ Seg get_segment(const SegTables &T, int32_t u) {
  Seg s;
  const int32_t nk = T.n * T.k;
  if (T.dedup) {
    const int32_t U = plan_U(T);
    if (u < U) {
      // a caller's plan is checked before its indices are used: an expert
      // id, a group inside [0, n*k) and slots below n*k, else skipped (-2)
      s.expert = __ldg(T.uniq + u);
      s.first = __ldg(T.offs + u);
      const int32_t last = __ldg(T.offs + u + 1);
      s.m = last - s.first;
      bool ok = s.expert >= 0 && s.expert < T.n_experts && s.first >= 0 && s.m >= 0 && last <= nk;
      for (int32_t i = 0; ok && i < s.m; ++i) {
        const int32_t p = __ldg(T.perm + s.first + i);
        ok = p >= 0 && p < nk;
      }
      if (!ok) {
        s.expert = -2;
        s.m = 0;
      }
    } else {
      s.expert = -1;
      s.first = 0;
      s.m = T.n;
    }
  } else {
    s.m = 1;
    s.first = u;
    if (u < nk) {
      const int32_t e = __ldg(T.ids + u);
      s.expert = (e >= 0 && e < T.n_experts) ? e : -2;
    } else {
      s.expert = -1;
    }
  }
  return s;
}

// Slot index of the i-th token of segment s.
__device__ __forceinline__ int32_t segment_slot(const SegTables &T, const Seg &s, int32_t i) {
  if (!T.dedup) return s.first;
  if (s.expert == -1) return T.n * T.k + i;
  return __ldg(T.perm + s.first + i);
}

__device__ __forceinline__ int32_t slot_token(const SegTables &T, int32_t slot) {
  const int32_t nk = T.n * T.k;
  return slot < nk ? slot / T.k : slot - nk;
}

}  // namespace moe
