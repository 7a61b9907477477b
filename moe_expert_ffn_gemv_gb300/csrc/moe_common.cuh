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
//                      route + plan kernel's ticket counter at byte 64,
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
struct Workspace {
  size_t inter, yslot, h16, hshift, ashift, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr size_t WS_TICKET_OFFSET = 64;
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
