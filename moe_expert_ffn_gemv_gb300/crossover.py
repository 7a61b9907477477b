"""Host-side analysis of the two engines' timings: the dedup-vs-per-slot
criterion and the crossover pass size.

"Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
Bandwidth and the Best Draft Length" (abstract; Table 1 and its note):
  - the per-slot engine requests n*m*b bytes per pass (m experts per token,
    b bytes per expert), the deduplicating engine the union bytes U*b;
  - effective bandwidth = requested bytes / time;
  - u_bar(n) = U*b / (n*m*b), the deduplicating engine's share of the
    per-slot bytes; r(n) = beta_dedup / beta_slot;
  - deduplication is faster exactly where u_bar(n) < r(n) (eq. (7));
  - the crossover is the first pass size at which deduplication is faster.
A shared expert counts as one more expert per token (m = k + 1) and one more
union member (U + 1).
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence


def requested_bytes_perslot(n: int, k: int, expert_bytes: int, n_shared: int = 0) -> int:
    return n * (k + n_shared) * expert_bytes


def union_bytes(U: int, expert_bytes: int, n_shared: int = 0) -> int:
    return (U + n_shared) * expert_bytes


def u_bar(U: int, n: int, k: int, n_shared: int = 0) -> float:
    """Share of the per-slot bytes that the deduplicating engine requests."""
    return (U + n_shared) / (n * (k + n_shared))


def effective_bandwidth(nbytes: float, seconds: float) -> float:
    return nbytes / seconds


def r_ratio(beta_dedup: float, beta_slot: float) -> float:
    return beta_dedup / beta_slot


def dedup_faster(ubar: float, r: float) -> bool:
    """Deduplication is faster exactly where u_bar < r."""
    return ubar < r


def crossover(ns: Sequence[int], t_dedup: Sequence[float], t_slot: Sequence[float]) -> Optional[int]:
    """First pass size n at which the deduplicating engine is faster."""
    for n, td, ts in zip(ns, t_dedup, t_slot):
        if td < ts:
            return n
    return None


def analyse(rows: Iterable[Dict], k: int, expert_bytes: int, n_shared: int = 0) -> List[Dict]:
    """rows: dicts with n, U, t_dedup, t_slot (seconds) -> adds u_bar, betas,
    r and whether the criterion and the timings agree."""
    out = []
    for row in rows:
        n, U = row["n"], row["U"]
        ub = union_bytes(U, expert_bytes, n_shared)
        rb = requested_bytes_perslot(n, k, expert_bytes, n_shared)
        bd = effective_bandwidth(ub, row["t_dedup"])
        bs = effective_bandwidth(rb, row["t_slot"])
        uu = u_bar(U, n, k, n_shared)
        r = r_ratio(bd, bs)
        out.append(dict(row, u_bar=uu, beta_dedup=bd, beta_slot=bs, r=r,
                        criterion_dedup_faster=dedup_faster(uu, r),
                        measured_dedup_faster=row["t_dedup"] < row["t_slot"]))
    return out
