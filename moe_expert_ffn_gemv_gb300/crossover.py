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

import math
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


def consecutive_reuse(ids: Sequence[Sequence[int]]) -> List[float]:
    """Consecutive-token reuse of one window of routed tokens, in the pass's
    token order: entry n - 2 (n = 2 .. len(ids)) is the share of token n's
    experts that the n - 1 tokens before it already selected ("Speculative
    Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel Bandwidth
    and the Best Draft Length", Fig. 1, rho_l(n) of one layer).  The page
    prints no formula; this reading is the one whose mean under independent
    uniform routing is the figure's dotted line (uniform_reuse)."""
    seen = set()
    out = []
    for t, row in enumerate(ids):
        row = list(row)
        if t > 0:
            out.append(sum(1 for e in row if e in seen) / len(row))
        seen.update(row)
    return out


def uniform_reuse(n: int, k: int, n_experts: int) -> float:
    """Mean consecutive-token reuse under independent uniform routing:
    1 - q^(n-1) with q = 1 - k/N, the chance that a given expert is missing
    from one token's k of N (same figure, dotted line)."""
    return 1.0 - (1.0 - k / n_experts) ** (n - 1)


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


# ---------------------------------------------------------------------------
# Bandwidth-fit cost model ("Expert Bytes, Kernel Bandwidth and the Best Draft
# Length", abstract, Fig. 2, Tables 1-3): each kernel's time on one layer's
# expert operation is its requested bytes over an effective bandwidth that
# already includes the operation's fixed work (Table 1 note).  The bandwidths
# are fitted per pass size n on one set of routing windows (median over the
# windows, as Fig. 2 plots); the bytes of other windows over those bandwidths
# predict each kernel's time and the saving of deduplication.  The error
# bounds of Table 2 are checked for a relative bandwidth error eps.

def fit_bandwidths(windows: Iterable[Dict], k: int, expert_bytes: int, n_shared: int = 0) -> Dict:
    """windows: dicts with n, U, t_dedup, t_slot (seconds).  Returns, per n,
    beta_slot and beta_dedup (median over the windows of bytes / time) and
    eps: the largest relative deviation of a window's bandwidth from the fit."""
    import statistics
    by_n: Dict[int, List[Dict]] = {}
    for w in windows:
        by_n.setdefault(w["n"], []).append(w)
    model = {}
    for n, ws in sorted(by_n.items()):
        bs = [requested_bytes_perslot(n, k, expert_bytes, n_shared) / w["t_slot"] for w in ws]
        bd = [union_bytes(w["U"], expert_bytes, n_shared) / w["t_dedup"] for w in ws]
        b_slot, b_dedup = statistics.median(bs), statistics.median(bd)
        eps = max([abs(x / b_slot - 1) for x in bs] + [abs(x / b_dedup - 1) for x in bd])
        model[n] = dict(beta_slot=b_slot, beta_dedup=b_dedup, eps=eps)
    return model


def fit_reread_cost(windows: Iterable[Dict], k: int, n_shared: int = 0) -> Dict:
    """The per-slot engine's cost of re-reading an expert against a unique
    read (the page's c_re / c_u of its eq. (4), given only as a range per
    engine in Table 1).  The page does not print eq. (4); the reading taken
    here is the linear step time
        t_slot = t0 + c_u * (U + shared) + c_re * (n*(k + shared) - U - shared):
    each pass reads its union's experts once at c_u each, and every further
    read of an expert another slot already named costs c_re.  Fitted by least
    squares over windows (dicts with n, U, t_slot in seconds); returns t0,
    c_u, c_re (seconds per expert read), their ratio and the fit's residual
    RMS (seconds)."""
    import numpy as np
    rows = list(windows)
    A, y = [], []
    for w in rows:
        unique = w["U"] + n_shared
        reads = w["n"] * (k + n_shared)
        A.append([1.0, float(unique), float(reads - unique)])
        y.append(float(w["t_slot"]))
    A, y = np.array(A), np.array(y)
    coef, *_ = np.linalg.lstsq(A, y, rcond=None)
    t0, c_u, c_re = (float(c) for c in coef)
    rms = float(np.sqrt(np.mean((A @ coef - y) ** 2)))
    return dict(t0=t0, c_u=c_u, c_re=c_re, ratio=c_re / c_u, rms=rms, points=len(rows))


def predict(model: Dict, n: int, U: int, k: int, expert_bytes: int, n_shared: int = 0) -> Dict:
    """Predicted time of each kernel (its memory term M = bytes / bandwidth)
    and predicted saving S = tau_slot - tau_dedup for one pass of n tokens with
    union size U."""
    m = model[n]
    m_slot = requested_bytes_perslot(n, k, expert_bytes, n_shared) / m["beta_slot"]
    m_dedup = union_bytes(U, expert_bytes, n_shared) / m["beta_dedup"]
    return dict(tau_slot=m_slot, tau_dedup=m_dedup, saving=m_slot - m_dedup)


def bound_verify_time(M: float, eps: float) -> float:
    """Table 2, (17): |tau_hat - tau| <= eps/(1-eps) * M."""
    return eps / (1.0 - eps) * M


def bound_saving(M_slot: float, M_dedup: float, eps: float) -> float:
    """Table 2, (18): |S_hat - S| <= eps/(1-eps) * (M_slot + M_dedup)."""
    return eps / (1.0 - eps) * (M_slot + M_dedup)


def faster_kernel_is_certain(r: float, ubar: float, eps: float) -> bool:
    """Table 2, (19): the two sides of u_bar < r cannot swap under relative
    bandwidth errors up to eps when |ln r - ln u_bar| > ln((1+eps)/(1-eps))."""
    return abs(math.log(r) - math.log(ubar)) > math.log((1.0 + eps) / (1.0 - eps))


def evaluate(model: Dict, windows: Iterable[Dict], k: int, expert_bytes: int,
             n_shared: int = 0) -> List[Dict]:
    """Held-out windows against the fitted model: predicted and measured
    saving, the saving bound (18) for the fit's eps, whether the measured
    saving lies inside it, and whether the faster kernel was predicted."""
    out = []
    for w in windows:
        n, U = w["n"], w["U"]
        if n not in model:
            continue
        pr = predict(model, n, U, k, expert_bytes, n_shared)
        eps = model[n]["eps"]
        S = w["t_slot"] - w["t_dedup"]
        bnd = bound_saving(pr["tau_slot"], pr["tau_dedup"], eps) if eps < 1 else math.inf
        out.append(dict(n=n, U=U, saving=S, saving_hat=pr["saving"], bound=bnd,
                        inside=abs(pr["saving"] - S) <= bnd,
                        sign_ok=(pr["saving"] > 0) == (S > 0)))
    return out
