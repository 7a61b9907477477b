"""Host-side model of a speculative step built from measured pass times: the
best draft length under geometric acceptance and the speedup it buys.

"Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
Bandwidth and the Best Draft Length" (abstract; appendix symbol table;
Table 2, rows (20)-(21)):
  - V(k) is the time of one step that verifies k drafts (k + 1 positions);
  - under geometric acceptance with rate a, a step commits
    E[G](k) = 1 + a + ... + a^k tokens on average (the drafts are accepted
    one after another until the first rejection, and the target always
    adds one token of its own);
  - the throughput is T_a(k) = E[G](k) / V(k), and the best draft length
    k*(a) is its arg-max: a staircase that never steps down as a grows;
  - a0 = V(1)/V(0) - 1 is the acceptance above which one draft beats none;
  - with every V off by a relative error of at most delta, the predicted
    best length loses at most 2 delta / (1 + delta) of the throughput (20),
    and the predicted best speedup is within a factor (1 +- delta)/(1 -+ delta)
    of the true one (21).
"The Limits of Speculation" (Sec. 3):
  - the MoESD speedup (eq. (2)): E[G] / (K T_D / T_T(0) + 1/eta(K)) with
    eta(K) = T_T(0) / T_T(K) (eq. (1)), T_T(K) the target model's pass time
    for K drafts and T_D the draft cost of one position;
  - U_bar_r, the number of distinct experts of the pass averaged over the
    MoE layers (eq. (5));
  - the cost model T_T = beta0(m) + alpha(m) U_bar, fitted for each
    microbatch size m = K + 1 (eq. (4); the context term c L_ctx is left
    out, since this path has no attention).
Readings: V(k) = T_T(k) + k T_D (the step is the draft's k positions and the
target's pass), which makes T_a(k)/T_a(0) equal the MoESD speedup; ties in
an arg-max go to the smaller k.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Sequence, Tuple


def expected_tokens(a: float, k: int) -> float:
    """E[G](k) = sum_{i=0..k} a^i under geometric acceptance."""
    if a == 1.0:
        return float(k + 1)
    return (1.0 - a ** (k + 1)) / (1.0 - a)


def step_time(t_target: Sequence[float], t_draft: float = 0.0) -> List[float]:
    """V(k) = T_T(k) + k T_D for k = 0..len(t_target)-1."""
    return [t + k * t_draft for k, t in enumerate(t_target)]


def throughput(a: float, V: Sequence[float], k: int) -> float:
    return expected_tokens(a, k) / V[k]


def best_draft_length(a: float, V: Sequence[float]) -> int:
    """k*(a): the k in 0..len(V)-1 of largest throughput, the smallest on a tie."""
    best, bt = 0, throughput(a, V, 0)
    for k in range(1, len(V)):
        t = throughput(a, V, k)
        if t > bt:
            best, bt = k, t
    return best


def a0(V: Sequence[float]) -> float:
    """The acceptance above which one draft is faster than none."""
    return V[1] / V[0] - 1.0


def speedup(a: float, V: Sequence[float], k: int) -> float:
    """T_a(k) / T_a(0): the step's speedup over plain decoding."""
    return throughput(a, V, k) / throughput(a, V, 0)


def moesd_speedup(eg: float, K: int, t_draft: float, t_target: Sequence[float]) -> float:
    """"The Limits of Speculation", eq. (2): E[G] / (K T_D/T_T(0) + 1/eta(K))."""
    eta = t_target[0] / t_target[K]
    return eg / (K * t_draft / t_target[0] + 1.0 / eta)


def staircase(V: Sequence[float], tol: float = 1e-12) -> List[Tuple[float, int]]:
    """The step points of k*(a) on [0, 1): a list of (a_j, k*(a) just above
    a_j), starting with (0.0, k*(0)).  A grid of 4096 points is scanned; each
    change is located by bisection to `tol`, and the scan restarts from the
    located point, so that several steps inside one grid cell are all found
    (k* never steps down, so k* equals the current value up to the next
    step)."""
    a_lo, k_lo = 0.0, best_draft_length(0.0, V)
    out = [(a_lo, k_lo)]
    for i in range(1, 4096):
        a = i / 4096
        while best_draft_length(a, V) != k_lo:
            lo, hi = a_lo, a
            while hi - lo > tol:
                mid = 0.5 * (lo + hi)
                if best_draft_length(mid, V) == k_lo:
                    lo = mid
                else:
                    hi = mid
            a_lo, k_lo = hi, best_draft_length(hi, V)
            out.append((a_lo, k_lo))
        a_lo = a
    return out


def bound_best_length(delta: float) -> float:
    """Table 2, (20): T_a(k_hat*) >= (1 - delta)/(1 + delta) T_a(k*)."""
    return (1.0 - delta) / (1.0 + delta)


def best_length_is_certain(a: float, V: Sequence[float], delta: float) -> bool:
    """Table 2, (20): k_hat* = k* if (1+delta)/(1-delta) T_a(i) < T_a(k*) for
    every i != k*."""
    ks = best_draft_length(a, V)
    tk = throughput(a, V, ks)
    f = (1.0 + delta) / (1.0 - delta)
    return all(f * throughput(a, V, i) < tk for i in range(len(V)) if i != ks)


def bound_best_speedup(delta: float) -> Tuple[float, float]:
    """Table 2, (21): the predicted best speedup over the true one lies in
    [(1 - delta)/(1 + delta), (1 + delta)/(1 - delta)]."""
    return (1.0 - delta) / (1.0 + delta), (1.0 + delta) / (1.0 - delta)


def layer_mean_union(unions: Iterable[int]) -> float:
    """"The Limits of Speculation", eq. (5): distinct experts of the pass,
    counted in each MoE layer and averaged over the layers."""
    u = list(unions)
    return sum(u) / len(u)


def fit_cost_model(rounds: Iterable[Dict]) -> Dict[int, Dict[str, float]]:
    """"The Limits of Speculation", eq. (4) without the context term: for
    each microbatch size m, least squares of T = beta0 + alpha U_bar over the
    rounds of that m.  rounds: dicts with m, u_bar, t.  Returns per m:
    alpha, beta0, r2 (1 when the fit is exact; alpha = 0 and r2 = nan when
    every round of that m has the same U_bar), rounds."""
    by_m: Dict[int, List[Tuple[float, float]]] = {}
    for r in rounds:
        by_m.setdefault(int(r["m"]), []).append((float(r["u_bar"]), float(r["t"])))
    out = {}
    for m, pts in sorted(by_m.items()):
        n = len(pts)
        mx = sum(x for x, _ in pts) / n
        my = sum(y for _, y in pts) / n
        sxx = sum((x - mx) ** 2 for x, _ in pts)
        sxy = sum((x - mx) * (y - my) for x, y in pts)
        syy = sum((y - my) ** 2 for _, y in pts)
        alpha = sxy / sxx if sxx > 0 else 0.0
        beta0 = my - alpha * mx
        if sxx > 0 and syy > 0:
            r2 = 1.0 - sum((y - beta0 - alpha * x) ** 2 for x, y in pts) / syy
        elif sxx > 0:
            r2 = 1.0
        else:
            r2 = math.nan
        out[m] = {"alpha": alpha, "beta0": beta0, "r2": r2, "rounds": n}
    return out
