"""The step-time model and best draft length (host), pinned against closed
forms and the properties the pages state.

"Speculative Decoding for MoE Models: Expert Bytes, ..." (abstract; symbol
table; Table 2 rows (20)-(21)); "The Limits of Speculation", Sec. 3,
eqs. (1), (2), (4), (5).
"""
import math
import random

import numpy as np
import pytest

from moe_expert_ffn_gemv_gb300 import draft_length as D


def test_expected_tokens_geometric():
    for a in (0.0, 0.3, 0.8, 0.999):
        for k in range(0, 12):
            assert math.isclose(D.expected_tokens(a, k), sum(a ** i for i in range(k + 1)),
                                rel_tol=1e-12)
    assert D.expected_tokens(1.0, 7) == 8.0
    assert D.expected_tokens(0.0, 5) == 1.0


def test_a0_is_where_one_draft_starts_to_win():
    V = [100.0, 125.0, 160.0, 210.0]
    assert math.isclose(D.a0(V), 0.25)
    assert D.throughput(0.2499, V, 1) < D.throughput(0.2499, V, 0)
    assert D.throughput(0.2501, V, 1) > D.throughput(0.2501, V, 0)


def test_flat_and_proportional_step_times():
    # a step that costs the same for any k: more drafts are always better
    # (a > 0); a step time proportional to k + 1: never better than none
    V = [50.0] * 9
    for a in (0.01, 0.5, 0.99):
        assert D.best_draft_length(a, V) == 8
    V = [50.0 * (k + 1) for k in range(9)]
    for a in (0.0, 0.5, 0.99):
        assert D.best_draft_length(a, V) == 0


def test_staircase_never_steps_down_and_step_points_are_ties():
    # the abstract: the best draft length is a monotone staircase in a
    rng = random.Random(3)
    for trial in range(40):
        K = rng.randint(2, 12)
        V = [1.0]
        for k in range(1, K + 1):
            V.append(V[-1] + rng.uniform(0.0, 0.6))
        steps = D.staircase(V)
        ks = [k for _, k in steps]
        assert ks == sorted(ks) and len(set(ks)) == len(ks)
        for a in np.linspace(0, 0.999, 200):
            k = D.best_draft_length(a, V)
            below = [kk for aa, kk in steps if aa <= a]
            assert k == below[-1] or abs(a - next(aa for aa, kk in steps if kk == k)) < 1e-9
        for a_j, k_j in steps[1:]:
            prev = [kk for aa, kk in steps if aa < a_j][-1]
            # at a step point the two lengths have equal throughput
            assert math.isclose(D.throughput(a_j, V, prev), D.throughput(a_j, V, k_j),
                                rel_tol=1e-9)
    # one draft: the single step is a0
    V = [100.0, 130.0]
    steps = D.staircase(V)
    assert steps[0] == (0.0, 0) and len(steps) == 2 and math.isclose(steps[1][0], D.a0(V))


def test_bound_20_and_21_under_step_time_error():
    # Table 2: V_hat within relative delta of V for every k
    rng = random.Random(5)
    for trial in range(300):
        K = rng.randint(1, 10)
        V = [1.0]
        for k in range(1, K + 1):
            V.append(V[-1] + rng.uniform(0.01, 0.5))
        delta = rng.choice([0.01, 0.05, 0.1, 0.2])
        Vh = [v * (1 + rng.uniform(-delta, delta)) for v in V]
        a = rng.uniform(0, 0.99)
        ks, kh = D.best_draft_length(a, V), D.best_draft_length(a, Vh)
        assert D.throughput(a, V, kh) >= D.bound_best_length(delta) * D.throughput(a, V, ks) * (1 - 1e-12)
        if D.best_length_is_certain(a, V, delta):
            assert kh == ks
        lo, hi = D.bound_best_speedup(delta)
        ratio = D.speedup(a, Vh, kh) / D.speedup(a, V, ks)
        assert lo * (1 - 1e-12) <= ratio <= hi * (1 + 1e-12)


def test_moesd_speedup_equals_the_step_model():
    # "The Limits of Speculation", eq. (2) with eta = T_T(0)/T_T(K), and the
    # step V(k) = T_T(k) + k T_D: the same number
    t_target = [300.0, 340.0, 390.0, 450.0, 520.0]
    for t_draft in (0.0, 12.5, 40.0):
        V = D.step_time(t_target, t_draft)
        for a in (0.3, 0.7, 0.9):
            for K in range(5):
                eg = D.expected_tokens(a, K)
                assert math.isclose(D.speedup(a, V, K), D.moesd_speedup(eg, K, t_draft, t_target),
                                    rel_tol=1e-12)


def test_layer_mean_union_and_cost_model_fit():
    assert D.layer_mean_union([8, 10, 12, 14]) == 11.0
    # exact linear data per m recovers alpha and beta0 with R^2 = 1
    rng = np.random.default_rng(7)
    rounds = []
    truth = {2: (3.0, 100.0), 5: (4.5, 120.0)}
    for m, (al, b0) in truth.items():
        for u in rng.uniform(10, 40, 20):
            rounds.append({"m": m, "u_bar": u, "t": b0 + al * u})
    fit = D.fit_cost_model(rounds)
    for m, (al, b0) in truth.items():
        assert math.isclose(fit[m]["alpha"], al, rel_tol=1e-9)
        assert math.isclose(fit[m]["beta0"], b0, rel_tol=1e-9)
        assert math.isclose(fit[m]["r2"], 1.0, rel_tol=1e-12) and fit[m]["rounds"] == 20
    # noise lowers R^2 below 1 but keeps the slope near the truth
    noisy = [dict(r, t=r["t"] + rng.normal(0, 2.0)) for r in rounds]
    fit = D.fit_cost_model(noisy)
    assert 0.5 < fit[2]["r2"] < 1.0 and abs(fit[2]["alpha"] - 3.0) < 0.5
