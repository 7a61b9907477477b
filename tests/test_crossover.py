"""The dedup-vs-per-slot criterion and crossover, against the numbers the
pages print (tests/golden/expertbytes_table1.txt) and closed cases."""
import os

from moe_expert_ffn_gemv_gb300 import crossover as X

GOLD = os.path.join(os.path.dirname(__file__), "golden", "expertbytes_table1.txt")


def rows():
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        yield f[0], f[1], [float(x) for x in f[2:]]


def test_r_is_the_bandwidth_ratio_to_printed_precision():
    for eng, model, v in rows():
        bs2, bd2, r2, u2, bs8, bd8, r8, u8 = v
        assert abs(X.r_ratio(bd2, bs2) - r2) <= 0.006, (eng, model, 2)
        assert abs(X.r_ratio(bd8, bs8) - r8) <= 0.006, (eng, model, 8)


def test_criterion_reproduces_which_kernel_the_table_says_is_faster():
    # abstract: deduplication is faster only from 5 to 8 tokens per pass, or
    # never -> at n = 2 the per-slot kernel wins on every row
    for eng, model, v in rows():
        bs2, bd2, r2, u2, bs8, bd8, r8, u8 = v
        assert not X.dedup_faster(u2, r2), (eng, model)
    faster8 = {(e, m): X.dedup_faster(v[7], v[6]) for e, m, v in rows()}
    assert faster8[("llama.cpp-CUDA", "OLMoE")] and faster8[("llama.cpp-CUDA", "gpt-oss")]
    assert not faster8[("llama.cpp-CUDA", "DeepSeek-V2-Lite")]
    assert not faster8[("llama.cpp-Metal", "Qwen3")]


def test_criterion_equals_timing_comparison():
    # u_bar < r  <=>  t_dedup < t_slot, for any positive bytes and times
    k, b = 8, 1000
    for n, U, td, ts in [(2, 15, 1.0, 1.2), (8, 39, 3.0, 2.9), (1, 8, 1.0, 1.0), (64, 173, 2.0, 9.0)]:
        a = X.analyse([dict(n=n, U=U, t_dedup=td, t_slot=ts)], k, b)[0]
        assert a["criterion_dedup_faster"] == a["measured_dedup_faster"]


def test_u_bar_bounds_and_shared_expert():
    # 1/n <= U/(nm) <= 1 ("Expert Bytes ...", Fig. 3)
    assert X.u_bar(8, 8, 8) == 1 / 8 and X.u_bar(64, 8, 8) == 1.0
    assert X.u_bar(39, 8, 8, n_shared=1) == 40 / 72
    assert X.crossover([1, 2, 3], [5, 4, 2], [5, 4.5, 3]) == 2
    assert X.crossover([1, 2], [5, 6], [4, 5]) is None


# ------------------------------------------------ cost model and Table 2 bounds
import math

import numpy as np


def test_bound_17_holds_for_any_bandwidth_error_within_eps():
    # tau = B / beta; an estimate beta_hat = beta (1 + e), |e| <= eps, predicts
    # tau_hat = B / beta_hat: |tau_hat - tau| <= eps/(1-eps) * tau
    rng = np.random.default_rng(1)
    for _ in range(2000):
        B = rng.uniform(1e6, 1e10)
        beta = rng.uniform(1e10, 1e13)
        eps = rng.uniform(0.0, 0.5)
        e = rng.uniform(-eps, eps)
        tau, tau_hat = B / beta, B / (beta * (1 + e))
        assert abs(tau_hat - tau) <= X.bound_verify_time(tau, eps) * (1 + 1e-12)
    # and the bound is reached at e = -eps
    B, beta, eps = 1e9, 5e12, 0.1
    tau, tau_hat = B / beta, B / (beta * (1 - eps))
    assert math.isclose(abs(tau_hat - tau), X.bound_verify_time(tau, eps), rel_tol=1e-12)


def test_bound_18_and_19_hold_for_any_bandwidth_errors_within_eps():
    rng = np.random.default_rng(2)
    for _ in range(2000):
        Bs, Bd = rng.uniform(1e8, 1e10, size=2)
        bs, bd = rng.uniform(1e11, 1e13, size=2)
        eps = rng.uniform(0.0, 0.4)
        es, ed = rng.uniform(-eps, eps, size=2)
        S = Bs / bs - Bd / bd
        S_hat = Bs / (bs * (1 + es)) - Bd / (bd * (1 + ed))
        assert abs(S_hat - S) <= X.bound_saving(Bs / bs, Bd / bd, eps) * (1 + 1e-12)
        # (19): r = bd/bs, u_bar = Bd/Bs; dedup faster <=> u_bar < r
        r, ub = bd / bs, Bd / Bs
        r_hat = bd * (1 + ed) / (bs * (1 + es))
        if X.faster_kernel_is_certain(r, ub, eps):
            assert (ub < r) == (ub < r_hat)


def test_fit_predict_evaluate_recovers_a_known_model():
    # windows generated from exact bandwidths: the fit recovers them, eps is 0,
    # predictions are exact and every point lies inside the (zero) bound
    k, b, sh = 8, 44_050_944, 1
    bslot = {2: 5.0e12, 8: 6.0e12}
    bded = {2: 4.5e12, 8: 5.8e12}
    wins = []
    for n in (2, 8):
        for U in (n * 3, n * 4, n * 5):
            wins.append(dict(n=n, U=U, t_slot=X.requested_bytes_perslot(n, k, b, sh) / bslot[n],
                             t_dedup=X.union_bytes(U, b, sh) / bded[n]))
    model = X.fit_bandwidths(wins, k, b, sh)
    for n in (2, 8):
        assert math.isclose(model[n]["beta_slot"], bslot[n], rel_tol=1e-12)
        assert math.isclose(model[n]["beta_dedup"], bded[n], rel_tol=1e-12)
        assert model[n]["eps"] < 1e-12
    ev = X.evaluate(model, wins, k, b, sh)
    assert all(e["inside"] and e["sign_ok"] for e in ev)
    assert all(abs(e["saving"] - e["saving_hat"]) < 1e-15 for e in ev)


# ------------------------------------------- re-read cost (eq. (4) reading)
def test_reread_fit_recovers_known_costs_and_the_no_cache_case():
    rng = np.random.default_rng(3)
    k, sh = 8, 1
    t0, c_u, c_re = 4e-6, 6.3e-6, 2.1e-6
    rows = []
    for n in range(1, 13):
        for _ in range(6):
            U = int(rng.integers(k, min(256, n * k) + 1))
            t = t0 + c_u * (U + sh) + c_re * (n * (k + sh) - U - sh)
            rows.append(dict(n=n, U=U, t_slot=t))
    f = X.fit_reread_cost(rows, k, sh)
    assert abs(f["c_u"] - c_u) < 1e-12 and abs(f["c_re"] - c_re) < 1e-12
    assert abs(f["t0"] - t0) < 1e-12 and abs(f["ratio"] - 1 / 3) < 1e-9 and f["rms"] < 1e-15
    # a per-slot engine with no cache benefit: time grows with the reads alone,
    # whether or not another slot named the expert -> c_re / c_u = 1
    flat = [dict(n=r["n"], U=r["U"], t_slot=t0 + c_u * r["n"] * (k + sh)) for r in rows]
    assert abs(X.fit_reread_cost(flat, k, sh)["ratio"] - 1) < 1e-9
    # noise of 1% moves the ratio only a little
    noisy = [dict(r, t_slot=r["t_slot"] * (1 + 0.01 * rng.standard_normal())) for r in rows]
    assert abs(X.fit_reread_cost(noisy, k, sh)["ratio"] - 1 / 3) < 0.1
