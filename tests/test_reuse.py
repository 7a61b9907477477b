"""Consecutive-token reuse rho(n) ("Speculative Decoding for Mixture-of-Experts
Models: Expert Bytes, Kernel Bandwidth and the Best Draft Length", Fig. 1):
a worked example, the degenerate windows, and the figure's closed form for
independent uniform routing, 1 - q^(n-1)."""
import math

import numpy as np

from moe_expert_ffn_gemv_gb300 import crossover as X
from moe_expert_ffn_gemv_gb300 import synth


def test_worked_example():
    # token 2 shares expert 1 with token 1; token 3 shares nothing; token 4's
    # experts 0 and 4 were both chosen before
    assert X.consecutive_reuse([[0, 1], [1, 2], [3, 4], [0, 4]]) == [0.5, 0.0, 1.0]
    assert X.consecutive_reuse([[5, 6, 7]]) == []


def test_identical_and_disjoint_windows():
    assert X.consecutive_reuse([[3, 1, 4, 9]] * 6) == [1.0] * 5
    assert X.consecutive_reuse([[4 * t + j for j in range(4)] for t in range(6)]) == [0.0] * 5


def test_mean_under_uniform_routing_is_the_dotted_line():
    n, k, N, W = 16, 8, 64, 600
    samples = np.array([X.consecutive_reuse(synth.uniform_ids(n, k, N, seed=100 + w).tolist())
                        for w in range(W)])
    for m in range(2, n + 1):
        col = samples[:, m - 2]
        se = col.std(ddof=1) / math.sqrt(W)
        expect = X.uniform_reuse(m, k, N)
        assert abs(col.mean() - expect) <= 4 * se + 1e-12, (m, col.mean(), expect)
    # the closed form's ends: nothing to reuse at n = 1, everything as n grows
    assert X.uniform_reuse(1, k, N) == 0.0
    assert X.uniform_reuse(200, k, N) > 0.999
    assert X.uniform_reuse(2, k, N) == k / N
