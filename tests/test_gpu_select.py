"""Pre-verification selection on the GPU against the oracle, bit for bit.

EVICT's utility-guided prefix ("Making Every Verified Token Count", Sec. 3)
and EcoSpec's cost-aware selection ("Less Experts, Faster Decoding",
Sec. 4.2) over batches of seeded synthetic draft trees.  Both sides decide
in double with the operations in the same order, so orders, arg-maxes,
prefix sums, utilities and expert buffers must be identical.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def random_tree(rng, K, kind):
    if kind == "bfs":
        return np.array(synth.tree_parents(K), dtype=np.int32)
    if kind == "chain":
        return np.arange(-1, K - 1, dtype=np.int32)
    par = [-1] + [int(rng.integers(0, v)) for v in range(1, K)]
    return np.array(par, dtype=np.int32)


def random_q(rng, K, kind):
    if kind == "uniform":
        return rng.uniform(0.0, 1.0, K).astype(np.float32)
    if kind == "ties":
        return np.full(K, 0.5, dtype=np.float32)
    if kind == "dyadic":
        return (rng.integers(0, 9, K) / 8.0).astype(np.float32)  # zeros and ones included
    # siblings share a Dirichlet draw, as draft probabilities of one parent's children do
    return np.clip(rng.dirichlet(np.ones(4), K)[:, 0] * 2, 0, 1).astype(np.float32)


EVICT_CASES = [(1, "rand", "uniform"), (2, "chain", "ties"), (7, "rand", "dyadic"),
               (61, "bfs", "dirichlet"), (64, "bfs", "uniform"), (64, "rand", "ties"),
               (100, "rand", "dyadic"), (256, "rand", "uniform"), (256, "chain", "dirichlet")]


@pytest.mark.parametrize("K,tree,qk", EVICT_CASES)
def test_evict_select_bit_exact(mv, K, tree, qk):
    rng = np.random.default_rng(1000 + K)
    T = 9
    par = np.stack([random_tree(rng, K, tree) for _ in range(T)])
    q = np.stack([random_q(rng, K, qk) for _ in range(T)])
    for cost_kind in ("linear", "flat", "affine_noise"):
        ks_ = np.arange(1, K + 1, dtype=np.float64)
        cost = {"linear": 2.0 * ks_, "flat": np.full(K, 5.0),
                "affine_noise": 40.0 + 1.5 * ks_ + rng.uniform(0, 3, K)}[cost_kind]
        cost = cost.astype(np.float32)
        k_star, order, exp_len, util = mv.evict_select(par, q, cost)
        torch.cuda.synchronize()
        for t in range(T):
            rk, rorder, rexp, rutil = oracle.evict_select(par[t], q[t], cost)
            assert int(k_star[t]) == rk, (cost_kind, t)
            assert np.array_equal(order[t].cpu().numpy(), rorder)
            assert np.array_equal(exp_len[t].cpu().numpy(), rexp)
            assert np.array_equal(util[t].cpu().numpy(), rutil)


def test_evict_malformed_tree_is_reported_and_others_unaffected(mv):
    rng = np.random.default_rng(5)
    K = 16
    par = np.stack([random_tree(rng, K, "rand") for _ in range(3)])
    q = rng.uniform(0, 1, (3, K)).astype(np.float32)
    par[1, 5] = 9  # a parent after its child
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    cost = np.arange(1, K + 1, dtype=np.float32)
    k_star, order, _, _ = mv.evict_select(par, q, cost, error_word=err)
    torch.cuda.synchronize()
    assert int(err[0]) == mv.MOE_ERR_DEVICE_INPUT
    assert int(k_star[1]) == 0 and bool((order[1] == -1).all())
    for t in (0, 2):
        assert int(k_star[t]) == oracle.evict_select(par[t], q[t], cost)[0]


def pack_bits(b):
    """[..., E] bool -> [..., ceil(E/32)] int32 words, bit e%32 of word e/32."""
    E = b.shape[-1]
    wpl = (E + 31) // 32
    pad = np.zeros(b.shape[:-1] + (wpl * 32,), dtype=np.uint64)
    pad[..., :E] = b
    words = (pad.reshape(b.shape[:-1] + (wpl, 32)) << np.arange(32, dtype=np.uint64)).sum(-1)
    return words.astype(np.uint32).view(np.int32)


def unpack_bits(w, E):
    u = np.asarray(w).view(np.uint32).astype(np.uint64)
    bits = (u[..., None] >> np.arange(32, dtype=np.uint64)) & 1
    return bits.reshape(u.shape[:-1] + (-1,))[..., :E].astype(bool)


ECO_CASES = [  # K, L, E, kp, gamma, eps, with_b0
    (1, 1, 64, 8, 1, 1e-6, False),
    (7, 1, 64, 8, 4, 1e-6, False),
    (16, 3, 100, 5, 6, 0.5, True),      # ragged last word
    (61, 1, 256, 8, 4, 1e-6, False),    # the 61-node tree, gamma = 4
    (64, 1, 256, 8, 16, 1e-6, True),
    (64, 1, 256, 8, 70, 1e-6, False),   # gamma > K: every node, in pick order
    (64, 61, 256, 8, 8, 1e-6, False),   # 61 layers: 125 KB of bitsets
    (200, 2, 128, 4, 12, 1e-3, True),
    (32, 2, 64, 3, 0, 1e-6, True),      # gamma = 0: only the buffer
]


@pytest.mark.parametrize("K,L,E,kp,gamma,eps,with_b0", ECO_CASES)
def test_ecospec_select_bit_exact(mv, K, L, E, kp, gamma, eps, with_b0):
    rng = np.random.default_rng(2000 + K * 7 + L)
    T = 5
    par = np.stack([random_tree(rng, K, "bfs" if t % 2 else "rand") for t in range(T)])
    q = np.stack([random_q(rng, K, "dyadic" if t == 3 else "dirichlet") for t in range(T)])
    # predicted sets: a few hot experts shared along branches, plus noise
    pred = rng.integers(0, E, (T, K, L, kp)).astype(np.int32)
    hot = rng.integers(0, E, (T, L, kp))
    for t in range(T):
        for v in range(1, K):
            if rng.random() < 0.5:
                pred[t, v] = pred[t, par[t, v]]
        pred[t, ::3] = hot[t]
    pred[0, 0, 0, 0] = -1        # ignored ids
    pred[0, min(1, K - 1), 0, 0] = E
    b0 = (rng.random((T, L, E)) < 0.1) if with_b0 else None
    sel, buf, usz = mv.ecospec_select(par, q, pred, E, gamma, eps,
                                      None if b0 is None else pack_bits(b0))
    torch.cuda.synchronize()
    for t in range(T):
        rsel, rbuf, rcnt = oracle.ecospec_select(par[t], q[t], pred[t], E, gamma, eps,
                                                 None if b0 is None else b0[t].astype(np.uint8))
        assert np.array_equal(sel[t].cpu().numpy(), rsel), t
        assert np.array_equal(unpack_bits(buf[t].cpu().numpy(), E), rbuf)
        assert int(usz[t]) == rcnt


def test_ecospec_malformed_tree_is_reported(mv):
    rng = np.random.default_rng(6)
    K, E = 12, 64
    par = np.stack([random_tree(rng, K, "rand") for _ in range(2)])
    par[0, 0] = 3  # the root must have no parent
    q = rng.uniform(0, 1, (2, K)).astype(np.float32)
    pred = rng.integers(0, E, (2, K, 1, 4)).astype(np.int32)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    sel, buf, usz = mv.ecospec_select(par, q, pred, E, 4, 1e-6, error_word=err)
    torch.cuda.synchronize()
    assert int(err[0]) == mv.MOE_ERR_DEVICE_INPUT
    assert int(usz[0]) == -1 and bool((sel[0] == -1).all())
    rsel, _, rcnt = oracle.ecospec_select(par[1], q[1], pred[1], E, 4, 1e-6)
    assert np.array_equal(sel[1].cpu().numpy(), rsel) and int(usz[1]) == rcnt


def test_ecospec_on_routed_expert_sets_shrinks_the_union(mv):
    # predicted sets = the layer's own top-k routing of the tree's hidden
    # states (a perfect predictor), computed by the oracle.  EcoSpec's
    # selection must match the oracle; its union is never larger than that
    # of the confidence-only choice of the same size at gamma = 1 and is
    # reported for the others
    cfg = synth.shrink(synth.DSV3, 1024, 128, 256, "dsv3-router")
    layer = synth.make_layer(cfg, seed=3)
    from tests.helpers import oracle_layer
    K = 61
    h = synth.make_hidden(cfg, K, seed=4)
    L = oracle_layer(layer)
    ids = np.stack([oracle.topk(oracle.router_scores(L, h[t].float().numpy()), cfg.top_k)
                    for t in range(K)]).astype(np.int32)
    par = np.array(synth.tree_parents(K), dtype=np.int32)[None]
    rng = np.random.default_rng(7)
    q = random_q(rng, K, "dirichlet")[None]
    pred = ids[None, :, None, :]
    for gamma in (1, 4, 8, 16):
        sel, _, usz = mv.ecospec_select(par, q, pred, cfg.n_experts, gamma, 1e-6)
        rsel, _, rcnt = oracle.ecospec_select(par[0], q[0], pred[0], cfg.n_experts, gamma, 1e-6)
        assert np.array_equal(sel[0].cpu().numpy(), rsel) and int(usz[0]) == rcnt
        conf = oracle.evict_select(par[0], q[0], np.ones(K))[1][:gamma]
        u_conf = len(set(ids[conf].ravel().tolist()))
        assert rcnt == len(set(ids[rsel].ravel().tolist()))
        if gamma == 1:
            assert rcnt == u_conf
