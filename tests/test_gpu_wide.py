"""The tcgen05 CTAs of the BF16 deduplicating engine against the oracle.

A BF16 pass of 25 tokens or more runs its segments of more than 8 tokens on
tensor-memory CTAs (the first W of the grid) while the rest run the mma.sync
path; smaller passes run the mma.sync path alone.  These cases aim at that
split: the segment-size boundary inside such a pass (8 tokens stay on the
mma.sync CTAs, 9 go to the tcgen05 ones), the pass-size boundary (24 and 25
tokens), a shared expert as a wide segment (its rows of the activation
buffer sit behind the routed slots), a down projection with an odd number
of 64-row blocks (the last row pair holds one tile), plans that mix wide and
narrow segments, and the largest segment (64 tokens).  The oracle gets the
GPU's routing (or the given one), as in the other expert tests.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import THREADS, TOL, np_bytes, oracle_layer, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


# d = 704: 11 row blocks in the down projection (odd), 11 columns of K of
# 64 elements; I = 192: 6 gate/up row blocks, 3 row pairs
SHARED = synth.LayerConfig("bf16-shared-d704-i192", 704, 12, 3, 192, synth.BF16, synth.BF16,
                           synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="tree_add", sigma=0.3)
PLAIN = synth.LayerConfig("bf16-d1024-i256", 1024, 16, 4, 256, synth.BF16, synth.BF16,
                          synth.GATE_SOFTMAX_RENORM, hidden="tree_add", sigma=0.3)

_LAYERS = {}


def get_layer(cfg):
    if cfg not in _LAYERS:
        _LAYERS.clear()
        cpu_layer = synth.make_layer(cfg, seed=1)
        _LAYERS[cfg] = (cpu_layer.to("cuda"), cpu_layer, oracle_layer(cpu_layer))
    return _LAYERS[cfg]


def run_routed(mv, cfg, h, ids, w, y_ref):
    dev_layer, _, _ = get_layer(cfg)
    n = h.shape[0]
    vl = mv.VerifyLayer(dev_layer, 64)
    vl.ids[:n * cfg.top_k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * cfg.top_k].copy_(torch.from_numpy(np.asarray(w).reshape(-1)).to(torch.float32))
    vl.union_plan(n)
    y = vl.dedup(h.cuda(), n)
    assert vl.last_error() == 0
    y = y.float().cpu().numpy().astype(np.float64)
    err = rel_err(y, y_ref)
    assert err <= TOL[cfg.wtype], f"{cfg.name} n={n}: rel err {err:.3g}"
    return y


def run(mv, cfg, n, kind=None, sigma=None):
    _, _, L = get_layer(cfg)
    h = synth.make_hidden(cfg, n, seed=5, kind=kind, sigma=sigma)
    ids, w, _, y_ref = oracle.verify(L, np_bytes(h), threads=THREADS)
    y = run_routed(mv, cfg, h, ids, w, y_ref)
    return y, np.bincount(ids.ravel(), minlength=cfg.n_experts)


def given_routing(n, k, n_experts, counts):
    """ids [n][k]: expert e on counts[e] tokens (sum = n*k), k distinct
    experts a token; each expert goes to the tokens with the fewest experts
    so far (lowest index first)."""
    assert sum(counts) == n * k and len(counts) == n_experts
    rows = [[] for _ in range(n)]
    for e in sorted(range(n_experts), key=lambda e: -counts[e]):
        order = sorted(range(n), key=lambda t: (len(rows[t]), t))
        picked = [t for t in order if len(rows[t]) < k][:counts[e]]
        assert len(picked) == counts[e]
        for t in picked:
            rows[t].append(e)
    assert all(len(r) == k for r in rows)
    return np.asarray(rows, dtype=np.int32)


def test_segment_size_boundary_inside_a_tcgen05_pass(mv):
    # 32 tokens, given routing: segments of 1, 2, 8 and 9, 16 and 17, and 24
    # tokens in one pass, so that 8 stays on the mma.sync CTAs and 9 goes to
    # the tcgen05 ones
    cfg, n = PLAIN, 32
    counts = [9, 8, 17, 16, 24, 1, 2, 12, 12, 8, 6, 5, 4, 2, 1, 1]
    ids = given_routing(n, cfg.top_k, cfg.n_experts, counts)
    assert np.array_equal(np.bincount(ids.ravel(), minlength=cfg.n_experts), counts)
    _, _, L = get_layer(cfg)
    h = synth.make_hidden(cfg, n, seed=7)
    w, _, y_ref = oracle.verify_routed(L, np_bytes(h), ids, threads=THREADS)
    run_routed(mv, cfg, h, ids, w, y_ref)


def test_down_projection_box_boundaries(mv):
    # 64 tokens, given routing: segments of 64, 49, 48, 33, 32 and 17 tokens,
    # each at or just past the edge of a 16/32/48/64-row activation box of
    # the down projection, beside narrow segments of 8 and 5
    cfg, n = PLAIN, 64
    counts = [64, 49, 48, 33, 32, 17, 8, 5] + [0] * 8
    ids = given_routing(n, cfg.top_k, cfg.n_experts, counts)
    assert np.array_equal(np.bincount(ids.ravel(), minlength=cfg.n_experts), counts)
    _, _, L = get_layer(cfg)
    h = synth.make_hidden(cfg, n, seed=8)
    w, _, y_ref = oracle.verify_routed(L, np_bytes(h), ids, threads=THREADS)
    run_routed(mv, cfg, h, ids, w, y_ref)


@pytest.mark.parametrize("n", [24, 25, 33, 64])
def test_identical_tokens(mv, n):
    # one segment of n tokens per chosen expert (and the shared expert's):
    # n = 24 runs on the mma.sync CTAs alone, n >= 25 on the tcgen05 ones
    y, counts = run(mv, SHARED, n, kind="identical")
    assert sorted(counts[counts > 0].tolist()) == [n] * SHARED.top_k
    assert np.array_equal(y[0], y[n - 1])


@pytest.mark.parametrize("n", [25, 40, 64])
def test_shared_expert_tree(mv, n):
    # the shared expert's segment (n tokens) is always wide here; the routed
    # segments of a correlated tree are a mix of both kinds
    run(mv, SHARED, n)


@pytest.mark.parametrize("n,sigma", [(28, 0.3), (48, 0.3), (64, 0.05), (64, 1.0)])
def test_mixed_segments(mv, n, sigma):
    _, counts = run(mv, PLAIN, n, sigma=sigma)
    if sigma <= 0.3:
        assert (counts > 8).any()


def test_repeat_is_bitwise_stable(mv):
    # the split of the grid and the accumulation order depend only on the
    # plan: the same pass twice gives the same bytes
    dev_layer, _, _ = get_layer(PLAIN)
    h = synth.make_hidden(PLAIN, 48, seed=6).cuda()
    vl = mv.VerifyLayer(dev_layer, 64)
    vl.route_plan(h, 48)
    y1 = vl.dedup(h, 48).clone()
    y2 = vl.dedup(h, 48).clone()
    assert vl.last_error() == 0
    assert torch.equal(y1, y2)


def test_pass_with_tcgen05_ctas_replays_from_a_cuda_graph(mv):
    # the tensor maps of the activation boxes are kernel parameters, recorded
    # with the graph: replays on new hidden states (written into the same
    # buffer) must match the eager pass bit for bit
    dev_layer, _, _ = get_layer(PLAIN)
    n = 48
    vl = mv.VerifyLayer(dev_layer, 64)
    h = torch.empty(n, PLAIN.d, dtype=torch.bfloat16, device="cuda")
    h.copy_(synth.make_hidden(PLAIN, n, seed=11))
    g = vl.capture_pass(h, n)
    for seed in (12, 13):
        h.copy_(synth.make_hidden(PLAIN, n, seed=seed))
        g.replay()
        y_graph = vl.y[:n].clone()
        y_eager = vl.verify_pass(h, n).clone()
        assert vl.last_error() == 0
        assert torch.equal(y_graph, y_eager)
