"""The tcgen05 CTAs of the BF16 deduplicating engine against the oracle.

A segment of more than 8 tokens of a BF16 pass runs on tensor-memory CTAs
(the first W of the grid) while the rest run the mma.sync path.  These cases
aim at that split: the boundary (m = 8 stays narrow, m = 9 goes wide), a
shared expert as a wide segment (its rows of the activation buffer sit behind
the routed slots), a down projection with an odd number of 64-row blocks (the
last row pair holds one tile), plans that mix wide and narrow segments, and
the largest segment (64 tokens).  The oracle gets the GPU's routing, as in
the other expert tests.
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


def run(mv, cfg, n, kind=None, sigma=None):
    dev_layer, _, L = get_layer(cfg)
    h = synth.make_hidden(cfg, n, seed=5, kind=kind, sigma=sigma)
    ids, w, _, y_ref = oracle.verify(L, np_bytes(h), threads=THREADS)
    vl = mv.VerifyLayer(dev_layer, 64)
    vl.ids[:n * cfg.top_k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * cfg.top_k].copy_(torch.from_numpy(w.reshape(-1)).to(torch.float32))
    vl.union_plan(n)
    y = vl.dedup(h.cuda(), n)
    assert vl.last_error() == 0
    y = y.float().cpu().numpy().astype(np.float64)
    err = rel_err(y, y_ref)
    assert err <= TOL[cfg.wtype], f"{cfg.name} n={n}: rel err {err:.3g}"
    counts = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    return y, counts


@pytest.mark.parametrize("n", [8, 9, 16, 33, 64])
def test_identical_tokens_boundary(mv, n):
    # one segment of n tokens per chosen expert (and the shared expert's):
    # n = 8 runs on the mma.sync CTAs, n >= 9 on the tensor-memory CTAs
    y, counts = run(mv, SHARED, n, kind="identical")
    assert sorted(counts[counts > 0].tolist()) == [n] * SHARED.top_k
    assert np.array_equal(y[0], y[n - 1])


@pytest.mark.parametrize("n", [12, 24, 40, 64])
def test_shared_expert_tree(mv, n):
    # the shared expert's segment (n tokens) is always wide here; the routed
    # segments of a correlated tree are a mix of both kinds
    run(mv, SHARED, n)


@pytest.mark.parametrize("n,sigma", [(20, 0.3), (48, 0.3), (64, 0.05), (64, 1.0)])
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
