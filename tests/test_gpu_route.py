"""Routing on the GPU against the oracle: top-k ids bit-exact, gate weights
and fp32 logits within fp32 rounding."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import oracle_gate, oracle_layer, tie_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def _topk_gpu(mv, cfg, scores: torch.Tensor):
    n = scores.shape[0]
    desc = mv.make_desc(cfg, max(n, 1))
    s = scores.cuda().contiguous()
    ids = torch.empty(max(n, 1), cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(max(n, 1), cfg.top_k, dtype=torch.float32, device="cuda")
    mv.moe_topk_from_logits(desc, s, n, ids, w)
    torch.cuda.synchronize()
    return ids[:n].cpu().numpy(), w[:n].cpu().numpy()


CASES = [(16, 2), (64, 8), (128, 8), (128, 4), (256, 8), (256, 32), (33, 5), (1, 1)]


@pytest.mark.parametrize("E,k", CASES)
@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("gate", [synth.GATE_SOFTMAX, synth.GATE_SOFTMAX_RENORM,
                                  synth.GATE_SIGMOID_RENORM])
def test_topk_from_logits_bit_exact(mv, E, k, ties, gate):
    cfg = synth.LayerConfig("t", 256, E, k, 128, synth.BF16, synth.BF16, gate)
    n = 64
    scores = synth.random_scores(n, E, seed=E * 7 + k + ties, ties=ties)
    if ties and gate != synth.GATE_SOFTMAX_RENORM:
        # keep the gate finite: the huge levels only matter for ordering
        scores = scores.clamp(-30, 30)
    ids, w = _topk_gpu(mv, cfg, scores)
    ref_ids, ref_w = oracle.topk_from_scores(scores.numpy(), k, oracle_gate(cfg))
    assert np.array_equal(ids, ref_ids)
    finite = np.isfinite(ref_w)
    np.testing.assert_allclose(w[finite], ref_w[finite], rtol=2e-6, atol=1e-7)


def test_topk_from_logits_empty_batch(mv):
    cfg = synth.LayerConfig("t", 256, 16, 2, 128, synth.BF16, synth.BF16, synth.GATE_SOFTMAX)
    ids, w = _topk_gpu(mv, cfg, torch.zeros(0, 16))
    assert ids.shape == (0, 2)


ROUTE_CASES = [
    (synth.TINY, 4), (synth.OLMOE, 8), (synth.QWEN3, 64), (synth.GPTOSS, 16), (synth.DSV3, 64),
    (synth.DSV3, 1), (synth.OLMOE, 61),
]


@pytest.mark.parametrize("cfg,n", ROUTE_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_route_from_hidden_states(mv, cfg, n):
    # only the router matters here: a layer with tiny experts and the real router
    small = synth.shrink(cfg, cfg.d, 128 if cfg.wtype == synth.E4M3 else 64)
    layer = synth.make_layer(small, seed=11)
    h = synth.make_hidden(small, n, seed=13)
    desc = mv.make_desc(small, n)
    wg = layer.wg.cuda()
    hd = h.cuda()
    ids = torch.empty(n, cfg.top_k, dtype=torch.int32, device="cuda")
    w = torch.empty(n, cfg.top_k, dtype=torch.float32, device="cuda")
    logits = torch.empty(n, cfg.n_experts, dtype=torch.float32, device="cuda")
    mv.moe_route_topk(desc, wg, hd, n, ids, w, logits)
    torch.cuda.synchronize()
    L = oracle_layer(layer)
    hv = h.double().numpy()
    rz = np.stack([oracle.router_scores(L, hv[t]) for t in range(n)])
    rids = np.stack([oracle.topk(rz[t], cfg.top_k) for t in range(n)])
    rw = np.stack([oracle.gate(rz[t], rids[t], oracle_gate(cfg)) for t in range(n)])
    # logits: fp32 accumulation of exact products
    z = logits.cpu().numpy().astype(np.float64)
    scale = np.abs(rz).max()
    assert np.max(np.abs(z - rz)) <= 2e-5 * scale
    margin = tie_margin(layer, h, rz, cfg.top_k)
    clear = margin > 1.0
    assert clear.mean() >= 0.9, f"too many near-ties ({(~clear).sum()} of {n})"
    got = ids.cpu().numpy()
    assert np.array_equal(got[clear], rids[clear])
    # the GPU's own ids are exactly the top-k of its own logits
    own_ids, own_w = oracle.topk_from_scores(logits.cpu().numpy(), cfg.top_k, oracle_gate(cfg))
    assert np.array_equal(got, own_ids)
    np.testing.assert_allclose(w.cpu().numpy(), own_w, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(w.cpu().numpy()[clear], rw[clear], rtol=1e-4, atol=1e-6)
