"""Degenerate routing through both expert engines and the whole pass, on the
GPU against the oracle.

  - one routed expert and top-1: every pass is a single segment holding all n
    tokens (up to 8 groups of 8 tokens at n = 64), and with one expert and
    k = 1 the layer is a dense SwiGLU MLP;
  - k = N: every token selects every expert, so U = N and every segment holds
    all n tokens.
The union plan must then be exactly: U = N, hist = n for every expert, and
each segment the slots t*k + j of its expert in ascending t.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import THREADS, TOL, np_bytes, oracle_layer, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    synth.LayerConfig("bf16-one-expert", 192, 1, 1, 64, synth.BF16, synth.BF16, synth.GATE_SOFTMAX,
                      hidden="chain", rho=0.5),
    synth.LayerConfig("fp8-one-expert-shared", 256, 1, 1, 128, synth.BF16, synth.E4M3,
                      synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="tree_ar", rho=0.6),
    synth.LayerConfig("bf16-k-equals-n", 192, 4, 4, 128, synth.BF16, synth.BF16,
                      synth.GATE_SOFTMAX_RENORM, hidden="chain", rho=0.0),
    synth.LayerConfig("fp8-k-equals-n-shared", 256, 3, 3, 128, synth.BF16, synth.E4M3,
                      synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="tree_ar", rho=0.6),
]


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


@pytest.mark.parametrize("n", [1, 9, 64])
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_degenerate_routing(mv, cfg, n):
    layer = synth.make_layer(cfg, seed=4, device="cpu")
    L = oracle_layer(layer)
    h = synth.make_hidden(cfg, n, seed=6)
    ids, w, _, y_ref = oracle.verify(L, np_bytes(h), threads=THREADS)
    N, k = cfg.n_experts, cfg.top_k
    assert all(sorted(row) == list(range(N)) for row in ids.tolist())   # every expert, every token

    dev = layer.to("cuda")
    vl = mv.VerifyLayer(dev, 64)
    hd = h.cuda()
    vl.ids[:n * k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * k].copy_(torch.from_numpy(w.reshape(-1)).to(torch.float32))
    vl.union_plan(n)
    torch.cuda.synchronize()
    assert int(vl.plan.n_uniq[0]) == N
    assert vl.plan.hist[:N].cpu().tolist() == [n] * N
    offs = vl.plan.offs[:N + 1].cpu().tolist()
    assert offs == [e * n for e in range(N + 1)]
    perm = vl.plan.perm[:n * k].cpu().numpy().reshape(N, n)
    for e in range(N):
        want = [t * k + int(np.nonzero(ids[t] == e)[0][0]) for t in range(n)]
        assert perm[e].tolist() == want

    for engine in ("dedup", "perslot"):
        y = (vl.dedup(hd, n) if engine == "dedup" else vl.perslot(hd, n)).float().cpu().numpy()
        assert vl.last_error() == mv.MOE_OK
        err = rel_err(y.astype(np.float64), y_ref)
        assert err <= TOL[cfg.wtype], f"{cfg.name} n={n} {engine}: rel err {err:.3g}"

    # the whole pass routes on the GPU: the same sets, the same outputs
    y = vl.verify_pass(hd, n).float().cpu().numpy()
    assert vl.last_error() == mv.MOE_OK
    assert int(vl.plan.n_uniq[0]) == N
    err = rel_err(y.astype(np.float64), y_ref)
    assert err <= TOL[cfg.wtype], f"{cfg.name} n={n} pass: rel err {err:.3g}"


LARGEST = [
    synth.LayerConfig("fp8-k32-shared", 256, 64, 32, 128, synth.BF16, synth.E4M3,
                      synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="tree_ar", rho=0.6),
    synth.LayerConfig("bf16-k32-shared", 256, 64, 32, 128, synth.BF16, synth.BF16,
                      synth.GATE_SOFTMAX_RENORM, n_shared=1, hidden="tree_add", sigma=0.3),
]


@pytest.mark.parametrize("cfg", LARGEST, ids=lambda c: c.name)
def test_largest_plan_the_abi_takes(mv, cfg):
    # n = 64 tokens, k = 32 (both at their limits) and a shared expert: 2048
    # routed slots and 64 shared ones, the most every table of the expert
    # kernels holds; with BF16 weights most segments (about 32 tokens each)
    # run on the tcgen05 CTAs, whose activation maps then span 2112 rows
    n = 64
    layer = synth.make_layer(cfg, seed=4, device="cpu")
    h = synth.make_hidden(cfg, n, seed=6)
    ids, w, _, y_ref = oracle.verify(oracle_layer(layer), np_bytes(h), threads=THREADS)
    dev = layer.to("cuda")
    vl = mv.VerifyLayer(dev, 64)
    hd = h.cuda()
    k = cfg.top_k
    vl.ids[:n * k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * k].copy_(torch.from_numpy(w.reshape(-1)).to(torch.float32))
    vl.union_plan(n)
    counts = np.bincount(ids.ravel(), minlength=cfg.n_experts)
    assert int(vl.plan.n_uniq[0]) == int((counts > 0).sum())
    for engine in ("dedup", "perslot"):
        y = (vl.dedup(hd, n) if engine == "dedup" else vl.perslot(hd, n)).float().cpu().numpy()
        assert vl.last_error() == mv.MOE_OK
        err = rel_err(y.astype(np.float64), y_ref)
        assert err <= TOL[cfg.wtype], f"{cfg.name} {engine}: rel err {err:.3g}"
