"""Full-size layers in the launch configuration bench.py times, checked
token by token against the oracle on every token of the pass (the oracle
splits the tokens over all host threads)."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import (THREADS, TOL, np_bytes, oracle_layer, rel_err, router_delta,
                           tie_margin, topk_within)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def full_pass_check(mv, cfg, n, n_max=64, seed=1):
    sample = list(range(n))
    layer = synth.make_layer(cfg, seed=seed, device="cuda")
    h_all = synth.make_hidden(cfg, n_max, seed=3, device="cuda")
    h = h_all[:n].contiguous()
    vl = mv.VerifyLayer(layer, n_max)
    y_dedup = vl.verify_pass(h, n, engine="dedup").float().cpu().numpy()
    assert vl.last_error() == 0
    ids_gpu = vl.ids_view(n).cpu().numpy().copy()
    U = int(vl.plan.n_uniq[0])
    ub = int(vl.plan.union_bytes[0])
    y_slot = vl.verify_pass(h, n, engine="perslot").float().cpu().numpy()
    assert vl.last_error() == 0
    cpu_layer = layer.to("cpu")
    del layer, vl
    torch.cuda.empty_cache()
    L = oracle_layer(cpu_layer)
    hb = np_bytes(h)
    ids, w, z, y_ref = oracle.verify(L, hb, tokens=sample, threads=THREADS)
    margin = tie_margin(cpu_layer, h.cpu()[sample], z, cfg.top_k)
    clear = margin > 1.0
    # a token whose oracle score gap exceeds the fp32 error bound delta is
    # routed exactly as the oracle routes it
    assert np.array_equal(ids_gpu[clear], ids[clear])
    # a near-tie token may take another top-k that fp32 rounding cannot tell
    # apart: it must be a top-k of the exact scores within 2 delta, and its
    # output is checked against the oracle on that same routing
    near = np.where(~clear)[0]
    assert near.size <= max(1, n // 8), f"{near.size} near-tie tokens of {n}"
    delta = router_delta(cpu_layer, h.cpu())
    for t in near:
        assert topk_within(z[t], ids_gpu[t], cfg.top_k, 2 * delta[t]), f"token {t}"
    if near.size:
        _, _, y_near = oracle.verify_routed(L, hb, ids_gpu[near], tokens=near.tolist(),
                                            threads=THREADS)
        y_ref = y_ref.copy()
        y_ref[near] = y_near
    assert rel_err(y_dedup[sample], y_ref) <= TOL[cfg.wtype]
    assert rel_err(y_slot[sample], y_ref) <= TOL[cfg.wtype]
    # and every token against its own scale
    for t in sample:
        assert rel_err(y_dedup[t], y_ref[t]) <= TOL[cfg.wtype], f"token {t}"
        assert rel_err(y_slot[t], y_ref[t]) <= TOL[cfg.wtype], f"token {t}"
    # union and byte count
    assert U == len(set(ids_gpu.ravel().tolist()))
    wb, sb = oracle.expert_bytes(cfg.d, cfg.inter, {synth.BF16: oracle.BF16,
                                                     synth.E4M3: oracle.E4M3}[cfg.wtype])
    assert ub == (U + cfg.n_shared) * (wb + sb)
    return U


def test_dsv3_fp8_n8_bench_workload(mv):
    # the bench's workload: n = 8 tokens of the 64-node tree, n_max = 64
    U = full_pass_check(mv, synth.DSV3, 8)
    assert 8 <= U <= 64


def test_dsv3_fp8_n64_tree(mv):
    full_pass_check(mv, synth.DSV3, 64)


def test_gptoss_bf16_n16_chain(mv):
    full_pass_check(mv, synth.GPTOSS, 16)


def test_qwen3_bf16_n61_tree(mv):
    full_pass_check(mv, synth.QWEN3, 61)
