"""A stack of MoE layers verified in one pass ("The Limits of Speculation",
Sec. 3.3, eq. (5)): every layer equals its own pass, the layer-averaged
union U_bar equals the oracle's, and the captured graph replays the stack."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import draft_length as D
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import THREADS, TOL, np_bytes, oracle_layer, rel_err, tie_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


CFG = synth.shrink(synth.DSV3, 640, 384, 32, "fp8-stack")
L_LAYERS, N_MAX = 4, 12


def stack_inputs(cfg, n_layers, n_max, seed):
    return torch.stack([synth.make_hidden(cfg, n_max, seed=seed + l) for l in range(n_layers)])


def test_stack_equals_layers_and_oracle_union(mv):
    layers = [synth.make_layer(CFG, seed=1 + 10 * l) for l in range(L_LAYERS)]
    st = mv.VerifyStack([mv.VerifyLayer(layer.to("cuda"), N_MAX) for layer in layers])
    hs = stack_inputs(CFG, L_LAYERS, N_MAX, 50)
    hs_d = hs.cuda()
    for n in (1, 5, 12):
        ys = [y.clone() for y in st.verify_pass(hs_d, n)]
        assert st.last_error() == 0
        unions = st.unions()
        u_ref = []
        for l, layer in enumerate(layers):
            # the same layer alone, in a fresh object: bitwise the same output
            vl = mv.VerifyLayer(layer.to("cuda"), N_MAX)
            assert torch.equal(vl.verify_pass(hs_d[l, :n], n), ys[l])
            L = oracle_layer(layer)
            ids, _, z, y_ref = oracle.verify(L, np_bytes(hs[l, :n]), threads=THREADS)
            assert (tie_margin(layer, hs[l, :n], z, CFG.top_k) > 1.0).all()
            assert rel_err(ys[l].float().cpu().numpy(), y_ref) <= TOL[CFG.wtype]
            u_ref.append(oracle.union_plan(ids, CFG.n_experts)[0])
        assert unions == u_ref
        assert D.layer_mean_union(unions) == np.mean(u_ref)
        if n == 1:
            assert unions == [CFG.top_k] * L_LAYERS


def test_stack_graph_replays_the_eager_pass(mv):
    st = mv.VerifyStack.synthetic(CFG, 3, N_MAX, seed=7)
    hs = stack_inputs(CFG, 3, N_MAX, 60).cuda()
    n = 9
    g = st.capture(hs, n)
    for seed in (61, 62):
        hs.copy_(stack_inputs(CFG, 3, N_MAX, seed))
        g.replay()
        y_graph = [vl.y[:n].clone() for vl in st.layers]
        u_graph = st.unions()
        y_eager = [y.clone() for y in st.verify_pass(hs, n)]
        assert st.last_error() == 0
        assert u_graph == st.unions()
        for a, b in zip(y_graph, y_eager):
            assert torch.equal(a, b)


def test_identical_tokens_give_u_bar_k(mv):
    st = mv.VerifyStack.synthetic(CFG, 3, N_MAX, seed=9)
    h = synth.make_hidden(CFG, N_MAX, seed=70, kind="identical")
    hs = torch.stack([h] * 3).cuda()
    st.verify_pass(hs, N_MAX)
    assert st.unions() == [CFG.top_k] * 3
