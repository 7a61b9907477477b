"""E4M3 layers whose activations leave fp16's range.

The E4M3 engines multiply on fp16 tensor cores.  Hidden states of magnitude
1e5 (beyond fp16's 65504) and 1e-6 (below its normal range), and weights
large enough that the intermediate silu(g) * u passes 65504, must still give
the oracle's output within the FP8 tolerance, token by token: each token's
row is checked against its own scale, so a token of tiny activations is not
hidden behind one of huge activations.  Full DeepSeek-V3 width and
intermediate size (d = 7168, I = 2048), a few experts, one shared expert.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import THREADS, TOL, np_bytes, oracle_layer, rel_err, tie_margin

pytestmark = pytest.mark.gpu

CFG = synth.LayerConfig("fp8-wide-range", 7168, 8, 2, 2048, synth.BF16, synth.E4M3,
                        synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="wide_range")
N = 8
WEIGHT_SCALE = 64.0  # multiplies every block scale: |w| of order 1


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


@pytest.fixture(scope="module")
def case():
    layer = synth.make_layer(CFG, seed=1, device="cuda")
    for t in (layer.s13, layer.s2, layer.sh_s13, layer.sh_s2):
        t.mul_(WEIGHT_SCALE)
    h = synth.make_hidden(CFG, N, seed=3, device="cuda")
    cpu = layer.to("cpu")
    ids, w, z, y_ref = oracle.verify(oracle_layer(cpu), np_bytes(h), threads=THREADS)
    return layer, h, cpu, ids, z, y_ref


def _dequant(codes, scales):
    w = codes.view(torch.float8_e4m3fn).to(torch.float64)
    R, C = w.shape
    return (w.view(R // 128, 128, C // 128, 128) * scales.to(torch.float64)[:, None, :, None]
            ).view(R, C)


def test_inputs_leave_fp16_range(case):
    layer, h, cpu, ids, z, y_ref = case
    hf = h.float().abs().cpu()
    assert float(hf.max()) > 65504.0
    assert 0.0 < float(hf[hf > 0].min()) < 2.0 ** -14
    # the shared expert's silu(g) * u on token 2 passes fp16's largest value
    w13 = _dequant(cpu.sh_w13, cpu.sh_s13)
    x = h[2].double().cpu()
    g, u = w13[:CFG.inter] @ x, w13[CFG.inter:] @ x
    a = g * torch.sigmoid(g) * u
    assert float(a.abs().max()) > 65504.0
    assert np.all(np.isfinite(y_ref))


def per_token_err(y, y_ref):
    return max(rel_err(y[t], y_ref[t]) for t in range(y_ref.shape[0]))


def check(y, case, ids_gpu):
    layer, h, cpu, ids, z, y_ref = case
    margin = tie_margin(cpu, h.cpu(), z, CFG.top_k)
    assert (margin > 1.0).all()
    assert np.array_equal(ids_gpu, ids)
    assert np.all(np.isfinite(y))
    err = per_token_err(y, y_ref)
    assert err <= TOL[synth.E4M3], f"per-token max rel err {err:.3g}"


def test_whole_pass(mv, case):
    layer, h = case[0], case[1]
    vl = mv.VerifyLayer(layer, N)
    y = vl.verify_pass(h, N).float().cpu().numpy()
    assert vl.last_error() == mv.MOE_OK
    check(y, case, vl.ids_view(N).cpu().numpy())


def test_dedup_call(mv, case):
    layer, h = case[0], case[1]
    vl = mv.VerifyLayer(layer, N)
    vl.route_plan(h, N)
    y = vl.dedup(h, N).float().cpu().numpy()
    assert vl.last_error() == mv.MOE_OK
    check(y, case, vl.ids_view(N).cpu().numpy())


def test_perslot(mv, case):
    layer, h = case[0], case[1]
    vl = mv.VerifyLayer(layer, N)
    y = vl.verify_pass(h, N, engine="perslot").float().cpu().numpy()
    assert vl.last_error() == mv.MOE_OK
    check(y, case, vl.ids_view(N).cpu().numpy())
