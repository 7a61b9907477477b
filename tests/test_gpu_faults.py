"""Failure handling on the GPU, without faulting it: bounded waits that run
out return an error status and leave the context usable; device-side bad
ids are reported, not followed."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import TOL, np_bytes, oracle_layer, rel_err

pytestmark = pytest.mark.gpu

SMALL = synth.LayerConfig("fp8-fault", 256, 8, 2, 128, synth.BF16, synth.E4M3,
                          synth.GATE_SIGMOID_RENORM, n_shared=1)


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def test_bounded_wait_runs_out_and_reports(mv):
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    mv.moe_selftest_bounded_wait(err, 2000)   # a barrier nothing arrives on; 2 ms limit
    torch.cuda.synchronize()
    assert int(err[0]) == mv.MOE_ERR_TIMEOUT
    # the context is still usable
    x = torch.arange(10, device="cuda").sum().item()
    assert x == 45


def _pass(mv, layer, h, n, timeout_us):
    vl = mv.VerifyLayer(layer, n, wait_timeout_us=timeout_us)
    vl.route(h, n)
    vl.union_plan(n)
    y = vl.dedup(h, n).float().cpu().numpy()
    return y, vl.last_error()


# A BF16 layer with a shared expert at 26 tokens: the shared expert's segment
# (and any routed one of more than 8 tokens) runs on the tcgen05 CTAs.
WIDE = synth.LayerConfig("bf16-wide-fault", 512, 12, 3, 192, synth.BF16, synth.BF16,
                         synth.GATE_SOFTMAX_RENORM, n_shared=1, hidden="tree_add", sigma=0.3)


@pytest.mark.parametrize("cfg,n", [(SMALL, 8), (WIDE, 26)], ids=["fp8-n8", "bf16-tcgen05-n26"])
def test_tiny_wait_limit_ends_cleanly_then_normal_call_is_right(mv, cfg, n):
    layer = synth.make_layer(cfg, seed=4).to("cuda")
    h = synth.make_hidden(cfg, n, seed=5)
    hd = h.cuda()
    # a 1 microsecond limit: waits may run out; the call must end with OK or
    # TIMEOUT, never hang (on the tcgen05 CTAs too: every wait bounded, the
    # tensor memory freed after the issued MMAs complete)
    for _ in range(3):
        _, status = _pass(mv, layer, hd, n, 1)
        assert status in (mv.MOE_OK, mv.MOE_ERR_TIMEOUT)
    y, status = _pass(mv, layer, hd, n, 0)
    assert status == mv.MOE_OK
    L = oracle_layer(layer.to("cpu"))
    _, _, _, y_ref = oracle.verify(L, np_bytes(h))
    assert rel_err(y, y_ref) <= TOL[cfg.wtype]


def test_out_of_range_ids_are_reported_by_both_engines(mv):
    layer = synth.make_layer(SMALL, seed=4).to("cuda")
    n = 4
    h = synth.make_hidden(SMALL, n, seed=5).cuda()
    vl = mv.VerifyLayer(layer, n)
    ids = np.array([[0, 1], [2, 99], [3, -5], [4, 5]], dtype=np.int32)
    vl.ids[:8].copy_(torch.from_numpy(ids.ravel()))
    vl.w[:8].fill_(0.5)
    vl.perslot(h, n)
    assert vl.last_error() == mv.MOE_ERR_DEVICE_INPUT
    vl.union_plan(n)
    vl.dedup(h, n)
    assert vl.last_error() == mv.MOE_ERR_DEVICE_INPUT
    # a clean call afterwards reports OK
    vl.route(h, n)
    vl.union_plan(n)
    vl.dedup(h, n)
    assert vl.last_error() == mv.MOE_OK


def test_pass_replays_from_a_cuda_graph(mv):
    # the pass is host-sync free: captured once, replays match the eager pass
    cfg = synth.LayerConfig("fp8-graph", 640, 10, 4, 384, synth.BF16, synth.E4M3,
                            synth.GATE_SIGMOID_RENORM, n_shared=1)
    layer = synth.make_layer(cfg, seed=8).to("cuda")
    n = 12
    vl = mv.VerifyLayer(layer, n)
    h = torch.empty(n, cfg.d, dtype=torch.bfloat16, device="cuda")
    h.copy_(synth.make_hidden(cfg, n, seed=9))
    g_route, g_exp = vl.capture(h, n)
    for seed in (10, 11):
        h.copy_(synth.make_hidden(cfg, n, seed=seed))
        g_route.replay()
        g_exp.replay()
        y_graph = vl.y[:n].clone()
        y_eager = vl.verify_pass(h, n).clone()
        assert vl.last_error() == mv.MOE_OK
        assert torch.equal(y_graph, y_eager)


MALFORMED = ["uniq_out_of_range", "perm_out_of_range", "u_too_large", "offs_decreasing",
             "offs_past_slots", "offs_negative"]


@pytest.mark.parametrize("cfg,n", [(SMALL, 6), (synth.shrink(synth.OLMOE, 512, 128), 6),
                                   (synth.TINY, 6), (WIDE, 26)],
                         ids=["fp8", "bf16", "f32", "bf16-tcgen05-n26"])
@pytest.mark.parametrize("kind", MALFORMED)
def test_a_malformed_caller_plan_is_reported_not_followed(mv, cfg, n, kind):
    # moe_verify_dedup takes any plan from its caller: the expert kernels
    # check it before using its indices and report MOE_ERR_DEVICE_INPUT
    layer = synth.make_layer(cfg, seed=4).to("cuda")
    h = synth.make_hidden(cfg, n, seed=5).cuda()
    vl = mv.VerifyLayer(layer, n)
    vl.route(h, n)
    vl.union_plan(n)
    y_ok = vl.dedup(h, n).clone()
    assert vl.last_error() == mv.MOE_OK
    U = int(vl.plan.n_uniq[0])
    if kind == "uniq_out_of_range":
        vl.plan.uniq[U // 2] = cfg.n_experts + 7
    elif kind == "perm_out_of_range":
        vl.plan.perm[1] = 1 << 20
    elif kind == "u_too_large":
        vl.plan.n_uniq[0] = cfg.n_experts + 1
    elif kind == "offs_decreasing":
        vl.plan.offs[1] = int(vl.plan.offs[2]) + 1
    elif kind == "offs_past_slots":
        vl.plan.offs[U] = n * cfg.top_k + 5
    else:
        vl.plan.offs[0] = -3
    vl.dedup(h, n)
    assert vl.last_error() == mv.MOE_ERR_DEVICE_INPUT
    # a good plan afterwards gives the right output again
    vl.union_plan(n)
    assert torch.equal(vl.dedup(h, n), y_ok)
    assert vl.last_error() == mv.MOE_OK
