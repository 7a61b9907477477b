"""moe_verify_dedup_noalloc: the deduplicating pass for callers that cannot
allocate device memory (their memory belongs to a framework allocator they
must not go around, or their hot path must never call cudaMalloc).  Its
scratch is a fixed array inside the library, so its output must equal
moe_verify_dedup's with a caller workspace, call after call, even though the
array keeps the previous call's contents.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import TOL, rel_err

pytestmark = pytest.mark.gpu

CASES = [
    synth.LayerConfig("fp8-noalloc", 640, 10, 4, 384, synth.BF16, synth.E4M3,
                      synth.GATE_SIGMOID_RENORM, n_shared=1, hidden="tree_ar", rho=0.6),
    synth.LayerConfig("bf16-noalloc", 704, 12, 3, 192, synth.BF16, synth.BF16,
                      synth.GATE_SOFTMAX, hidden="chain", rho=0.5),
    synth.TINY,
]


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_matches_workspace_pass_on_two_calls_in_a_row(mv, cfg):
    layer = synth.make_layer(cfg, seed=21, device="cuda")
    vl = mv.VerifyLayer(layer, 64)
    err = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    # two calls in a row with different tokens; the second must not see the
    # first call's leftovers in the shared scratch.  Both entry points run
    # the same kernels in the same order, so their outputs are identical.
    for n, seed in ((24, 5), (7, 6)):
        h = synth.make_hidden(cfg, n, seed=seed, device="cuda")
        vl.route_plan(h, n)
        y_ref = vl.dedup(h, n).clone()
        assert vl.last_error() == mv.MOE_OK
        y = torch.full((n, cfg.d), float("nan"), dtype=synth.torch_dtype(cfg.act), device="cuda")
        mv.moe_verify_dedup_noalloc(vl.desc, vl.weights, h, n, vl.ids, vl.w, vl._cplan, y, err)
        torch.cuda.synchronize()
        assert int(err[0]) == mv.MOE_OK
        assert torch.equal(y, y_ref)
        # (identical outputs are within every tolerance of the parity tests)
        assert rel_err(y.float().cpu().numpy(), y_ref.float().cpu().numpy()) <= TOL[cfg.wtype]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_noalloc_reports_a_device_error_then_recovers(mv, cfg):
    # a malformed plan (an expert id out of range) is reported through
    # error_word, copied out of the shared scratch; the next, clean call
    # starts from a cleared error word and gives the right output again
    layer = synth.make_layer(cfg, seed=22, device="cuda")
    n = 6
    vl = mv.VerifyLayer(layer, n)
    h = synth.make_hidden(cfg, n, seed=7, device="cuda")
    vl.route_plan(h, n)
    y_ref = vl.dedup(h, n).clone()
    assert vl.last_error() == mv.MOE_OK
    err = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    y = torch.empty(n, cfg.d, dtype=synth.torch_dtype(cfg.act), device="cuda")
    U = int(vl.plan.n_uniq[0])
    good = int(vl.plan.uniq[U // 2])
    vl.plan.uniq[U // 2] = cfg.n_experts + 7
    mv.moe_verify_dedup_noalloc(vl.desc, vl.weights, h, n, vl.ids, vl.w, vl._cplan, y, err)
    torch.cuda.synchronize()
    assert int(err[0]) == mv.MOE_ERR_DEVICE_INPUT
    vl.plan.uniq[U // 2] = good
    mv.moe_verify_dedup_noalloc(vl.desc, vl.weights, h, n, vl.ids, vl.w, vl._cplan, y, err)
    torch.cuda.synchronize()
    assert int(err[0]) == mv.MOE_OK
    assert torch.equal(y, y_ref)


def test_noalloc_rejects_a_call_beyond_its_fixed_scratch(mv):
    # DeepSeek-V3 shapes: 64 tokens x 9 slots need about 19 MB of scratch
    desc = mv.make_desc(synth.DSV3, 64)
    fake = 0x10000  # never dereferenced: the size check comes before any launch
    W = mv.moe_expert_weights(fake, fake, fake, fake)
    plan = mv.moe_plan(fake, fake, fake, fake, fake, fake)
    p = ctypes.c_void_p(fake)
    st = mv._lib.moe_verify_dedup_noalloc(ctypes.byref(desc), ctypes.byref(W), p, 64, p, p,
                                          ctypes.byref(plan), p, None, ctypes.c_void_p(0))
    assert st == mv.MOE_ERR_WORKSPACE
    # 8 tokens fit
    assert mv.moe_workspace_bytes(mv.make_desc(synth.DSV3, 8)) < (16 << 20)
