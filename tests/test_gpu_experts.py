"""Both expert engines on the GPU against the oracle.

The GPU engines get the oracle's own routing (ids, and gate weights rounded
to fp32) so that these tests isolate the expert arithmetic; routing has its
own tests.  Sizes span several stages of the weight pipeline, ragged K
tails, and segments of more than 8 tokens (the width of one MMA token tile,
so such a segment takes several passes over its weights).
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


_LAYERS = {}


def get_layer(cfg, seed=1):
    key = (cfg, seed)
    if key not in _LAYERS:
        _LAYERS.clear()
        big = cfg.n_experts * cfg.d * cfg.inter > 64 * 2048 * 1024
        dev_layer = synth.make_layer(cfg, seed=seed, device="cuda" if big else "cpu").to("cuda")
        cpu_layer = dev_layer.to("cpu")
        _LAYERS[key] = (dev_layer, cpu_layer, oracle_layer(cpu_layer))
    return _LAYERS[key]


def run_gpu(mv, dev_layer, h, n, ids, w, engine, n_max=None):
    vl = mv.VerifyLayer(dev_layer, n_max or max(n, 1))
    if n:
        vl.ids[:n * dev_layer.cfg.top_k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
        vl.w[:n * dev_layer.cfg.top_k].copy_(torch.from_numpy(w.reshape(-1)).to(torch.float32))
    hd = h.cuda()
    if engine == "dedup":
        vl.union_plan(n)
        y = vl.dedup(hd, n)
    else:
        y = vl.perslot(hd, n)
    assert vl.last_error() == 0
    return y.float().cpu().numpy().astype(np.float64), vl


def check_layer(mv, cfg, n, seed=1, kind=None, rho=None, sigma=None, engines=("dedup", "perslot"),
                tokens=None):
    dev_layer, cpu_layer, L = get_layer(cfg, seed)
    h = synth.make_hidden(cfg, n, seed=seed + 2, kind=kind, rho=rho, sigma=sigma)
    ids, w, _, y_ref = oracle.verify(L, np_bytes(h), threads=THREADS)
    out = {}
    for eng in engines:
        y, _ = run_gpu(mv, dev_layer, h, n, ids, w, eng)
        err = rel_err(y, y_ref)
        assert err <= TOL[cfg.wtype], f"{cfg.name} n={n} {eng}: rel err {err:.3g}"
        out[eng] = y
    return out, ids


BF16_SMALL = synth.shrink(synth.OLMOE, d=704, inter=192, n_experts=12, name="bf16-d704-i192")
BF16_SMALL = synth.LayerConfig(**{**BF16_SMALL.__dict__, "top_k": 3})
FP8_SMALL = synth.shrink(synth.DSV3, d=640, inter=384, n_experts=10, name="fp8-d640-i384")
FP8_SMALL = synth.LayerConfig(**{**FP8_SMALL.__dict__, "top_k": 4})
F32_SMALL = synth.shrink(synth.TINY, d=264, inter=36, n_experts=9, name="f32-d264-i36")


@pytest.mark.parametrize("n", [1, 4, 9, 64])
def test_tiny_fp32_layer(mv, n):
    check_layer(mv, synth.TINY, n)


@pytest.mark.parametrize("n", [1, 3, 17])
def test_f32_ragged(mv, n):
    check_layer(mv, F32_SMALL, n)


@pytest.mark.parametrize("n", [1, 5, 8, 13, 24, 40, 64])
def test_bf16_small(mv, n):
    check_layer(mv, BF16_SMALL, n)


@pytest.mark.parametrize("n", [1, 4, 8, 17, 33, 64])
def test_fp8_small_with_shared_expert(mv, n):
    check_layer(mv, FP8_SMALL, n)


@pytest.mark.parametrize("cfg", [BF16_SMALL, FP8_SMALL, F32_SMALL], ids=lambda c: c.name)
def test_identical_tokens(mv, cfg):
    # every token routes to the same k experts: U = k, each segment holds all 64
    out, ids = check_layer(mv, cfg, 64, kind="identical")
    assert len(set(ids.ravel().tolist())) == cfg.top_k
    for eng in out:
        assert np.array_equal(out[eng][0], out[eng][63])


@pytest.mark.parametrize("cfg", [BF16_SMALL, FP8_SMALL, F32_SMALL, synth.TINY], ids=lambda c: c.name)
def test_engines_agree_and_match_bitwise_at_one_token(mv, cfg):
    # "Expert Bytes ...", Table 6: at n = 1 an engine runs the same kernel with
    # deduplication off and on
    out, _ = check_layer(mv, cfg, 1)
    assert np.array_equal(out["dedup"], out["perslot"])
    out, _ = check_layer(mv, cfg, 12)
    assert rel_err(out["dedup"], out["perslot"]) <= TOL[cfg.wtype]


@pytest.mark.parametrize("n,rho", [(1, 0.0), (2, 0.5), (4, 0.9), (8, 0.0), (8, 0.9)])
def test_olmoe_layer(mv, n, rho):
    check_layer(mv, synth.OLMOE, n, rho=rho)


@pytest.mark.parametrize("n,sigma", [(16, 0.3), (16, 1.0)])
def test_qwen3_tree(mv, n, sigma):
    check_layer(mv, synth.QWEN3, n, sigma=sigma)


def test_gptoss_chain(mv):
    check_layer(mv, synth.GPTOSS, 3)


def test_dsv3_fp8_layer(mv):
    check_layer(mv, synth.DSV3, 2)


def test_empty_pass(mv):
    dev_layer, _, _ = get_layer(BF16_SMALL)
    h = synth.make_hidden(BF16_SMALL, 1)
    vl = mv.VerifyLayer(dev_layer, 4)
    vl.y.fill_(7)
    vl.union_plan(0)
    vl.dedup(h.cuda(), 0)
    vl.perslot(h.cuda(), 0)
    assert vl.last_error() == 0
    assert torch.all(vl.y == 7)
