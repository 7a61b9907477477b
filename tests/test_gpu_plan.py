"""The union planner on the GPU against the oracle's plain counting: hist,
uniq, U, offsets, permutation and union bytes bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def run_plan(mv, cfg, ids: np.ndarray):
    n = ids.shape[0]
    k, E = cfg.top_k, cfg.n_experts
    desc = mv.make_desc(cfg, max(n, 1))
    dev = "cuda"
    pb = mv.PlanBuffers(torch.full((E,), -7, dtype=torch.int32, device=dev),
                        torch.full((E,), -7, dtype=torch.int32, device=dev),
                        torch.full((4,), -7, dtype=torch.int32, device=dev),
                        torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                        torch.full((max(n * k, 4),), -7, dtype=torch.int32, device=dev),
                        torch.full((2,), -7, dtype=torch.int64, device=dev))
    err = torch.zeros(4, dtype=torch.int32, device=dev)
    ids_d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)).to(dev)
    if ids_d.numel() == 0:
        ids_d = torch.zeros(4, dtype=torch.int32, device=dev)
    mv.moe_union_plan(desc, ids_d, n, pb.c(), err)
    torch.cuda.synchronize()
    U = int(pb.n_uniq[0])
    return (U, pb.hist.cpu().numpy(), pb.uniq[:U].cpu().numpy(), pb.offs[:U + 1].cpu().numpy(),
            pb.perm[:n * k].cpu().numpy(), int(pb.union_bytes[0]), int(err[0]))


def check(mv, cfg, ids):
    U, hist, uniq, offs, perm, ub, err = run_plan(mv, cfg, ids)
    rU, rhist, runiq, roffs, rperm = oracle.union_plan(ids, cfg.n_experts)
    assert err == 0
    assert U == rU
    assert np.array_equal(hist, rhist)
    assert np.array_equal(uniq, runiq)
    assert np.array_equal(offs, roffs)
    assert np.array_equal(perm, rperm)
    wtype = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.E4M3: oracle.E4M3}[cfg.wtype]
    wb, sb = oracle.expert_bytes(cfg.d, cfg.inter, wtype)
    assert ub == (U + cfg.n_shared) * (wb + sb)
    return U


PLAN_CONFIGS = [synth.TINY, synth.OLMOE, synth.QWEN3, synth.GPTOSS, synth.DSV3]


@pytest.mark.parametrize("cfg", PLAN_CONFIGS, ids=lambda c: c.name)
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 31, 64])
def test_plan_uniform_ids(mv, cfg, n):
    ids = synth.uniform_ids(n, cfg.top_k, cfg.n_experts, seed=100 + n).numpy()
    check(mv, cfg, ids)


@pytest.mark.parametrize("cfg", PLAN_CONFIGS, ids=lambda c: c.name)
def test_plan_identical_tokens_union_is_k(mv, cfg):
    row = synth.uniform_ids(1, cfg.top_k, cfg.n_experts, seed=3).numpy()
    for n in (1, 2, 8, 64):
        assert check(mv, cfg, np.tile(row, (n, 1))) == cfg.top_k


def test_plan_skewed_and_full_coverage(mv):
    cfg = synth.DSV3
    # every expert used (64 tokens x 8 slots cover 256 experts twice)
    ids = np.arange(512, dtype=np.int32).reshape(64, 8) % 256
    assert check(mv, cfg, ids) == 256
    # all tokens share 7 experts and differ in the 8th
    ids = np.tile(np.arange(7, dtype=np.int32), (64, 1))
    ids = np.concatenate([ids, (np.arange(64, dtype=np.int32) + 100)[:, None]], axis=1)
    assert check(mv, cfg, ids) == 7 + 64


def test_plan_k32(mv):
    cfg = synth.LayerConfig("k32", 256, 256, 32, 128, synth.BF16, synth.BF16, synth.GATE_SOFTMAX)
    ids = synth.uniform_ids(64, 32, 256, seed=9).numpy()
    check(mv, cfg, ids)


def test_plan_empty(mv):
    cfg = synth.OLMOE
    U, hist, uniq, offs, perm, ub, err = run_plan(mv, cfg, np.zeros((0, 8), np.int32))
    assert U == 0 and offs[0] == 0 and hist.sum() == 0 and ub == 0


def test_plan_flags_out_of_range_ids(mv):
    cfg = synth.OLMOE
    ids = synth.uniform_ids(4, 8, 64, seed=1).numpy()
    ids[2, 3] = 64
    ids[0, 0] = -1
    U, hist, uniq, offs, perm, ub, err = run_plan(mv, cfg, ids)
    assert err == 7  # MOE_ERR_DEVICE_INPUT
    valid = ids[(ids >= 0) & (ids < 64)]
    assert U == len(set(valid.tolist())) and hist.sum() == valid.size


ROUTE_PLAN_CASES = [(synth.TINY, 4), (synth.OLMOE, 8), (synth.QWEN3, 61), (synth.GPTOSS, 16),
                    (synth.DSV3, 8), (synth.DSV3, 64), (synth.DSV3, 1)]


@pytest.mark.parametrize("cfg,n", ROUTE_PLAN_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_fused_route_plan_equals_separate_calls(mv, cfg, n):
    # one launch (scores, top-k, gate, plan) == moe_route_topk then moe_union_plan, bit for bit,
    # on three calls in a row (the ticket counter must reset itself)
    small = synth.shrink(cfg, cfg.d, 128 if cfg.wtype == synth.E4M3 else 64)
    layer = synth.make_layer(small, seed=31).to("cuda")
    vl = mv.VerifyLayer(layer, 64)
    for rep in range(3):
        h = synth.make_hidden(small, n, seed=40 + rep).cuda()
        vl.route(h, n)
        vl.union_plan(n)
        torch.cuda.synchronize()
        ref = [t.clone() for t in (vl.ids, vl.w, vl.logits, vl.plan.hist, vl.plan.uniq,
                                   vl.plan.n_uniq, vl.plan.offs, vl.plan.perm,
                                   vl.plan.union_bytes)]
        for t in (vl.ids, vl.plan.perm, vl.plan.uniq):
            t.fill_(-3)
        vl.route_plan(h, n)
        torch.cuda.synchronize()
        U = int(vl.plan.n_uniq[0])
        k = small.top_k
        got = [vl.ids[:n * k], vl.w[:n * k], vl.logits[:n * small.n_experts], vl.plan.hist,
               vl.plan.uniq[:U], vl.plan.n_uniq[:1], vl.plan.offs[:U + 1], vl.plan.perm[:n * k],
               vl.plan.union_bytes[:1]]
        want = [ref[0][:n * k], ref[1][:n * k], ref[2][:n * small.n_experts], ref[3], ref[4][:U],
                ref[5][:1], ref[6][:U + 1], ref[7][:n * k], ref[8][:1]]
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        assert vl.last_error() == 0
        # the ticket counter in the workspace header is back at zero
        assert int(vl.workspace[64:68].view(torch.int32)[0]) == 0


def test_fused_route_plan_empty(mv):
    layer = synth.make_layer(synth.shrink(synth.OLMOE, 2048, 64), seed=3).to("cuda")
    vl = mv.VerifyLayer(layer, 8)
    vl.plan.n_uniq.fill_(5)
    vl.route_plan(torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda"), 0)
    torch.cuda.synchronize()
    assert int(vl.plan.n_uniq[0]) == 0 and int(vl.plan.offs[0]) == 0
