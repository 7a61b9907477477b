"""The expert-budgeted plan and pass on the GPU against the oracle.

MoE-Spec's verification-time expert budget (its abstract, as listed on
"Speculative Decoding for MoE Models: Expert Bytes, ..."; "The Limits of
Speculation", Sec. 2.4): at most B routed experts are loaded; the kept ones
are those of largest summed gate weight (ties to the lower id); a dropped
slot's term is left out.  The plan is bit-exact from identical (ids, w); the
pass is compared with the oracle's budgeted pass wherever the kept set is
decided with a margin larger than the error bound of the GPU's weights.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth
from tests.helpers import THREADS, TOL, np_bytes, oracle_layer, rel_err, tie_margin

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def _w_uniform(n, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(n, k, generator=g, dtype=torch.float32).numpy()


def run_budget_plan(mv, cfg, ids: np.ndarray, w: np.ndarray, budget: int):
    n = ids.shape[0]
    k, E = cfg.top_k, cfg.n_experts
    desc = mv.make_desc(cfg, max(n, 1))
    dev = "cuda"
    fill = lambda m, dt=torch.int32: torch.full((m,), -7, dtype=dt, device=dev)
    pb = mv.PlanBuffers(fill(E), fill(E), fill(4), fill(E + 1), fill(max(n * k, 4)),
                        fill(2, torch.int64))
    w_kept = torch.full((max(n * k, 4),), -5.0, dtype=torch.float32, device=dev)
    routed = fill(4)
    err = torch.zeros(4, dtype=torch.int32, device=dev)
    ids_d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)).to(dev)
    w_d = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32).reshape(-1)).to(dev)
    mv.moe_union_plan_budgeted(desc, ids_d, w_d, n, budget, pb.c(), w_kept, routed, err)
    torch.cuda.synchronize()
    U = int(pb.n_uniq[0])
    return dict(U=U, hist=pb.hist.cpu().numpy(), uniq=pb.uniq[:U].cpu().numpy(),
                offs=pb.offs[:U + 1].cpu().numpy(),
                perm=pb.perm[:int(pb.offs[U]) if U else 0].cpu().numpy(),
                ub=int(pb.union_bytes[0]), w_kept=w_kept[:n * k].cpu().numpy(),
                routed=int(routed[0]), err=int(err[0]))


def check_budget_plan(mv, cfg, ids, w, budget):
    g = run_budget_plan(mv, cfg, ids, w, budget)
    rU, rhist, runiq, roffs, rperm, rw_kept, rkeep = oracle.budget_plan(
        ids, w.astype(np.float64), cfg.n_experts, budget)
    assert g["err"] == 0
    assert g["routed"] == oracle.union_plan(ids, cfg.n_experts)[0]
    assert g["U"] == rU == min(budget, g["routed"])
    assert np.array_equal(g["hist"], rhist)
    assert np.array_equal(g["uniq"], runiq)
    assert np.array_equal(g["offs"], roffs)
    assert np.array_equal(g["perm"], rperm)
    assert np.array_equal(g["w_kept"].astype(np.float64), rw_kept)
    wtype = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.E4M3: oracle.E4M3}[cfg.wtype]
    wb, sb = oracle.expert_bytes(cfg.d, cfg.inter, wtype)
    assert g["ub"] == (rU + cfg.n_shared) * (wb + sb)
    return g


PLAN_CONFIGS = [synth.TINY, synth.OLMOE, synth.QWEN3, synth.GPTOSS, synth.DSV3]


@pytest.mark.parametrize("cfg", PLAN_CONFIGS, ids=lambda c: c.name)
@pytest.mark.parametrize("n", [1, 3, 8, 31, 64])
def test_budget_plan_bit_exact_from_identical_inputs(mv, cfg, n):
    ids = synth.uniform_ids(n, cfg.top_k, cfg.n_experts, seed=300 + n).numpy()
    w = _w_uniform(n, cfg.top_k, seed=400 + n)
    U = oracle.union_plan(ids, cfg.n_experts)[0]
    for B in sorted({0, 1, U // 2, max(U - 1, 0), U, U + 3, cfg.n_experts}):
        check_budget_plan(mv, cfg, ids, w, B)


@pytest.mark.parametrize("n", [4, 16, 64])
@pytest.mark.parametrize("signed", [False, True])
def test_budget_plan_ties_break_to_the_lower_id(mv, n, signed):
    # weights in multiples of 1/8 make many contributions exactly equal; the
    # signed case also orders negative and zero contributions (weights any
    # caller may pass, not gate outputs)
    cfg = synth.DSV3
    ids = synth.uniform_ids(n, cfg.top_k, cfg.n_experts, seed=500 + n).numpy()
    rng = np.random.default_rng(600 + n)
    lo = -8 if signed else 1
    w = (rng.integers(lo, 9, size=ids.shape) / 8.0).astype(np.float32)
    U = oracle.union_plan(ids, cfg.n_experts)[0]
    for B in range(0, U + 1, max(1, U // 16)):
        check_budget_plan(mv, cfg, ids, w, B)


def test_budget_plan_with_identical_tokens_and_bad_ids(mv):
    cfg = synth.OLMOE
    row = synth.uniform_ids(1, 8, 64, seed=3).numpy()
    ids = np.tile(row, (16, 1))
    w = _w_uniform(16, 8, seed=4)
    for B in (0, 3, 8):
        g = check_budget_plan(mv, cfg, ids, w, B)
        assert g["U"] == min(B, 8)
    # an invalid id is reported, left out of the plan and given weight 0
    ids = synth.uniform_ids(4, 8, 64, seed=1).numpy()
    ids[1, 2] = 64
    g = run_budget_plan(mv, cfg, ids, _w_uniform(4, 8, seed=2), 3)
    assert g["err"] == mv.MOE_ERR_DEVICE_INPUT and g["w_kept"][1 * 8 + 2] == 0.0
    assert g["U"] == 3 and g["hist"].sum() == g["offs"][-1]


def test_budget_plan_empty(mv):
    g = run_budget_plan(mv, synth.OLMOE, np.zeros((0, 8), np.int32), np.zeros((0, 8), np.float32), 4)
    assert g["U"] == 0 and g["offs"][0] == 0 and g["hist"].sum() == 0 and g["ub"] == 0
    assert g["routed"] == 0


FUSED_CASES = [(synth.TINY, 4, 3), (synth.OLMOE, 8, 20), (synth.QWEN3, 61, 40),
               (synth.GPTOSS, 16, 10), (synth.DSV3, 8, 16), (synth.DSV3, 64, 64)]


@pytest.mark.parametrize("cfg,n,B", FUSED_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_fused_budgeted_route_plan_equals_separate_calls(mv, cfg, n, B):
    small = synth.shrink(cfg, cfg.d, 128 if cfg.wtype == synth.E4M3 else 64)
    layer = synth.make_layer(small, seed=31).to("cuda")
    vl = mv.VerifyLayer(layer, 64)
    k = small.top_k
    for rep in range(3):
        h = synth.make_hidden(small, n, seed=40 + rep).cuda()
        vl.route(h, n)
        vl.union_plan(n, budget=B)
        torch.cuda.synchronize()
        U = int(vl.plan.n_uniq[0])
        want = [t.clone() for t in (vl.ids[:n * k], vl.w[:n * k], vl.logits[:n * small.n_experts],
                                    vl.plan.hist, vl.plan.uniq[:U], vl.plan.n_uniq[:1],
                                    vl.plan.offs[:U + 1], vl.plan.perm[:int(vl.plan.offs[U])],
                                    vl.plan.union_bytes[:1], vl.w_kept[:n * k], vl.routed_u[:1])]
        for t in (vl.ids, vl.plan.perm, vl.plan.uniq, vl.routed_u):
            t.fill_(-3)
        vl.w_kept.fill_(-1.0)
        vl.route_plan(h, n, budget=B)
        torch.cuda.synchronize()
        got = [vl.ids[:n * k], vl.w[:n * k], vl.logits[:n * small.n_experts], vl.plan.hist,
               vl.plan.uniq[:U], vl.plan.n_uniq[:1], vl.plan.offs[:U + 1],
               vl.plan.perm[:int(vl.plan.offs[U])], vl.plan.union_bytes[:1], vl.w_kept[:n * k],
               vl.routed_u[:1]]
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        assert vl.last_error() == 0
        assert int(vl.workspace[64:68].view(torch.int32)[0]) == 0


# ------------------------------------------------------------- the pass

def cut_margin(ids, w, E, B, slot_err):
    """(kept-set decision margin) for the oracle's weights w: the smallest
    lower bound of a kept contribution minus the largest upper bound of a
    dropped one, where each contribution may be off by the sum of slot_err
    over its slots.  Positive: any weights within slot_err of w keep the same
    experts."""
    keep, score, _ = oracle.expert_budget(ids, w, E, B)
    used = np.zeros(E, dtype=bool)
    used[np.asarray(ids).ravel()] = True
    err = np.zeros(E)
    np.add.at(err, np.asarray(ids).ravel(), np.broadcast_to(slot_err, np.shape(ids)).ravel())
    kept, dropped = keep & used, ~keep & used
    if not kept.any() or not dropped.any():
        return np.inf
    return (score[kept] - err[kept]).min() - (score[dropped] + err[dropped]).max()


def gpu_budgeted_pass_from(mv, dev_layer, h, n, ids, w, B):
    """The budgeted plan and the dedup engine on the given routing."""
    k = dev_layer.cfg.top_k
    vl = mv.VerifyLayer(dev_layer, max(n, 1))
    vl.ids[:n * k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * k].copy_(torch.from_numpy(w.reshape(-1)).to(torch.float32))
    vl.union_plan(n, budget=B)
    y = vl.dedup(h.cuda(), n, kept=True)
    assert vl.last_error() == 0
    U = int(vl.plan.n_uniq[0])
    return y.float().cpu().numpy().astype(np.float64), set(vl.plan.uniq[:U].cpu().tolist())


PASS_CASES = [
    (synth.shrink(synth.DSV3, 1024, 256, 32, "dsv3-small"), 8),
    (synth.shrink(synth.DSV3, 1024, 256, 32, "dsv3-small"), 33),
    (synth.shrink(synth.OLMOE, 512, 128), 16),
    (synth.shrink(synth.QWEN3, 512, 192), 61),
    (synth.TINY, 4),
]


@pytest.mark.parametrize("cfg,n", PASS_CASES, ids=lambda x: getattr(x, "name", str(x)))
def test_budgeted_pass_against_oracle(mv, cfg, n):
    # the oracle's routing, gate weights rounded to fp32, goes to the GPU
    layer = synth.make_layer(cfg, seed=5)
    L = oracle_layer(layer)
    h = synth.make_hidden(cfg, n, seed=6)
    hb = np_bytes(h)
    ids, w, _, _ = oracle.verify(L, hb, threads=THREADS)
    w32 = w.astype(np.float32)
    U = oracle.union_plan(ids, cfg.n_experts)[0]
    dev_layer = layer.to("cuda")
    checked = 0
    for B in sorted({0, 1, U // 4, U // 2, U - 1, U}):
        # the GPU decides on fp32 weights: each is within 2^-24 relative of w
        if cut_margin(ids, w, cfg.n_experts, B, np.abs(w) * 2.0 ** -23) <= 0:
            continue
        _, _, _, y_ref, keep = oracle.verify_budget(L, hb, B, threads=THREADS)
        y, kept = gpu_budgeted_pass_from(mv, dev_layer, h, n, ids, w32, B)
        assert kept == set(np.flatnonzero(keep).tolist())
        if np.any(y_ref != 0):
            assert rel_err(y, y_ref) <= TOL[cfg.wtype], B
        else:
            assert np.all(y == 0)
        checked += 1
    assert checked >= 4


def test_budget_at_or_above_the_union_is_bitwise_the_plain_pass(mv):
    cfg = synth.shrink(synth.DSV3, 1024, 256, 32, "dsv3-small")
    layer = synth.make_layer(cfg, seed=7).to("cuda")
    n = 12
    h = synth.make_hidden(cfg, n, seed=8).cuda()
    vl = mv.VerifyLayer(layer, n)
    y_plain = vl.verify_pass(h, n).clone()
    U = int(vl.plan.n_uniq[0])
    for B in (U, U + 1, cfg.n_experts):
        y_b = vl.verify_pass(h, n, budget=B).clone()
        assert vl.last_error() == 0 and int(vl.plan.n_uniq[0]) == U
        assert torch.equal(y_b, y_plain)
        assert torch.equal(vl.w_kept[:n * cfg.top_k], vl.w[:n * cfg.top_k])


def test_budget_zero_applies_only_the_shared_expert(mv):
    for cfg in (synth.shrink(synth.DSV3, 1024, 256, 32, "dsv3-small"),
                synth.shrink(synth.OLMOE, 512, 128)):
        layer = synth.make_layer(cfg, seed=9)
        n = 6
        h = synth.make_hidden(cfg, n, seed=10)
        vl = mv.VerifyLayer(layer.to("cuda"), n)
        y = vl.verify_pass(h.cuda(), n, budget=0).float().cpu().numpy()
        assert vl.last_error() == 0 and int(vl.plan.n_uniq[0]) == 0
        assert int(vl.routed_u[0]) >= cfg.top_k
        if cfg.n_shared:
            _, _, _, y_ref, keep = oracle.verify_budget(oracle_layer(layer), np_bytes(h), 0)
            assert not keep.any()
            assert rel_err(y, y_ref) <= TOL[cfg.wtype]
        else:
            assert np.all(y == 0)


def test_budgeted_pass_replays_from_a_cuda_graph(mv):
    cfg = synth.LayerConfig("fp8-graph-budget", 640, 10, 4, 384, synth.BF16, synth.E4M3,
                            synth.GATE_SIGMOID_RENORM, n_shared=1)
    layer = synth.make_layer(cfg, seed=8).to("cuda")
    n = 12
    vl = mv.VerifyLayer(layer, n)
    h = torch.empty(n, cfg.d, dtype=torch.bfloat16, device="cuda")
    h.copy_(synth.make_hidden(cfg, n, seed=9))
    g_route, g_exp = vl.capture(h, n, budget=5)
    for seed in (10, 11):
        h.copy_(synth.make_hidden(cfg, n, seed=seed))
        g_route.replay()
        g_exp.replay()
        y_graph = vl.y[:n].clone()
        assert int(vl.plan.n_uniq[0]) == 5
        y_eager = vl.verify_pass(h, n, budget=5).clone()
        assert vl.last_error() == mv.MOE_OK
        assert torch.equal(y_graph, y_eager)


# ------------------------------------------------ full size, sampled tokens

def router_delta(layer, h):
    """Per token: 1e-5 * max_e sum_i |Wg[e][i] h[i]|, the bound on the GPU's
    fp32 router-score error that tie_margin uses."""
    wg = np.asarray(layer.wg.float().cpu().numpy(), dtype=np.float64)
    hh = np.asarray(h.float().cpu().numpy(), dtype=np.float64)
    return 1e-5 * (np.abs(hh) @ np.abs(wg).T).max(axis=1)


@pytest.mark.parametrize("n,sample", [(8, [0, 3, 7]), (64, [0, 63])])
def test_dsv3_fp8_budgeted_pass_full_size(mv, n, sample):
    # the bench's layer and launch configuration (n_max = 64, fused
    # route + budgeted plan, graph-free here); B is the largest cut at or
    # below U/2 that the routing error bound cannot move
    cfg = synth.DSV3
    layer = synth.make_layer(cfg, seed=1, device="cuda")
    h = synth.make_hidden(cfg, 64, seed=3, device="cuda")[:n].contiguous()
    cpu_layer = layer.to("cpu")
    L = oracle_layer(cpu_layer)
    hb = np_bytes(h)
    ids, w, z, _, _ = oracle.verify_budget(L, hb, cfg.n_experts, tokens=[], threads=THREADS)
    clear = tie_margin(cpu_layer, h.cpu(), z, cfg.top_k) > 1.0
    # a score error below delta moves a renormalised gate weight by < 2 delta (+ fp32 rounding)
    slot_err = (2.0 * router_delta(cpu_layer, h.cpu())[:, None] + 1e-6) * np.ones_like(w)
    U = oracle.union_plan(ids, cfg.n_experts)[0]
    B = next(b for b in range(U // 2, 0, -1) if cut_margin(ids, w, cfg.n_experts, b, slot_err) > 0)
    vl = mv.VerifyLayer(layer, 64)
    y = vl.verify_pass(h, n, budget=B).float().cpu().numpy()
    assert vl.last_error() == 0
    # the kept set depends on every token's routing: the GPU must route all
    # n tokens as the oracle does (certain where the gap exceeds the error
    # bound; a token inside the bound may legitimately differ, and is named)
    ids_gpu = vl.ids_view(n).cpu().numpy()
    assert np.array_equal(ids_gpu[clear], ids[clear])
    assert np.array_equal(ids_gpu, ids), f"near-tie tokens routed differently: {np.flatnonzero(~clear)}"
    assert int(vl.routed_u[0]) == U and int(vl.plan.n_uniq[0]) == B
    kept_gpu = set(vl.plan.uniq[:B].cpu().tolist())
    del vl, layer
    torch.cuda.empty_cache()
    _, _, _, y_ref, keep = oracle.verify_budget(L, hb, B, tokens=sample, threads=THREADS)
    assert kept_gpu == set(np.flatnonzero(keep).tolist())
    assert rel_err(y[sample], y_ref) <= TOL[cfg.wtype]
