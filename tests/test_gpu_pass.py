"""moe_verify_pass, the whole pass in one call, against the separate calls
(moe_route_plan [budgeted] + moe_verify_dedup), bit for bit.  Inside it the
first expert kernel starts on the shared expert while routing still runs;
the outputs must not change, and work enqueued before the call (a write of
the hidden states) must be seen."""
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


# d = 8192: the widest E4M3 rows, every thread of the row-scaling CTAs on
# its last 16-byte word (the pass scales rows in its plan kernel, the dedup
# call in a kernel of its own: both must give the same rows and shifts)
CASES = [synth.TINY, synth.shrink(synth.OLMOE, 512, 128),
         synth.shrink(synth.DSV3, 1024, 256, 64, "dsv3-pass"),
         synth.shrink(synth.DSV3, 7168, 256, 16, "dsv3-wide"),
         synth.shrink(synth.DSV3, 8192, 256, 16, "dsv3-d8192")]


def separate(vl, h, n, budget):
    vl.route_plan(h, n, budget)
    return vl.dedup(h, n, kept=budget is not None).clone()


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
@pytest.mark.parametrize("n", [1, 3, 8, 17, 64])
def test_verify_pass_equals_separate_calls(mv, cfg, n):
    layer = synth.make_layer(cfg, seed=21).to("cuda")
    vl = mv.VerifyLayer(layer, 64)
    h = synth.make_hidden(cfg, n, seed=22).cuda()
    for budget in (None, 3):
        want = separate(vl, h, n, budget)
        plan_want = [t.clone() for t in (vl.plan.hist, vl.plan.n_uniq[:1], vl.ids[:n * cfg.top_k],
                                         vl.w[:n * cfg.top_k], vl.w_kept[:n * cfg.top_k])]
        vl.y.fill_(0)
        got = vl.verify_pass(h, n, budget=budget).clone()
        assert vl.last_error() == 0
        assert torch.equal(got, want), (budget,)
        plan_got = [vl.plan.hist, vl.plan.n_uniq[:1], vl.ids[:n * cfg.top_k],
                    vl.w[:n * cfg.top_k], vl.w_kept[:n * cfg.top_k]]
        for a, b in zip(plan_got, plan_want if budget is not None else plan_want[:4]):
            assert torch.equal(a, b)


def test_verify_pass_sees_the_hidden_states_written_just_before(mv):
    # the write of h is a device copy enqueued right before the call, with no
    # synchronisation in between; the pass must read the new values
    cfg = synth.shrink(synth.DSV3, 1024, 256, 64, "dsv3-pass")
    layer = synth.make_layer(cfg, seed=23).to("cuda")
    vl = mv.VerifyLayer(layer, 16)
    n = 12
    h_new = synth.make_hidden(cfg, n, seed=24).cuda()
    ref = separate(vl, h_new, n, None)
    h = synth.make_hidden(cfg, n, seed=25).cuda()
    torch.cuda.synchronize()
    big = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        big.fill_(1)          # keep the stream busy ahead of the write
        h.copy_(h_new)        # the write
        got = vl.verify_pass(h, n).clone()
        assert torch.equal(got, ref)
        h.copy_(synth.make_hidden(cfg, n, seed=25).cuda())
    assert vl.last_error() == 0


def test_verify_pass_empty(mv):
    layer = synth.make_layer(synth.shrink(synth.OLMOE, 512, 128), seed=3).to("cuda")
    vl = mv.VerifyLayer(layer, 8)
    vl.plan.n_uniq.fill_(5)
    vl.verify_pass(torch.empty(0, 512, dtype=torch.bfloat16, device="cuda"), 0)
    torch.cuda.synchronize()
    assert int(vl.plan.n_uniq[0]) == 0


@pytest.mark.parametrize("d,n", [(8192, 8), (8064, 13)])
def test_widest_e4m3_rows_match_the_oracle(mv, d, n):
    # the largest hidden size E4M3 layers take (8192), and one whose rows
    # end inside the row-scaling threads' last word, over two token groups
    cfg = synth.shrink(synth.DSV3, d, 256, 8, f"dsv3-d{d}")
    layer = synth.make_layer(cfg, seed=26)
    h = synth.make_hidden(cfg, n, seed=27)
    ids, w, _, y_ref = oracle.verify(oracle_layer(layer), np_bytes(h), threads=THREADS)
    vl = mv.VerifyLayer(layer.to("cuda"), 16)
    hd = h.cuda()
    vl.ids[:n * cfg.top_k].copy_(torch.from_numpy(ids.reshape(-1)).to(torch.int32))
    vl.w[:n * cfg.top_k].copy_(torch.from_numpy(np.asarray(w).reshape(-1)).to(torch.float32))
    vl.union_plan(n)
    y = vl.dedup(hd, n).float().cpu().numpy().astype(np.float64)
    assert vl.last_error() == 0
    err = rel_err(y, y_ref)
    assert err <= TOL[synth.E4M3], f"d={d} n={n}: rel err {err:.3g}"
