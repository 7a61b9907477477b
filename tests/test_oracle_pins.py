"""Pins of the CPU oracle against facts fixed by the pages or by mathematics.

Nothing here compares the oracle with itself: each check uses a closed form,
a brute-force enumeration, an independent library routine (torch's float8 /
bfloat16 casts, scipy's softmax and expit, numpy's matmul), an invariant, or
a number the pages print.  Each is chosen so that a plausible slip in the
oracle (a swapped gate/up, a transposed down projection, a wrong scale block
index, a tie broken the other way, a dropped shared expert) fails it.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O


# ----------------------------------------------------------------- decoding

def test_e4m3_decode_all_256_codes_against_torch_cast():
    codes = np.arange(256, dtype=np.uint8)
    ours = O.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # zero's sign survives
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_decode_format_facts():
    # OCP E4M3: bias 7, largest finite 448, smallest subnormal 2^-9,
    # smallest normal 2^-6, only S.1111.111 is NaN, no infinities.
    d = O.decode_e4m3(np.arange(256, dtype=np.uint8))
    assert d[0x38] == 1.0
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0
    assert d[0x01] == 2.0 ** -9 and d[0x07] == 7 * 2.0 ** -9
    assert d[0x08] == 2.0 ** -6
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.sum(np.isnan(d)) == 2 and not np.any(np.isinf(d))
    finite = d[~np.isnan(d)]
    assert np.max(finite) == 448.0


def test_bf16_decode_against_torch():
    g = torch.Generator().manual_seed(11)
    x = (torch.randn(4096, generator=g) * 10).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_to_double(bits), x.to(torch.float64).numpy())


# ------------------------------------------------------------------- top-k

def _brute_topk(z, k):
    """The unique k-subset S whose members all beat every non-member under
    (larger score, then lower id), listed in that order."""
    E = len(z)
    beats = lambda i, j: z[i] > z[j] or (z[i] == z[j] and i < j)
    found = [S for S in itertools.combinations(range(E), k)
             if all(beats(i, j) for i in S for j in range(E) if j not in S)]
    assert len(found) == 1
    return sorted(found[0], key=lambda i: (-z[i], i))


@pytest.mark.parametrize("ties", [False, True])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_topk_brute_force_on_16_experts(ties, k):
    rng = np.random.default_rng(100 + k + 10 * ties)
    for _ in range(40):
        z = (rng.integers(-3, 4, size=16).astype(np.float64) if ties
             else rng.standard_normal(16))
        assert list(O.topk(z, k)) == _brute_topk(list(z), k)


def test_topk_matches_numpy_lexsort():
    rng = np.random.default_rng(3)
    for E, k in [(64, 8), (128, 8), (128, 4), (256, 8)]:
        z = np.round(rng.standard_normal(E), 1)     # many ties
        expect = np.lexsort((np.arange(E), -z))[:k]
        assert np.array_equal(O.topk(z, k), expect)


def test_topk_from_scores_signed_zero_is_a_tie():
    s = np.array([[0.0, -0.0, -1.0, 0.0]], dtype=np.float32)
    ids, _ = O.topk_from_scores(s, 3, O.GATE_SOFTMAX_RENORM)
    assert list(ids[0]) == [0, 1, 3]


# -------------------------------------------------------------------- gates

def test_gates_against_scipy():
    rng = np.random.default_rng(4)
    for E, k in [(16, 2), (64, 8), (256, 8)]:
        z = rng.standard_normal(E) * 3
        ids = O.topk(z, k)
        p = scipy.special.softmax(z)
        w = O.gate(z, ids, O.GATE_SOFTMAX)
        np.testing.assert_allclose(w, p[ids], rtol=1e-13)
        assert w.sum() < 1.0
        w = O.gate(z, ids, O.GATE_SOFTMAX_RENORM)
        np.testing.assert_allclose(w, scipy.special.softmax(z[ids]), rtol=1e-13)
        np.testing.assert_allclose(w, p[ids] / p[ids].sum(), rtol=1e-12)
        assert abs(w.sum() - 1.0) < 1e-14
        w = O.gate(z, ids, O.GATE_SIGMOID_RENORM)
        sg = scipy.special.expit(z[ids])
        np.testing.assert_allclose(w, sg / sg.sum(), rtol=1e-13)


# ----------------------------------------------------------------- the FFN

def _f32_layer(d, I, E, k, gate, wg, w13, w2, sh=None):
    f = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)
    return O.Layer(d, E, k, I, O.F32, O.F32, gate, f(wg), f(w13), f(w2),
                   sh_w13=f(sh[0]) if sh else None, sh_w2=f(sh[1]) if sh else None)


def test_swiglu_closed_form_gate_rows_first_and_down_layout():
    # one expert, h = e_0: gate pre-activations g_i = W1[i][0], up = W3[i][0] = 1,
    # so a_i = silu(g_i); W2 = [[1,0,0],[0,1,0],[0,0,1],[1,1,1]] reads a back.
    d, I = 4, 3
    g = [1.0, -2.0, 0.5]
    w13 = np.zeros((1, 2 * I, d))
    for i in range(I):
        w13[0, i, 0] = g[i]       # gate rows first
        w13[0, I + i, 0] = 1.0    # then up rows
    w2 = np.zeros((1, d, I))
    w2[0, :I, :] = np.eye(I)
    w2[0, I, :] = 1.0
    wg = np.ones((1, d))
    L = _f32_layer(d, I, 1, 1, O.GATE_SOFTMAX_RENORM, wg, w13, w2)
    h = np.array([[1.0, 0.0, 0.0, 0.0]], dtype=np.float32)
    ids, w, z, y = O.verify(L, h)
    silu = [0.7310585786300049, -0.2384058440442351, 0.31122966560092724]  # x / (1 + e^-x)
    np.testing.assert_allclose(y[0], silu + [sum(silu)], rtol=1e-15, atol=1e-16)
    assert w[0, 0] == 1.0 and z[0, 0] == 1.0


def test_router_scores_and_selection_closed_form():
    # W_g = identity on 4 experts: scores equal h; experts 2 and 0 win.
    d = I = 4
    E, k = 4, 2
    wg = np.eye(E, d)
    w13 = np.zeros((E, 2 * I, d))
    w2 = np.zeros((E, d, I))
    for e in range(E):          # expert e: a_0 = silu(1)*1 at h[0]=1 -> y = (e+1) e_0
        w13[e, 0, 0] = 1.0
        w13[e, I, 0] = 1.0
        w2[e, 0, 0] = e + 1.0
    h = np.array([[1.0, -0.5, 3.0, 0.25]], dtype=np.float32)
    L = _f32_layer(d, I, E, k, O.GATE_SOFTMAX_RENORM, wg, w13, w2)
    ids, w, z, y = O.verify(L, h)
    np.testing.assert_array_equal(z[0], h[0])
    assert list(ids[0]) == [2, 0]
    e3, e1 = math.exp(3.0), math.exp(1.0)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    expect = (e3 * 3.0 + e1 * 1.0) / (e3 + e1) * silu1
    assert abs(y[0, 0] - expect) < 1e-14 and np.all(y[0, 1:] == 0)


def _dense_numpy(wg, w13, w2, h, k, gate, sh=None, ids_given=None):
    """Every expert applied to every token with numpy matmuls, then the top-k
    picked by numpy's lexsort (or the given ids) and gated with scipy."""
    I = w13.shape[1] // 2
    z = h @ wg.T
    out = np.zeros((h.shape[0], w2.shape[1]))
    for t in range(h.shape[0]):
        ids = np.lexsort((np.arange(z.shape[1]), -z[t]))[:k] if ids_given is None else ids_given[t]
        if gate == O.GATE_SOFTMAX:
            wts = scipy.special.softmax(z[t])[ids]
        elif gate == O.GATE_SOFTMAX_RENORM:
            wts = scipy.special.softmax(z[t, ids])
        else:
            s = scipy.special.expit(z[t, ids])
            wts = s / s.sum()
        allo = []
        for e in range(wg.shape[0]):
            gu = w13[e] @ h[t]
            a = gu[:I] * scipy.special.expit(gu[:I]) * gu[I:]
            allo.append(w2[e] @ a)
        out[t] = sum(wts[j] * allo[ids[j]] for j in range(k))
        if sh is not None:
            gu = sh[0] @ h[t]
            out[t] += sh[1] @ (gu[:I] * scipy.special.expit(gu[:I]) * gu[I:])
    return out


@pytest.mark.parametrize("gate", [O.GATE_SOFTMAX, O.GATE_SOFTMAX_RENORM, O.GATE_SIGMOID_RENORM])
@pytest.mark.parametrize("shared", [False, True])
def test_layer_against_dense_numpy_formulation(gate, shared):
    rng = np.random.default_rng(9 + gate + 3 * shared)
    d, I, E, k, n = 24, 10, 6, 2, 5           # d != I catches a transposed W2
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d) * 0.3, f(E, d, I) * 0.3, f(n, d)
    sh = (f(2 * I, d) * 0.3, f(d, I) * 0.3) if shared else None
    L = _f32_layer(d, I, E, k, gate, wg, w13, w2, sh)
    _, _, _, y = O.verify(L, h)
    ref = _dense_numpy(wg.astype(np.float64), w13.astype(np.float64), w2.astype(np.float64),
                       h.astype(np.float64), k, gate,
                       None if sh is None else tuple(s.astype(np.float64) for s in sh))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("gate", [O.GATE_SOFTMAX, O.GATE_SOFTMAX_RENORM, O.GATE_SIGMOID_RENORM])
@pytest.mark.parametrize("shared", [False, True])
def test_given_routing_against_dense_numpy_formulation(gate, shared):
    # verify_routed: any distinct ids in any order (here mostly not the top-k)
    rng = np.random.default_rng(19 + gate + 3 * shared)
    d, I, E, k, n = 24, 10, 7, 3, 6
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d) * 0.3, f(E, d, I) * 0.3, f(n, d)
    sh = (f(2 * I, d) * 0.3, f(d, I) * 0.3) if shared else None
    L = _f32_layer(d, I, E, k, gate, wg, w13, w2, sh)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(n)]).astype(np.int32)
    w, z, y = O.verify_routed(L, h, ids.copy())  # the reference keeps its own copy of the routing
    ref = _dense_numpy(wg.astype(np.float64), w13.astype(np.float64), w2.astype(np.float64),
                       h.astype(np.float64), k, gate,
                       None if sh is None else tuple(s.astype(np.float64) for s in sh),
                       ids_given=ids)
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(z, h.astype(np.float64) @ wg.astype(np.float64).T, rtol=1e-12)
    # a subset of tokens, threads: the same rows
    w2_, z2, y2 = O.verify_routed(L, h, ids[[4, 1]].copy(), tokens=[4, 1], threads=2)
    np.testing.assert_array_equal(y2, y[[4, 1]])


def test_layer_is_linear_in_down_weights_and_invariant_to_expert_relabeling():
    rng = np.random.default_rng(21)
    d, I, E, k, n = 16, 8, 8, 3, 4
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d), f(E, d, I), f(n, d)
    _, _, _, y = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM, wg, w13, w2), h)
    _, _, _, y4 = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM, wg, w13, 4 * w2), h)
    np.testing.assert_allclose(y4, 4 * y, rtol=1e-12)
    p = rng.permutation(E)
    ids0, _, _, _ = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM, wg, w13, w2), h)
    idsp, _, _, yp = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM,
                                         wg[p], w13[p], w2[p]), h)
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-14)
    # new expert i is old expert p[i]
    assert sorted(p[idsp].ravel().tolist()) == sorted(ids0.ravel().tolist())


def test_bf16_layer_reads_the_stored_bits():
    # a bf16 layer equals the f32 layer built from the same (exact) values
    rng = np.random.default_rng(31)
    d, I, E, k, n = 16, 8, 4, 2, 3
    tb = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float32)).to(torch.bfloat16)
    wg, w13, w2, h = tb(E, d), tb(E, 2 * I, d), tb(E, d, I), tb(n, d)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    Lb = O.Layer(d, E, k, I, O.BF16, O.BF16, O.GATE_SOFTMAX, bits(wg), bits(w13), bits(w2))
    _, _, _, yb = O.verify(Lb, bits(h))
    f = lambda t: t.to(torch.float32).numpy()
    _, _, _, yf = O.verify(_f32_layer(d, I, E, k, O.GATE_SOFTMAX, f(wg), f(w13), f(w2)), f(h))
    np.testing.assert_array_equal(yb, yf)


def test_e4m3_block_scale_indexing_one_hot():
    # One nonzero code per matrix, placed in a chosen 128x128 block whose scale
    # differs from every other block: the output isolates scale[row/128][col/128]
    # of both W13 (gate and up) and W2.
    d, I, E = 256, 256, 1
    w13 = np.zeros((1, 2 * I, d), np.uint8)
    w2 = np.zeros((1, d, I), np.uint8)
    s13 = (np.arange(4 * 2, dtype=np.float32).reshape(1, 4, 2) + 1.0) * 0.5  # [2I/128][d/128]
    s2 = (np.arange(2 * 2, dtype=np.float32).reshape(1, 2, 2) + 1.0) * 0.25  # [d/128][I/128]
    i, c, r = 131, 200, 7                    # gate row i (block 1), column c (block 1)
    w13[0, i, c] = 0x38                      # 1.0
    w13[0, I + i, c] = 0x40                  # 2.0 (up row I+i sits in row block 3)
    w2[0, r, i] = 0x30                       # 0.5, row block 0, column block 1
    L = O.Layer(d, E, 1, I, O.F32, O.E4M3, O.GATE_SOFTMAX_RENORM,
                np.zeros((1, d), np.float32), w13, w2, s13, s2)
    h = np.zeros((1, d), np.float32)
    h[0, c] = 0.75
    _, _, _, y = O.verify(L, h)
    g = 1.0 * float(s13[0, 1, 1]) * 0.75
    u = 2.0 * float(s13[0, 3, 1]) * 0.75
    a = g / (1 + math.exp(-g)) * u
    expect = np.zeros(d)
    expect[r] = 0.5 * float(s2[0, 0, 1]) * a
    np.testing.assert_allclose(y[0], expect, rtol=1e-15, atol=0)


def test_shared_expert_adds_with_weight_one():
    rng = np.random.default_rng(41)
    d, I, E, k, n = 8, 4, 4, 2, 3
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d), f(E, d, I), f(n, d)
    sh13, sh2 = f(2 * I, d), f(d, I)
    _, _, _, y0 = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM, wg, w13, w2), h)
    # the shared expert alone: a one-expert layer with k = 1 and weight 1
    _, _, _, ys = O.verify(_f32_layer(d, I, 1, 1, O.GATE_SOFTMAX_RENORM, wg[:1],
                                      sh13[None], sh2[None]), h)
    _, _, _, y1 = O.verify(_f32_layer(d, I, E, k, O.GATE_SIGMOID_RENORM, wg, w13, w2,
                                      (sh13, sh2)), h)
    np.testing.assert_allclose(y1, y0 + ys, rtol=1e-12, atol=1e-14)


def test_token_subset_and_threads_do_not_change_results():
    rng = np.random.default_rng(51)
    d, I, E, k, n = 16, 8, 8, 2, 7
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    L = _f32_layer(d, I, E, k, O.GATE_SOFTMAX, f(E, d), f(E, 2 * I, d), f(E, d, I))
    h = f(n, d)
    ids, w, z, y = O.verify(L, h)
    ids3, w3, z3, y3 = O.verify(L, h, threads=3)
    assert np.array_equal(y, y3) and np.array_equal(ids, ids3)
    sel = [6, 2, 2]
    idss, _, _, ys = O.verify(L, h, tokens=sel, threads=2)
    assert np.array_equal(ys, y[sel]) and np.array_equal(idss, ids[sel])


# -------------------------------------------------------------- union plan

def _check_plan(ids, E, k):
    U, hist, uniq, offs, perm = O.union_plan(ids, E)
    flat = np.asarray(ids).ravel()
    n = flat.size // k
    assert U == len(set(flat.tolist()))
    assert hist.sum() == flat.size
    assert np.all(np.diff(uniq) > 0)
    assert sorted(perm.tolist()) == list(range(flat.size))
    for u in range(U):
        seg = perm[offs[u]:offs[u + 1]]
        assert np.all(flat[seg] == uniq[u]) and np.all(np.diff(seg) > 0)
        assert offs[u + 1] - offs[u] == hist[uniq[u]]
    assert k <= U <= min(E, n * k)
    # "Expert Bytes ...", Fig. 3: U/(nm) lies between 1/n and 1
    assert 1.0 / n - 1e-15 <= U / (n * k) <= 1.0
    return U


def test_union_plan_invariants_random_ids():
    for (n, k, E, seed) in [(1, 2, 16, 1), (4, 2, 16, 2), (8, 8, 64, 3), (16, 8, 128, 4),
                            (64, 8, 256, 5), (13, 4, 128, 6)]:
        ids = torch.stack([torch.randperm(E, generator=torch.Generator().manual_seed(seed * 100 + t))[:k]
                           for t in range(n)]).numpy()
        _check_plan(ids, E, k)


def test_identical_tokens_give_a_union_of_exactly_k():
    row = np.array([5, 17, 3, 250, 9, 0, 128, 77], dtype=np.int32)
    for n in (1, 2, 8, 64):
        ids = np.tile(row, (n, 1))
        assert _check_plan(ids, 256, 8) == 8


def test_disjoint_tokens_give_a_union_of_nk():
    ids = np.arange(64, dtype=np.int32).reshape(8, 8)
    assert _check_plan(ids, 64, 8) == 64


def test_uniform_routing_mean_union_matches_closed_form():
    # independent uniform k-subsets: P(e unused by all n tokens) = (1-k/E)^n,
    # so E[U] = E (1 - (1 - k/E)^n)   ("Expert Bytes ...", Fig. 1: 1 - q^(n-1))
    from moe_expert_ffn_gemv_gb300 import synth
    for n, k, E in [(2, 8, 64), (8, 8, 256), (16, 4, 128), (64, 8, 256)]:
        Us = []
        for rep in range(300):
            ids = synth.uniform_ids(n, k, E, seed=1000 * n + rep).numpy()
            Us.append(O.union_plan(ids, E)[0])
        Us = np.array(Us, dtype=np.float64)
        expect = E * (1 - (1 - k / E) ** n)
        se = Us.std(ddof=1) / math.sqrt(len(Us))
        assert abs(Us.mean() - expect) < 3.5 * se + 1e-9, (n, k, E, Us.mean(), expect, se)


# -------------------------------------------------------------- byte counts

def test_expert_bytes_printed_on_the_pages():
    # "Less Experts, Faster Decoding", Fig. 1(c): one DeepSeek-V3.1 FP8 expert
    # moves 44.04 MB; 3 * 7168 * 2048 * 1 B = 44,040,192 B.
    wb, sb = O.expert_bytes(7168, 2048, O.E4M3)
    assert wb == 44_040_192 and round(wb / 1e6, 2) == 44.04
    assert sb == 4 * (32 * 56 + 56 * 16) == 10_752
    # "The Limits of Speculation", App. A.6: 9.4 MB per Qwen3-30B-A3B bf16 expert
    wb, sb = O.expert_bytes(2048, 768, O.BF16)
    assert wb == 9_437_184 and round(wb / 1e6, 1) == 9.4 and sb == 0
    # and 48 layers of it is about 0.45 GB
    assert round(48 * wb / 1e9, 2) == 0.45


# ------------------------------------------------------------ expert budget
# Verification-time expert budgeting (MoE-Spec, as its abstract is listed on
# "Speculative Decoding for MoE Models: Expert Bytes, ..."; "The Limits of
# Speculation", Sec. 2.4): keep the `budget` most useful experts,
# drop the rest.  Contribution = summed gate weight (a reading).

def test_budget_hand_worked_example():
    # slots (token, slot): expert ids and weights
    #   t0: e0 .625  e1 .375      contributions: e0 .625, e1 .375 + .75 = 1.125,
    #   t1: e1 .75   e2 .25                      e2 .25 + .875 = 1.125, e3 .125
    #   t2: e2 .875  e3 .125      e1 and e2 tie: the lower id ranks first
    ids = np.array([[0, 1], [1, 2], [2, 3]], dtype=np.int32)
    w = np.array([[.625, .375], [.75, .25], [.875, .125]])
    keep, score, kept = O.expert_budget(ids, w, 5, 2)
    assert score.tolist() == [.625, 1.125, 1.125, .125, 0.0]
    assert keep.tolist() == [False, True, True, False, False] and kept == 2
    assert O.expert_budget(ids, w, 5, 1)[0].tolist() == [False, True, False, False, False]
    assert O.expert_budget(ids, w, 5, 3)[0].tolist() == [True, True, True, False, False]
    assert O.expert_budget(ids, w, 5, 0)[2] == 0
    # the kept plan: experts 1 and 2; slots 1, 2 (e1) and 3, 4 (e2)
    U, hist, uniq, offs, perm, w_kept, _ = O.budget_plan(ids, w, 5, 2)
    assert U == 2 and hist.tolist() == [0, 2, 2, 0, 0]
    assert uniq.tolist() == [1, 2] and offs.tolist() == [0, 2, 4] and perm.tolist() == [1, 2, 3, 4]
    assert w_kept.tolist() == [0.0, .375, .75, .25, .875, 0.0]


def test_budget_brute_force_max_total_contribution():
    # dyadic weights (multiples of 1/8) make every sum exact and create ties;
    # the kept set must have the largest total contribution of any set of
    # min(B, U) used experts, and must precede every dropped expert in the
    # order (contribution descending, id ascending)
    rng = np.random.default_rng(77)
    for trial in range(60):
        E = int(rng.integers(4, 11))
        k = int(rng.integers(1, min(E, 4) + 1))
        n = int(rng.integers(1, 6))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(n)]).astype(np.int32)
        w = rng.integers(1, 9, size=(n, k)) / 8.0
        used = sorted(set(ids.ravel().tolist()))
        contrib = {e: math.fsum(w.ravel()[ids.ravel() == e]) for e in used}
        for B in range(0, len(used) + 2):
            keep, score, kept = O.expert_budget(ids, w, E, B)
            m = min(B, len(used))
            assert kept == m and keep.sum() == m
            for e in range(E):
                assert score[e] == contrib.get(e, 0.0)
            best = max((sum(contrib[e] for e in c) for c in itertools.combinations(used, m)),
                       default=0.0)
            assert sum(contrib[e] for e in used if keep[e]) == best
            kept_ids = [e for e in used if keep[e]]
            dropped = [e for e in used if not keep[e]]
            for a in kept_ids:
                for b in dropped:
                    assert contrib[a] > contrib[b] or (contrib[a] == contrib[b] and a < b)
            assert not keep[[e for e in range(E) if e not in contrib]].any()


def test_budget_kept_sets_are_nested():
    from moe_expert_ffn_gemv_gb300 import synth
    ids = synth.uniform_ids(16, 8, 128, seed=5).numpy()
    w = np.random.default_rng(6).random(ids.shape)
    prev = np.zeros(128, dtype=bool)
    for B in range(0, 129):
        keep = O.expert_budget(ids, w, 128, B)[0]
        assert np.all(keep[prev]) and keep.sum() == min(B, O.union_plan(ids, 128)[0])
        prev = keep


def test_budget_at_or_above_the_union_is_the_plain_plan():
    rng = np.random.default_rng(8)
    ids = np.stack([rng.permutation(64)[:8] for _ in range(12)]).astype(np.int32)
    w = rng.random(ids.shape)
    U, hist, uniq, offs, perm = O.union_plan(ids, 64)
    for B in (U, U + 1, 64, 1000):
        Ub, histb, uniqb, offsb, permb, w_kept, keep = O.budget_plan(ids, w, 64, B)
        assert Ub == U and np.array_equal(histb, hist) and np.array_equal(uniqb, uniq)
        assert np.array_equal(offsb, offs) and np.array_equal(permb, perm)
        assert np.array_equal(w_kept, w.ravel())
    # one below the union drops exactly the expert of least contribution
    Ub, histb, uniqb, offsb, permb, w_kept, keep = O.budget_plan(ids, w, 64, U - 1)
    score = O.expert_budget(ids, w, 64, U)[1]
    least = min(uniq.tolist(), key=lambda e: (score[e], -e))
    assert Ub == U - 1 and sorted(set(uniq.tolist()) - set(uniqb.tolist())) == [least]
    assert np.all(w_kept[ids.ravel() == least] == 0.0) and permb.size == ids.size - hist[least]


def test_budget_pass_equals_full_pass_with_dropped_experts_zeroed():
    # a dropped expert's term is absent: the same as running the unbudgeted
    # pass on a layer whose dropped experts have all-zero weights (the router
    # does not read expert weights, so the routing is unchanged)
    rng = np.random.default_rng(61)
    d, I, E, k, n = 16, 8, 12, 3, 6
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d), f(E, d, I), f(n, d)
    sh = (f(2 * I, d), f(d, I))
    for gate in (O.GATE_SOFTMAX, O.GATE_SIGMOID_RENORM):
        L = _f32_layer(d, I, E, k, gate, wg, w13, w2, sh)
        ids, w, _, y_full = O.verify(L, h)
        U = O.union_plan(ids, E)[0]
        for B in (0, 1, 3, U - 1, U):
            idsb, wb, _, yb, keep = O.verify_budget(L, h, B, threads=2)
            assert np.array_equal(idsb, ids) and np.array_equal(wb, w)
            assert np.array_equal(keep, O.expert_budget(ids, w, E, B)[0])
            w13z, w2z = w13.copy(), w2.copy()
            w13z[~keep] = 0.0
            w2z[~keep] = 0.0
            _, _, _, yz = O.verify(_f32_layer(d, I, E, k, gate, wg, w13z, w2z, sh), h)
            assert np.array_equal(yb, yz), (gate, B)
            if B >= U:
                assert np.array_equal(yb, y_full)
            # a token subset gives the same rows (the kept set still comes from all tokens)
            sel = [5, 0, 5]
            _, _, _, ys, keeps = O.verify_budget(L, h, B, tokens=sel, threads=2)
            assert np.array_equal(keeps, keep) and np.array_equal(ys, yb[sel])


def test_budget_zero_leaves_only_the_shared_expert():
    rng = np.random.default_rng(62)
    d, I, E, k, n = 8, 4, 6, 2, 5
    f = lambda *s: rng.standard_normal(s).astype(np.float32)
    wg, w13, w2, h = f(E, d), f(E, 2 * I, d), f(E, d, I), f(n, d)
    sh13, sh2 = f(2 * I, d), f(d, I)
    y0 = O.verify_budget(_f32_layer(d, I, E, k, O.GATE_SOFTMAX, wg, w13, w2), h, 0)[3]
    assert np.array_equal(y0, np.zeros((n, d)))
    ys = O.verify(_f32_layer(d, I, 1, 1, O.GATE_SOFTMAX_RENORM, wg[:1], sh13[None], sh2[None]),
                  h)[3]
    y1 = O.verify_budget(_f32_layer(d, I, E, k, O.GATE_SOFTMAX, wg, w13, w2, (sh13, sh2)), h, 0)[3]
    assert np.array_equal(y1, ys)


def test_budget_e4m3_layer_zeroed_codes():
    # the same identity on an FP8 layer with block scales: zero codes (+0)
    # for the dropped experts, scales untouched
    from moe_expert_ffn_gemv_gb300 import synth
    from tests.helpers import np_bytes, oracle_layer
    cfg = synth.LayerConfig("fp8-budget", 256, 8, 3, 128, synth.BF16, synth.E4M3,
                            synth.GATE_SIGMOID_RENORM, n_shared=1)
    layer = synth.make_layer(cfg, seed=12)
    h = np_bytes(synth.make_hidden(cfg, 4, seed=13))
    L = oracle_layer(layer)
    U = O.union_plan(O.verify(L, h)[0], 8)[0]
    assert U >= 4
    for B in (1, 3):
        _, _, _, yb, keep = O.verify_budget(L, h, B)
        lz = synth.make_layer(cfg, seed=12)
        lz.w13[torch.from_numpy(~keep)] = 0
        lz.w2[torch.from_numpy(~keep)] = 0
        _, _, _, yz = O.verify(oracle_layer(lz), h)
        assert np.array_equal(yb, yz)


# ------------------------------------------------ pre-verification selection
# "Making Every Verified Token Count", Sec. 3 (EVICT) and "Less Experts,
# Faster Decoding", Sec. 4.2 (EcoSpec).  Trees: node 0 is the root
# (factor 1), parent[v] < v.

def _random_tree(rng, K, max_children=3):
    par = [-1]
    for v in range(1, K):
        par.append(int(rng.integers(0, v)) if rng.random() < 0.7 else v - 1)
    return np.array(par, dtype=np.int32)


def _ancestor_closed(par, nodes):
    s = set(int(v) for v in nodes)
    return all(v == 0 or par[v] in s for v in s)


def test_tree_scores_chain_and_log_sum():
    # a chain with constant acceptance alpha: node i scores alpha^i
    K, a = 12, 0.75
    par = np.arange(-1, K - 1, dtype=np.int32)
    q = np.full(K, a, dtype=np.float32)
    s = O.tree_scores(par, q)
    np.testing.assert_allclose(s, [a ** i for i in range(K)], rtol=1e-14)
    # any tree: the score is exp(sum of log q over the path), the root excluded
    rng = np.random.default_rng(5)
    par = _random_tree(rng, 30)
    q = rng.uniform(0.05, 1.0, 30).astype(np.float32)
    s = O.tree_scores(par, q)
    for v in range(30):
        lg, u = 0.0, v
        while u > 0:
            lg += math.log(float(q[u]))
            u = par[u]
        assert abs(s[v] - math.exp(lg)) <= 1e-13 * math.exp(lg)


def test_evict_chain_closed_forms():
    # geometric chain: E_hat[A(T_k)] = (1 - a^k) / (1 - a); a constant cost
    # makes the whole tree best (k* = K); a cost proportional to k makes the
    # root alone best (k* = 1); C(k) = c0 + c1 k has the closed-form argmax
    K, a = 16, 0.8
    par = np.arange(-1, K - 1, dtype=np.int32)
    q = np.full(K, a, dtype=np.float32)
    aa = float(np.float32(a))
    closed = np.array([(1 - aa ** k) / (1 - aa) for k in range(1, K + 1)])
    ks, order, exp_len, util = O.evict_select(par, q, np.full(K, 3.0))
    assert ks == K and order.tolist() == list(range(K))
    np.testing.assert_allclose(exp_len, closed, rtol=1e-13)
    assert O.evict_select(par, q, 2.5 * np.arange(1, K + 1))[0] == 1
    for c0, c1 in [(10.0, 1.0), (4.0, 1.0), (1.0, 1.0), (30.0, 0.5)]:
        f = closed / (c0 + c1 * np.arange(1, K + 1))
        assert O.evict_select(par, q, c0 + c1 * np.arange(1, K + 1))[0] == int(np.argmax(f)) + 1


def test_evict_top_k_is_the_best_subtree_brute_force():
    # Sec. 3.2.1: the top-k nodes by cumulative score form a valid (ancestor-
    # closed) subtree whose estimated accepted length is the largest of any
    # k-node subtree containing the root
    rng = np.random.default_rng(9)
    for trial in range(25):
        K = int(rng.integers(2, 10))
        par = _random_tree(rng, K)
        q = rng.uniform(0.05, 1.0, K).astype(np.float32)
        if trial % 3 == 0:
            q[:] = 0.5  # ties everywhere
        s = O.tree_scores(par, q)
        ks, order, exp_len, util = O.evict_select(par, q, np.ones(K))
        for k in range(1, K + 1):
            assert _ancestor_closed(par, order[:k])
            best = max(sum(s[list(c)]) for c in itertools.combinations(range(K), k)
                       if 0 in c and _ancestor_closed(par, c))
            assert abs(exp_len[k - 1] - best) <= 1e-12 * best


def test_evict_utility_and_ties():
    par = np.array([-1, 0, 0, 1, 2], dtype=np.int32)
    q = np.array([1.0, 0.5, 0.5, 0.5, 0.5], dtype=np.float32)
    # scores 1, .5, .5, .25, .25: equal scores rank by lower node index
    ks, order, exp_len, util = O.evict_select(par, q, [1.0, 1.5, 2.0, 2.5, 3.0])
    assert order.tolist() == [0, 1, 2, 3, 4]
    assert exp_len.tolist() == [1.0, 1.5, 2.0, 2.25, 2.5]
    assert util.tolist() == [1.0, 1.0, 1.0, 0.9, 2.5 / 3.0]
    assert ks == 1  # three-way tie at utility 1: the smallest k
    # scaling every cost by a constant leaves k* alone
    rng = np.random.default_rng(10)
    par = _random_tree(rng, 40)
    q = rng.uniform(0.1, 1.0, 40).astype(np.float32)
    cost = 100 + 3.0 * np.arange(1, 41) + rng.uniform(0, 5, 40)
    assert O.evict_select(par, q, cost)[0] == O.evict_select(par, q, 4.0 * cost)[0]


def test_ecospec_hand_worked_example():
    # root {0,1}; 1 {1,2}; 2 {3,4}; 3 {2,5}; 4 {6,7}; 5 {3,8}; P = 1, .5, .25, .25, .125, .125
    # step 1: costs 2,3,4,4,5,5 -> node 0;  B = {0,1}
    # step 2: node 1 costs 1 (.5)                -> node 1;  B = {0,1,2}
    # step 3: node 2 costs 2 (.125), node 3 costs 1 (.25)   -> node 3;  B += {5}
    # step 4: node 2 (.125) beats 4 (.0625) and 5 (.125/3)  -> node 2;  B += {3,4}
    par = [-1, 0, 0, 1, 1, 2]
    q = [1, .5, .25, .5, .25, .5]
    pred = np.array([[[0, 1]], [[1, 2]], [[3, 4]], [[2, 5]], [[6, 7]], [[3, 8]]])
    sel, buf, cnt = O.ecospec_select(par, q, pred, 16, 4, 1e-6)
    assert sel.tolist() == [0, 1, 3, 2] and cnt == 6
    assert np.flatnonzero(buf[0]).tolist() == [0, 1, 2, 3, 4, 5]
    # gamma = 3: confidence order would take node 2 (union 5); EcoSpec takes 3 (union 4)
    sel, buf, cnt = O.ecospec_select(par, q, pred, 16, 3, 1e-6)
    assert sel.tolist() == [0, 1, 3] and cnt == 4
    # eps: a free node wins over a costlier one of larger P when P0/eps > P1/(c+eps)
    sel, _, _ = O.ecospec_select([-1, 0, 0], [1, .9, .1], np.array([[[0]], [[1]], [[0]]]), 4, 2, 1e-3)
    assert sel.tolist() == [0, 2]
    sel, _, _ = O.ecospec_select([-1, 0, 0], [1, .9, .1], np.array([[[0]], [[1]], [[0]]]), 4, 2, 100.0)
    assert sel.tolist() == [0, 1]


def test_ecospec_reduces_to_confidence_order_without_new_experts():
    # identical predicted sets, or a buffer that already holds every expert:
    # every cost after the first pick is 0, so the order is by P (ties to
    # the lower index), the same as EVICT's ranking
    rng = np.random.default_rng(11)
    for trial in range(10):
        K, L, E, kp = 24, 3, 32, 4
        par = _random_tree(rng, K)
        q = rng.uniform(0.1, 1.0, K).astype(np.float32)
        if trial % 2:
            q[:] = 0.5  # siblings tie: the lower index goes first
        order = O.evict_select(par, q, np.ones(K))[1]
        same = np.broadcast_to(rng.integers(0, E, (1, L, kp)), (K, L, kp))
        for gamma in (1, 5, K, K + 3):
            sel, buf, cnt = O.ecospec_select(par, q, same, E, gamma, 1e-6)
            assert sel.tolist() == order[:min(gamma, K)].tolist()
        pred = rng.integers(0, E, (K, L, kp))
        full = np.ones((L, E), dtype=np.uint8)
        sel, buf, cnt = O.ecospec_select(par, q, pred, E, 7, 1e-6, buf0=full)
        assert sel.tolist() == order[:7].tolist() and cnt == L * E


def test_ecospec_selection_is_prefix_closed_and_buffer_is_the_union():
    # "Less Experts, Faster Decoding", Sec. 4.2 (prefix consistency): a child
    # never outscores its parent under the same buffer, so the selected set
    # stays ancestor-closed; the final buffer is B0 plus the predicted sets
    # of the selected nodes
    rng = np.random.default_rng(12)
    for trial in range(20):
        K, L, E, kp = int(rng.integers(2, 40)), int(rng.integers(1, 4)), 64, 6
        par = _random_tree(rng, K)
        q = rng.uniform(0.05, 1.0, K).astype(np.float32)
        pred = rng.integers(0, E, (K, L, kp))
        b0 = (rng.random((L, E)) < 0.2).astype(np.uint8)
        gamma = int(rng.integers(1, K + 2))
        sel, buf, cnt = O.ecospec_select(par, q, pred, E, gamma, 1e-6, buf0=b0)
        assert len(set(sel.tolist())) == len(sel) == min(gamma, K)
        for i in range(1, len(sel) + 1):
            assert _ancestor_closed(par, sel[:i])
        want = b0.astype(bool).copy()
        for v in sel:
            for l in range(L):
                want[l, pred[v, l]] = True
        assert np.array_equal(buf, want) and cnt == want.sum()


def test_layer_mean_union_closed_forms():
    # "The Limits of Speculation", eq. (5), over per-layer oracle unions
    from moe_expert_ffn_gemv_gb300 import draft_length as D
    from moe_expert_ffn_gemv_gb300 import synth
    row = np.array([3, 9, 27, 81, 100, 5, 6, 7], dtype=np.int32)
    assert D.layer_mean_union([O.union_plan(np.tile(row, (n, 1)), 128)[0]
                               for n in (1, 4, 16)]) == 8
    n, k, E, Lyr = 6, 8, 128, 400
    us = [O.union_plan(synth.uniform_ids(n, k, E, seed=9000 + l).numpy(), E)[0]
          for l in range(Lyr)]
    expect = E * (1 - (1 - k / E) ** n)
    se = np.std(us, ddof=1) / math.sqrt(Lyr)
    assert abs(D.layer_mean_union(us) - expect) < 3.5 * se
