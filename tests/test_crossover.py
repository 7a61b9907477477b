"""The dedup-vs-per-slot criterion and crossover, against the numbers the
pages print (tests/golden/expertbytes_table1.txt) and closed cases."""
import os

from moe_expert_ffn_gemv_gb300 import crossover as X

GOLD = os.path.join(os.path.dirname(__file__), "golden", "expertbytes_table1.txt")


def rows():
    for line in open(GOLD):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        yield f[0], f[1], [float(x) for x in f[2:]]


def test_r_is_the_bandwidth_ratio_to_printed_precision():
    for eng, model, v in rows():
        bs2, bd2, r2, u2, bs8, bd8, r8, u8 = v
        assert abs(X.r_ratio(bd2, bs2) - r2) <= 0.006, (eng, model, 2)
        assert abs(X.r_ratio(bd8, bs8) - r8) <= 0.006, (eng, model, 8)


def test_criterion_reproduces_which_kernel_the_table_says_is_faster():
    # abstract: deduplication is faster only from 5 to 8 tokens per pass, or
    # never -> at n = 2 the per-slot kernel wins on every row
    for eng, model, v in rows():
        bs2, bd2, r2, u2, bs8, bd8, r8, u8 = v
        assert not X.dedup_faster(u2, r2), (eng, model)
    faster8 = {(e, m): X.dedup_faster(v[7], v[6]) for e, m, v in rows()}
    assert faster8[("llama.cpp-CUDA", "OLMoE")] and faster8[("llama.cpp-CUDA", "gpt-oss")]
    assert not faster8[("llama.cpp-CUDA", "DeepSeek-V2-Lite")]
    assert not faster8[("llama.cpp-Metal", "Qwen3")]


def test_criterion_equals_timing_comparison():
    # u_bar < r  <=>  t_dedup < t_slot, for any positive bytes and times
    k, b = 8, 1000
    for n, U, td, ts in [(2, 15, 1.0, 1.2), (8, 39, 3.0, 2.9), (1, 8, 1.0, 1.0), (64, 173, 2.0, 9.0)]:
        a = X.analyse([dict(n=n, U=U, t_dedup=td, t_slot=ts)], k, b)[0]
        assert a["criterion_dedup_faster"] == a["measured_dedup_faster"]


def test_u_bar_bounds_and_shared_expert():
    # 1/n <= U/(nm) <= 1 ("Expert Bytes ...", Fig. 3)
    assert X.u_bar(8, 8, 8) == 1 / 8 and X.u_bar(64, 8, 8) == 1.0
    assert X.u_bar(39, 8, 8, n_shared=1) == 40 / 72
    assert X.crossover([1, 2, 3], [5, 4, 2], [5, 4.5, 3]) == 2
    assert X.crossover([1, 2], [5, 6], [4, 5]) is None
