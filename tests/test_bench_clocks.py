"""The bench's host-side rules: rejecting a timed region by its clock
samples (a hardware or thermal slowdown, or SM clocks well below their
maximum with no reason reported, i.e. a leftover clock lock; power capping
alone is kept), and the source hash that gates the recorded DRAM traffic."""
import bench


def test_clean_and_power_capped_regions_are_kept():
    assert not bench.clocks_rejected({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []})
    assert not bench.clocks_rejected({"sm_mhz": 1492, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"]})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]})


def test_slowdowns_and_unexplained_low_clocks_are_rejected():
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": [r]})
    assert bench.clocks_rejected({"sm_mhz": 1200, "sm_max_mhz": 2070, "reasons": []})


def test_code_hash_ignores_comments_and_keeps_code_and_literals():
    # the recorded DRAM traffic is tied to the kernels' code: a comment edit
    # keeps the hash, a code edit (or a literal's text) changes it
    src = 'int a = 1; // one\n/* block\n comment */ const char *s = "x // y";\nint b;\n'
    assert bench.strip_comments(src) == 'int a = 1; const char *s = "x // y"; int b;'
    assert bench.strip_comments("a /* x */ b") == "a b"
    assert bench.strip_comments("c = '/'; // q") == "c = '/';"
    assert bench.strip_comments('s = "a\\"//b";') == 's = "a\\"//b";'
    assert bench.strip_comments(src.replace("// one", "// two")) == bench.strip_comments(src)
    assert bench.strip_comments(src.replace("int b;", "int c;")) != bench.strip_comments(src)
    assert len(bench.code_hash(bench.DEDUP_KERNEL_SOURCES)) == 16
