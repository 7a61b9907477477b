"""The C-ABI library loads and exports every symbol include/moe_verify.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_verify.h")


@pytest.fixture(scope="module")
def lib():
    from moe_expert_ffn_gemv_gb300 import build
    build.build()
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_four_calls_of_the_path():
    names = declared_functions()
    for f in ("moe_route_topk", "moe_union_plan", "moe_verify_dedup", "moe_verify_perslot"):
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    cdll = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(cdll, name), name
    assert sorted(lib.EXPORTED) == declared_functions()


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    ours = sorted(l.split()[-1] for l in out.splitlines() if " T " in l and "moe_" in l)
    assert ours == declared_functions()


def _desc(lib, **kw):
    base = dict(d=7168, n_experts=256, top_k=8, inter=2048, n_shared=1, n_max=64,
                act_dtype=lib.MOE_BF16, w_dtype=lib.MOE_E4M3_B128,
                gate=lib.MOE_GATE_SIGMOID_RENORM, wait_timeout_us=0)
    base.update(kw)
    return lib.moe_layer_desc(**base)


def test_expert_bytes_through_the_abi(lib):
    # one DeepSeek-V3 FP8 expert: 44,040,192 weight bytes + 10,752 scale bytes
    assert lib.moe_expert_bytes(_desc(lib)) == (44_040_192, 10_752)
    # one Qwen3-30B-A3B bf16 expert: 9,437,184 bytes
    d = _desc(lib, d=2048, n_experts=128, inter=768, n_shared=0, w_dtype=lib.MOE_BF16)
    assert lib.moe_expert_bytes(d) == (9_437_184, 0)


def test_packed_bytes_through_the_abi(lib):
    # DeepSeek-V3 FP8: W13 2I x d = 4096 x 7168 bytes in 64 x 14 tiles of 64 rows x 512 bytes,
    # W2 d x I = 7168 x 2048 bytes in 112 x 4 tiles; each tile carries 32 bytes of scales
    assert lib.moe_packed_bytes(_desc(lib)) == (4096 * 7168 + 64 * 14 * 32,
                                                7168 * 2048 + 112 * 4 * 32)
    # a ragged E4M3 shape: K = 640 bytes is 2 tiles a row block, K = 384 one
    assert lib.moe_packed_bytes(_desc(lib, d=640, inter=384)) == (768 * 640 + 12 * 2 * 32,
                                                                 640 * 384 + 10 * 1 * 32)
    # bf16: the row-major size
    d = _desc(lib, d=2048, n_experts=128, inter=768, n_shared=0, w_dtype=lib.MOE_BF16)
    assert lib.moe_packed_bytes(d) == (2 * 768 * 2048 * 2, 2048 * 768 * 2)


def test_workspace_bytes_and_desc_checks(lib):
    assert lib.moe_workspace_bytes(_desc(lib)) > 0
    bad = [dict(d=0), dict(top_k=0), dict(top_k=300), dict(n_experts=-1), dict(n_shared=-1),
           dict(act_dtype=9), dict(w_dtype=7), dict(gate=5), dict(wait_timeout_us=-3)]
    for kw in bad:
        assert lib.moe_workspace_bytes(_desc(lib, **kw)) == 0, kw
    unsupported = [dict(n_experts=512, top_k=8), dict(top_k=33, n_experts=64), dict(n_max=65),
                   dict(n_shared=2), dict(d=7200), dict(inter=2000), dict(act_dtype=lib.MOE_F32),
                   dict(w_dtype=lib.MOE_BF16, d=2080)]
    for kw in unsupported:
        with pytest.raises(lib.MoeError) as e:
            lib.moe_expert_bytes(_desc(lib, **kw))
        assert e.value.status == lib.MOE_ERR_UNSUPPORTED, kw


def test_launching_calls_reject_bad_arguments_before_any_launch(lib):
    D = _desc(lib)
    P = ctypes.c_void_p
    r = lib._lib
    s0 = P(0)
    assert r.moe_route_topk(ctypes.byref(D), None, None, 4, None, None, None, s0) == lib.MOE_ERR_INVALID_ARG
    # misaligned pointers
    x = P(0x1008)
    assert r.moe_route_topk(ctypes.byref(D), x, x, 4, x, x, x, s0) == lib.MOE_ERR_ALIGNMENT
    # n beyond n_max
    y = P(0x1000)
    assert r.moe_route_topk(ctypes.byref(D), y, y, 65, y, y, y, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_topk_from_logits(ctypes.byref(D), y, -1, y, y, s0) == lib.MOE_ERR_INVALID_ARG
    W = lib.moe_expert_weights(0x1000, 0x1000, 0x1000, 0x1000)
    plan = lib.moe_plan(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    nb = lib.moe_workspace_bytes(D)
    # workspace too small
    assert r.moe_verify_dedup(ctypes.byref(D), ctypes.byref(W), y, 8, y, y, ctypes.byref(plan), y,
                              nb - 1, y, s0) == lib.MOE_ERR_WORKSPACE
    # E4M3 weights packed without their scales
    z = P(0x2000)
    assert r.moe_pack_expert_weights(ctypes.byref(D), y, y, None, None, 2, z, z,
                                     s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_pack_expert_weights(ctypes.byref(D), y, y, x, y, 2, z, z,
                                     s0) == lib.MOE_ERR_ALIGNMENT
    # missing shared expert when the desc has one
    W3 = lib.moe_expert_weights(0x1000, 0x1000, None, None)
    assert r.moe_verify_perslot(ctypes.byref(D), ctypes.byref(W3), y, 8, y, y, y, nb, y,
                                s0) == lib.MOE_ERR_INVALID_ARG
    # plan without arrays
    empty_plan = lib.moe_plan(None, None, None, None, None, None)
    assert r.moe_union_plan(ctypes.byref(D), y, 8, ctypes.byref(empty_plan), None,
                            s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_selftest_bounded_wait(y, 0, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_last_error(None, s0) == lib.MOE_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(8):
        assert lib.moe_status_string(s) not in ("", "unknown status")
    assert lib.moe_status_string(99) == "unknown status"


def test_budgeted_plan_calls_reject_bad_arguments_before_any_launch(lib):
    D = _desc(lib)
    P = ctypes.c_void_p
    r = lib._lib
    s0 = P(0)
    y = P(0x1000)
    plan = lib.moe_plan(0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    nb = lib.moe_workspace_bytes(D)
    # a negative budget
    assert r.moe_union_plan_budgeted(ctypes.byref(D), y, y, 8, -1, ctypes.byref(plan), y, None,
                                     None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_route_plan_budgeted(ctypes.byref(D), y, y, 8, -2, y, y, y, ctypes.byref(plan),
                                     y, None, y, nb, s0) == lib.MOE_ERR_INVALID_ARG
    # missing weights or kept-weight output
    assert r.moe_union_plan_budgeted(ctypes.byref(D), y, None, 8, 4, ctypes.byref(plan), y, None,
                                     None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_union_plan_budgeted(ctypes.byref(D), y, y, 8, 4, ctypes.byref(plan), None, None,
                                     None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_route_plan_budgeted(ctypes.byref(D), y, y, 8, 4, y, y, y, ctypes.byref(plan),
                                     None, None, y, nb, s0) == lib.MOE_ERR_INVALID_ARG
    # misaligned kept weights; n beyond n_max; a workspace below its header
    x = P(0x1004)
    assert r.moe_union_plan_budgeted(ctypes.byref(D), y, y, 8, 4, ctypes.byref(plan), x, None,
                                     None, s0) == lib.MOE_ERR_ALIGNMENT
    assert r.moe_union_plan_budgeted(ctypes.byref(D), y, y, 65, 4, ctypes.byref(plan), y, None,
                                     None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_route_plan_budgeted(ctypes.byref(D), y, y, 8, 4, y, y, y, ctypes.byref(plan),
                                     y, None, y, 255, s0) == lib.MOE_ERR_WORKSPACE


def test_selection_calls_reject_bad_arguments_before_any_launch(lib):
    P = ctypes.c_void_p
    r = lib._lib
    s0 = P(0)
    y = P(0x1000)
    x = P(0x1004)
    # EVICT: node count out of range, missing outputs, misaligned arrays; no trees is a no-op
    assert r.moe_evict_select(y, y, 2, 0, y, y, None, None, y, None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_evict_select(y, y, 2, 257, y, y, None, None, y, None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_evict_select(y, y, 2, 8, y, None, None, None, y, None, s0) == lib.MOE_ERR_INVALID_ARG
    assert r.moe_evict_select(y, x, 2, 8, y, y, None, None, y, None, s0) == lib.MOE_ERR_ALIGNMENT
    assert r.moe_evict_select(None, None, 0, 8, None, None, None, None, None, None, s0) == lib.MOE_OK
    # EcoSpec: eps must be positive; gamma >= 0; bitsets beyond shared memory are unsupported
    eco = lambda *a: r.moe_ecospec_select(*a)
    assert eco(y, y, y, 1, 8, 1, 64, 4, 2, ctypes.c_double(0.0), None, y, None, y, None,
               s0) == lib.MOE_ERR_INVALID_ARG
    assert eco(y, y, y, 1, 8, 1, 64, 4, -1, ctypes.c_double(1e-6), None, y, None, y, None,
               s0) == lib.MOE_ERR_INVALID_ARG
    assert eco(y, y, y, 1, 256, 64, 256, 8, 4, ctypes.c_double(1e-6), None, y, None, y, None,
               s0) == lib.MOE_ERR_UNSUPPORTED
    assert eco(y, y, None, 1, 8, 1, 64, 4, 2, ctypes.c_double(1e-6), None, y, None, y, None,
               s0) == lib.MOE_ERR_INVALID_ARG
    assert eco(y, y, y, 1, 8, 1, 64, 4, 2, ctypes.c_double(1e-6), x, y, None, y, None,
               s0) == lib.MOE_ERR_ALIGNMENT


def test_binding_fails_loudly_without_the_library(tmp_path):
    # a copy of the package with no libmoe_verify.so: importing the binding
    # must raise, not fall back to anything on the CPU
    import shutil
    import subprocess
    import sys
    src = os.path.join(ROOT, "moe_expert_ffn_gemv_gb300")
    dst = tmp_path / "moe_expert_ffn_gemv_gb300"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.so", "__pycache__", "csrc"))
    code = ("import sys; sys.path.insert(0, sys.argv[1])\n"
            "try:\n"
            "    import moe_expert_ffn_gemv_gb300.binding\n"
            "except ImportError as e:\n"
            "    print('IMPORT-ERROR', 'no CPU fallback' in str(e))\n"
            "else:\n"
            "    print('IMPORTED')\n")
    r = subprocess.run([sys.executable, "-c", code, str(tmp_path)], capture_output=True, text=True,
                       timeout=300)
    assert r.stdout.strip() == "IMPORT-ERROR True", (r.stdout, r.stderr[-2000:])
