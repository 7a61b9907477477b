"""Plain CPU oracle for the MoE verification-pass layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  It shares no
code with the CUDA library (``moe_expert_ffn_gemv_gb300``) and imports
nothing from it.

The arithmetic lives in ``moe_oracle.c`` (double precision, one token at a
time); this module compiles it with gcc and marshals numpy arrays into it.
Every function is pinned by ``tests/test_oracle_pins.py`` against facts the
pages or mathematics fix (closed forms, brute force, library routines,
invariants, the byte counts the pages print).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liborc.so")
# A test may point this at a deliberately broken build of the oracle to show
# that the pins catch the break.
_LIB_OVERRIDE = os.environ.get("MOE_ORACLE_LIB")

# element types and gate variants, as numbered in moe_oracle.c
F32, BF16, E4M3 = 0, 1, 2
GATE_SOFTMAX, GATE_SOFTMAX_RENORM, GATE_SIGMOID_RENORM = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liborc.so next to it (plain -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


class _Layer(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("n_experts", ctypes.c_int), ("top_k", ctypes.c_int),
                ("inter", ctypes.c_int), ("n_shared", ctypes.c_int), ("act_type", ctypes.c_int),
                ("w_type", ctypes.c_int), ("gate", ctypes.c_int),
                ("wg", ctypes.c_void_p), ("w13", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("s13", ctypes.c_void_p), ("s2", ctypes.c_void_p),
                ("sh_w13", ctypes.c_void_p), ("sh_w2", ctypes.c_void_p),
                ("sh_s13", ctypes.c_void_p), ("sh_s2", ctypes.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_LIB_OVERRIDE or build())
        p = ctypes.c_void_p
        L.orc_e4m3_to_double.restype = ctypes.c_double
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_router_scores.argtypes = [ctypes.POINTER(_Layer), p, p]
        L.orc_topk.argtypes = [p, ctypes.c_int, ctypes.c_int, p]
        L.orc_gate.argtypes = [p, ctypes.c_int, p, ctypes.c_int, ctypes.c_int, p]
        L.orc_verify.restype = ctypes.c_int
        L.orc_verify.argtypes = [ctypes.POINTER(_Layer), p, p, ctypes.c_int, ctypes.c_int,
                                 p, p, p, p]
        L.orc_verify_routed.restype = ctypes.c_int
        L.orc_verify_routed.argtypes = [ctypes.POINTER(_Layer), p, p, ctypes.c_int, ctypes.c_int,
                                        p, p, p, p]
        L.orc_topk_from_scores.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, p, p]
        L.orc_union_plan.restype = ctypes.c_int
        L.orc_union_plan.argtypes = [p, ctypes.c_int, ctypes.c_int, p, p, p, p]
        L.orc_expert_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_int64),
                                       ctypes.POINTER(ctypes.c_int64)]
        L.orc_expert_budget.restype = ctypes.c_int
        L.orc_expert_budget.argtypes = [p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, p]
        L.orc_budget_plan.restype = ctypes.c_int
        L.orc_budget_plan.argtypes = [p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      p, p, p, p, p, p, p]
        L.orc_tree_scores.argtypes = [p, p, ctypes.c_int, p]
        L.orc_evict_select.restype = ctypes.c_int
        L.orc_evict_select.argtypes = [p, p, ctypes.c_int, p, p, p, p]
        L.orc_ecospec_select.restype = ctypes.c_int
        L.orc_ecospec_select.argtypes = [p, p, p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, p, ctypes.c_double, p, p]
        L.orc_verify_budget.restype = ctypes.c_int
        L.orc_verify_budget.argtypes = [ctypes.POINTER(_Layer), p, ctypes.c_int, p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, p, p, p, p, p]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


@dataclass
class Layer:
    """A MoE layer as the oracle reads it.

    Arrays hold the stored bytes: float32 for F32, uint16 bit patterns for
    BF16, uint8 codes for E4M3 (with float32 block scales).  Shapes:
    wg [N][d], w13 [N][2I][d] (gate rows first), w2 [N][d][I],
    s13 [N][2I/128][d/128], s2 [N][d/128][I/128]; shared expert without the
    leading N.
    """
    d: int
    n_experts: int
    top_k: int
    inter: int
    act_type: int
    w_type: int
    gate: int
    wg: np.ndarray
    w13: np.ndarray
    w2: np.ndarray
    s13: Optional[np.ndarray] = None
    s2: Optional[np.ndarray] = None
    sh_w13: Optional[np.ndarray] = None
    sh_w2: Optional[np.ndarray] = None
    sh_s13: Optional[np.ndarray] = None
    sh_s2: Optional[np.ndarray] = None

    @property
    def n_shared(self) -> int:
        return 0 if self.sh_w13 is None else 1

    def _c(self) -> _Layer:
        return _Layer(self.d, self.n_experts, self.top_k, self.inter, self.n_shared,
                      self.act_type, self.w_type, self.gate,
                      _ptr(self.wg), _ptr(self.w13), _ptr(self.w2), _ptr(self.s13),
                      _ptr(self.s2), _ptr(self.sh_w13), _ptr(self.sh_w2),
                      _ptr(self.sh_s13), _ptr(self.sh_s2))


def decode_e4m3(codes) -> np.ndarray:
    """Decode E4M3 codes (uint8) to float64 from the OCP bit-field definition."""
    codes = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_e4m3_to_double
    return np.array([f(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def bf16_to_double(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    f = lib().orc_bf16_to_double
    return np.array([f(int(b)) for b in bits.ravel()], dtype=np.float64).reshape(bits.shape)


def topk(z: np.ndarray, k: int) -> np.ndarray:
    z = np.ascontiguousarray(z, dtype=np.float64)
    ids = np.zeros(k, dtype=np.int32)
    lib().orc_topk(_ptr(z), z.shape[0], k, _ptr(ids))
    return ids


def gate(z: np.ndarray, ids: np.ndarray, mode: int) -> np.ndarray:
    z = np.ascontiguousarray(z, dtype=np.float64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.zeros(ids.shape[0], dtype=np.float64)
    lib().orc_gate(_ptr(z), z.shape[0], _ptr(ids), ids.shape[0], mode, _ptr(w))
    return w


def router_scores(layer: Layer, h_row: np.ndarray) -> np.ndarray:
    """Scores of one token given as float64 values (already decoded)."""
    h_row = np.ascontiguousarray(h_row, dtype=np.float64)
    z = np.zeros(layer.n_experts, dtype=np.float64)
    c = layer._c()
    lib().orc_router_scores(ctypes.byref(c), _ptr(h_row), _ptr(z))
    return z


def verify(layer: Layer, h: np.ndarray, tokens=None, threads: int = 1):
    """The layer's outputs for the listed tokens (all tokens if None).

    h holds the stored hidden states [n][d] (float32, or uint16 bf16 bits).
    Returns (ids [m][k] int32, w [m][k] f64, z [m][N] f64, y [m][d] f64),
    row i for token tokens[i].
    """
    h = np.ascontiguousarray(h)
    n = h.shape[0]
    if tokens is None:
        tok = None
        m = n
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        assert tok.size == 0 or (tok.min() >= 0 and tok.max() < n)
        m = tok.shape[0]
    ids = np.zeros((m, layer.top_k), dtype=np.int32)
    w = np.zeros((m, layer.top_k), dtype=np.float64)
    z = np.zeros((m, layer.n_experts), dtype=np.float64)
    y = np.zeros((m, layer.d), dtype=np.float64)
    c = layer._c()
    lib().orc_verify(ctypes.byref(c), _ptr(h), _ptr(tok), m, threads,
                     _ptr(ids), _ptr(w), _ptr(z), _ptr(y))
    return ids, w, z, y


def verify_routed(layer: Layer, h: np.ndarray, ids: np.ndarray, tokens=None, threads: int = 1):
    """verify() on a given routing: ids [m][k] int32 (row i the experts of
    token tokens[i], all tokens if None; distinct ids in [0, N)) replace the
    top-k.  Returns (w [m][k] f64, the gate of those ids on the fp64 scores;
    z [m][N] f64; y [m][d] f64)."""
    h = np.ascontiguousarray(h)
    n = h.shape[0]
    if tokens is None:
        tok, m = None, n
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        assert tok.size == 0 or (tok.min() >= 0 and tok.max() < n)
        m = tok.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    assert ids.shape == (m, layer.top_k)
    assert ids.size == 0 or (ids.min() >= 0 and ids.max() < layer.n_experts)
    assert all(len(set(r.tolist())) == layer.top_k for r in ids)
    w = np.zeros((m, layer.top_k), dtype=np.float64)
    z = np.zeros((m, layer.n_experts), dtype=np.float64)
    y = np.zeros((m, layer.d), dtype=np.float64)
    c = layer._c()
    lib().orc_verify_routed(ctypes.byref(c), _ptr(h), _ptr(tok), m, threads, _ptr(ids),
                            _ptr(w), _ptr(z), _ptr(y))
    return w, z, y


def topk_from_scores(scores: np.ndarray, k: int, mode: int):
    """Top-k and gate on given float32 scores [n][N] (widened exactly)."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    n, E = s.shape
    ids = np.zeros((n, k), dtype=np.int32)
    w = np.zeros((n, k), dtype=np.float64)
    lib().orc_topk_from_scores(_ptr(s), n, E, k, mode, _ptr(ids), _ptr(w))
    return ids, w


def union_plan(ids: np.ndarray, n_experts: int):
    """(U, hist [N], uniq [U], offs [U+1], perm [n*k]) of the routed ids."""
    flat = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).ravel())
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < n_experts)
    hist = np.zeros(n_experts, dtype=np.int32)
    uniq = np.zeros(n_experts, dtype=np.int32)
    offs = np.zeros(n_experts + 1, dtype=np.int32)
    perm = np.zeros(max(flat.size, 1), dtype=np.int32)
    U = lib().orc_union_plan(_ptr(flat), flat.size, n_experts, _ptr(hist), _ptr(uniq),
                             _ptr(offs), _ptr(perm))
    return U, hist, uniq[:U].copy(), offs[:U + 1].copy(), perm[:flat.size].copy()


def expert_bytes(d: int, inter: int, w_type: int):
    """(weight bytes, scale bytes) of one expert."""
    wb, sb = ctypes.c_int64(), ctypes.c_int64()
    lib().orc_expert_bytes(d, inter, w_type, ctypes.byref(wb), ctypes.byref(sb))
    return wb.value, sb.value


def expert_budget(ids: np.ndarray, w: np.ndarray, n_experts: int, budget: int):
    """Verification-time expert budget (MoE-Spec): (keep [N] bool, score [N]
    f64, number kept).  score[e] sums the weights of the slots naming e in
    ascending slot order; the kept experts are the first `budget` used ones
    by (score descending, id ascending).  w is widened to double exactly."""
    flat = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).ravel())
    wf = np.ascontiguousarray(np.asarray(w).ravel(), dtype=np.float64)
    assert flat.size == wf.size and budget >= 0
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < n_experts)
    keep = np.zeros(n_experts, dtype=np.uint8)
    score = np.zeros(n_experts, dtype=np.float64)
    kept = lib().orc_expert_budget(_ptr(flat), _ptr(wf), flat.size, n_experts, budget,
                                   _ptr(keep), _ptr(score))
    return keep.astype(bool), score, kept


def budget_plan(ids: np.ndarray, w: np.ndarray, n_experts: int, budget: int):
    """The union plan of the kept slots under an expert budget:
    (U, hist [N], uniq [U], offs [U+1], perm [kept slots], w_kept [n*k] f64,
    keep [N] bool)."""
    flat = np.ascontiguousarray(np.asarray(ids, dtype=np.int32).ravel())
    wf = np.ascontiguousarray(np.asarray(w).ravel(), dtype=np.float64)
    assert flat.size == wf.size and budget >= 0
    assert flat.size == 0 or (flat.min() >= 0 and flat.max() < n_experts)
    keep = np.zeros(n_experts, dtype=np.uint8)
    score = np.zeros(n_experts, dtype=np.float64)
    hist = np.zeros(n_experts, dtype=np.int32)
    uniq = np.zeros(n_experts, dtype=np.int32)
    offs = np.zeros(n_experts + 1, dtype=np.int32)
    perm = np.zeros(max(flat.size, 1), dtype=np.int32)
    w_kept = np.zeros(max(flat.size, 1), dtype=np.float64)
    U = lib().orc_budget_plan(_ptr(flat), _ptr(wf), flat.size, n_experts, budget, _ptr(keep),
                              _ptr(score), _ptr(hist), _ptr(uniq), _ptr(offs), _ptr(perm),
                              _ptr(w_kept))
    return (U, hist, uniq[:U].copy(), offs[:U + 1].copy(), perm[:offs[U]].copy(),
            w_kept[:flat.size].copy(), keep.astype(bool))


def verify_budget(layer: Layer, h: np.ndarray, budget: int, tokens=None, threads: int = 1):
    """The pass of n tokens under an expert budget: (ids [n][k], w [n][k]
    f64, z [n][N] f64, y [m][d] f64, keep [N] bool).  Routing is the same as
    verify() and covers all n tokens (the kept experts depend on all of
    them); y row i is token tokens[i] (all tokens if None) and sums only its
    slots whose expert is kept (plus the shared expert), with the weights not
    renormalised."""
    h = np.ascontiguousarray(h)
    n = h.shape[0]
    assert budget >= 0
    if tokens is None:
        tok, m = None, n
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        assert tok.size == 0 or (tok.min() >= 0 and tok.max() < n)
        m = tok.shape[0]
    ids = np.zeros((n, layer.top_k), dtype=np.int32)
    w = np.zeros((n, layer.top_k), dtype=np.float64)
    z = np.zeros((n, layer.n_experts), dtype=np.float64)
    y = np.zeros((m, layer.d), dtype=np.float64)
    keep = np.zeros(layer.n_experts, dtype=np.uint8)
    c = layer._c()
    lib().orc_verify_budget(ctypes.byref(c), _ptr(h), n, _ptr(tok), m, threads, budget, _ptr(ids),
                            _ptr(w), _ptr(z), _ptr(y), _ptr(keep))
    return ids, w, z, y, keep.astype(bool)


def _tree(parent, q):
    par = np.ascontiguousarray(np.asarray(parent, dtype=np.int32))
    qq = np.ascontiguousarray(np.asarray(q, dtype=np.float32))
    K = par.shape[0]
    assert qq.shape == (K,) and K >= 1 and par[0] == -1
    assert all(0 <= par[v] < v for v in range(1, K)), "parent[v] must precede v"
    return par, qq, K


def tree_scores(parent, q) -> np.ndarray:
    """Cumulative draft score of every node: the product of q along the path
    from the root (factor 1) to the node ("Making Every Verified Token Count",
    eq. (7))."""
    par, qq, K = _tree(parent, q)
    out = np.zeros(K, dtype=np.float64)
    lib().orc_tree_scores(_ptr(par), _ptr(qq), K, _ptr(out))
    return out


def evict_select(parent, q, cost):
    """EVICT's best verification prefix: (k*, order [K], exp_len [K],
    utility [K]); cost[k-1] = C(k) (float32, widened)."""
    par, qq, K = _tree(parent, q)
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.float32))
    assert c.shape == (K,)
    order = np.zeros(K, dtype=np.int32)
    exp_len = np.zeros(K, dtype=np.float64)
    util = np.zeros(K, dtype=np.float64)
    ks = lib().orc_evict_select(_ptr(par), _ptr(qq), K, _ptr(c), _ptr(order), _ptr(exp_len),
                                _ptr(util))
    return ks, order, exp_len, util


def ecospec_select(parent, q, pred_ids, n_experts: int, gamma: int, eps: float, buf0=None):
    """EcoSpec's cost-aware selection: (selected [min(gamma, K)], buffer
    [L][E] bool, |buffer|).  pred_ids: [K][L][kp] int32 predicted experts."""
    par, qq, K = _tree(parent, q)
    pid = np.ascontiguousarray(np.asarray(pred_ids, dtype=np.int32))
    assert pid.ndim == 3 and pid.shape[0] == K
    L, kp = pid.shape[1], pid.shape[2]
    b0 = None
    if buf0 is not None:
        b0 = np.ascontiguousarray(np.asarray(buf0, dtype=np.uint8))
        assert b0.shape == (L, n_experts)
    n_sel = min(gamma, K)
    sel = np.zeros(max(n_sel, 1), dtype=np.int32)
    buf = np.zeros((L, n_experts), dtype=np.uint8)
    cnt = lib().orc_ecospec_select(_ptr(par), _ptr(qq), _ptr(pid), K, L, n_experts, kp, gamma,
                                   _ptr(b0), ctypes.c_double(eps), _ptr(sel), _ptr(buf))
    return sel[:n_sel].copy(), buf.astype(bool), cnt
