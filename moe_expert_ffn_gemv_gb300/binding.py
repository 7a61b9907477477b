"""Python binding of libmoe_verify.so (include/moe_verify.h).

Argument marshalling only: every step of the verification pass runs in the
library's CUDA kernels.  PyTorch provides device memory and the current CUDA
stream.  Importing this module loads the library and raises if it is missing
(build it with ``python -m moe_expert_ffn_gemv_gb300.build``): there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import synth

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_verify.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m moe_expert_ffn_gemv_gb300.build` "
                      "(needs the CUDA toolkit); there is no CPU fallback")
_lib = ctypes.CDLL(LIB_PATH)

# status codes, dtypes and gates as numbered in include/moe_verify.h
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_ALIGNMENT = 0, 1, 2, 3
MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_INPUT = 4, 5, 6, 7
MOE_F32, MOE_BF16, MOE_E4M3_B128 = 0, 1, 2
MOE_GATE_SOFTMAX, MOE_GATE_SOFTMAX_RENORM, MOE_GATE_SIGMOID_RENORM = 0, 1, 2

EXPORTED = ["moe_workspace_bytes", "moe_expert_bytes", "moe_route_topk", "moe_topk_from_logits",
            "moe_union_plan", "moe_verify_dedup", "moe_verify_perslot", "moe_workspace_init",
            "moe_last_error", "moe_selftest_bounded_wait", "moe_status_string",
            "moe_pack_expert_weights", "moe_verify_dedup_noalloc", "moe_route_plan",
            "moe_union_plan_budgeted", "moe_route_plan_budgeted", "moe_evict_select",
            "moe_ecospec_select", "moe_verify_pass", "moe_packed_bytes"]


class moe_layer_desc(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in
                ("d", "n_experts", "top_k", "inter", "n_shared", "n_max", "act_dtype", "w_dtype",
                 "gate", "wait_timeout_us")]


class moe_expert_weights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in
                ("w13", "w2", "sh_w13", "sh_w2")]


class moe_plan(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in
                ("hist", "uniq", "n_uniq", "offs", "perm", "union_bytes")]


_P = ctypes.c_void_p
_D = ctypes.POINTER(moe_layer_desc)
_lib.moe_workspace_bytes.restype = ctypes.c_size_t
_lib.moe_workspace_bytes.argtypes = [_D]
_lib.moe_expert_bytes.restype = ctypes.c_int
_lib.moe_expert_bytes.argtypes = [_D, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
_lib.moe_route_topk.restype = ctypes.c_int
_lib.moe_route_topk.argtypes = [_D, _P, _P, ctypes.c_int32, _P, _P, _P, _P]
_lib.moe_topk_from_logits.restype = ctypes.c_int
_lib.moe_topk_from_logits.argtypes = [_D, _P, ctypes.c_int32, _P, _P, _P]
_lib.moe_union_plan.restype = ctypes.c_int
_lib.moe_union_plan.argtypes = [_D, _P, ctypes.c_int32, ctypes.POINTER(moe_plan), _P, _P]
_lib.moe_route_plan.restype = ctypes.c_int
_lib.moe_route_plan.argtypes = [_D, _P, _P, ctypes.c_int32, _P, _P, _P, ctypes.POINTER(moe_plan), _P,
                                ctypes.c_size_t, _P]
_lib.moe_union_plan_budgeted.restype = ctypes.c_int
_lib.moe_union_plan_budgeted.argtypes = [_D, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.POINTER(moe_plan), _P, _P, _P, _P]
_lib.moe_route_plan_budgeted.restype = ctypes.c_int
_lib.moe_route_plan_budgeted.argtypes = [_D, _P, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                         ctypes.POINTER(moe_plan), _P, _P, _P, ctypes.c_size_t,
                                         _P]
_lib.moe_evict_select.restype = ctypes.c_int
_lib.moe_evict_select.argtypes = [_P, _P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                  _P]
_lib.moe_ecospec_select.restype = ctypes.c_int
_lib.moe_ecospec_select.argtypes = [_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_double, _P, _P, _P, _P, _P, _P]
_lib.moe_verify_pass.restype = ctypes.c_int
_lib.moe_verify_pass.argtypes = [_D, ctypes.POINTER(moe_expert_weights), _P, _P, ctypes.c_int32,
                                 ctypes.c_int32, _P, _P, _P, ctypes.POINTER(moe_plan), _P, _P, _P,
                                 ctypes.c_size_t, _P, _P]
_lib.moe_verify_dedup.restype = ctypes.c_int
_lib.moe_verify_dedup.argtypes = [_D, ctypes.POINTER(moe_expert_weights), _P, ctypes.c_int32, _P,
                                  _P, ctypes.POINTER(moe_plan), _P, ctypes.c_size_t, _P, _P]
_lib.moe_verify_perslot.restype = ctypes.c_int
_lib.moe_verify_perslot.argtypes = [_D, ctypes.POINTER(moe_expert_weights), _P, ctypes.c_int32,
                                    _P, _P, _P, ctypes.c_size_t, _P, _P]
_lib.moe_verify_dedup_noalloc.restype = ctypes.c_int
_lib.moe_verify_dedup_noalloc.argtypes = [_D, ctypes.POINTER(moe_expert_weights), _P, ctypes.c_int32,
                                          _P, _P, ctypes.POINTER(moe_plan), _P, _P, _P]
_lib.moe_pack_expert_weights.restype = ctypes.c_int
_lib.moe_pack_expert_weights.argtypes = [_D, _P, _P, _P, _P, ctypes.c_int32, _P, _P, _P]
_lib.moe_packed_bytes.restype = ctypes.c_int
_lib.moe_packed_bytes.argtypes = [_D, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
_lib.moe_workspace_init.restype = ctypes.c_int
_lib.moe_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
_lib.moe_last_error.restype = ctypes.c_int
_lib.moe_last_error.argtypes = [_P, _P]
_lib.moe_selftest_bounded_wait.restype = ctypes.c_int
_lib.moe_selftest_bounded_wait.argtypes = [_P, ctypes.c_int32, _P]
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_status_string.argtypes = [ctypes.c_int]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {moe_status_string(status)} (status {status})")


def _check(status: int, where: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------- the C calls

def moe_status_string(status: int) -> str:
    return _lib.moe_status_string(status).decode()


def moe_workspace_bytes(desc: moe_layer_desc) -> int:
    return int(_lib.moe_workspace_bytes(ctypes.byref(desc)))


def moe_expert_bytes(desc: moe_layer_desc):
    wb, sb = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.moe_expert_bytes(ctypes.byref(desc), ctypes.byref(wb), ctypes.byref(sb)),
           "moe_expert_bytes")
    return wb.value, sb.value


def moe_route_topk(desc, router_w, h, n, ids, w, logits, stream=None) -> None:
    _check(_lib.moe_route_topk(ctypes.byref(desc), _ptr(router_w), _ptr(h), n, _ptr(ids), _ptr(w),
                               _ptr(logits), _stream(stream)), "moe_route_topk")


def moe_topk_from_logits(desc, logits, n, ids, w, stream=None) -> None:
    _check(_lib.moe_topk_from_logits(ctypes.byref(desc), _ptr(logits), n, _ptr(ids), _ptr(w),
                                     _stream(stream)), "moe_topk_from_logits")


def moe_union_plan(desc, ids, n, plan: moe_plan, error_word=None, stream=None) -> None:
    _check(_lib.moe_union_plan(ctypes.byref(desc), _ptr(ids), n, ctypes.byref(plan),
                               _ptr(error_word), _stream(stream)), "moe_union_plan")


def moe_route_plan(desc, router_w, h, n, ids, w, logits, plan: moe_plan, workspace,
                   stream=None) -> None:
    _check(_lib.moe_route_plan(ctypes.byref(desc), _ptr(router_w), _ptr(h), n, _ptr(ids), _ptr(w),
                               _ptr(logits), ctypes.byref(plan), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_route_plan")


def moe_union_plan_budgeted(desc, ids, w, n, budget, plan: moe_plan, w_kept, routed_union=None,
                            error_word=None, stream=None) -> None:
    _check(_lib.moe_union_plan_budgeted(ctypes.byref(desc), _ptr(ids), _ptr(w), n, budget,
                                        ctypes.byref(plan), _ptr(w_kept), _ptr(routed_union),
                                        _ptr(error_word), _stream(stream)),
           "moe_union_plan_budgeted")


def moe_route_plan_budgeted(desc, router_w, h, n, budget, ids, w, logits, plan: moe_plan, w_kept,
                            routed_union, workspace, stream=None) -> None:
    _check(_lib.moe_route_plan_budgeted(ctypes.byref(desc), _ptr(router_w), _ptr(h), n, budget,
                                        _ptr(ids), _ptr(w), _ptr(logits), ctypes.byref(plan),
                                        _ptr(w_kept), _ptr(routed_union), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)), "moe_route_plan_budgeted")


def moe_evict_select(parent, q, n_trees, n_nodes, cost, order, exp_len, utility, k_star,
                     error_word=None, stream=None) -> None:
    _check(_lib.moe_evict_select(_ptr(parent), _ptr(q), n_trees, n_nodes, _ptr(cost), _ptr(order),
                                 _ptr(exp_len), _ptr(utility), _ptr(k_star), _ptr(error_word),
                                 _stream(stream)), "moe_evict_select")


def moe_ecospec_select(parent, q, pred_ids, n_trees, n_nodes, n_layers, n_experts, pred_k, gamma,
                       eps, buffer0, selected, buffer_out, union_size, error_word=None,
                       stream=None) -> None:
    _check(_lib.moe_ecospec_select(_ptr(parent), _ptr(q), _ptr(pred_ids), n_trees, n_nodes,
                                   n_layers, n_experts, pred_k, gamma, ctypes.c_double(eps),
                                   _ptr(buffer0), _ptr(selected), _ptr(buffer_out),
                                   _ptr(union_size), _ptr(error_word), _stream(stream)),
           "moe_ecospec_select")


def moe_verify_pass(desc, weights: moe_expert_weights, router_w, h, n, budget, ids, w, logits,
                    plan: moe_plan, w_kept, routed_union, workspace, y, stream=None) -> None:
    _check(_lib.moe_verify_pass(ctypes.byref(desc), ctypes.byref(weights), _ptr(router_w), _ptr(h),
                                n, budget, _ptr(ids), _ptr(w), _ptr(logits), ctypes.byref(plan),
                                _ptr(w_kept), _ptr(routed_union), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _ptr(y),
                                _stream(stream)), "moe_verify_pass")


def moe_verify_dedup(desc, weights: moe_expert_weights, h, n, ids, w, plan: moe_plan, workspace,
                     y, stream=None) -> None:
    _check(_lib.moe_verify_dedup(ctypes.byref(desc), ctypes.byref(weights), _ptr(h), n, _ptr(ids),
                                 _ptr(w), ctypes.byref(plan), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(y),
                                 _stream(stream)), "moe_verify_dedup")


def moe_verify_dedup_noalloc(desc, weights: moe_expert_weights, h, n, ids, w, plan: moe_plan, y,
                             error_word=None, stream=None) -> None:
    """The deduplicating pass with the library's own fixed scratch (no
    workspace): for callers that cannot allocate device memory themselves."""
    _check(_lib.moe_verify_dedup_noalloc(ctypes.byref(desc), ctypes.byref(weights), _ptr(h), n,
                                         _ptr(ids), _ptr(w), ctypes.byref(plan), _ptr(y),
                                         _ptr(error_word), _stream(stream)),
           "moe_verify_dedup_noalloc")


def moe_verify_perslot(desc, weights: moe_expert_weights, h, n, ids, w, workspace, y,
                       stream=None) -> None:
    _check(_lib.moe_verify_perslot(ctypes.byref(desc), ctypes.byref(weights), _ptr(h), n,
                                   _ptr(ids), _ptr(w), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(y),
                                   _stream(stream)), "moe_verify_perslot")


def moe_packed_bytes(desc) -> Tuple[int, int]:
    """(W13, W2) bytes of one packed expert."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    _check(_lib.moe_packed_bytes(ctypes.byref(desc), ctypes.byref(a), ctypes.byref(b)),
           "moe_packed_bytes")
    return a.value, b.value


def moe_pack_expert_weights(desc, w13, w2, s13, s2, n_matrices, w13_packed, w2_packed,
                            stream=None) -> None:
    _check(_lib.moe_pack_expert_weights(ctypes.byref(desc), _ptr(w13), _ptr(w2), _ptr(s13),
                                        _ptr(s2), n_matrices, _ptr(w13_packed), _ptr(w2_packed),
                                        _stream(stream)),
           "moe_pack_expert_weights")


def moe_workspace_init(workspace, stream=None) -> None:
    _check(_lib.moe_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                   _stream(stream)), "moe_workspace_init")


def moe_last_error(workspace, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device error word."""
    return int(_lib.moe_last_error(_ptr(workspace), _stream(stream)))


def moe_selftest_bounded_wait(error_word, limit_us: int, stream=None) -> None:
    _check(_lib.moe_selftest_bounded_wait(_ptr(error_word), limit_us, _stream(stream)),
           "moe_selftest_bounded_wait")


# ------------------------------------------------------- layer convenience

_DT = {synth.F32: MOE_F32, synth.BF16: MOE_BF16, synth.E4M3: MOE_E4M3_B128}
_GATE = {synth.GATE_SOFTMAX: MOE_GATE_SOFTMAX, synth.GATE_SOFTMAX_RENORM: MOE_GATE_SOFTMAX_RENORM,
         synth.GATE_SIGMOID_RENORM: MOE_GATE_SIGMOID_RENORM}


def make_desc(cfg: synth.LayerConfig, n_max: int, wait_timeout_us: int = 0) -> moe_layer_desc:
    return moe_layer_desc(cfg.d, cfg.n_experts, cfg.top_k, cfg.inter, cfg.n_shared, n_max,
                          _DT[cfg.act], _DT[cfg.wtype], _GATE[cfg.gate], wait_timeout_us)


@dataclass
class PackedWeights:
    """A layer's expert weights in the library's packed tile layout (device)."""
    w13: torch.Tensor
    w2: torch.Tensor
    sh_w13: Optional[torch.Tensor]
    sh_w2: Optional[torch.Tensor]

    def c(self) -> moe_expert_weights:
        return moe_expert_weights(_ptr(self.w13), _ptr(self.w2), _ptr(self.sh_w13),
                                  _ptr(self.sh_w2))


def pack_weights(layer: synth.Layer, desc: moe_layer_desc) -> PackedWeights:
    """Repack a layer's (device, row-major) expert weights, and for E4M3 their
    block scales, with moe_pack_expert_weights."""
    b13, b2 = moe_packed_bytes(desc)
    dev = layer.w13.device
    N = layer.cfg.n_experts
    w13 = torch.empty(N * b13, dtype=torch.uint8, device=dev)
    w2 = torch.empty(N * b2, dtype=torch.uint8, device=dev)
    moe_pack_expert_weights(desc, layer.w13, layer.w2, layer.s13, layer.s2, N, w13, w2)
    sh13 = sh2 = None
    if layer.sh_w13 is not None:
        sh13 = torch.empty(b13, dtype=torch.uint8, device=dev)
        sh2 = torch.empty(b2, dtype=torch.uint8, device=dev)
        moe_pack_expert_weights(desc, layer.sh_w13, layer.sh_w2, layer.sh_s13, layer.sh_s2, 1,
                                sh13, sh2)
    return PackedWeights(w13, w2, sh13, sh2)


@dataclass
class PlanBuffers:
    hist: torch.Tensor
    uniq: torch.Tensor
    n_uniq: torch.Tensor
    offs: torch.Tensor
    perm: torch.Tensor
    union_bytes: torch.Tensor

    def c(self) -> moe_plan:
        return moe_plan(*(_ptr(t) for t in (self.hist, self.uniq, self.n_uniq, self.offs,
                                            self.perm, self.union_bytes)))


def _aligned_empty(count: int, dtype, device) -> torch.Tensor:
    # torch allocations start on 512-byte boundaries; keep each array separate
    return torch.empty(max(count, 4), dtype=dtype, device=device)


class VerifyLayer:
    """Device buffers of one layer and the calls of one verification pass.

    Owns nothing but torch tensors (its packed copy of the expert weights,
    the workspace, routing and plan buffers); every method is one or more C
    calls on the current stream.
    """

    def __init__(self, layer: synth.Layer, n_max: int, device="cuda", wait_timeout_us: int = 0):
        cfg = layer.cfg
        self.layer = layer
        self.cfg = cfg
        self.n_max = n_max
        self.desc = make_desc(cfg, n_max, wait_timeout_us)
        self.packed = pack_weights(layer, self.desc)
        self.weights = self.packed.c()
        nb = moe_workspace_bytes(self.desc)
        if nb == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED, "moe_workspace_bytes")
        self.workspace = torch.empty(nb, dtype=torch.uint8, device=device)
        moe_workspace_init(self.workspace)
        k, E = cfg.top_k, cfg.n_experts
        i32 = torch.int32
        self.ids = _aligned_empty(n_max * k, i32, device)
        self.w = _aligned_empty(n_max * k, torch.float32, device)
        self.logits = _aligned_empty(n_max * E, torch.float32, device)
        self.plan = PlanBuffers(_aligned_empty(E, i32, device), _aligned_empty(E, i32, device),
                                _aligned_empty(1, i32, device), _aligned_empty(E + 1, i32, device),
                                _aligned_empty(n_max * k, i32, device),
                                _aligned_empty(1, torch.int64, device))
        self._cplan = self.plan.c()
        self.w_kept = _aligned_empty(n_max * k, torch.float32, device)  # budgeted weights
        self.routed_u = _aligned_empty(1, i32, device)                   # U before a budget
        self.error_word = self.workspace[:4].view(torch.int32)
        self.y = torch.empty(n_max, cfg.d, dtype=synth.torch_dtype(cfg.act), device=device)

    def route(self, h: torch.Tensor, n: int) -> None:
        moe_route_topk(self.desc, self.layer.wg, h, n, self.ids, self.w, self.logits)

    def union_plan(self, n: int, budget: Optional[int] = None) -> None:
        """The union plan of the routed ids; with `budget`, the plan of the
        kept experts only, and self.w_kept / self.routed_u written."""
        if budget is None:
            moe_union_plan(self.desc, self.ids, n, self._cplan, self.error_word)
        else:
            moe_union_plan_budgeted(self.desc, self.ids, self.w, n, budget, self._cplan,
                                    self.w_kept, self.routed_u, self.error_word)

    def route_plan(self, h: torch.Tensor, n: int, budget: Optional[int] = None) -> None:
        """route + union_plan (budgeted when `budget` is given) in one launch."""
        if budget is None:
            moe_route_plan(self.desc, self.layer.wg, h, n, self.ids, self.w, self.logits,
                           self._cplan, self.workspace)
        else:
            moe_route_plan_budgeted(self.desc, self.layer.wg, h, n, budget, self.ids, self.w,
                                    self.logits, self._cplan, self.w_kept, self.routed_u,
                                    self.workspace)

    def dedup(self, h: torch.Tensor, n: int, y: Optional[torch.Tensor] = None,
              kept: bool = False) -> torch.Tensor:
        """The deduplicating engine on the current plan; kept=True combines
        with the budgeted weights self.w_kept."""
        y = self.y if y is None else y
        moe_verify_dedup(self.desc, self.weights, h, n, self.ids, self.w_kept if kept else self.w,
                         self._cplan, self.workspace, y)
        return y[:n]

    def perslot(self, h: torch.Tensor, n: int, y: Optional[torch.Tensor] = None) -> torch.Tensor:
        y = self.y if y is None else y
        moe_verify_perslot(self.desc, self.weights, h, n, self.ids, self.w, self.workspace, y)
        return y[:n]

    def verify_pass(self, h: torch.Tensor, n: int, engine: str = "dedup",
                    y: Optional[torch.Tensor] = None,
                    budget: Optional[int] = None) -> torch.Tensor:
        """Route, plan and run the experts: one MoE verification pass (the
        deduplicating engine through moe_verify_pass, optionally under an
        expert budget; the per-slot engine through route + per-slot)."""
        if engine == "dedup":
            y = self.y if y is None else y
            moe_verify_pass(self.desc, self.weights, self.layer.wg, h, n,
                            -1 if budget is None else budget, self.ids, self.w, self.logits,
                            self._cplan, self.w_kept, self.routed_u, self.workspace, y)
            return y[:n]
        assert budget is None, "the expert budget applies to the deduplicating engine"
        self.route(h, n)
        return self.perslot(h, n, y)

    def capture(self, h: torch.Tensor, n: int, engine: str = "dedup",
                budget: Optional[int] = None):
        """Record one verification pass (route, plan, experts, combine) on `h`
        (a fixed device buffer) into CUDA graphs; returns (route_and_plan,
        experts), two torch.cuda.CUDAGraph objects replayed in that order.
        Every call of the pass is asynchronous and host-sync free, so it can
        be captured; replays read whatever `h` holds and write self.y."""
        # one eager pass first: sets kernel attributes and warms the library
        self.verify_pass(h, n, engine, budget=budget)
        torch.cuda.synchronize()
        g_route = torch.cuda.CUDAGraph()
        g_experts = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_route):
            if engine == "dedup":
                self.route_plan(h, n, budget)
            else:
                self.route(h, n)
        with torch.cuda.graph(g_experts):
            if engine == "dedup":
                self.dedup(h, n, kept=budget is not None)
            else:
                self.perslot(h, n)
        return g_route, g_experts

    def capture_pass(self, h: torch.Tensor, n: int, budget: Optional[int] = None,
                     y: Optional[torch.Tensor] = None):
        """The whole deduplicating pass (fused route + plan, then the expert
        call) on `h` (a fixed device buffer) as one CUDA graph writing `y`
        (self.y by default), so that the expert kernels launch as
        programmatic dependents of the routing."""
        self.verify_pass(h, n, y=y, budget=budget)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.verify_pass(h, n, y=y, budget=budget)
        return g

    def last_error(self) -> int:
        return moe_last_error(self.workspace)

    def release_unpacked(self) -> None:
        """Drop this object's references to the row-major expert weights
        (the packed copy is what the kernels read); the router weights and
        the scale tables stay."""
        L = self.layer
        self.layer = synth.Layer(L.cfg, L.wg, None, None, L.s13, L.s2, None, None, L.sh_s13,
                                 L.sh_s2)

    # views of the routing results
    def ids_view(self, n):
        return self.ids[:n * self.cfg.top_k].view(n, self.cfg.top_k)

    def w_view(self, n):
        return self.w[:n * self.cfg.top_k].view(n, self.cfg.top_k)

    def logits_view(self, n):
        return self.logits[:n * self.cfg.n_experts].view(n, self.cfg.n_experts)


# -------------------------------------------------- pre-verification selection

def _i32(x, device):
    return torch.as_tensor(x, dtype=torch.int32).contiguous().to(device)


def evict_select(parent, q, cost, error_word=None):
    """EVICT's best prefix for a batch of trees on the GPU.  parent, q:
    [trees][K] (int32 / float32 tensors or arrays, moved to the GPU); cost:
    [K] C(k).  Returns (k_star [trees], order [trees][K], exp_len, utility)
    as device tensors."""
    parent = _i32(parent, "cuda")
    q = torch.as_tensor(q, dtype=torch.float32).contiguous().cuda()
    cost = torch.as_tensor(cost, dtype=torch.float32).contiguous().cuda()
    T, K = parent.shape
    order = torch.empty(T, K, dtype=torch.int32, device="cuda")
    exp_len = torch.empty(T, K, dtype=torch.float64, device="cuda")
    util = torch.empty(T, K, dtype=torch.float64, device="cuda")
    k_star = torch.empty(max(T, 1), dtype=torch.int32, device="cuda")
    moe_evict_select(parent, q, T, K, cost, order, exp_len, util, k_star, error_word)
    return k_star[:T], order, exp_len, util


def ecospec_select(parent, q, pred_ids, n_experts: int, gamma: int, eps: float, buffer0=None,
                   error_word=None):
    """EcoSpec's cost-aware selection for a batch of trees on the GPU.
    pred_ids: [trees][K][L][kp]; buffer0: [trees][L][ceil(E/32)] uint32 bit
    words (as int32) or None.  Returns (selected [trees][min(gamma,K)],
    buffer [trees][L][words] (int32 view of the bits), union_size [trees])."""
    parent = _i32(parent, "cuda")
    q = torch.as_tensor(q, dtype=torch.float32).contiguous().cuda()
    pred = _i32(pred_ids, "cuda")
    T, K, L, kp = pred.shape
    wpl = (n_experts + 31) // 32
    n_sel = min(gamma, K)
    sel = torch.empty(T, max(n_sel, 1), dtype=torch.int32, device="cuda")
    buf = torch.empty(T, L, wpl, dtype=torch.int32, device="cuda")
    usz = torch.empty(max(T, 1), dtype=torch.int32, device="cuda")
    b0 = None if buffer0 is None else _i32(buffer0, "cuda")
    moe_ecospec_select(parent, q, pred, T, K, L, n_experts, kp, gamma, eps, b0, sel, buf, usz,
                       error_word)
    return sel[:, :n_sel], buf, usz[:T]


class VerifyStack:
    """L MoE layers verified in one pass ("The Limits of Speculation",
    Sec. 3.3: the pass's cost follows the distinct experts counted in each
    MoE layer).  Each layer routes its own hidden states, plans its union and
    runs the deduplicating engine; the whole stack is captured in one CUDA
    graph.  What sits between two MoE layers (attention, norms, the residual
    stream) is not on this path, so each layer's input is given: hs is
    [L][n_max][d], one row block per layer."""

    def __init__(self, vls):
        self.layers = list(vls)
        self.cfg = self.layers[0].cfg
        self.n_max = self.layers[0].n_max

    @classmethod
    def synthetic(cls, cfg: synth.LayerConfig, n_layers: int, n_max: int, seed: int = 1):
        """n_layers seeded layers of one shape (weights seed + 10 l), each
        generated on the device, packed, then freed of its row-major copy, so
        that at most one row-major layer is held at a time."""
        vls = []
        for l in range(n_layers):
            layer = synth.make_layer(cfg, seed=seed + 10 * l, device="cuda")
            vl = VerifyLayer(layer, n_max)
            vl.release_unpacked()
            del layer
            vls.append(vl)
            torch.cuda.empty_cache()
        return cls(vls)

    def verify_pass(self, hs: torch.Tensor, n: int, budget: Optional[int] = None):
        """Every layer's pass on its own rows of hs; returns the outputs."""
        return [vl.verify_pass(hs[l, :n], n, budget=budget) for l, vl in enumerate(self.layers)]

    def capture(self, hs: torch.Tensor, n: int, budget: Optional[int] = None):
        """The whole stack's pass on hs (a fixed device buffer) as one CUDA
        graph; replays read whatever hs holds and write each layer's y."""
        self.verify_pass(hs, n, budget)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l, vl in enumerate(self.layers):
                vl.verify_pass(hs[l, :n], n, budget=budget)
        return g

    def unions(self):
        """U of each layer's last plan (synchronises)."""
        return [int(vl.plan.n_uniq[0]) for vl in self.layers]

    def last_error(self) -> int:
        errs = [vl.last_error() for vl in self.layers]
        return next((e for e in errs if e), MOE_OK)
