"""Seeded synthetic inputs for the MoE verification-pass layer.

This module only draws numbers: layer weights, hidden states of draft chains
and draft trees, and random routing ids.  It holds none of the layer's
arithmetic (no routing, gating, FFN or union), so the CUDA path and the CPU
oracle can both be fed from it without sharing any code of the method.

Distributions (readings of the workload descriptions, stated once here):
  expert weights  N(0, 0.02^2);  router weights N(0, 1/d);
  chain           h_0 ~ N(0, I), h_t = rho h_{t-1} + sqrt(1 - rho^2) eps_t;
  wide range      unit normal elements multiplied by 1e5 or 1e-6 (a test of
                  the fp16 range handling; see make_hidden);
  tree            BFS-numbered, node 0 the root, 4 children under the root
                  and 2 under every deeper node; child = parent + sigma eps
                  ("parent + N(0, sigma^2)") or, for the FP8 layer,
                  child = rho parent + sqrt(1 - rho^2) eps;
  FP8 weights     per 128 x 128 block: s = amax / 448, q = E4M3(w / s) with
                  round-to-nearest-even, stored as uint8 codes and fp32 s.
Seeds: expert weights `seed`, router `seed + 1`, hidden states `seed + 2`.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

F32, BF16, E4M3 = "f32", "bf16", "e4m3"
GATE_SOFTMAX, GATE_SOFTMAX_RENORM, GATE_SIGMOID_RENORM = "softmax", "softmax_renorm", "sigmoid_renorm"


@dataclass(frozen=True)
class LayerConfig:
    name: str
    d: int
    n_experts: int
    top_k: int
    inter: int
    act: str          # dtype of hidden states, router weights and outputs
    wtype: str        # dtype of expert weights
    gate: str
    n_shared: int = 0
    hidden: str = "chain"   # "chain" or "tree"
    rho: float = 0.0
    sigma: float = 0.0


# The five layer shapes of the workload.
TINY = LayerConfig("tiny-f32", 256, 16, 2, 128, F32, F32, GATE_SOFTMAX_RENORM,
                   hidden="chain", rho=0.8)
OLMOE = LayerConfig("olmoe-bf16", 2048, 64, 8, 1024, BF16, BF16, GATE_SOFTMAX,
                    hidden="chain", rho=0.5)
QWEN3 = LayerConfig("qwen3-30b-a3b-bf16", 2048, 128, 8, 768, BF16, BF16, GATE_SOFTMAX_RENORM,
                    hidden="tree_add", sigma=0.3)
GPTOSS = LayerConfig("gpt-oss-120b-bf16", 2880, 128, 4, 2880, BF16, BF16, GATE_SOFTMAX_RENORM,
                     hidden="chain", rho=0.7)
DSV3 = LayerConfig("deepseek-v3-fp8", 7168, 256, 8, 2048, BF16, E4M3, GATE_SIGMOID_RENORM,
                   n_shared=1, hidden="tree_ar", rho=0.6)

CONFIGS: Dict[str, LayerConfig] = {c.name: c for c in (TINY, OLMOE, QWEN3, GPTOSS, DSV3)}


def shrink(cfg: LayerConfig, d: int, inter: int, n_experts: Optional[int] = None,
           name: Optional[str] = None) -> LayerConfig:
    """The same layer kind with smaller sizes (for fast parity cases)."""
    from dataclasses import replace
    return replace(cfg, d=d, inter=inter, n_experts=n_experts or cfg.n_experts,
                   name=name or f"{cfg.name}-d{d}-i{inter}")


def torch_dtype(kind: str) -> torch.dtype:
    return {F32: torch.float32, BF16: torch.bfloat16, E4M3: torch.uint8}[kind]


@dataclass
class Layer:
    cfg: LayerConfig
    wg: torch.Tensor                 # [N][d] act dtype
    w13: torch.Tensor                # [N][2I][d] (uint8 codes for E4M3)
    w2: torch.Tensor                 # [N][d][I]
    s13: Optional[torch.Tensor] = None   # [N][2I/128][d/128] float32
    s2: Optional[torch.Tensor] = None    # [N][d/128][I/128] float32
    sh_w13: Optional[torch.Tensor] = None
    sh_w2: Optional[torch.Tensor] = None
    sh_s13: Optional[torch.Tensor] = None
    sh_s2: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)

    def tensors(self) -> List[torch.Tensor]:
        return [t for t in (self.wg, self.w13, self.w2, self.s13, self.s2, self.sh_w13,
                            self.sh_w2, self.sh_s13, self.sh_s2) if t is not None]

    def to(self, device) -> "Layer":
        f = lambda t: None if t is None else t.to(device)
        return Layer(self.cfg, f(self.wg), f(self.w13), f(self.w2), f(self.s13), f(self.s2),
                     f(self.sh_w13), f(self.sh_w2), f(self.sh_s13), f(self.sh_s2))


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _quantise_e4m3(w: torch.Tensor):
    """Per 128 x 128 block: s = amax / 448, codes = E4M3(w / s) (RNE)."""
    R, C = w.shape
    blocks = w.reshape(R // 128, 128, C // 128, 128)
    amax = blocks.abs().amax(dim=(1, 3))
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    q = (blocks / s[:, None, :, None]).clamp(-448.0, 448.0).reshape(R, C)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), s.contiguous()


def _expert_matrix(rows: int, cols: int, wtype: str, g: torch.Generator, device):
    w = torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * 0.02
    if wtype == E4M3:
        return _quantise_e4m3(w)
    return w.to(torch_dtype(wtype)).contiguous(), None


def make_layer(cfg: LayerConfig, seed: int = 1, device="cpu") -> Layer:
    """All N routed experts (+ the shared expert), expert-major."""
    d, I, N = cfg.d, cfg.inter, cfg.n_experts
    if cfg.wtype == E4M3:
        assert d % 128 == 0 and I % 128 == 0, "E4M3 layers need d and I multiples of 128"
    g = _gen(seed, device)
    wdt = torch_dtype(cfg.wtype)
    w13 = torch.empty(N, 2 * I, d, dtype=wdt, device=device)
    w2 = torch.empty(N, d, I, dtype=wdt, device=device)
    s13 = s2 = None
    if cfg.wtype == E4M3:
        s13 = torch.empty(N, 2 * I // 128, d // 128, dtype=torch.float32, device=device)
        s2 = torch.empty(N, d // 128, I // 128, dtype=torch.float32, device=device)
    for e in range(N):
        a, sa = _expert_matrix(2 * I, d, cfg.wtype, g, device)
        b, sb = _expert_matrix(d, I, cfg.wtype, g, device)
        w13[e].copy_(a)
        w2[e].copy_(b)
        if s13 is not None:
            s13[e].copy_(sa)
            s2[e].copy_(sb)
    sh = [None] * 4
    if cfg.n_shared:
        a, sa = _expert_matrix(2 * I, d, cfg.wtype, g, device)
        b, sb = _expert_matrix(d, I, cfg.wtype, g, device)
        sh = [a, b, sa, sb]
    gr = _gen(seed + 1, device)
    wg = (torch.randn(N, d, generator=gr, device=device, dtype=torch.float32)
          / math.sqrt(d)).to(torch_dtype(cfg.act)).contiguous()
    return Layer(cfg, wg, w13, w2, s13, s2, *sh)


def tree_parents(n: int, root_children: int = 4, branching: int = 2) -> List[int]:
    """Parent of each node of a BFS-numbered draft tree (root's parent = -1)."""
    parents = [-1]
    frontier = [0]
    while len(parents) < n:
        nxt = []
        for p in frontier:
            for _ in range(root_children if p == 0 else branching):
                if len(parents) == n:
                    break
                parents.append(p)
                nxt.append(len(parents) - 1)
        frontier = nxt
    return parents[:n]


def make_hidden(cfg: LayerConfig, n: int, seed: int = 3, device="cpu", kind: Optional[str] = None,
                rho: Optional[float] = None, sigma: Optional[float] = None) -> torch.Tensor:
    """Hidden states [n][d] of n draft tokens, in the layer's act dtype."""
    kind = kind or cfg.hidden
    rho = cfg.rho if rho is None else rho
    sigma = cfg.sigma if sigma is None else sigma
    g = _gen(seed, device)
    eps = torch.randn(max(n, 1), cfg.d, generator=g, device=device, dtype=torch.float64)
    h = torch.empty(max(n, 1), cfg.d, dtype=torch.float64, device=device)
    h[0] = eps[0]
    if kind == "chain":
        c = math.sqrt(max(0.0, 1.0 - rho * rho))
        for t in range(1, n):
            h[t] = rho * h[t - 1] + c * eps[t]
    elif kind == "tree_add":
        par = tree_parents(n)
        for t in range(1, n):
            h[t] = h[par[t]] + sigma * eps[t]
    elif kind == "tree_ar":
        par = tree_parents(n)
        c = math.sqrt(max(0.0, 1.0 - rho * rho))
        for t in range(1, n):
            h[t] = rho * h[par[t]] + c * eps[t]
    elif kind == "identical":
        h[:] = eps[0]
    elif kind == "wide_range":
        # magnitudes far outside fp16's range, for the E4M3 engines' scaling:
        # token 0 all x1e5, token 1 all x1e-6, the others a mix per element
        # (2% x1e5, 40% x1e-6, the rest unit normal)
        h[:] = eps[:max(n, 1)]
        u = torch.rand(max(n, 1), cfg.d, generator=g, device=device, dtype=torch.float64)
        mul = torch.where(u < 0.02, 1e5, torch.where(u < 0.42, 1e-6, 1.0))
        mul[0] = 1e5
        if n > 1:
            mul[1] = 1e-6
        h *= mul
    else:
        raise ValueError(kind)
    return h[:n].to(torch_dtype(cfg.act)).contiguous()


def uniform_ids(n: int, k: int, n_experts: int, seed: int = 5) -> torch.Tensor:
    """n independent uniformly random k-subsets of the experts, int32 [n][k]."""
    g = _gen(seed, "cpu")
    keys = torch.rand(n, n_experts, generator=g)
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


def random_scores(n: int, n_experts: int, seed: int = 7, ties: bool = False) -> torch.Tensor:
    """float32 scores [n][N]; with ties=True values are drawn from a few levels
    so that equal scores are common (and include both signs of zero)."""
    g = _gen(seed, "cpu")
    if not ties:
        return torch.randn(n, n_experts, generator=g, dtype=torch.float32)
    levels = torch.tensor([-1.5, -0.0, 0.0, 0.25, 0.25, 2.0, 3.0e38, -3.0e38], dtype=torch.float32)
    idx = torch.randint(0, levels.numel(), (n, n_experts), generator=g)
    return levels[idx].contiguous()
