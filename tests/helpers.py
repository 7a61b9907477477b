"""Test helpers: hand the same synthetic bytes to the oracle and the GPU path,
and the error measure used for floating-point parity."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from moe_expert_ffn_gemv_gb300 import synth

# Floating-point parity bars (max element error of the layer output, see rel_err):
# fp32 1e-4, bf16 2e-2, FP8-E4M3 5e-2.
TOL = {synth.F32: 1e-4, synth.BF16: 2e-2, synth.E4M3: 5e-2}

_OT = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.E4M3: oracle.E4M3}
_OG = {synth.GATE_SOFTMAX: oracle.GATE_SOFTMAX, synth.GATE_SOFTMAX_RENORM: oracle.GATE_SOFTMAX_RENORM,
       synth.GATE_SIGMOID_RENORM: oracle.GATE_SIGMOID_RENORM}

THREADS = max(1, os.cpu_count() or 1)


def np_bytes(t):
    """The stored bytes of a tensor as a numpy array (bf16 -> uint16 bits)."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_layer(layer: synth.Layer) -> oracle.Layer:
    c = layer.cfg
    return oracle.Layer(c.d, c.n_experts, c.top_k, c.inter, _OT[c.act], _OT[c.wtype], _OG[c.gate],
                        np_bytes(layer.wg), np_bytes(layer.w13), np_bytes(layer.w2),
                        np_bytes(layer.s13), np_bytes(layer.s2), np_bytes(layer.sh_w13),
                        np_bytes(layer.sh_w2), np_bytes(layer.sh_s13), np_bytes(layer.sh_s2))


def oracle_gate(cfg) -> int:
    return _OG[cfg.gate]


def rel_err(y, y_ref) -> float:
    """max_i |y_i - yref_i| / max(|yref_i|, rms(yref)): element-relative error,
    floored at the output RMS so that near-zero outputs do not dominate."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if y_ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    den = np.maximum(np.abs(y_ref), rms if rms > 0 else 1.0)
    return float(np.max(np.abs(y - y_ref) / den))


def router_delta(layer: synth.Layer, h: torch.Tensor) -> np.ndarray:
    """Per token: delta = 1e-5 * max_e sum_i |Wg[e][i] h[i]|, a bound on the
    error of an fp32 accumulation of its router dot products (see tie_margin)."""
    wg = np.asarray(layer.wg.float().cpu().numpy(), dtype=np.float64)
    hh = np.asarray(h.float().cpu().numpy(), dtype=np.float64)
    return 1e-5 * (np.abs(hh) @ np.abs(wg).T).max(axis=1)


def topk_within(z_row: np.ndarray, ids: np.ndarray, k: int, tol: float) -> bool:
    """ids (k distinct experts, in the order a GPU emitted them) are a top-k
    of the exact scores z_row up to score errors of tol: every selected
    score is at least the exact k-th largest minus tol, every other score at
    most the k-th largest plus tol, and the order descends up to tol."""
    ids = np.asarray(ids)
    if len(set(ids.tolist())) != k:
        return False
    zk = np.sort(z_row)[::-1][k - 1]
    sel = np.zeros(z_row.shape[0], dtype=bool)
    sel[ids] = True
    return bool(np.all(z_row[sel] >= zk - tol) and np.all(z_row[~sel] <= zk + tol)
                and np.all(z_row[ids[:-1]] >= z_row[ids[1:]] - tol))


def tie_margin(layer: synth.Layer, h: torch.Tensor, z: np.ndarray, k: int) -> np.ndarray:
    """Per token: the smallest gap between consecutive oracle scores among the
    first k+1 (in sorted order), over delta = 1e-5 * max_e sum_i |Wg[e][i] h[i]|,
    a bound on the error of an fp32 accumulation of the router dot products
    (it exceeds (terms per accumulator + tree depth) * 2^-24 * sum |.| by
    several times at d <= 8192).  A token with margin > 1 must be routed
    exactly as the oracle routes it."""
    delta = router_delta(layer, h)
    out = np.empty(z.shape[0])
    for t in range(z.shape[0]):
        s = np.sort(z[t])[::-1][:k + 1]
        out[t] = np.min(s[:-1] - s[1:]) / delta[t] if len(s) > 1 else np.inf
    return out
