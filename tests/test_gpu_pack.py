"""moe_pack_expert_weights writes the tile layout include/moe_verify.h states,
checked piece by piece against a numpy transcription of that statement."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def expected_packed(mat: np.ndarray, gate_up: bool, inter: int) -> np.ndarray:
    """mat: one expert matrix as uint8 [rows][K bytes] -> packed bytes."""
    rows, K = mat.shape
    out = np.empty(rows * K, dtype=np.uint8)
    pos = 0
    for rb in range(rows // 64):
        for kc in range((K + 511) // 512):
            width = min(512, K - 512 * kc)
            for w in range(width // 64):
                for mt in range(4):
                    for h in range(2):
                        for lane in range(32):
                            rit = 16 * mt + lane // 4 + 8 * h
                            if gate_up:
                                row = 32 * rb + rit if rit < 32 else inter + 32 * rb + rit - 32
                            else:
                                row = 64 * rb + rit
                            col = 512 * kc + 64 * w + 16 * (lane % 4)
                            out[pos:pos + 16] = mat[row, col:col + 16]
                            pos += 16
    assert pos == rows * K
    return out


@pytest.mark.parametrize("wtype,d,inter", [(synth.BF16, 704, 96), (synth.E4M3, 640, 384),
                                           (synth.BF16, 2880, 96)])
def test_pack_layout(mv, wtype, d, inter):
    cfg = synth.LayerConfig("pack", d, 3, 2, inter, synth.BF16, wtype, synth.GATE_SOFTMAX)
    layer = synth.make_layer(cfg, seed=9, device="cuda")
    desc = mv.make_desc(cfg, 4)
    packed = mv.pack_weights(layer, desc)
    torch.cuda.synchronize()
    es = 1 if wtype == synth.E4M3 else 2
    for e in range(cfg.n_experts):
        for src, dst, gate_up in ((layer.w13[e], packed.w13[e], True),
                                  (layer.w2[e], packed.w2[e], False)):
            m = src.contiguous().view(torch.uint8).cpu().numpy().reshape(src.shape[0], -1)
            assert m.shape[1] == src.shape[1] * es
            got = dst.contiguous().view(torch.uint8).cpu().numpy().ravel()
            assert np.array_equal(got, expected_packed(m, gate_up, inter))


def test_pack_fp32_is_a_copy(mv):
    cfg = synth.shrink(synth.TINY, d=64, inter=16, n_experts=2)
    layer = synth.make_layer(cfg, device="cuda")
    packed = mv.pack_weights(layer, mv.make_desc(cfg, 2))
    torch.cuda.synchronize()
    assert torch.equal(packed.w13, layer.w13) and torch.equal(packed.w2, layer.w2)
