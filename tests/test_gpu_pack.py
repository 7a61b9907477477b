"""moe_pack_expert_weights writes the tile layout include/moe_verify.h states
(BF16: 128-byte swizzled K-major columns; E4M3: fragment-ordered pieces, each
tile followed by its 8 block scales), checked piece by piece against a numpy
transcription of that statement."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_gemv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mv():
    from moe_expert_ffn_gemv_gb300 import binding
    return binding


def expected_packed(mat: np.ndarray, gate_up: bool, inter: int, scales=None) -> np.ndarray:
    """mat: one expert matrix as uint8 [rows][K bytes] -> packed bytes; scales:
    its E4M3 block scales [rows/128][K/128] (float32) or None."""
    rows, K = mat.shape
    tiles = (rows // 64) * ((K + 511) // 512)
    out = np.empty(rows * K + (32 * tiles if scales is not None else 0), dtype=np.uint8)
    pos = 0
    def row_of(rit, rb):
        if gate_up:
            return 32 * rb + rit if rit < 32 else inter + 32 * rb + rit - 32
        return 64 * rb + rit

    for rb in range(rows // 64):
        for kc in range((K + 511) // 512):
            width = min(512, K - 512 * kc)
            if scales is None:
                # BF16: [128-byte column q][8-row group m][row r][position], chunk j
                # of row 8m+r at position j XOR r
                for q in range(width // 128):
                    for m in range(8):
                        for r in range(8):
                            for p in range(8):
                                col = 512 * kc + 128 * q + 16 * (p ^ r)
                                out[pos:pos + 16] = mat[row_of(8 * m + r, rb), col:col + 16]
                                pos += 16
                continue
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
            if scales is not None:
                # the 128-row blocks of the tile's first and last 32 rows
                blocks = ((32 * rb) // 128, (inter + 32 * rb) // 128) if gate_up else \
                    ((64 * rb) // 128,) * 2
                tr = np.zeros(8, dtype=np.float32)
                for half, br in enumerate(blocks):
                    for t in range(4):
                        c = 4 * kc + t
                        if c < scales.shape[1]:
                            tr[4 * half + t] = scales[br, c]
                out[pos:pos + 32] = tr.view(np.uint8)
                pos += 32
    assert pos == out.size
    return out


@pytest.mark.parametrize("wtype,d,inter", [(synth.BF16, 704, 192), (synth.E4M3, 640, 384),
                                           (synth.BF16, 2880, 192)])
def test_pack_layout(mv, wtype, d, inter):
    cfg = synth.LayerConfig("pack", d, 3, 2, inter, synth.BF16, wtype, synth.GATE_SOFTMAX)
    layer = synth.make_layer(cfg, seed=9, device="cuda")
    desc = mv.make_desc(cfg, 4)
    packed = mv.pack_weights(layer, desc)
    torch.cuda.synchronize()
    es = 1 if wtype == synth.E4M3 else 2
    b13, b2 = mv.moe_packed_bytes(desc)
    fp8 = wtype == synth.E4M3
    for e in range(cfg.n_experts):
        for src, dst, sc, gate_up in (
                (layer.w13[e], packed.w13[e * b13:(e + 1) * b13], layer.s13, True),
                (layer.w2[e], packed.w2[e * b2:(e + 1) * b2], layer.s2, False)):
            m = src.contiguous().view(torch.uint8).cpu().numpy().reshape(src.shape[0], -1)
            assert m.shape[1] == src.shape[1] * es
            got = dst.cpu().numpy()
            scales = sc[e].cpu().numpy() if fp8 else None
            assert np.array_equal(got, expected_packed(m, gate_up, inter, scales))


def test_pack_fp32_is_a_copy(mv):
    cfg = synth.shrink(synth.TINY, d=64, inter=16, n_experts=2)
    layer = synth.make_layer(cfg, device="cuda")
    packed = mv.pack_weights(layer, mv.make_desc(cfg, 2))
    torch.cuda.synchronize()
    assert torch.equal(packed.w13, layer.w13.contiguous().view(torch.uint8).ravel())
    assert torch.equal(packed.w2, layer.w2.contiguous().view(torch.uint8).ravel())
