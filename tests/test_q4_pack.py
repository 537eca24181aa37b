"""The library's 4-bit packer (host code) against the oracle's quantiser: the
same codes and block scales bit for bit, read back from the documented
layout (no GPU)."""
import numpy as np
import pytest
import torch

import oracle


@pytest.fixture(scope="module")
def es():
    from routed_expert_ffn_topk_gb300 import estream
    estream.lib()
    return estream


def decode_plane(raw, rows, cols, tile_rows, fp16):
    """Codes [rows][cols] and scales [rows][cols/32] (fp32) of one packed
    plane: tile-major boxes of tile_rows x 64 weights, each two column blocks
    of codes (block j: every row's 16 bytes of weights 32j..32j+31; byte-word w:
    bits 4i.. weight 32j+8w+2i, bits 16+4i.. weight 32j+8w+2i+1) then the
    rows' two scales."""
    box = tile_rows * 36
    codes = np.zeros((rows, cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.float32)
    o = 0
    for nb in range(rows // tile_rows):
        for kb in range(cols // 64):
            b = raw[o:o + box]
            for j in range(2):
                words = b[j * tile_rows * 16:(j + 1) * tile_rows * 16].view(np.uint32).reshape(tile_rows, 4)
                c0 = kb * 64 + 32 * j
                for i in range(4):
                    codes[nb * tile_rows:(nb + 1) * tile_rows, c0 + 2 * i:c0 + 32:8] = (words >> (4 * i)) & 0xF
                    codes[nb * tile_rows:(nb + 1) * tile_rows, c0 + 2 * i + 1:c0 + 32:8] = (words >> (16 + 4 * i)) & 0xF
            sb = b[tile_rows * 32:].view(np.uint16).reshape(tile_rows, 2)
            if fp16:
                sv = sb.view(np.float16).astype(np.float32)
            else:
                sv = (sb.astype(np.uint32) << 16).view(np.float32)
            scales[nb * tile_rows:(nb + 1) * tile_rows, kb * 2:kb * 2 + 2] = sv
            o += box
    return codes, scales


@pytest.mark.parametrize("G", [1, 3])
def test_q4_pack_matches_oracle(es, G):
    E, H, F = 4, 256, 128
    g = torch.Generator().manual_seed(8)
    Wg = (torch.randn(E, F, H, generator=g) * 0.02).bfloat16()
    Wu = (torch.randn(E, F, H, generator=g) * 0.02).bfloat16()
    Wd = (torch.randn(E, H, F, generator=g) * 0.02).bfloat16()
    Wd[1] *= 300.0
    Wg[2, :5] = 0.0          # whole zero blocks
    Wu[3, 7, 40] = -1.0      # one dominant weight
    perm = torch.randperm(E, generator=g).to(torch.int32)
    d, keep = es.make_desc(1, E, H, F, G, 1, es.Q4, None, [None], perm=perm)
    pool = torch.zeros(es.pool_bytes(E, H, F, es.Q4), dtype=torch.uint8)
    es.pack_experts(d, 0, Wg, Wu, Wd, pool)
    raw = pool.numpy()
    S = H * F * 9 // 16
    W = 3 * S
    assert es.pool_bytes(E, H, F, es.Q4) == E * W + 16
    scales = raw[E * W:E * W + 4 * E].view(np.float32)
    for e in range(E):
        pos = int(perm[e])
        q, r = divmod(pos, G)
        n_q = min(G, E - q * G)
        base = q * G * W
        for name, Wm, off, rows, cols, tr, fp16 in (
                ("gate", Wg, base + r * S, F, H, 128, False),
                ("up", Wu, base + n_q * S + r * S, F, H, 128, False),
                ("down", Wd, base + 2 * n_q * S + r * S, H, F, 256, True)):
            c, s = decode_plane(raw[off:off + S], rows, cols, tr, fp16)
            sexp = oracle.down_scale_exp(Wm[e]) if name == "down" else 0
            co, so = oracle.q4_quantize(Wm[e], fp16=fp16, scale_exp=sexp)
            np.testing.assert_array_equal(c, co, err_msg=f"{name} codes, expert {e}")
            np.testing.assert_array_equal(s, so, err_msg=f"{name} scales, expert {e}")
            if name == "down":
                assert scales[pos] == np.float32(2.0 ** -sexp)
