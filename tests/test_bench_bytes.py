"""Algorithmic bytes of the bench's roofline, against the block format worked by hand.

A 32-weight block is 16 bytes of nibbles plus a 2-byte fp16 scale (18 bytes, 0.5625
byte per weight); a union expert streams its gate, up and down matrices (3 * H * I
weights) once per layer, the router is E * H fp32, and each row brings H bf16
activations in and takes H fp32 outputs out.
"""
import pytest

import bench
import syngen


def _by_hand(H, E, I, U, R):
    blocks = 3 * H * I // 32
    return U * blocks * 18 + E * H * 4 + R * H * (2 + 4)


def test_a3b_one_row_layer_is_22_29_mb():
    cfg = syngen.CONFIGS["a3b_r1"]
    # 8 experts x 2,654,208 B + the 1 MiB router + 4 KB in and 8 KB out
    assert bench.layer_bytes(cfg, 8, 1) == 21_233_664 + 1_048_576 + 12_288
    assert cfg.expert_bytes == 2_654_208


def test_e512_three_row_layer():
    cfg = syngen.CONFIGS["e512_r3"]
    assert cfg.expert_bytes == 1_769_472
    assert bench.layer_bytes(cfg, 10, 3) == 10 * 1_769_472 + 4_194_304 + 36_864


@pytest.mark.parametrize("name", ["tiny", "a3b_r1", "a3b_r4", "a3b_r16", "e512_r3"])
@pytest.mark.parametrize("U,R", [(1, 1), (8, 1), (17, 4), (28, 16)])
def test_layer_bytes_match_the_block_format(name, U, R):
    cfg = syngen.CONFIGS[name]
    assert bench.layer_bytes(cfg, U, R) == _by_hand(cfg.hidden, cfg.experts, cfg.inter, U, R)
