"""Pins of the LM-head oracle (oracle/lmhead.py): the bf16 rounding against
hand-computed encodings, and the projection against a triple loop."""
import numpy as np
import pytest

from oracle import lmhead as LM

# (value, bf16 bits): encodings written out by hand from the format (1 sign,
# 8 exponent bits with bias 127, 7 stored fraction bits)
CASES = [
    (1.0, 0x3F80),
    (-2.5, 0xC020),                      # -1.25 * 2^1
    (1.0 + 2.0 ** -8, 0x3F80),           # halfway between 1 and 1 + 2^-7: ties to even (down)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),       # halfway between 1 + 2^-7 and 1 + 2^-6: ties to even (up)
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # just above the tie: up
    (1.0 + 2.0 ** -8 - 2.0 ** -30, 0x3F80),  # just below the tie: down
    (float.fromhex("0x1.fep127"), 0x7F7F),   # largest finite
    (float.fromhex("0x1.fep127") + float.fromhex("0x1p119"), 0x7F80),  # tie at the top: infinity
    (float.fromhex("0x1.fep127") + float.fromhex("0x0.fp119"), 0x7F7F),  # below that tie
    (-3.0e38 * 2, 0xFF80),
    (2.0 ** -126, 0x0080),               # smallest normal
    (2.0 ** -130, 0x0008),               # subnormal: 8 * 2^-133
    (2.0 ** -133, 0x0001),               # smallest subnormal
    (2.0 ** -134, 0x0000),               # half of it: ties to even (zero)
    (3 * 2.0 ** -134, 0x0002),           # 1.5 quanta: ties to even (2)
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (float("inf"), 0x7F80),
    (65504.0, 0x4780),                   # 1.9990234375 * 2^15 -> 2^16 after rounding
    (0.1, 0x3DCD),                       # 0x3DCCCCCD in f32 rounds up
]


@pytest.mark.parametrize("x,bits", CASES)
def test_bf16_rounding(x, bits):
    assert int(LM.f64_to_bf16_bits(np.array([x]))[0]) == bits


def test_bf16_nan_and_roundtrip():
    assert int(LM.f64_to_bf16_bits(np.array([float("nan")]))[0]) & 0x7FFF > 0x7F80
    every = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = LM.bf16_bits_to_f64(every)
    fin = np.isfinite(vals)
    back = LM.f64_to_bf16_bits(vals[fin])
    # every finite encoding is its own rounding, except -0 / +0 keep their sign
    assert np.array_equal(back, every[fin])


def test_projection_matches_triple_loop():
    rng = np.random.default_rng(0)
    R, H, V = 3, 7, 5
    h = LM.f64_to_bf16_bits(rng.normal(0, 1, (R, H)))
    w = LM.f64_to_bf16_bits(rng.normal(0, 1, (V, H)))
    hf, wf = LM.bf16_bits_to_f64(h), LM.bf16_bits_to_f64(w)
    ref = np.zeros((R, V))
    for r in range(R):
        for v in range(V):
            s = 0.0
            for k in range(H):
                s += hf[r, k] * wf[v, k]
            ref[r, v] = s
    got = LM.lmhead_logits_f64(h, w)
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-15)
    assert np.array_equal(LM.lmhead_logits(h, w), LM.f64_to_bf16_bits(ref))
    # operands are not swapped: a non-square case keeps [R, V]
    assert LM.lmhead_logits(h, w).shape == (R, V)
