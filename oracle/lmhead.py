"""Float64 oracle of the LM-head projection that produces the target's logits.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same rule as the rest of ``oracle/``:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
use it).

The target scores the drafts with one forward pass whose last step is the
vocabulary projection ("投机采样", 第二步: one target pass yields the
distributions p_1 .. p_{gamma+1}); the logits are the last hidden state times
the LM-head matrix.  Here that is written out plainly: both bf16 operands are
widened to float64, multiplied with a library matmul (exact products,
float64 sums), and every logit is rounded once to the nearest bf16 value,
ties to even, as a bf16 logits tensor stores it.

Pins (tests/test_oracle_lmhead.py): the rounding against hand-computed bf16
encodings (ties to even both ways, the overflow threshold, subnormals, signs,
NaN), and the matmul path against a triple loop on tiny shapes.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")      # largest finite bf16 (0x7F7F)
_HALF_ULP_AT_MAX = float.fromhex("0x1p119")  # half an ulp at the top binade


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even) -> uint16 bits.

    bf16 has 8 significant bits; normal numbers from 2^-126, subnormals
    down to 2^-133 in steps of 2^-133.  Values whose magnitude reaches
    BF16_MAX + half an ulp round to infinity (the tie there goes to the even
    encoding, which is infinity).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    nan = np.isnan(x)
    ax = np.abs(x)
    big = ax >= BF16_MAX + _HALF_ULP_AT_MAX
    fin = ~nan & ~big & np.isfinite(x)
    # quantum of the bf16 grid at each magnitude: 2^(e - 8) for 2^(e-1) <= |x| < 2^e
    # (frexp gives |x| = m 2^e with 0.5 <= m < 1), never finer than 2^-133
    _, e = np.frexp(np.where(fin & (ax > 0), ax, 1.0))
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(np.where(fin, x, 0.0) / q) * q  # np.rint: ties to even
    out[fin] = r[fin]
    out[big] = np.copysign(np.inf, x[big])
    out[~nan & np.isinf(x)] = x[~nan & np.isinf(x)]
    bits = (out.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits[nan] = 0x7FC0
    return bits


def lmhead_logits(hidden_bits: np.ndarray, weight_bits: np.ndarray) -> np.ndarray:
    """logits[r, v] = bf16( sum_h hidden[r, h] * W[v, h] ) from bf16 bit patterns.

    hidden_bits: [R, H] uint16; weight_bits: [V, H] uint16; returns [R, V] uint16.
    """
    h = bf16_bits_to_f64(hidden_bits)
    w = bf16_bits_to_f64(weight_bits)
    return f64_to_bf16_bits(h @ w.T)


def lmhead_logits_f64(hidden_bits: np.ndarray, weight_bits: np.ndarray) -> np.ndarray:
    """The same projection before the bf16 rounding (float64)."""
    return bf16_bits_to_f64(hidden_bits) @ bf16_bits_to_f64(weight_bits).T
