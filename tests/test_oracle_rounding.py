"""Direct pins of the oracle's fp64 -> bf16 rounding (one rounding to nearest,
ties to even, with bf16's subnormal quantum 2^-133 and overflow to infinity).

Two independent sources: hand-derived values (ties on both sides, the
subnormal range, the overflow threshold) and torch's float32 -> bfloat16
conversion (a library routine, round to nearest even) on float32-representable
inputs, where one rounding of the fp64 value and one of the float32 value
coincide."""
import numpy as np
import torch

import oracle


def _bits(x):
    return oracle.round_to_bf16(np.asarray(x, dtype=np.float64))


def _val(bits):
    return float((np.asarray(bits, np.uint32).reshape(-1) << 16).view(np.float32)[0])


def test_ties_go_to_even_on_both_sides():
    # 1 + 2^-8 lies halfway between 1 (even) and 1 + 2^-7 (odd): down to 1
    assert _val(_bits(1.0 + 2.0 ** -8)) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 (odd) and 1 + 2^-6 (even): up
    assert _val(_bits(1.0 + 3 * 2.0 ** -8)) == 1.0 + 2.0 ** -6
    # a hair off the tie decides by distance (values only fp64 can hold)
    assert _val(_bits(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 1.0 + 2.0 ** -7
    assert _val(_bits(1.0 + 3 * 2.0 ** -8 - 2.0 ** -40)) == 1.0 + 2.0 ** -7
    # signs are symmetric
    assert _val(_bits(-(1.0 + 3 * 2.0 ** -8))) == -(1.0 + 2.0 ** -6)
    assert _val(_bits(-(1.0 + 2.0 ** -8))) == -1.0


def test_subnormal_quantum_and_the_clamp():
    q = 2.0 ** -133  # smallest bf16 subnormal; the quantum of the whole subnormal range
    assert _bits(q) == 0x0001
    assert _bits(2.0 ** -134) == 0x0000          # halfway 0 / q: to even (0)
    assert _bits(3 * 2.0 ** -134) == 0x0002      # halfway q / 2q: to even (2q)
    assert _bits(0.75 * q) == 0x0001             # above half: up to q
    assert _bits(2.0 ** -140) == 0x0000          # far below half: 0
    assert _bits(-2.0 ** -140) == 0x8000         # negative zero keeps its sign
    assert _bits(5 * q + 0.5 * q) == 0x0006      # 5.5 q: halfway 5q / 6q, to even
    # the largest subnormal and the smallest normal
    assert _bits(127 * q) == 0x007F
    assert _bits(2.0 ** -126) == 0x0080
    # a value between them that needs the clamp (exponent below -126 but
    # eight significant bits would ask for a finer quantum than 2^-133)
    assert _bits(2.0 ** -127 + 2.0 ** -134) == 0x0040  # halfway 64q / 65q: to even (64q)


def test_overflow_threshold():
    maxbf = (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert _bits(maxbf) == 0x7F7F
    half_ulp = 2.0 ** (127 - 8)
    assert _bits(maxbf + half_ulp - 2.0 ** 100) == 0x7F7F  # below the midpoint
    assert _bits(maxbf + half_ulp) == 0x7F80                # midpoint: to even, which is infinity
    assert _bits(1e300) == 0x7F80
    assert _bits(-1e300) == 0xFF80
    assert _bits(np.inf) == 0x7F80
    assert np.isnan(_val(_bits(np.nan)))


def test_agrees_with_torch_float32_to_bfloat16():
    rng = np.random.default_rng(5)
    # every exponent band, subnormal floats included, and exact ties
    mant = rng.integers(0, 1 << 23, size=40000, dtype=np.uint32)
    expo = rng.integers(0, 255, size=40000, dtype=np.uint32)
    sign = rng.integers(0, 2, size=40000, dtype=np.uint32)
    f = ((sign << 31) | (expo << 23) | mant).view(np.float32)
    ties = ((rng.integers(0, 1 << 15, size=2000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, np.float32([3.3e38, 3.39e38, -3.4e38, 1e-45, -1e-40])])
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(_bits(f.astype(np.float64)), ref)
