"""Pins of the oracle's Q/K RMSNorm -> bf16 boundary -> partial RoPE step.

The oracle is checked against things other than itself: torch's float64
``rms_norm`` (a library routine), closed forms (constant rows, quarter-turn
and half-turn rotations), numpy complex multiplication (rotation of a
complex number), invariants (unit RMS, pair norms, pass-through channels,
position 0) and the rounding bound between the fp64 definition and the
float32 emulation that the CUDA kernel must match bit for bit.
"""
import numpy as np
import pytest
import torch

import h3inputs as gen
import oracle

D = 128
R = 96
HALF = R // 2


def _x(B=2, S=16, H=3, seed=0, std=1.0, off=0.0):
    return gen.normal_bshd(B, S, H, D, seed, gen.STREAM_Q, std, off)


def _f64(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


def _bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def test_rmsnorm_matches_torch_rms_norm_f64():
    x = _x(seed=1)
    w = gen.uniform_f32(D, 1, gen.STREAM_WQ, 0.5, 1.5)
    y = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=False)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(_f64(x)), (D,), weight=torch.from_numpy(w.astype(np.float64)),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_unit_rms_before_weight():
    x = _x(seed=2, std=3.0)
    y = oracle.qk_norm_rope_f64(x, np.ones(D, np.float32), None, None, 0, 1e-6, round_boundary=False)
    xf = _f64(x)
    ms = (xf ** 2).mean(-1)
    rms_y = np.sqrt((y ** 2).mean(-1))
    np.testing.assert_allclose(rms_y ** 2, ms / (ms + 1e-6), rtol=1e-12)
    np.testing.assert_allclose(rms_y, 1.0, rtol=1e-6)


def test_constant_row_closed_form():
    c = 0.75  # exact in bf16
    x = np.full((1, 4, 2, D), np.float32(c).view(np.uint32) >> 16, dtype=np.uint16)
    w = gen.uniform_f32(D, 3, gen.STREAM_WQ, 0.5, 1.5)
    eps = 1e-3
    y = oracle.qk_norm_rope_f64(x, w, None, None, 0, eps, round_boundary=False)
    expect = c / np.sqrt(c * c + eps) * w.astype(np.float64)
    np.testing.assert_allclose(y, np.broadcast_to(expect, y.shape), rtol=1e-14)


def test_scale_invariance_eps0():
    x = _x(seed=4)
    x2 = (gen.bf16_bits_to_f32(x) * 2.0).view(np.uint32) >> 16  # exact doubling
    x2 = x2.astype(np.uint16)
    w = gen.uniform_f32(D, 4, gen.STREAM_WQ, 0.5, 1.5)
    a = oracle.qk_norm_rope_f64(x, w, None, None, 0, 0.0, round_boundary=False)
    b = oracle.qk_norm_rope_f64(x2, w, None, None, 0, 0.0, round_boundary=False)
    np.testing.assert_allclose(a, b, rtol=1e-14)


def test_boundary_is_a_bf16_rounding_of_the_norm():
    x = _x(seed=5)
    w = gen.uniform_f32(D, 5, gen.STREAM_WQ, 0.5, 1.5)
    exact = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=False)
    bounded = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=True)
    # With no rotation the output is the boundary value itself: the nearest
    # bf16 of the exact norm (ties to even).
    np.testing.assert_array_equal(oracle.round_to_bf16(exact), oracle.round_to_bf16(bounded))
    np.testing.assert_array_equal(bounded, _f64(oracle.round_to_bf16(exact)))


def _tables(S, cval, sval):
    return np.full((S, HALF), cval, np.float32), np.full((S, HALF), sval, np.float32)


def test_quarter_turn_and_half_turn():
    S = 4
    x = _x(B=1, S=S, H=2, seed=6)
    w = np.ones(D, np.float32)
    n = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=True)
    c, s = _tables(S, 0.0, 1.0)  # +90 degrees: (a, b) -> (-b, a)
    y = oracle.qk_norm_rope_f64(x, w, c, s, R, 1e-6, round_boundary=True)
    np.testing.assert_array_equal(y[..., :HALF], -n[..., HALF:R])
    np.testing.assert_array_equal(y[..., HALF:R], n[..., :HALF])
    np.testing.assert_array_equal(y[..., R:], n[..., R:])
    c, s = _tables(S, -1.0, 0.0)  # 180 degrees: negation
    y = oracle.qk_norm_rope_f64(x, w, c, s, R, 1e-6, round_boundary=True)
    np.testing.assert_array_equal(y[..., :R], -n[..., :R])


def test_rotation_is_complex_multiplication():
    S = 64
    x = _x(B=1, S=S, H=3, seed=7)
    w = gen.uniform_f32(D, 7, gen.STREAM_WQ, 0.5, 1.5)
    c, s = gen.rope_tables(S, R)
    n = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=True)
    y = oracle.qk_norm_rope_f64(x, w, c, s, R, 1e-6, round_boundary=True)
    z = (n[..., :HALF] + 1j * n[..., HALF:R]) * (c.astype(np.float64) + 1j * s.astype(np.float64))[None, :, None, :]
    np.testing.assert_allclose(y[..., :HALF], z.real, rtol=0, atol=1e-14)
    np.testing.assert_allclose(y[..., HALF:R], z.imag, rtol=0, atol=1e-14)


def test_pair_norm_preserved_and_position_zero_identity():
    S = 128
    x = _x(B=2, S=S, H=2, seed=8, off=0.5)
    w = gen.uniform_f32(D, 8, gen.STREAM_WK, 0.5, 1.5)
    c, s = gen.rope_tables(S, R)
    # the table itself: cos^2 + sin^2 = 1 to float rounding
    np.testing.assert_allclose(c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2, 1.0, atol=2e-7)
    n = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6, round_boundary=True)
    y = oracle.qk_norm_rope_f64(x, w, c, s, R, 1e-6, round_boundary=True)
    cs2 = (c.astype(np.float64) ** 2 + s.astype(np.float64) ** 2)[None, :, None, :]
    lhs = y[..., :HALF] ** 2 + y[..., HALF:R] ** 2
    rhs = (n[..., :HALF] ** 2 + n[..., HALF:R] ** 2) * cs2
    np.testing.assert_allclose(lhs, rhs, rtol=1e-13, atol=1e-300)
    np.testing.assert_array_equal(y[..., R:], n[..., R:])  # channels 96..127 untouched
    np.testing.assert_array_equal(y[:, 0], n[:, 0])        # position 0: identity


def test_positions_follow_sequence_index_not_head_or_batch():
    S, H = 8, 3
    x = _x(B=2, S=S, H=H, seed=9)
    w = np.ones(D, np.float32)
    c, s = gen.rope_tables(S, R)
    y = oracle.qk_norm_rope_f64(x, w, c, s, R, 1e-6)
    for b in range(2):
        for pos in range(S):
            for h in range(H):
                xs = x[b:b + 1, pos:pos + 1, h:h + 1]
                one = oracle.qk_norm_rope_f64(xs, w, c[pos:pos + 1], s[pos:pos + 1], R, 1e-6)
                np.testing.assert_array_equal(one[0, 0, 0], y[b, pos, h])


@pytest.mark.parametrize("Dd,Rr", [(128, 96), (64, 32), (256, 96), (128, 128), (128, 0),
                                   # rotary_dim even but not a multiple of 16
                                   (128, 2), (128, 24), (128, 40), (128, 94), (64, 62), (256, 250)])
def test_emulation_within_rounding_bound_of_fp64(Dd, Rr):
    B, S, H = 2, 96, 4
    half = Rr // 2
    x = gen.normal_bshd(B, S, H, Dd, 10, gen.STREAM_Q, 1.0, 0.5)
    w = gen.uniform_f32(Dd, 10, gen.STREAM_WQ, 0.5, 1.5)
    c, s = gen.rope_tables(S, Rr) if Rr else (None, None)
    exact = oracle.qk_norm_rope_f64(x, w, c, s, Rr, 1e-6)
    emu = _f64(oracle.qk_norm_rope_emulate(x, w, c, s, Rr, 1e-6))
    n = oracle.qk_norm_rope_f64(x, w, None, None, 0, 1e-6)  # boundary values
    # The emulation's boundary value can land one bf16 step from the fp64 one
    # when the norm sits next to a rounding tie.  After the rotation that step
    # is carried by a pair of magnitude |(a, b)|, and the final store adds at
    # most half a step of the output: |emu - exact| <= ulp(y) + 2 ulp(|(a,b)|).
    mag = np.abs(n).copy()
    if half:
        pair = np.sqrt(n[..., :half] ** 2 + n[..., half:Rr] ** 2)
        mag[..., :half] = pair
        mag[..., half:Rr] = pair
    bound = _bf16_ulp(exact) + 2.0 * _bf16_ulp(mag)
    assert np.all(np.abs(emu - exact) <= bound)
    # and a disagreement with the correctly rounded fp64 value is rare
    mismatch = np.mean(oracle.round_to_bf16(exact) != oracle.round_to_bf16(emu))
    assert mismatch < 1e-3, mismatch
    # channels that are not rotated differ by at most the boundary rounding
    assert np.all(np.abs(emu - exact)[..., Rr:] <= _bf16_ulp(exact)[..., Rr:])


def test_emulation_exact_on_closed_forms():
    c0 = 0.75
    x = np.full((1, 2, 1, D), np.float32(c0).view(np.uint32) >> 16, dtype=np.uint16)
    w = np.ones(D, np.float32)
    cos, sin = _tables(2, 0.0, 1.0)
    out = _f64(oracle.qk_norm_rope_emulate(x, w, cos, sin, R, 0.0))
    # a constant row normalises to exactly 1; the quarter turn maps (1, 1) -> (-1, 1)
    np.testing.assert_array_equal(out[..., :HALF], -1.0)
    np.testing.assert_array_equal(out[..., HALF:], 1.0)


def test_emulation_reduction_order_is_the_specified_tree():
    """Cross-check (not a pin): the emulation follows the stated lane/butterfly
    order, which can differ from a left-to-right float32 sum."""
    rng = np.random.default_rng(0)
    vals = rng.standard_normal((1, 1, 64, D)).astype(np.float32) * np.float32(3.0)
    x = (vals.view(np.uint32) >> 16).astype(np.uint16)
    w = np.ones(D, np.float32)
    emu = oracle.qk_norm_rope_emulate(x, w, None, None, 0, 1e-6)
    xf = gen.bf16_bits_to_f32(x)
    # Independent restatement of the tree in numpy float32
    parts = np.zeros(x.shape[:-1] + (D // 8,), np.float32)
    for e in range(8):
        xe = xf.reshape(x.shape[:-1] + (D // 8, 8))[..., e]
        parts = (xe.astype(np.float64) * xe + parts).astype(np.float32)  # fma: exact product, one rounding
    L = D // 8
    off = L // 2
    while off >= 1:
        parts = (parts + parts[..., np.arange(L) ^ off]).astype(np.float32)
        off //= 2
    ms = parts[..., 0] * np.float32(1.0 / D)
    r = np.float32(1.0) / np.sqrt(ms + np.float32(1e-6), dtype=np.float32)
    n = (xf * r[..., None]).astype(np.float32) * w
    ref = ((n.view(np.uint32) + 0x7FFF + ((n.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)
    np.testing.assert_array_equal(emu, ref)
