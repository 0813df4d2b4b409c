"""Pins of the oracle's RMSNorm -> indexed AdaLN scale/shift modulation step
(TeleFuser PR #37 section 2.5: RMSNorm then indexed scale/shift, bf16
store/load boundaries of the unfused path preserved).

Checked against things other than the function itself: torch's float64
``rms_norm`` and ``addcmul`` (library routines) with the same bf16 boundaries,
the Q/K norm oracle (separate code) for the norm part, closed forms
(scale = -1 leaves exactly the shift, scale = 1 doubles the norm, zero
modulation leaves the norm), index semantics (a table whose row i is the
constant i), unit RMS, and the rounding bound between the fp64 definition
and the float32 emulation that the CUDA kernel must match bit for bit.
"""
import numpy as np
import torch

import h3inputs as gen
import oracle


def _f32(bits):
    return gen.bf16_bits_to_f32(bits)


def _bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _case(T=40, C=264, N=5, seed=0):
    x = gen.normal_bshd(1, T, 1, C, seed, gen.STREAM_Q)[0, :, 0].copy()
    sc = gen.normal_bshd(1, N, 1, C, seed, gen.STREAM_K, 0.3)[0, :, 0].copy()
    sh = gen.normal_bshd(1, N, 1, C, seed, gen.STREAM_V, 0.3)[0, :, 0].copy()
    idx = gen.uniform_int(T, seed, gen.STREAM_KVLEN, 0, N - 1).astype(np.int32)
    w = gen.uniform_f32(C, seed, gen.STREAM_WQ, 0.5, 1.5)
    return x, w, sc, sh, idx


def _to_bf16(t):
    return t.to(torch.bfloat16).double()


def test_matches_torch_library_path_f64():
    x, w, sc, sh, idx = _case(seed=1)
    C = x.shape[1]
    xt = torch.from_numpy(_f32(x).astype(np.float64))
    n = _to_bf16(torch.nn.functional.rms_norm(xt, (C,), weight=torch.from_numpy(w.astype(np.float64)), eps=1e-6))
    it = torch.from_numpy(idx.astype(np.int64))
    a = _to_bf16(1.0 + torch.from_numpy(_f32(sc).astype(np.float64))[it])
    m = _to_bf16(n * a)
    y = _to_bf16(torch.addcmul(torch.from_numpy(_f32(sh).astype(np.float64))[it], m, torch.ones_like(m)))
    got = oracle.rmsnorm_modulate_f64(x, w, sc, sh, idx, 1e-6)
    np.testing.assert_array_equal(_f32(got).astype(np.float64), y.numpy())


def test_norm_part_matches_qk_norm_oracle():
    # zero modulation leaves bf16(x * r * w); the Q/K norm oracle (separate code,
    # rotary_dim 0) computes the same norm over rows of 128 channels
    x, w, sc, sh, idx = _case(T=12, C=128, N=1, seed=2)
    zero = np.zeros((1, 128), np.uint16)
    got = oracle.rmsnorm_modulate_f64(x, w, zero, zero, None, 1e-6)
    ref = oracle.round_to_bf16(oracle.qk_norm_rope_f64(x[None, :, None, :], w, None, None, 0, 1e-6,
                                                       round_boundary=False))[0, :, 0]
    np.testing.assert_array_equal(got, ref)


def test_scale_minus_one_leaves_the_shift_and_scale_one_doubles():
    x, w, _, sh, idx = _case(T=16, C=64, N=3, seed=3)
    minus1 = np.full((3, 64), _bits([-1.0])[0], np.uint16)
    for fn in (oracle.rmsnorm_modulate_f64, oracle.rmsnorm_modulate_emulate):
        y = fn(x, w, minus1, sh, idx, 1e-6)
        np.testing.assert_array_equal(y, sh[idx], err_msg=fn.__name__)
    one = np.full((1, 64), _bits([1.0])[0], np.uint16)
    zero = np.zeros((1, 64), np.uint16)
    n = oracle.rmsnorm_modulate_f64(x, w, zero, zero, None, 1e-6)
    y = oracle.rmsnorm_modulate_f64(x, w, one, zero, None, 1e-6)
    np.testing.assert_array_equal(_f32(y), 2.0 * _f32(n))


def test_index_selects_table_rows_and_out_of_range_rows_are_zero():
    T, C, N = 9, 32, 4
    x, w, _, _, _ = _case(T=T, C=C, N=N, seed=4)
    minus1 = np.full((N, C), _bits([-1.0])[0], np.uint16)
    rows = np.repeat(_bits(np.arange(N, dtype=np.float32))[:, None], C, axis=1)  # table row i is the constant i
    idx = np.array([3, 0, 2, 1, 3, -1, 4, 2, 0], np.int32)
    for fn in (oracle.rmsnorm_modulate_f64, oracle.rmsnorm_modulate_emulate):
        y = _f32(fn(x, w, minus1, rows, idx, 1e-6))
        for t in range(T):
            want = float(idx[t]) if 0 <= idx[t] < N else 0.0
            assert np.all(y[t] == want), (fn.__name__, t, y[t][:3])
    # no index array == every row uses table row 0
    a = oracle.rmsnorm_modulate_f64(x, w, minus1, rows, None, 1e-6)
    b = oracle.rmsnorm_modulate_f64(x, w, minus1, rows, np.zeros(T, np.int32), 1e-6)
    np.testing.assert_array_equal(a, b)


def test_unit_rms_without_weight():
    x, _, _, _, _ = _case(T=8, C=4096, N=1, seed=5)
    zero = np.zeros((1, 4096), np.uint16)
    y = _f32(oracle.rmsnorm_modulate_f64(x, None, zero, zero, None, 0.0)).astype(np.float64)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1.0, rtol=2e-3)  # bf16 rounding of each element


def test_emulation_within_rounding_of_definition():
    x, w, sc, sh, idx = _case(T=2000, C=264, N=5, seed=6)
    e = _f32(oracle.rmsnorm_modulate_emulate(x, w, sc, sh, idx, 1e-6)).astype(np.float64)
    d = _f32(oracle.rmsnorm_modulate_f64(x, w, sc, sh, idx, 1e-6)).astype(np.float64)
    # the float32 norm value can round to the neighbouring bf16 number near a
    # tie; the later steps carry at most a few bf16 quanta of that
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(d), 2.0 ** -126))) - 7)
    assert np.all(np.abs(e - d) <= 4 * ulp + 2.0 ** -24)
    assert np.mean(e != d) < 2e-3
