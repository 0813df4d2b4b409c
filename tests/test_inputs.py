"""The seeded input generator: deterministic, thread-count independent,
distributed as stated, and the workload table matches the stated shapes."""
import numpy as np

import h3inputs as gen


def test_deterministic_and_thread_independent():
    a = gen.normal_bshd(2, 64, 3, 128, 42, gen.STREAM_Q, nthreads=1)
    b = gen.normal_bshd(2, 64, 3, 128, 42, gen.STREAM_Q, nthreads=7)
    np.testing.assert_array_equal(a, b)
    c = gen.normal_bshd(2, 64, 3, 128, 42, gen.STREAM_K)
    d = gen.normal_bshd(2, 64, 3, 128, 43, gen.STREAM_Q)
    assert np.mean(a == c) < 0.05 and np.mean(a == d) < 0.05


def test_normal_moments_and_offsets():
    x = gen.bf16_bits_to_f32(gen.normal_bshd(1, 4096, 4, 128, 0, gen.STREAM_Q)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    y = gen.bf16_bits_to_f32(gen.normal_bshd(1, 4096, 4, 128, 0, gen.STREAM_Q, 1.0, 0.5)).astype(np.float64)
    off = (y - x).mean(axis=(0, 1))  # per (head, channel) offset, shared by all tokens
    assert abs(off.std() - 0.5) < 0.05
    np.testing.assert_allclose((y - x).std(axis=(0, 1)), 0.0, atol=0.02)


def test_uniform_ranges_and_tables():
    w = gen.uniform_f32(10000, 1, gen.STREAM_WQ, 0.5, 1.5)
    assert w.min() >= 0.5 and w.max() < 1.5 and abs(w.mean() - 1.0) < 0.01
    n = gen.uniform_int(10000, 1, gen.STREAM_KVLEN, 4096, 8192)
    assert n.min() >= 4096 and n.max() <= 8192
    c, s = gen.rope_tables(16, 96)
    assert c.shape == (16, 48)
    np.testing.assert_array_equal(c[0], 1.0)
    np.testing.assert_array_equal(s[0], 0.0)
    np.testing.assert_allclose(c[3, 0], np.float32(np.cos(3.0)))
    np.testing.assert_allclose(s[5, 47], np.float32(np.sin(5.0 * 10000.0 ** (-94.0 / 96.0))))


def test_bits_layout():
    m = gen.bernoulli_bits(2, 5, 70, 0, gen.STREAM_BITS, 0.5)
    assert m.shape == (2, 5, 3)
    assert np.all(m[:, :, 2] >> np.uint32(6) == 0)  # keys >= 70 are clear


def test_workload_shapes():
    wl = gen.WORKLOADS
    assert (wl["long_video_h24"].Sq, wl["long_video_h24"].Hq, wl["long_video_h24"].D) == (32760, 24, 128)
    assert (wl["padded_gqa"].Hq, wl["padded_gqa"].Hkv, wl["padded_gqa"].B) == (16, 4, 4)
    assert wl["packed_clip_cross"].Sk == 512 and wl["packed_clip_self"].kv_len_range == (100000, 100000)
    inp = gen.make_inputs(wl["tiny_mha"], 0)
    assert inp.q.shape == (1, 256, 4, 128) and inp.cos.shape == (256, 48)
