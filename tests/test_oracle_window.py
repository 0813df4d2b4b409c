"""Pins of the oracle's chunked-window attention (SGLang PR #37903
"[diffusion] model: support VDN-H3 ...", section "Modifications",
hybrid_window_attn_h3: chunk-5 / radius-1 window with anchor frames,
dense-query rows against all keys; "Accuracy Tests": the anchor frames shift
the chunk grid).

Checked against things other than the window code itself: a boolean mask
enumerated frame by frame on tiny inputs and run through the oracle's
bit-mask path (separate code), dense attention where the window covers
everything, anchor rows equal to dense rows, keys outside every window
poisoned with NaN, and the interval count of allowed pairs against the
enumerated mask."""
import numpy as np
import pytest

import h3inputs as gen
import oracle


def _mask_by_frames(S, F, A, K, r):
    """allowed[i, j], enumerated from frames: frame f = t // F; frames < A
    are anchors; other frames belong to chunk (f - A) // K."""
    frame = np.arange(S) // F
    anchor = frame < A
    chunk = np.where(anchor, -1, (frame - A) // K)
    m = np.zeros((S, S), dtype=bool)
    for i in range(S):
        for j in range(S):
            m[i, j] = anchor[i] or anchor[j] or abs(chunk[i] - chunk[j]) <= r
    return m


def _pack(m):
    S, Sk = m.shape
    W = (Sk + 31) // 32
    bits = np.zeros((S, W), np.uint32)
    for j in range(Sk):
        bits[:, j >> 5] |= (m[:, j].astype(np.uint32) << np.uint32(j & 31))
    return bits


def _qkv(B, S, H, D, seed):
    return (gen.normal_bshd(B, S, H, D, seed, gen.STREAM_Q), gen.normal_bshd(B, S, H, D, seed, gen.STREAM_K),
            gen.normal_bshd(B, S, H, D, seed, gen.STREAM_V))


@pytest.mark.parametrize("S,F,A,K,r", [(60, 4, 1, 2, 1), (77, 5, 2, 3, 0), (64, 8, 0, 1, 1), (50, 3, 0, 5, 2)])
def test_window_equals_enumerated_mask(S, F, A, K, r):
    q, k, v = _qkv(2, S, 2, 64, S + F)
    m = _mask_by_frames(S, F, A, K, r)
    bits = np.broadcast_to(_pack(m), (2,) + _pack(m).shape).copy()
    ref = oracle.attention_f64(q, k, v, 0.125, bits=bits)
    got = oracle.attention_window_f64(q, k, v, 0.125, F, A, K, r)
    np.testing.assert_array_equal(got, ref)
    assert oracle.window_allowed_pairs(S, S, F, A, K, r) == int(m.sum())


def test_window_covering_everything_is_dense():
    q, k, v = _qkv(1, 90, 3, 64, 1)
    dense = oracle.attention_f64(q, k, v, 0.1)
    np.testing.assert_array_equal(oracle.attention_window_f64(q, k, v, 0.1, 10, 1, 2, 5), dense)
    np.testing.assert_array_equal(oracle.attention_window_f64(q, k, v, 0.1, 3, 0, 30, 0), dense)


def test_anchor_rows_are_dense_and_padding_applies():
    S, F, A = 80, 8, 2
    q, k, v = _qkv(1, S, 2, 64, 2)
    kv_len = np.array([70], np.int32)
    dense = oracle.attention_f64(q, k, v, 0.1, kv_len=kv_len)
    win = oracle.attention_window_f64(q, k, v, 0.1, F, A, 1, 1, kv_len=kv_len)
    np.testing.assert_array_equal(win[:, :A * F], dense[:, :A * F])
    assert oracle.window_allowed_pairs(S, 70, F, A, 1, 1) == int(
        (_mask_by_frames(S, F, A, 1, 1) & (np.arange(S)[None, :] < 70)).sum())


def test_keys_outside_every_window_never_attended():
    S, F, A, K, r = 96, 8, 1, 2, 0
    q, k, v = _qkv(1, S, 1, 64, 3)
    base = oracle.attention_window_f64(q, k, v, 0.2, F, A, K, r)
    # query rows of chunk 0 (tokens 8..23) see anchors 0..7 and chunk 0 only:
    # poison every key of chunks >= 1 (tokens >= 24)
    k2, v2 = k.copy(), v.copy()
    k2[:, 24:] = 0x7FC0
    v2[:, 24:] = 0x7FC0
    poisoned = oracle.attention_window_f64(q, k2, v2, 0.2, F, A, K, r)
    np.testing.assert_array_equal(poisoned[:, 8:24], base[:, 8:24])
