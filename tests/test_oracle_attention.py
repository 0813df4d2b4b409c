"""Pins of the oracle's dense prefill attention.

Brute force: the definition written out on tiny inputs in long double,
materialising each score matrix (separate code from the oracle's row loop).
Against a library routine: torch's ``scaled_dot_product_attention`` in
float64 on the CPU, with GQA expressed as K/V heads repeated, and the boolean
[Q, K] mask (True = attend) that FastVideo PR #1799 ("Add opt-in FlashInfer
attention backend for Wan", section "Implementation") converts every padding
and causal mask into.  Closed forms: one key, zero scale, constant V, one
dominant key.  Invariants: key permutation, poisoned masked keys, GQA vs
repeated heads, packed-bit mask vs structured mask, fully masked rows.
"""
import zlib

import numpy as np
import pytest
import torch

import h3inputs as gen
import oracle


def _bf(x):
    return gen.bf16_bits_to_f32(x).astype(np.float64)


def _to_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _rand(B, Sq, Sk, Hq, Hkv, D, seed):
    q = gen.normal_bshd(B, Sq, Hq, D, seed, gen.STREAM_Q)
    k = gen.normal_bshd(B, Sk, Hkv, D, seed, gen.STREAM_K)
    v = gen.normal_bshd(B, Sk, Hkv, D, seed, gen.STREAM_V)
    return q, k, v


def _mask_matrix(B, Sq, Sk, causal=False, kv_len=None, q_len=None, causal_b=None, bits=None):
    """Boolean [B, Sq, Sk] attend-mask from the structured fields (test-side)."""
    m = np.ones((B, Sq, Sk), bool)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    for b in range(B):
        if kv_len is not None:
            m[b] &= j < kv_len[b]
        if causal or (causal_b is not None and causal_b[b]):
            m[b] &= j <= i
        if bits is not None:
            m[b] &= ((bits[b][:, j[0] >> 5] >> (j[0] & 31)) & 1).astype(bool)
    return m


def _pack(m):
    B, Sq, Sk = m.shape
    W = (Sk + 31) // 32
    out = np.zeros((B, Sq, W), np.uint32)
    for j in range(Sk):
        out[:, :, j >> 5] |= (m[:, :, j].astype(np.uint32) << np.uint32(j & 31))
    return out


def _sdpa_f64(q, k, v, scale, mask):
    """torch SDPA in float64; q [B,Sq,Hq,D], k/v [B,Sk,Hkv,D] bf16 bits; mask [B,Sq,Sk] bool."""
    Hq, Hkv = q.shape[2], k.shape[2]
    tq = torch.from_numpy(_bf(q)).permute(0, 2, 1, 3)
    tk = torch.from_numpy(_bf(k)).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    tv = torch.from_numpy(_bf(v)).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    tm = torch.from_numpy(mask)[:, None, :, :]
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=tm, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


CASES = [
    # name, B, Sq, Sk, Hq, Hkv, D, causal, kv_len, causal_b, bit-density
    ("self_mha", 1, 48, 48, 2, 2, 32, False, None, None, None),
    ("cross_gqa", 2, 40, 24, 4, 2, 16, False, None, None, None),
    ("causal", 1, 37, 37, 2, 1, 16, True, None, None, None),
    ("causal_padding", 2, 33, 33, 4, 2, 16, False, [20, 33], [1, 0], None),
    ("bits", 2, 29, 45, 2, 2, 16, False, None, None, 0.6),
    ("bits_and_padding_causal", 2, 31, 31, 2, 1, 32, False, [17, 30], [0, 1], 0.7),
]


def _brute_longdouble(q, k, v, scale, mask):
    """The definition written out on tiny inputs, separate from the oracle's
    code: per (sample, head) the whole score matrix in long double, then per
    row the softmax over the allowed keys and the weighted sum of their value
    rows; a row with no allowed key is 0."""
    B, Sq, Hq, D = q.shape
    Hkv = k.shape[2]
    qf, kf, vf = (_bf(x).astype(np.longdouble) for x in (q, k, v))
    out = np.zeros((B, Sq, Hq, D), np.longdouble)
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            scores = (qf[b, :, h, :] @ kf[b, :, kvh, :].T) * np.longdouble(scale)
            for i in range(Sq):
                allowed = mask[b, i]
                if not allowed.any():
                    continue
                s = scores[i, allowed]
                p = np.exp(s - s.max())
                out[b, i, h] = (p[:, None] * vf[b, allowed, kvh, :]).sum(axis=0) / p.sum()
    return out


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_long_double_brute_force(case):
    name, B, Sq, Sk, Hq, Hkv, D, causal, kv_len, causal_b, dens = case
    q, k, v = _rand(B, Sq, Sk, Hq, Hkv, D, seed=zlib.crc32(name.encode()) % 997 + 1)
    kv_len = None if kv_len is None else np.array(kv_len, np.int32)
    causal_b = None if causal_b is None else np.array(causal_b, np.uint8)
    bits = None if dens is None else gen.bernoulli_bits(B, Sq, Sk, 5, gen.STREAM_BITS, dens)
    scale = 1.0 / np.sqrt(D)
    o = oracle.attention_f64(q, k, v, scale, causal, kv_len, None, causal_b, bits)
    ref = _brute_longdouble(q, k, v, scale, _mask_matrix(B, Sq, Sk, causal, kv_len, None, causal_b, bits))
    np.testing.assert_allclose(o, ref.astype(np.float64), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_matches_torch_sdpa_float64(case):
    name, B, Sq, Sk, Hq, Hkv, D, causal, kv_len, causal_b, dens = case
    q, k, v = _rand(B, Sq, Sk, Hq, Hkv, D, seed=zlib.crc32(name.encode()) % 1000)
    kv_len = None if kv_len is None else np.array(kv_len, np.int32)
    causal_b = None if causal_b is None else np.array(causal_b, np.uint8)
    bits = None if dens is None else gen.bernoulli_bits(B, Sq, Sk, 3, gen.STREAM_BITS, dens)
    scale = 1.0 / np.sqrt(D)
    o = oracle.attention_f64(q, k, v, scale, causal, kv_len, None, causal_b, bits)
    m = _mask_matrix(B, Sq, Sk, causal, kv_len, None, causal_b, bits)
    ref = _sdpa_f64(q, k, v, scale, m)
    live = m.any(-1)  # rows with at least one allowed key
    np.testing.assert_allclose(o[live], ref[live], rtol=1e-11, atol=1e-12)
    # rows with no allowed key are 0 (SDPA would give NaN there)
    np.testing.assert_array_equal(o[~live], 0.0)


def test_single_key_returns_its_value():
    q, k, v = _rand(2, 7, 1, 4, 2, 16, seed=11)
    o = oracle.attention_f64(q, k, v, 0.3)
    vv = _bf(v)
    for h in range(4):
        np.testing.assert_array_equal(o[:, :, h, :], np.broadcast_to(vv[:, 0:1, h // 2, :], (2, 7, 16)))


def test_causal_row_zero_returns_first_value():
    q, k, v = _rand(1, 9, 9, 2, 2, 16, seed=12)
    o = oracle.attention_f64(q, k, v, 0.25, causal=True)
    np.testing.assert_array_equal(o[0, 0], _bf(v)[0, 0])


def test_zero_scale_is_mean_of_allowed_values():
    B, S, H, D = 2, 30, 2, 16
    q, k, v = _rand(B, S, S, H, H, D, seed=13)
    kv_len = np.array([11, 30], np.int32)
    o = oracle.attention_f64(q, k, v, 0.0, kv_len=kv_len, causal_b=np.array([1, 0], np.uint8))
    vv = _bf(v)
    for i in range(S):
        lim = min(11, i + 1)
        np.testing.assert_allclose(o[0, i], vv[0, :lim].mean(0), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(o[1], np.broadcast_to(vv[1].mean(0), (S, H, D)), rtol=1e-13, atol=1e-15)


def test_constant_v_gives_constant_output_and_weights_sum_to_one():
    B, Sq, Sk, H, D = 1, 20, 50, 2, 16
    q, k, _ = _rand(B, Sq, Sk, H, H, D, seed=14)
    ones = _to_bits(np.ones((B, Sk, H, D), np.float32))
    o = oracle.attention_f64(q, k, ones, 0.9)
    np.testing.assert_allclose(o, 1.0, rtol=1e-14)  # softmax weights sum to one
    cst = _to_bits(np.full((B, Sk, H, D), -2.5, np.float32))
    o = oracle.attention_f64(q, k, cst, 0.9, kv_len=np.array([7], np.int32))
    np.testing.assert_allclose(o, -2.5, rtol=1e-14)


def test_dominant_key_is_selected():
    """q aligned with one key and a large scale: the softmax is one-hot."""
    B, Sk, H, D = 1, 16, 1, 16
    k = np.zeros((B, Sk, H, D), np.float32)
    for j in range(Sk):
        k[0, j, 0, j % D] = 1.0
    q = np.zeros((B, 1, H, D), np.float32)
    q[0, 0, 0, 5] = 1.0
    v = gen.normal_bshd(B, Sk, H, D, 15, gen.STREAM_V)
    o = oracle.attention_f64(_to_bits(q), _to_bits(k), v, 1000.0)
    np.testing.assert_allclose(o[0, 0, 0], _bf(v)[0, 5, 0], rtol=0, atol=1e-300)


def test_key_permutation_invariance():
    q, k, v = _rand(1, 12, 40, 2, 2, 16, seed=16)
    perm = np.random.default_rng(0).permutation(40)
    o1 = oracle.attention_f64(q, k, v, 0.4)
    o2 = oracle.attention_f64(q, k[:, perm].copy(), v[:, perm].copy(), 0.4)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)


def test_masked_keys_are_never_attended_even_if_poisoned():
    B, S, Hq, Hkv, D = 2, 24, 4, 2, 16
    q, k, v = _rand(B, S, S, Hq, Hkv, D, seed=17)
    kv_len = np.array([13, 24], np.int32)
    bits = gen.bernoulli_bits(B, S, S, 4, gen.STREAM_BITS, 0.5)
    ref = oracle.attention_f64(q, k, v, 0.3, kv_len=kv_len, bits=bits)
    kp, vp = k.copy(), v.copy()
    kp[0, 13:] = 0x7FC0  # NaN
    vp[0, 13:] = 0x7F80  # +inf
    o = oracle.attention_f64(q, kp, vp, 0.3, kv_len=kv_len, bits=bits)
    np.testing.assert_array_equal(o, ref)
    assert np.all(np.isfinite(o))


def test_gqa_equals_mha_with_repeated_heads():
    B, Sq, Sk, Hq, Hkv, D = 2, 18, 26, 6, 2, 16
    q, k, v = _rand(B, Sq, Sk, Hq, Hkv, D, seed=18)
    o1 = oracle.attention_f64(q, k, v, 0.25, kv_len=np.array([26, 9], np.int32))
    kr = np.repeat(k, Hq // Hkv, axis=2).copy()
    vr = np.repeat(v, Hq // Hkv, axis=2).copy()
    o2 = oracle.attention_f64(q, kr, vr, 0.25, kv_len=np.array([26, 9], np.int32))
    np.testing.assert_array_equal(o1, o2)


def test_packed_bits_equal_structured_masks():
    B, S, H, D = 2, 70, 2, 16
    q, k, v = _rand(B, S, S, H, H, D, seed=19)
    kv_len = np.array([41, 70], np.int32)
    causal_b = np.array([1, 0], np.uint8)
    o1 = oracle.attention_f64(q, k, v, 0.3, kv_len=kv_len, causal_b=causal_b)
    bits = _pack(_mask_matrix(B, S, S, False, kv_len, None, causal_b))
    o2 = oracle.attention_f64(q, k, v, 0.3, bits=bits)
    np.testing.assert_array_equal(o1, o2)


def test_row_subset_equals_full_rows_and_q_len_zero_tail():
    B, Sq, Sk, Hq, Hkv, D = 2, 20, 30, 4, 2, 16
    q, k, v = _rand(B, Sq, Sk, Hq, Hkv, D, seed=20)
    q_len = np.array([20, 7], np.int32)
    full = oracle.attention_f64(q, k, v, 0.3, q_len=q_len)
    ids = np.array([0, 5, 79, (1 * Sq + 6) * Hq + 3, (1 * Sq + 7) * Hq + 0, B * Sq * Hq - 1], np.int64)
    sub = oracle.attention_f64(q, k, v, 0.3, q_len=q_len, row_ids=ids)
    np.testing.assert_array_equal(sub, full.reshape(-1, D)[ids])
    np.testing.assert_array_equal(full[1, 7:], 0.0)
    assert np.all(np.abs(full[1, :7]) > 0)


def test_allowed_pair_count():
    B, S = 3, 57
    kv_len = np.array([57, 30, 1], np.int32)
    causal_b = np.array([1, 0, 1], np.uint8)
    n = oracle.allowed_pairs(B, S, S, False, kv_len, None, causal_b)
    assert n == int(_mask_matrix(B, S, S, False, kv_len, None, causal_b).sum())
    assert oracle.allowed_pairs(1, 10, 10, True) == 55  # triangle: 10*11/2
