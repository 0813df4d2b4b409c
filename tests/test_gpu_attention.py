"""GPU parity of the prefill attention kernel against the fp64 oracle, called
through the C ABI.  Full comparison where the oracle finishes in seconds;
sampled rows (each row is independent, so a sampled row is compared
exactly) at the full workload sizes, in the same launch configuration the
bench times.  Bound: max |err| <= 2e-2 and relative RMS <= 5e-3."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import (assert_convex_bound, check_close, from_dev, sample_rows, to_dev, to_dev_f32, to_dev_i32,
                     to_dev_u8)


def gpu_attention(h3, q, k, v, scale, causal=False, kv_len=None, q_len=None, causal_b=None, bits=None):
    import torch
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    do = torch.full(dq.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    mask = None
    if any(x is not None for x in (kv_len, q_len, causal_b, bits)):
        mask = h3.Mask(kv_len=None if kv_len is None else to_dev_i32(kv_len),
                       q_len=None if q_len is None else to_dev_i32(q_len),
                       causal_b=None if causal_b is None else to_dev_u8(causal_b),
                       bits=None if bits is None else torch.from_numpy(bits.view(np.int32)).cuda())
    h3.h3attn_prefill(dq, dk, dv, do, scale, mask, causal)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    return from_dev(do)


def full_case(h3, B, Sq, Sk, Hq, Hkv, D, seed=0, causal=False, kv_len=None, q_len=None, causal_b=None,
              bits_density=None, std=1.0, what=""):
    q = gen.normal_bshd(B, Sq, Hq, D, seed, gen.STREAM_Q, std)
    k = gen.normal_bshd(B, Sk, Hkv, D, seed, gen.STREAM_K, std)
    v = gen.normal_bshd(B, Sk, Hkv, D, seed, gen.STREAM_V)
    bits = None if bits_density is None else gen.bernoulli_bits(B, Sq, Sk, seed, gen.STREAM_BITS, bits_density)
    scale = 1.0 / np.sqrt(D)
    got = gpu_attention(h3, q, k, v, scale, causal, kv_len, q_len, causal_b, bits)
    ref = oracle.attention_f64(q, k, v, scale, causal, kv_len, q_len, causal_b, bits)
    return check_close(got, ref, what)


# ---------------------------------------------------------------- small / edge cases
# Every edge case runs on every attention kernel: "1" = one query tile per CTA
# (Q in tensor memory), "2" = two query tiles per CTA, "3" = the persistent
# kernel (one CTA per SM over all units), "4" = one query tile per CTA, two
# CTAs per SM (head_dim 256 falls back to "2" for "3" and "4"), "5" = the
# head-dim-256 kernel with double-buffered scores, "6" = the head-dim-128
# kernel that chains its work units, one CTA per SM (other head dims take the
# library's choice for "5" and "6").  Without the override the library picks
# by shape.
@pytest.fixture(params=["1", "2", "3", "4", "5", "6"],
                ids=["one_tile", "two_tiles", "persistent", "two_ctas", "wide", "chain"])
def kernel(request, monkeypatch):
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", request.param)
    return request.param

@pytest.mark.gpu
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,D", [
    (1, 128, 128, 1, 1, 128),    # one tile
    (1, 256, 256, 2, 2, 128),    # one CTA, two query tiles
    (1, 300, 300, 2, 2, 128),    # ragged query and key tails
    (2, 77, 200, 4, 2, 128),     # cross-attention + GQA, short query
    (1, 1, 1, 1, 1, 128),        # single row, single key
    (1, 513, 129, 3, 1, 128),    # ragged both sides, MQA
    (1, 190, 333, 2, 2, 64),
    (2, 130, 260, 4, 2, 256),
])
def test_dense_shapes(h3, kernel, B, Sq, Sk, Hq, Hkv, D):
    full_case(h3, B, Sq, Sk, Hq, Hkv, D, seed=B * 1000 + Sq, what=f"dense {B},{Sq},{Sk},{Hq},{Hkv},{D}")


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128, 256])
def test_causal_and_padding(h3, kernel, D):
    B, S = 3, 389
    kv_len = np.array([389, 150, 1], np.int32)
    causal_b = np.array([1, 0, 1], np.uint8)
    full_case(h3, B, S, S, 4, 2, D, seed=3, kv_len=kv_len, causal_b=causal_b, what=f"causal+pad D={D}")
    full_case(h3, 1, 300, 300, 2, 1, D, seed=4, causal=True, what=f"causal D={D}")


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128, 256])
def test_bit_mask_and_q_len_and_degenerate(h3, kernel, D):
    # random packed boolean [Q, K] mask, combined with key padding
    full_case(h3, 2, 200, 333, 2, 2, D, seed=5, bits_density=0.3, kv_len=np.array([333, 100], np.int32),
              what=f"bits+pad D={D}")
    # very sparse mask: many rows fully masked -> zero rows
    full_case(h3, 1, 140, 140, 2, 2, D, seed=6, bits_density=0.002, what=f"sparse bits D={D}")
    # zero-tail mode and kv_len <= 0 (every key masked -> zeros)
    full_case(h3, 3, 270, 270, 2, 2, D, seed=7, q_len=np.array([270, 13, 0], np.int32),
              kv_len=np.array([-5, 270, 100], np.int32), what=f"q_len/kv_len edge D={D}")


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128, 256])
def test_poisoned_key_padding_is_never_attended(h3, kernel, D):
    """Keys past kv_len hold NaN and Inf in K and V (as uninitialised padding
    may): they must not reach the output.  kv_len falls inside a key tile, so
    the tile that straddles it is loaded with its poisoned rows; the oracle
    skips masked keys outright."""
    B, S, Hq, Hkv = 2, 1300, 2, 1
    kv_len = np.array([1000, 777], np.int32)
    q = gen.normal_bshd(B, S, Hq, D, 21, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, 21, gen.STREAM_K)
    v = gen.normal_bshd(B, S, Hkv, D, 21, gen.STREAM_V)
    for b in range(B):
        for x in (k, v):
            x[b, kv_len[b]:, :, 0::2] = 0x7FC0  # NaN
            x[b, kv_len[b]:, :, 1::2] = 0x7F80  # +Inf
    scale = 1.0 / np.sqrt(D)
    got = gpu_attention(h3, q, k, v, scale, kv_len=kv_len)
    ref = oracle.attention_f64(q, k, v, scale, False, kv_len, None, None)
    assert np.all(np.isfinite(ref))
    check_close(got, ref, f"poisoned padding D={D}")


@pytest.mark.gpu
def test_peaky_scores_exercise_rescaling(h3, kernel):
    """Large-magnitude inputs: maxima grow across key tiles, forcing O rescales."""
    full_case(h3, 1, 256, 1024, 2, 2, 128, seed=8, std=4.0, what="peaky")


@pytest.mark.gpu
def test_gqa_equals_repeated_heads_on_gpu(h3, kernel):
    B, S, Hq, Hkv, D = 1, 256, 8, 2, 128
    q = gen.normal_bshd(B, S, Hq, D, 9, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, 9, gen.STREAM_K)
    v = gen.normal_bshd(B, S, Hkv, D, 9, gen.STREAM_V)
    o1 = gpu_attention(h3, q, k, v, 0.1)
    o2 = gpu_attention(h3, q, np.repeat(k, 4, axis=2).copy(), np.repeat(v, 4, axis=2).copy(), 0.1)
    np.testing.assert_array_equal(o1, o2)


# ---------------------------------------------------------------- the workloads
def _workload_inputs(name, seed):
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl, seed)
    q, k = inp.q, inp.k
    if wl.norm_rope:
        # The attention oracle consumes the oracle's own norm/RoPE output
        # (the GPU kernel is bit-exact to it, see test_gpu_norm_rope.py).
        q = oracle.qk_norm_rope_emulate(inp.q, inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
        if not wl.cross:
            k = oracle.qk_norm_rope_emulate(inp.k, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    return wl, inp, q, k


def _gpu_step(h3, wl, inp):
    """The whole step on the GPU: norm/RoPE in place, then attention."""
    import torch
    dq, dk, dv = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
    if wl.norm_rope:
        h3.h3attn_qk_norm_rope(dq, None if wl.cross else dk, to_dev_f32(inp.wq),
                               None if wl.cross else to_dev_f32(inp.wk), to_dev_f32(inp.cos),
                               to_dev_f32(inp.sin), wl.rotary_dim, wl.eps)
    mask = None
    if inp.kv_len is not None or inp.causal_b is not None:
        mask = h3.Mask(kv_len=None if inp.kv_len is None else to_dev_i32(inp.kv_len),
                       causal_b=None if inp.causal_b is None else to_dev_u8(inp.causal_b))
    do = torch.empty_like(dq)
    h3.h3attn_prefill(dq, dk, dv, do, wl.scale, mask, False)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    assert_convex_bound(dv, do, wl.Hq // wl.Hkv, wl.name)
    return from_dev(do)



FULL = ["tiny_mha", "dit_block", "padded_gqa_d64", "padded_gqa_d256"]
# random rows per (sample, head) on top of the fixed rows of sample_rows()
SAMPLED = {"long_video_h12": 24, "long_video_h24": 64, "padded_gqa": 24, "packed_clip_self": 8,
           "packed_clip_cross": 48}
SEEDS = [0, 42, 1234]


@pytest.mark.gpu
@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("name", FULL)
def test_workload_full(h3, name, seed):
    wl, inp, q, k = _workload_inputs(name, seed=seed)
    got = _gpu_step(h3, wl, inp)
    ref = oracle.attention_f64(q, k, inp.v, wl.scale, False, inp.kv_len, None, inp.causal_b)
    check_close(got, ref, f"{name} seed {seed}")


@pytest.mark.gpu
@pytest.mark.parametrize("seed", SEEDS)
@pytest.mark.parametrize("name", list(SAMPLED))
def test_workload_sampled_rows(h3, name, seed):
    wl, inp, q, k = _workload_inputs(name, seed=seed)
    got = _gpu_step(h3, wl, inp)
    ids = sample_rows(wl.B, wl.Sq, wl.Hq, SAMPLED[name], seed=seed + 1, kv_len=inp.kv_len)
    ref = oracle.attention_f64(q, k, inp.v, wl.scale, False, inp.kv_len, None, inp.causal_b, row_ids=ids)
    check_close(got.reshape(-1, wl.D)[ids], ref, f"{name} seed {seed}")


@pytest.mark.gpu
@pytest.mark.parametrize("kern", ["3", "6"], ids=["persistent", "chain"])
def test_persistent_kernel_on_long_video(h3, monkeypatch, kern):
    """The kernels with one CTA per SM walking the unit list (the persistent
    and the unit-chaining one) at a full workload size: sampled rows against
    the oracle."""
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", kern)
    wl, inp, q, k = _workload_inputs("long_video_h12", seed=42)
    got = _gpu_step(h3, wl, inp)
    ids = sample_rows(wl.B, wl.Sq, wl.Hq, 24, seed=43)
    ref = oracle.attention_f64(q, k, inp.v, wl.scale, row_ids=ids)
    check_close(got.reshape(-1, wl.D)[ids], ref, f"kernel {kern} long_video_h12")


# The kernels with one CTA per SM take several units per CTA only when the
# grid has several times more units than the GPU has SMs; the edge-case shapes
# above give each CTA one unit at most.  These shapes give each 3 to 10, with
# the unit changes the chaining kernel hands over between its warps: one- and
# two-tile units, units with no key tile (rows past q_len), a padded tile in
# every unit of a sample, cross-attention, per-sample causal masks, GQA and a
# packed mask.
@pytest.mark.gpu
@pytest.mark.parametrize("kern", ["3", "6"], ids=["persistent", "chain"])
def test_unit_walking_kernels_over_many_units(h3, monkeypatch, kern):
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", kern)
    full_case(h3, 4, 256, 256, 96, 96, 128, seed=31, causal=True, what=f"kernel {kern} short causal units")
    B, Sq, Sk, Hq, Hkv, D = 2, 4096, 300, 24, 8, 128
    kv_len = np.array([300, 173], np.int32)
    q_len = np.array([4096, 1000], np.int32)
    q = gen.normal_bshd(B, Sq, Hq, D, 32, gen.STREAM_Q)
    k = gen.normal_bshd(B, Sk, Hkv, D, 32, gen.STREAM_K)
    v = gen.normal_bshd(B, Sk, Hkv, D, 32, gen.STREAM_V)
    scale = 1.0 / np.sqrt(D)
    got = gpu_attention(h3, q, k, v, scale, kv_len=kv_len, q_len=q_len)
    ids = sample_rows(B, Sq, Hq, 12, seed=33, extra_rows=(172, 173, 999, 1000, 1023, 1024, 2047, 2048))
    ref = oracle.attention_f64(q, k, v, scale, False, kv_len, q_len, None, row_ids=np.asarray(ids, np.int64))
    check_close(got.reshape(-1, D)[ids], ref, f"kernel {kern} cross-attention units")
    assert not np.any(got[1, 1000:]), "rows past q_len are zeros"
    full_case(h3, 2, 1024, 1024, 48, 16, 128, seed=35, kv_len=np.array([1024, 700], np.int32),
              q_len=np.array([1024, 600], np.int32), causal_b=np.array([1, 0], np.uint8),
              what=f"kernel {kern} per-sample causal units")
    full_case(h3, 2, 1024, 1024, 32, 32, 128, seed=34, bits_density=0.5, kv_len=np.array([1024, 700], np.int32),
              what=f"kernel {kern} packed mask units")


def _structured_as_bits(B, Sq, Sk, kv_len, causal_b):
    """The key-padding + per-sample causal pattern written out as the packed
    [B, Sq, ceil(Sk/32)] bit mask (bit j & 31 of word j >> 5, 1 = attend)."""
    words = (Sk + 31) // 32
    out = np.zeros((B, Sq, words), np.uint32)
    j = np.arange(words * 32)
    for b in range(B):
        for i0 in range(0, Sq, 1024):
            i = np.arange(i0, min(i0 + 1024, Sq))[:, None]
            allowed = (j[None, :] < min(int(kv_len[b]), Sk)) & np.ones_like(i, dtype=bool)
            if causal_b[b]:
                allowed &= j[None, :] <= i
            out[b, i0:i0 + len(i)] = np.packbits(allowed, axis=1, bitorder="little").view("<u4")
    return out


@pytest.mark.gpu
def test_full_length_bit_mask_equals_structured_mask(h3):
    """padded_gqa's key padding and causal samples given as a packed bit mask
    over 8192 keys (64 key tiles of word loads per row) on the long-sequence
    kernel: sampled rows against the oracle, and every output element against
    the run with the structured mask.  The two runs need not be bit-identical:
    with bits the kernel visits every key tile (the mask is not read on the
    host), so its start tile and its running max can differ; both sit within
    the oracle tolerance, and of each other."""
    import torch
    wl, inp, q, k = _workload_inputs("padded_gqa", seed=42)
    bits = _structured_as_bits(wl.B, wl.Sq, wl.Sk, inp.kv_len, inp.causal_b)
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(inp.v)
    o_bits = torch.empty_like(dq)
    o_struct = torch.empty_like(dq)
    h3.h3attn_prefill(dq, dk, dv, o_bits, wl.scale, h3.Mask(bits=torch.from_numpy(bits.view(np.int32)).cuda()))
    h3.h3attn_prefill(dq, dk, dv, o_struct, wl.scale,
                      h3.Mask(kv_len=to_dev_i32(inp.kv_len), causal_b=to_dev_u8(inp.causal_b)))
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    got = from_dev(o_bits)
    ids = sample_rows(wl.B, wl.Sq, wl.Hq, 24, seed=7, kv_len=inp.kv_len)
    ref = oracle.attention_f64(q, k, inp.v, wl.scale, False, inp.kv_len, None, inp.causal_b, row_ids=ids)
    check_close(got.reshape(-1, wl.D)[ids], ref, "padded_gqa as bits")
    diff = (o_bits.float() - o_struct.float()).abs().max().item()
    assert diff <= 2e-2, f"bit-mask run differs from the structured run by {diff:.3e}"


# The epilogues write o as whole 128-row tiles with TMA stores (rows past Sq
# fall outside the tensor map and are dropped); the split tail's combine and
# the zero rows of empty units write rows directly.  o here is a window into
# a larger buffer whose bytes on both sides hold a sentinel: a write outside
# o shows up there.
@pytest.mark.gpu
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,D,split", [
    (2, 300, 500, 3, 1, 128, False),   # ragged query tail, short keys (two CTAs per SM)
    (1, 1100, 1100, 2, 2, 128, False),  # one query tile per CTA
    (1, 1100, 1100, 2, 2, 128, True),   # ... with the split-key tail and its combine
    (1, 77, 900, 2, 2, 64, False),
    (2, 130, 260, 2, 1, 256, False),
])
def test_prefill_writes_nothing_outside_o(h3, kernel, B, Sq, Sk, Hq, Hkv, D, split):
    import torch
    q = gen.normal_bshd(B, Sq, Hq, D, 51, gen.STREAM_Q)
    k = gen.normal_bshd(B, Sk, Hkv, D, 51, gen.STREAM_K)
    v = gen.normal_bshd(B, Sk, Hkv, D, 51, gen.STREAM_V)
    n, pad = B * Sq * Hq * D, 8192
    sentinel = 0x7FA5  # a NaN pattern no kernel writes
    buf = torch.full((pad + n + pad,), sentinel, dtype=torch.int16, device="cuda")
    o = buf[pad:pad + n].view(torch.bfloat16).view(B, Sq, Hq, D)
    ws = None
    if split:
        nbytes = h3.h3attn_prefill_workspace_size(B, Sq, Sk, Hq, Hkv, D)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    h3.h3attn_prefill(to_dev(q), to_dev(k), to_dev(v), o, 1.0 / np.sqrt(D), workspace=ws)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    guard = torch.cat([buf[:pad], buf[pad + n:]])
    assert bool((guard == sentinel).all()), "bytes outside o were written"
    got = from_dev(o)
    ref = oracle.attention_f64(q, k, v, 1.0 / np.sqrt(D))
    check_close(got, ref, f"guarded o {B},{Sq},{Sk},{Hq},{Hkv},{D} split={split}")
