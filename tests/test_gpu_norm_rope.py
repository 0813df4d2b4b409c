"""GPU parity of the fused Q/K RMSNorm + bf16 boundary + partial RoPE kernel:
bit-exact against the oracle's float32 fixed-order emulation, called through
the C ABI, on every workload that runs the step and on edge cases."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import bf16_f64, bf16_ulp, from_dev, to_dev, to_dev_f32

NORM_WORKLOADS = ["tiny_mha", "dit_block", "long_video_h12", "long_video_h24", "padded_gqa",
                  "packed_clip_self"]


def _run(h3, q_bits, k_bits, wq, wk, cos, sin, rot, eps):
    import torch
    q = to_dev(q_bits) if q_bits is not None else None
    k = to_dev(k_bits) if k_bits is not None else None
    h3.h3attn_qk_norm_rope(q, k, to_dev_f32(wq) if wq is not None else None,
                           to_dev_f32(wk) if wk is not None else None,
                           to_dev_f32(cos) if cos is not None else None,
                           to_dev_f32(sin) if sin is not None else None, rot, eps)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    return (from_dev(q) if q is not None else None), (from_dev(k) if k is not None else None)


def _assert_bits_equal(got, ref, what):
    bad = np.flatnonzero(got.reshape(-1) != ref.reshape(-1))
    assert bad.size == 0, f"{what}: {bad.size} of {got.size} elements differ, first at flat index {bad[:5]}"


@pytest.mark.gpu
@pytest.mark.parametrize("name", NORM_WORKLOADS)
def test_bit_exact_on_workloads(h3, name):
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl, seed=42)
    gq, gk = _run(h3, inp.q, inp.k, inp.wq, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    _assert_bits_equal(gq, oracle.qk_norm_rope_emulate(inp.q, inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps),
                       f"{name} q")
    _assert_bits_equal(gk, oracle.qk_norm_rope_emulate(inp.k, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps),
                       f"{name} k")


@pytest.mark.gpu
def test_bit_exact_cross_attention_query_only(h3):
    wl = gen.WORKLOADS["packed_clip_cross"]
    inp = gen.make_inputs(wl, seed=0)
    gq, _ = _run(h3, inp.q, None, inp.wq, None, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    _assert_bits_equal(gq, oracle.qk_norm_rope_emulate(inp.q, inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps),
                       "cross q")


@pytest.mark.gpu
@pytest.mark.parametrize("D,rot,eps,B,S,Hq,Hkv", [
    (128, 96, 1e-6, 2, 37, 3, 1),     # ragged rows, GQA head counts
    (128, 128, 1e-6, 1, 64, 4, 4),    # full rotation
    (128, 0, 1e-6, 1, 64, 4, 4),      # norm only
    (128, 32, 1e-2, 1, 50, 2, 2),     # short rotation, large eps
    (64, 32, 1e-6, 3, 33, 4, 2),
    (64, 64, 0.0, 1, 31, 2, 2),
    (256, 96, 1e-6, 2, 29, 2, 2),
    (256, 256, 1e-6, 1, 17, 3, 3),
    # table rows staged with the chunk, chunks crossing sample boundaries
    (128, 96, 1e-6, 3, 5, 24, 12),
    (64, 64, 1e-6, 2, 9, 20, 20),
    (256, 128, 1e-6, 2, 7, 12, 12),
    # chunks spanning more tokens than a sample has positions: tables read directly
    (128, 96, 1e-6, 4, 2, 16, 8),
])
def test_bit_exact_edge_shapes(h3, D, rot, eps, B, S, Hq, Hkv):
    q = gen.normal_bshd(B, S, Hq, D, 7, gen.STREAM_Q, 2.0, 0.5)
    k = gen.normal_bshd(B, S, Hkv, D, 7, gen.STREAM_K, 0.25, 0.0)
    wq = gen.uniform_f32(D, 7, gen.STREAM_WQ, 0.5, 1.5)
    wk = gen.uniform_f32(D, 7, gen.STREAM_WK, 0.5, 1.5)
    cos, sin = gen.rope_tables(S, rot) if rot else (None, None)
    gq, gk = _run(h3, q, k, wq, wk, cos, sin, rot, eps)
    _assert_bits_equal(gq, oracle.qk_norm_rope_emulate(q, wq, cos, sin, rot, eps), "q")
    _assert_bits_equal(gk, oracle.qk_norm_rope_emulate(k, wk, cos, sin, rot, eps), "k")


@pytest.mark.gpu
@pytest.mark.parametrize("D,rot", [(128, 2), (128, 24), (128, 40), (128, 94), (64, 2), (64, 62),
                                   (256, 18), (256, 250)])
def test_any_even_rotary_dim(h3, D, rot):
    """rotary_dim even but not a multiple of 16: rotation pairs straddle the
    lanes' channel groups (the kernel's channel-by-channel path).  Bit-exact
    against the emulation, within the emulation's rounding bound of the fp64
    definition, and the out-of-place call bit-equal to the in-place one."""
    B, S, Hq, Hkv = 2, 41, 3, 1
    q = gen.normal_bshd(B, S, Hq, D, 13, gen.STREAM_Q, 1.0, 0.5)
    k = gen.normal_bshd(B, S, Hkv, D, 13, gen.STREAM_K)
    wq = gen.uniform_f32(D, 13, gen.STREAM_WQ, 0.5, 1.5)
    wk = gen.uniform_f32(D, 13, gen.STREAM_WK, 0.5, 1.5)
    cos, sin = gen.rope_tables(S, rot)
    gq, gk = _run(h3, q, k, wq, wk, cos, sin, rot, 1e-6)
    eq = oracle.qk_norm_rope_emulate(q, wq, cos, sin, rot, 1e-6)
    _assert_bits_equal(gq, eq, f"q rot {rot}")
    _assert_bits_equal(gk, oracle.qk_norm_rope_emulate(k, wk, cos, sin, rot, 1e-6), f"k rot {rot}")
    # |gpu - fp64| <= ulp(y) + 2 ulp(|(a, b)|): a boundary value one bf16 step
    # off, carried through the rotation by the pair's magnitude, plus the store
    exact = oracle.qk_norm_rope_f64(q, wq, cos, sin, rot, 1e-6)
    n = oracle.qk_norm_rope_f64(q, wq, None, None, 0, 1e-6)
    half = rot // 2
    mag = np.abs(n).copy()
    pair = np.sqrt(n[..., :half] ** 2 + n[..., half:rot] ** 2)
    mag[..., :half] = pair
    mag[..., half:rot] = pair
    assert np.all(np.abs(bf16_f64(gq) - exact) <= bf16_ulp(exact) + 2.0 * bf16_ulp(mag))
    _, _, oq, ok_ = _run_out(h3, q, k, wq, wk, cos, sin, rot, 1e-6)
    _assert_bits_equal(oq, gq, f"q_out rot {rot}")
    _assert_bits_equal(ok_, gk, f"k_out rot {rot}")


@pytest.mark.gpu
def test_zero_rows_and_tiny_values(h3):
    """Rows of zeros (r = 1/sqrt(eps)) and subnormal-scale inputs."""
    D, S = 128, 8
    q = gen.normal_bshd(1, S, 2, D, 3, gen.STREAM_Q)
    q[0, 0] = 0
    q[0, 1, 0] = 0x0001  # tiniest subnormal bf16
    k = (gen.normal_bshd(1, S, 2, D, 3, gen.STREAM_K).astype(np.uint32) & 0x80FF) .astype(np.uint16)  # tiny values
    w = gen.uniform_f32(D, 3, gen.STREAM_WQ, 0.5, 1.5)
    cos, sin = gen.rope_tables(S, 96)
    gq, gk = _run(h3, q, k, w, w, cos, sin, 96, 1e-6)
    _assert_bits_equal(gq, oracle.qk_norm_rope_emulate(q, w, cos, sin, 96, 1e-6), "q")
    _assert_bits_equal(gk, oracle.qk_norm_rope_emulate(k, w, cos, sin, 96, 1e-6), "k")


# ---------------------------------------------------------------- out of place
def _run_out(h3, q_bits, k_bits, wq, wk, cos, sin, rot, eps, alias=False):
    import torch
    q, k = to_dev(q_bits), to_dev(k_bits)
    q_out = q if alias else torch.full_like(q, float("nan"))
    k_out = k if alias else torch.full_like(k, float("nan"))
    h3.h3attn_qk_norm_rope_out(q, k, q_out, k_out, to_dev_f32(wq), to_dev_f32(wk),
                               to_dev_f32(cos) if cos is not None else None,
                               to_dev_f32(sin) if sin is not None else None, rot, eps)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    return from_dev(q), from_dev(k), from_dev(q_out), from_dev(k_out)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny_mha", "dit_block", "padded_gqa"])
def test_out_of_place_bit_equal_and_inputs_kept(h3, name):
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl, seed=1234)
    gq, gk, oq, ok_ = _run_out(h3, inp.q, inp.k, inp.wq, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    # the raw inputs are untouched
    _assert_bits_equal(gq, inp.q, f"{name} q input")
    _assert_bits_equal(gk, inp.k, f"{name} k input")
    # the outputs equal the emulation and the in-place kernel bit for bit
    eq = oracle.qk_norm_rope_emulate(inp.q, inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    ek = oracle.qk_norm_rope_emulate(inp.k, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    _assert_bits_equal(oq, eq, f"{name} q_out")
    _assert_bits_equal(ok_, ek, f"{name} k_out")
    iq, ik = _run(h3, inp.q, inp.k, inp.wq, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    _assert_bits_equal(oq, iq, f"{name} q_out vs in place")
    _assert_bits_equal(ok_, ik, f"{name} k_out vs in place")


@pytest.mark.gpu
@pytest.mark.parametrize("D,rot,B,S,Hq,Hkv", [(128, 96, 2, 37, 3, 1), (64, 32, 3, 9, 20, 4), (256, 128, 1, 17, 3, 3)])
def test_out_of_place_edge_shapes_and_alias(h3, D, rot, B, S, Hq, Hkv):
    q = gen.normal_bshd(B, S, Hq, D, 11, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, 11, gen.STREAM_K)
    w = gen.uniform_f32(D, 11, gen.STREAM_WQ, 0.5, 1.5)
    cos, sin = gen.rope_tables(S, rot)
    eq = oracle.qk_norm_rope_emulate(q, w, cos, sin, rot, 1e-6)
    ek = oracle.qk_norm_rope_emulate(k, w, cos, sin, rot, 1e-6)
    gq, gk, oq, ok_ = _run_out(h3, q, k, w, w, cos, sin, rot, 1e-6)
    _assert_bits_equal(gq, q, "q input kept")
    _assert_bits_equal(oq, eq, "q_out")
    _assert_bits_equal(ok_, ek, "k_out")
    # outputs that are their own inputs: the in-place call
    gq, gk, _, _ = _run_out(h3, q, k, w, w, cos, sin, rot, 1e-6, alias=True)
    _assert_bits_equal(gq, eq, "aliased q")
    _assert_bits_equal(gk, ek, "aliased k")


@pytest.mark.gpu
def test_binding_rejects_short_weights_and_missing_tables(h3):
    """Arguments the kernel would read past (a weight vector shorter than D,
    absent RoPE tables, a strided per-sample length vector) are refused by the
    binding before any launch, and the device status stays clean."""
    import torch
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, dtype=torch.float32, device="cuda")
    cos = torch.ones(8, 48, dtype=torch.float32, device="cuda")
    with pytest.raises(h3.H3AttnError, match="wq must be"):
        h3.h3attn_qk_norm_rope(q, None, w[:64], None, cos, cos)
    with pytest.raises(h3.H3AttnError, match="cos and sin are required"):
        h3.h3attn_qk_norm_rope(q, None, w, None, None, None, rotary_dim=96)
    h3.h3attn_qk_norm_rope(q, None, w, None, None, None, rotary_dim=0)   # no rotation: no tables needed
    q2 = torch.zeros(2, 8, 2, 128, dtype=torch.bfloat16, device="cuda")
    kv_len = torch.full((4,), 8, dtype=torch.int32, device="cuda")[::2]    # [2], stride 2
    with pytest.raises(h3.H3AttnError, match="kv_len must be"):
        h3.h3attn_prefill_window(q2, q2, q2, torch.empty_like(q2), h3.Window(4, 0, 1, 0),
                                 mask=h3.Mask(kv_len=kv_len))
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
