"""Tensors past 2^31 elements (byte offsets past 2^32): the norm/RoPE kernel
and the attention kernels the library picks for head dim 128 (one query tile
per CTA; two CTAs per SM), on a cross-attention shape whose query has
2^31 + 4.2 M elements (4.3 GB per tensor), and the RMSNorm -> AdaLN kernel on
hidden rows of the same size, compared with the oracle on rows on both sides
of the 2^31-element line.  Only the compared rows come back to the host."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import assert_convex_bound, check_close, sample_rows, to_dev, to_dev_f32

B, SQ, SK, H, D = 1, (1 << 21) + 4133, 128 + 77, 8, 128
ROT, EPS = 96, 1e-6
LINE = (1 << 31) // (H * D)   # first token whose rows start past 2^31 elements


@pytest.fixture(scope="module")
def big_inputs():
    q = gen.normal_bshd(B, SQ, H, D, 21, gen.STREAM_Q)
    k = gen.normal_bshd(B, SK, H, D, 21, gen.STREAM_K)
    v = gen.normal_bshd(B, SK, H, D, 21, gen.STREAM_V)
    assert q.size > (1 << 31)
    return q, k, v


def _rows_back(t, ids):
    """The sampled (token, head) rows of a BSHD device tensor, as bf16 bits on the host."""
    import torch
    sel = t.view(-1, D)[torch.from_numpy(ids).cuda()]
    return sel.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.gpu
def test_norm_rope_past_2_to_the_31_elements(h3, big_inputs):
    import torch
    q, _, _ = big_inputs
    w = gen.uniform_f32(D, 21, gen.STREAM_WQ, 0.5, 1.5)
    cos, sin = gen.rope_tables(SQ, ROT)
    dq = to_dev(q)
    dq_out = torch.empty_like(dq)
    h3.h3attn_qk_norm_rope_out(dq, None, dq_out, None, to_dev_f32(w), None, to_dev_f32(cos), to_dev_f32(sin),
                               ROT, EPS)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    for s0, s1 in ((0, 64), (LINE - 40, LINE + 40), (SQ - 300, SQ)):
        ref = oracle.qk_norm_rope_emulate(np.ascontiguousarray(q[:, s0:s1]), w, cos[s0:s1], sin[s0:s1], ROT, EPS)
        ids = np.arange(s0 * H, s1 * H, dtype=np.int64)
        got = _rows_back(dq_out, ids)
        np.testing.assert_array_equal(got, ref.reshape(-1, D), err_msg=f"tokens {s0}..{s1}")


@pytest.mark.gpu
@pytest.mark.parametrize("kern", ["1", "4"], ids=["one_tile", "two_ctas"])
def test_attention_past_2_to_the_31_elements(h3, big_inputs, monkeypatch, kern):
    import torch
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", kern)
    q, k, v = big_inputs
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    do = torch.full_like(dq, float("nan"))
    scale = 1.0 / np.sqrt(D)
    h3.h3attn_prefill(dq, dk, dv, do, scale)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    assert_convex_bound(dv, do, 1, "past 2^31 elements")
    extra = (LINE - 1, LINE, LINE + 1, SQ - 129, SQ - 128, SQ - 2)
    ids = sample_rows(B, SQ, H, 16, seed=3, extra_rows=extra)
    ref = oracle.attention_f64(q, k, v, scale, row_ids=ids)
    check_close(_rows_back(do, ids), ref, f"cross past 2^31 elements, kernel {kern}")


@pytest.mark.gpu
def test_rmsnorm_modulate_past_2_to_the_31_elements(h3):
    """Hidden rows of 2^31 + 3.1 M elements (700 k rows of 3072 channels), bit-exact
    on row ranges at the start, across the 2^31-element line and at the end."""
    import torch
    C, N = 3072, 21
    T = (1 << 31) // C + 1024
    inp = gen.make_modulate_inputs(T, C, N, seed=23)
    assert inp.x.size > (1 << 31)

    def dev2(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    x = dev2(inp.x)
    y = torch.empty_like(x)
    h3.h3attn_rmsnorm_modulate(x, y, to_dev_f32(inp.w), dev2(inp.scale), dev2(inp.shift),
                               torch.from_numpy(inp.idx).cuda(), 1e-6)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    line = (1 << 31) // C
    for t0, t1 in ((0, 64), (line - 50, line + 50), (T - 200, T)):
        ref = oracle.rmsnorm_modulate_emulate(np.ascontiguousarray(inp.x[t0:t1]), inp.w, inp.scale, inp.shift,
                                              np.ascontiguousarray(inp.idx[t0:t1]), 1e-6)
        got = y[t0:t1].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(got, ref, err_msg=f"rows {t0}..{t1}")


@pytest.mark.gpu
def test_head_dim_256_attention_past_2_to_the_31_elements(h3):
    """The head-dim-256 kernel (double-buffered scores) on a cross-attention
    query of 2^31 + 8.5 M elements (4.3 GB): sampled rows on both sides of the
    2^31-element line against the oracle, and the convex bound everywhere."""
    import torch
    D2, H2 = 256, 8
    SQ2, SK2 = (1 << 20) + 4133, 128 + 77
    line2 = (1 << 31) // (H2 * D2)
    q = gen.normal_bshd(1, SQ2, H2, D2, 25, gen.STREAM_Q)
    k = gen.normal_bshd(1, SK2, H2, D2, 25, gen.STREAM_K)
    v = gen.normal_bshd(1, SK2, H2, D2, 25, gen.STREAM_V)
    assert q.size > (1 << 31)
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    do = torch.full_like(dq, float("nan"))
    scale = 1.0 / np.sqrt(D2)
    h3.h3attn_prefill(dq, dk, dv, do, scale)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    assert_convex_bound(dv, do, 1, "head dim 256 past 2^31 elements")
    extra = (line2 - 1, line2, line2 + 1, SQ2 - 129, SQ2 - 128, SQ2 - 2)
    ids = sample_rows(1, SQ2, H2, 16, seed=5, extra_rows=extra)
    ref = oracle.attention_f64(q, k, v, scale, row_ids=ids)
    got = do.view(-1, D2)[torch.from_numpy(ids).cuda()].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(got, ref, "head dim 256 cross past 2^31 elements")
