"""GPU parity of the split-key tail (h3attn_prefill_ws): the last partial wave
of work units cut into key ranges whose partial (O, m, l) a combine kernel
merges.  Compared with the fp64 oracle (max |err| 2e-2, relative RMS 5e-3),
called through the C ABI, on the Video-DiT block workload and on small shapes
that force the split onto ragged tails, key padding, zero tails, bit masks,
GQA and head dim 64."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import check_close, from_dev, to_dev, to_dev_i32


def _run(h3, q, k, v, scale, mask=None, ws="auto", poison_ws=True):
    import torch
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    do = torch.full(dq.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    if ws == "auto":
        ws = h3.prefill_workspace(dq, dk, mask)
        assert ws is not None, "this shape is expected to split"
        if poison_ws:
            ws.view(torch.float32).fill_(float("nan"))  # contents on entry must not matter
    h3.h3attn_prefill(dq, dk, dv, do, scale, mask, workspace=ws)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    return from_dev(do)


@pytest.mark.gpu
@pytest.mark.parametrize("seed", [0, 42])
def test_dit_block_split_full_parity(h3, seed):
    """dit_block: 768 units on 152 SMs leave 8 units for a sixth wave; with
    the workspace they run as key-range pieces.  Every output element."""
    wl = gen.WORKLOADS["dit_block"]
    inp = gen.make_inputs(wl, seed)
    q = oracle.qk_norm_rope_emulate(inp.q, inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    k = oracle.qk_norm_rope_emulate(inp.k, inp.wk, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
    got = _run(h3, q, k, inp.v, wl.scale)
    ref = oracle.attention_f64(q, k, inp.v, wl.scale)
    check_close(got, ref, f"dit_block split seed {seed}")
    # deterministic: a second call gives the same bits
    np.testing.assert_array_equal(_run(h3, q, k, inp.v, wl.scale), got)


@pytest.fixture
def one_tile(monkeypatch):
    # the split lives in the one-query-tile kernel; small shapes (and head dim
    # 64) reach it only when it is forced
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", "1")


@pytest.mark.gpu
@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,D", [
    (1, 1100, 1100, 2, 2, 128),   # 18 units: every unit split, ragged query and key tails
    (2, 300, 1500, 4, 2, 128),    # cross-attention shape, GQA
    (1, 128, 512, 1, 1, 128),     # one unit of four key tiles: two pieces of two
    (1, 700, 2000, 3, 1, 64),     # head dim 64, MQA
])
def test_split_small_shapes(h3, one_tile, B, Sq, Sk, Hq, Hkv, D):
    q = gen.normal_bshd(B, Sq, Hq, D, 31, gen.STREAM_Q)
    k = gen.normal_bshd(B, Sk, Hkv, D, 31, gen.STREAM_K)
    v = gen.normal_bshd(B, Sk, Hkv, D, 31, gen.STREAM_V)
    scale = 1.0 / np.sqrt(D)
    got = _run(h3, q, k, v, scale)
    check_close(got, oracle.attention_f64(q, k, v, scale), f"split {B},{Sq},{Sk},{Hq},{Hkv},{D}")


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
def test_split_with_padding_zero_tail_and_bits(h3, one_tile, D):
    """Key padding that ends inside a piece (NaN/Inf past kv_len), a sample
    with kv_len 0 (pieces with no allowed key), q_len zero tails, and a packed
    bit mask that leaves some rows fully masked."""
    import torch
    B, S, Hq, Hkv = 3, 1300, 2, 1
    kv_len = np.array([1000, 0, 777], np.int32)
    q_len = np.array([1300, 900, 5], np.int32)
    q = gen.normal_bshd(B, S, Hq, D, 32, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, 32, gen.STREAM_K)
    v = gen.normal_bshd(B, S, Hkv, D, 32, gen.STREAM_V)
    for b in range(B):
        for x in (k, v):
            x[b, kv_len[b]:, :, 0::2] = 0x7FC0
            x[b, kv_len[b]:, :, 1::2] = 0x7F80
    bits = gen.bernoulli_bits(B, S, S, 32, gen.STREAM_BITS, 0.02)
    scale = 1.0 / np.sqrt(D)
    mask = h3.Mask(kv_len=to_dev_i32(kv_len), q_len=to_dev_i32(q_len),
                   bits=torch.from_numpy(bits.view(np.int32)).cuda())
    got = _run(h3, q, k, v, scale, mask)
    ref = oracle.attention_f64(q, k, v, scale, False, kv_len, q_len, None, bits)
    check_close(got, ref, f"split padding/q_len/bits D={D}")


@pytest.mark.gpu
def test_split_matches_unsplit_and_rejects_short_workspace(h3, one_tile):
    import torch
    B, S, H, D = 1, 1100, 2, 128
    q = gen.normal_bshd(B, S, H, D, 33, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, H, D, 33, gen.STREAM_K)
    v = gen.normal_bshd(B, S, H, D, 33, gen.STREAM_V)
    scale = 1.0 / np.sqrt(D)
    split = _run(h3, q, k, v, scale)
    whole = _run(h3, q, k, v, scale, ws=None)
    d = np.abs(gen.bf16_bits_to_f32(split).astype(np.float64) - gen.bf16_bits_to_f32(whole))
    assert d.max() <= 2e-2
    dq, dk = to_dev(q), to_dev(k)
    n = h3.h3attn_prefill_workspace_size(B, S, S, H, H, D)
    assert n > 0
    short = torch.empty(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(h3.H3AttnError, match="invalid argument"):
        h3.h3attn_prefill(dq, dk, to_dev(v), torch.empty_like(dq), scale, workspace=short)
    # causal calls and the other kernels need no workspace
    assert h3.h3attn_prefill_workspace_size(B, S, S, H, H, D, causal=True) == 0
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
