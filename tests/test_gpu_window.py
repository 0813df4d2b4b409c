"""GPU parity of the chunked-window prefill (SGLang PR #37903, section
"Modifications", hybrid_window_attn_h3) against the fp64 oracle, called
through the C ABI: full comparison on small clips with chunk and anchor
boundaries off the 128-key tile grid, GQA, D = 64 and 128, key padding and a
zero tail; sampled rows (exact per row) on the full packed clip in the launch
configuration the bench times.  Bound: max |err| <= 2e-2, relative RMS <= 5e-3."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import assert_convex_bound, check_close, from_dev, sample_rows, to_dev, to_dev_i32


def gpu_window(h3, q, k, v, scale, win, kv_len=None, q_len=None):
    import torch
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    do = torch.full(dq.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    mask = None
    if kv_len is not None or q_len is not None:
        mask = h3.Mask(kv_len=None if kv_len is None else to_dev_i32(kv_len),
                       q_len=None if q_len is None else to_dev_i32(q_len))
    h3.h3attn_prefill_window(dq, dk, dv, do, h3.Window(*win), scale, mask)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    assert_convex_bound(dv, do, dq.shape[2] // dk.shape[2], "window")   # every row written, none out of range
    return from_dev(do)


@pytest.mark.gpu
@pytest.mark.parametrize("B,S,Hq,Hkv,D,win", [
    (1, 700, 2, 2, 128, (16, 2, 5, 1)),     # chunks of 80 tokens, anchors of 32
    (2, 1000, 4, 2, 64, (50, 0, 3, 0)),     # no anchors, radius 0, GQA
    (1, 2000, 2, 1, 128, (100, 1, 5, 1)),   # MQA, the chunk-5 / radius-1 pattern
    (1, 130, 1, 1, 128, (7, 1, 2, 1)),      # ragged tail, tiny frames
    (1, 1, 1, 1, 128, (4, 0, 1, 0)),        # one token
    (1, 600, 2, 2, 128, (10, 1, 2, 50)),    # radius past the clip: dense
])
def test_window_full(h3, B, S, Hq, Hkv, D, win):
    q = gen.normal_bshd(B, S, Hq, D, S, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, S, gen.STREAM_K)
    v = gen.normal_bshd(B, S, Hkv, D, S, gen.STREAM_V)
    scale = 1.0 / np.sqrt(D)
    got = gpu_window(h3, q, k, v, scale, win)
    ref = oracle.attention_window_f64(q, k, v, scale, *win)
    check_close(got, ref, f"window {win}")


@pytest.mark.gpu
def test_window_with_padding_and_zero_tail(h3):
    B, S, H, D, win = 2, 900, 2, 128, (30, 1, 4, 1)
    q = gen.normal_bshd(B, S, H, D, 7, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, H, D, 7, gen.STREAM_K)
    v = gen.normal_bshd(B, S, H, D, 7, gen.STREAM_V)
    kv_len = np.array([900, 400], np.int32)
    q_len = np.array([850, 900], np.int32)
    got = gpu_window(h3, q, k, v, 0.09, win, kv_len=kv_len, q_len=q_len)
    ref = oracle.attention_window_f64(q, k, v, 0.09, *win, kv_len=kv_len, q_len=q_len)
    check_close(got, ref, "window + padding + zero tail")


@pytest.mark.gpu
def test_window_packed_clip_sampled_rows(h3):
    wl = gen.WINDOW_WORKLOADS["packed_clip_window"]
    q = gen.normal_bshd(wl.B, wl.S, wl.H, wl.D, 0, gen.STREAM_Q)
    k = gen.normal_bshd(wl.B, wl.S, wl.H, wl.D, 0, gen.STREAM_K)
    v = gen.normal_bshd(wl.B, wl.S, wl.H, wl.D, 0, gen.STREAM_V)
    win = (wl.frame_tokens, wl.anchor_frames, wl.chunk_frames, wl.radius)
    scale = 1.0 / np.sqrt(wl.D)
    got = gpu_window(h3, q, k, v, scale, win)
    af, ct = wl.anchor_frames * wl.frame_tokens, wl.chunk_frames * wl.frame_tokens
    rng = np.random.default_rng(0)
    rows = set(rng.integers(0, wl.S, 120).tolist())
    rows |= {0, af - 1, af, af + ct - 1, af + ct, wl.S - 1, wl.S // 2}
    rows = np.array(sorted(r for r in rows if 0 <= r < wl.S))
    heads = np.array([0, 7, 23])
    ids = (rows[:, None] * wl.H + heads[None, :]).reshape(-1).astype(np.int64)
    ref = oracle.attention_window_f64(q, k, v, scale, *win, row_ids=ids)
    check_close(got.reshape(-1, wl.D)[ids], ref, "packed clip window, sampled rows")


@pytest.mark.gpu
@pytest.mark.parametrize("B,S,Hq,Hkv,D,win", [
    (1, 700, 2, 2, 128, (16, 2, 5, 1)),
    (2, 1000, 4, 2, 64, (50, 0, 3, 0)),
])
def test_window_writes_nothing_outside_o(h3, B, S, Hq, Hkv, D, win):
    """o as a window into a larger buffer with sentinel bytes on both sides:
    the epilogue's TMA stores of whole 128-row tiles stay inside o."""
    import torch
    q = gen.normal_bshd(B, S, Hq, D, 61, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, Hkv, D, 61, gen.STREAM_K)
    v = gen.normal_bshd(B, S, Hkv, D, 61, gen.STREAM_V)
    n, pad, sentinel = B * S * Hq * D, 8192, 0x7FA5
    buf = torch.full((pad + n + pad,), sentinel, dtype=torch.int16, device="cuda")
    o = buf[pad:pad + n].view(torch.bfloat16).view(B, S, Hq, D)
    scale = 1.0 / np.sqrt(D)
    h3.h3attn_prefill_window(to_dev(q), to_dev(k), to_dev(v), o, h3.Window(*win), scale)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    assert bool((torch.cat([buf[:pad], buf[pad + n:]]) == sentinel).all()), "bytes outside o were written"
    ref = oracle.attention_window_f64(q, k, v, scale, *win)
    check_close(from_dev(o), ref, f"guarded window o {B},{S},{Hq},{Hkv},{D},{win}")
