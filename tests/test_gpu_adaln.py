"""GPU parity of the fused RMSNorm -> indexed AdaLN scale/shift modulation
kernel, called through the C ABI: bit-exact against the oracle's float32
fixed-order emulation (the contract of TeleFuser PR #37 section 2.5:
element-wise bit-exact with the unfused path), on the hidden-row workload and
on edge cases (ragged group counts, the largest C, no weight, no index, in
place, an index outside the table)."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import from_dev, to_dev_f32, to_dev_i32


def _dev2(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(h3, inp, with_w=True, with_idx=True, in_place=False, eps=1e-6):
    import torch
    x = _dev2(inp.x)
    y = x if in_place else torch.full_like(x, float("nan"))
    h3.h3attn_rmsnorm_modulate(x, y, to_dev_f32(inp.w) if with_w else None, _dev2(inp.scale), _dev2(inp.shift),
                               to_dev_i32(inp.idx) if with_idx else None, eps)
    torch.cuda.synchronize()
    return from_dev(y)


def _expect(inp, with_w=True, with_idx=True, eps=1e-6):
    return oracle.rmsnorm_modulate_emulate(inp.x, inp.w if with_w else None, inp.scale, inp.shift,
                                           inp.idx if with_idx else None, eps)


def _assert_bits_equal(got, ref, what):
    bad = np.flatnonzero(got.reshape(-1) != ref.reshape(-1))
    assert bad.size == 0, f"{what}: {bad.size} of {got.size} elements differ, first at {bad[:5]}"


@pytest.mark.gpu
def test_bit_exact_on_hidden_row_workload(h3):
    wl = gen.MOD_WORKLOADS["dit_hidden_adaln"]
    inp = gen.make_modulate_inputs(wl.T, wl.C, wl.frames, seed=42)
    got = _run(h3, inp, eps=wl.eps)
    assert h3.h3attn_check_device_status() == 0
    _assert_bits_equal(got, _expect(inp, eps=wl.eps), wl.name)


@pytest.mark.gpu
@pytest.mark.parametrize("T,C,N", [(1, 8, 1), (7, 264, 3), (33, 1536, 5), (9, 8192, 2), (130, 5120, 4)])
def test_bit_exact_edge_shapes(h3, T, C, N):
    inp = gen.make_modulate_inputs(T, C, N, seed=T + C)
    for with_w in (True, False):
        got = _run(h3, inp, with_w=with_w)
        assert h3.h3attn_check_device_status() == 0
        _assert_bits_equal(got, _expect(inp, with_w=with_w), f"T={T} C={C} w={with_w}")


# Every ring shape the launcher picks, with many rows per CTA so that each
# compute warp goes round its CTA's ring several times (C 1536: 16 warps, 35
# stages, 2 CTAs per SM; 3072: 14 warps, 16 stages, 2 CTAs, weight staged;
# 3456: 14 warps, 16 stages, 2 CTAs, weight through L1; 4096 / 5120: 16 warps,
# 1 CTA; 8192: 8 warps, 12 stages, 1 CTA); every stage is refilled at least
# twice, so a warp that took a stale fill of its stage (phase aliasing) would
# show here as a wrong row.  Without the weight the same sizes take the other
# shapes.
@pytest.mark.gpu
@pytest.mark.parametrize("with_w", [True, False], ids=["weight", "no_weight"])
@pytest.mark.parametrize("T,C,N", [(24000, 1536, 4), (20000, 3072, 4), (11000, 3456, 3), (9000, 4096, 3),
                                   (7000, 5120, 3), (6000, 6144, 3), (4500, 8192, 2)])
def test_bit_exact_rows_lap_the_ring(h3, T, C, N, with_w):
    inp = gen.make_modulate_inputs(T, C, N, seed=T ^ C)
    got = _run(h3, inp, with_w=with_w)
    assert h3.h3attn_check_device_status() == 0
    _assert_bits_equal(got, _expect(inp, with_w=with_w), f"T={T} C={C} weight={with_w}")


@pytest.mark.gpu
def test_no_index_and_in_place(h3):
    inp = gen.make_modulate_inputs(50, 3072, 4, seed=5)
    got = _run(h3, inp, with_idx=False)
    _assert_bits_equal(got, _expect(inp, with_idx=False), "no index")
    got = _run(h3, inp, in_place=True)
    _assert_bits_equal(got, _expect(inp), "in place")
    assert h3.h3attn_check_device_status() == 0


@pytest.mark.gpu
def test_index_outside_the_table_gives_zero_rows_and_an_error_status(h3):
    inp = gen.make_modulate_inputs(12, 256, 3, seed=9)
    inp.idx[[2, 7]] = [3, -1]
    got = _run(h3, inp)
    assert h3.h3attn_check_device_status() == h3.H3ATTN_ERR_INVALID_ARG
    assert h3.h3attn_check_device_status() == 0  # the status word is cleared once read
    _assert_bits_equal(got, _expect(inp), "bad index rows")
    assert np.all(got[[2, 7]] == 0)


# The kernel is launched as a programmatic dependent of the previous kernel
# of the stream and reads or writes global memory only once that kernel has
# completed.  Chained calls with no host synchronisation between them, each
# reading what the one before wrote (out of place, in place, and after a
# PyTorch kernel that rewrites the buffer), give the emulation applied in the
# same order.
@pytest.mark.gpu
def test_back_to_back_calls_read_the_previous_output(h3):
    import torch
    inp = gen.make_modulate_inputs(20000, 3072, 4, seed=77)
    w, idx = to_dev_f32(inp.w), to_dev_i32(inp.idx)
    sc, sh = _dev2(inp.scale), _dev2(inp.shift)
    x = _dev2(inp.x)
    y = torch.full_like(x, float("nan"))
    z = torch.full_like(x, float("nan"))
    h3.h3attn_rmsnorm_modulate(x, y, w, sc, sh, idx, 1e-6)  # y = f(x)
    h3.h3attn_rmsnorm_modulate(y, y, w, sc, sh, idx, 1e-6)  # y = f(f(x)), in place
    y.neg_()                                                # a PyTorch kernel in between
    h3.h3attn_rmsnorm_modulate(y, z, w, sc, sh, idx, 1e-6)  # z = f(-f(f(x)))
    h3.h3attn_rmsnorm_modulate(z, x, w, sc, sh, idx, 1e-6)  # x = f(z), over the first input
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0

    def f(bits):
        return oracle.rmsnorm_modulate_emulate(bits, inp.w, inp.scale, inp.shift, inp.idx, 1e-6)
    ref_y = f(f(inp.x)) ^ np.uint16(0x8000)
    ref_z = f(ref_y)
    _assert_bits_equal(from_dev(y), ref_y, "in place, then negated")
    _assert_bits_equal(from_dev(z), ref_z, "after a PyTorch kernel")
    _assert_bits_equal(from_dev(x), f(ref_z), "over the first call's input")
