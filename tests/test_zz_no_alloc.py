"""h3attn_prefill_noalloc: prefill for callers that cannot allocate device
memory (frameworks and plugins that own every allocation, serving paths that
keep allocation out, code running during stream capture).  Its split-key
scratch is the library's fixed device array, so the call takes only the
inputs and outputs.  Called through the C ABI and compared with the
workspace entry point (h3attn_prefill_ws, torch-allocated workspace) within
the attention tolerance of the other tests, on two calls in a row with
different inputs (the second must not see the first call's partials).

The file sorts last so that a run stopping at the first failure has run
every other test first."""
import ctypes

import numpy as np
import pytest

import h3inputs as gen
from helpers import bf16_f64, check_close, from_dev, to_dev


def _noalloc(h3, dq, dk, dv, do, scale, causal=False):
    import torch
    lib = h3.load()
    B, Sq, Hq, D = dq.shape
    Sk, Hkv = dk.shape[1], dk.shape[2]
    st = lib.h3attn_prefill_noalloc(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), B, Sq, Sk, Hq,
                                    Hkv, D, ctypes.c_float(scale), None, int(causal),
                                    torch.cuda.current_stream().cuda_stream)
    assert st == h3.H3ATTN_OK, h3.h3attn_status_string(st)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(h3):
    import torch
    B, S, H, D = 1, 4096, 24, 128  # the Video-DiT block shape: 768 units, the last 8 split into pieces
    scale = 1.0 / np.sqrt(D)
    need = h3.h3attn_prefill_workspace_size(B, S, S, H, H, D)
    assert 0 < need <= h3.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((101, 202)):
        dq = to_dev(gen.normal_bshd(B, S, H, D, seed, gen.STREAM_Q))
        dk = to_dev(gen.normal_bshd(B, S, H, D, seed, gen.STREAM_K))
        dv = to_dev(gen.normal_bshd(B, S, H, D, seed, gen.STREAM_V))
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        o_ref = torch.empty_like(dq)
        h3.h3attn_prefill(dq, dk, dv, o_ref, scale, workspace=ws)
        o = torch.full_like(dq, float("nan"))
        _noalloc(h3, dq, dk, dv, o, scale)
        torch.cuda.synchronize()
        assert h3.h3attn_check_device_status() == 0
        check_close(from_dev(o), bf16_f64(from_dev(o_ref)), f"noalloc call {call + 1}")


@pytest.mark.gpu
def test_noalloc_without_scratch_runs_like_prefill(h3):
    """A causal call needs no scratch: it runs exactly as h3attn_prefill."""
    import torch
    B, S, H, D = 1, 1300, 2, 128
    assert h3.h3attn_prefill_workspace_size(B, S, S, H, H, D, causal=True) == 0
    dq = to_dev(gen.normal_bshd(B, S, H, D, 303, gen.STREAM_Q))
    dk = to_dev(gen.normal_bshd(B, S, H, D, 303, gen.STREAM_K))
    dv = to_dev(gen.normal_bshd(B, S, H, D, 303, gen.STREAM_V))
    o_ref = torch.empty_like(dq)
    h3.h3attn_prefill(dq, dk, dv, o_ref, 1.0 / np.sqrt(D), causal=True)
    o = torch.full_like(dq, float("nan"))
    _noalloc(h3, dq, dk, dv, o, 1.0 / np.sqrt(D), causal=True)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == 0
    check_close(from_dev(o), bf16_f64(from_dev(o_ref)), "noalloc causal")
