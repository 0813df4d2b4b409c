"""Failure detection without a GPU fault: the attention kernel's waits are
bounded.  With the producer told to issue no copies (a flag that makes a
wait run out), every waiting role gives up after the wait limit, the kernel
exits normally, the device status word reports H3ATTN_ERR_TIMEOUT, the
output is left untouched, and the context stays usable."""
import numpy as np
import pytest

import h3inputs as gen
import oracle
from helpers import check_close, from_dev, to_dev


@pytest.mark.gpu
@pytest.mark.parametrize("kernel,D", [("1", 128), ("2", 128), ("3", 128), ("4", 128), ("6", 128), ("5", 256), ("4", 64)],
                         ids=["one_tile", "two_tiles", "persistent", "two_ctas", "chain", "wide_d256", "two_ctas_sep_p_d64"])
def test_stalled_producer_times_out_and_context_survives(h3, monkeypatch, kernel, D):
    import torch
    B, S, H = 1, 256, 1  # two query tiles: one wait limit of runtime
    q = gen.normal_bshd(B, S, H, D, 5, gen.STREAM_Q)
    k = gen.normal_bshd(B, S, H, D, 5, gen.STREAM_K)
    v = gen.normal_bshd(B, S, H, D, 5, gen.STREAM_V)
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full(dq.shape, 7.0, dtype=torch.bfloat16, device="cuda")
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK

    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", kernel)
    monkeypatch.setenv("H3ATTN_FAULT_INJECT_STALL_PRODUCER", "1")
    monkeypatch.setenv("H3ATTN_WAIT_LIMIT_MS", "200")
    h3.h3attn_prefill(dq, dk, dv, o, 1.0 / np.sqrt(D))
    assert h3.h3attn_check_device_status() == h3.H3ATTN_ERR_TIMEOUT
    assert torch.all(o == 7.0), "an aborted launch must not write its output"
    # the status word was cleared by the read
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK

    monkeypatch.delenv("H3ATTN_FAULT_INJECT_STALL_PRODUCER")
    h3.h3attn_prefill(dq, dk, dv, o, 1.0 / np.sqrt(D))
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK
    check_close(from_dev(o), oracle.attention_f64(q, k, v, 1.0 / np.sqrt(D)), "after timeout")


@pytest.mark.gpu
def test_stalled_split_launch_reports_the_timeout(h3, monkeypatch):
    """The split-key tail: the split kernel's waits run out the same way and
    the call reports H3ATTN_ERR_TIMEOUT.  Its combine kernel still runs and
    writes o from whatever partials the workspace holds, so here the status
    word, not the output, carries the failure; the next call is correct."""
    import torch
    B, Sq, Sk, H, D = 1, 128, 512, 1, 128  # one unit of four key tiles: two pieces
    q = gen.normal_bshd(B, Sq, H, D, 6, gen.STREAM_Q)
    k = gen.normal_bshd(B, Sk, H, D, 6, gen.STREAM_K)
    v = gen.normal_bshd(B, Sk, H, D, 6, gen.STREAM_V)
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    o = torch.empty_like(dq)
    monkeypatch.setenv("H3ATTN_ATTN_KERNEL", "1")
    ws = h3.prefill_workspace(dq, dk)
    assert ws is not None, "this shape is expected to split"
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK

    monkeypatch.setenv("H3ATTN_FAULT_INJECT_STALL_PRODUCER", "1")
    monkeypatch.setenv("H3ATTN_WAIT_LIMIT_MS", "200")
    h3.h3attn_prefill(dq, dk, dv, o, 1.0 / np.sqrt(D), workspace=ws)
    assert h3.h3attn_check_device_status() == h3.H3ATTN_ERR_TIMEOUT
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK

    monkeypatch.delenv("H3ATTN_FAULT_INJECT_STALL_PRODUCER")
    h3.h3attn_prefill(dq, dk, dv, o, 1.0 / np.sqrt(D), workspace=ws)
    torch.cuda.synchronize()
    assert h3.h3attn_check_device_status() == h3.H3ATTN_OK
    check_close(from_dev(o), oracle.attention_f64(q, k, v, 1.0 / np.sqrt(D)), "split after timeout")
