"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side argument validation answers before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

import video_dit_dense_gb300 as h3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h3attn.h")


@pytest.fixture(scope="module")
def lib():
    h3.build()
    return h3.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("h3attn_qk_norm_rope", "h3attn_qk_norm_rope_out", "h3attn_prefill", "h3attn_prefill_window",
              "h3attn_rmsnorm_modulate", "h3attn_status_string", "h3attn_check_device_status", "h3attn_version"):
        assert n in names
    assert set(names) == set(h3.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", h3.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(h3attn_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert lib.h3attn_version() == 10000
    for code in range(8):
        s = lib.h3attn_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.h3attn_status_string(99).decode() == "unknown status"


FAKE = 0x10000  # 16-byte aligned fake device address; validation fails before any use


def prefill(lib, q=FAKE, k=FAKE * 2, v=FAKE * 3, o=FAKE * 4, B=1, Sq=256, Sk=256, Hq=4, Hkv=4, D=128,
            scale=0.088, mask=None, causal=0):
    return lib.h3attn_prefill(q, k, v, o, B, Sq, Sk, Hq, Hkv, D, scale, mask, causal, None)


def test_prefill_validation(lib):
    assert prefill(lib, D=96) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert prefill(lib, D=512) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert prefill(lib, Hq=6, Hkv=4) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, scale=-1.0) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, scale=float("nan")) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, scale=0.0) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, Sk=0) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, Sq=100, Sk=200, causal=1) == h3.H3ATTN_ERR_INVALID_ARG
    m = h3.h3attn_mask_t(None, None, FAKE, None)
    assert prefill(lib, Sq=100, Sk=200, mask=ctypes.pointer(m)) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, q=FAKE + 8) == h3.H3ATTN_ERR_MISALIGNED
    assert prefill(lib, o=FAKE * 4 + 2) == h3.H3ATTN_ERR_MISALIGNED
    m = h3.h3attn_mask_t(None, None, None, FAKE + 2)
    assert prefill(lib, mask=ctypes.pointer(m)) == h3.H3ATTN_ERR_MISALIGNED
    assert prefill(lib, q=None) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, o=FAKE) == h3.H3ATTN_ERR_INVALID_ARG  # o aliases q
    assert prefill(lib, B=65536) == h3.H3ATTN_ERR_INVALID_ARG
    # 2^31 work units (128-row query blocks x heads x batch) do not fit 32 bits
    assert prefill(lib, B=4096, Sq=2**23, Sk=2**23, Hq=64, Hkv=64) == h3.H3ATTN_ERR_INVALID_ARG
    assert prefill(lib, B=0) == h3.H3ATTN_OK  # empty batch: no-op, nothing launched
    assert prefill(lib, Sq=0) == h3.H3ATTN_OK


def norm(lib, q=FAKE, k=FAKE * 64, wq=FAKE * 200, wk=FAKE * 201, cos=FAKE * 202, sin=FAKE * 203, B=1, S=16,
         Hq=2, Hkv=2, D=128, rot=96, eps=1e-6):
    return lib.h3attn_qk_norm_rope(q, k, wq, wk, cos, sin, B, S, Hq, Hkv, D, rot, eps, None)


def test_norm_rope_validation(lib):
    assert norm(lib, D=80) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert norm(lib, rot=95) == h3.H3ATTN_ERR_INVALID_ARG  # odd
    assert norm(lib, rot=-2) == h3.H3ATTN_ERR_INVALID_ARG
    assert norm(lib, rot=144) == h3.H3ATTN_ERR_INVALID_ARG  # > D
    assert norm(lib, eps=-1.0) == h3.H3ATTN_ERR_INVALID_ARG
    assert norm(lib, eps=float("inf")) == h3.H3ATTN_ERR_INVALID_ARG
    assert norm(lib, cos=None) == h3.H3ATTN_ERR_INVALID_ARG
    assert norm(lib, wq=None) == h3.H3ATTN_ERR_INVALID_ARG
    assert norm(lib, q=None) == h3.H3ATTN_ERR_INVALID_ARG  # q absent but Hq > 0
    assert norm(lib, q=FAKE + 4) == h3.H3ATTN_ERR_MISALIGNED
    assert norm(lib, cos=FAKE * 202 + 4) == h3.H3ATTN_ERR_MISALIGNED
    assert norm(lib, k=FAKE + 256) == h3.H3ATTN_ERR_INVALID_ARG  # k overlaps q
    assert norm(lib, B=0) == h3.H3ATTN_OK
    assert norm(lib, q=None, Hq=0, k=None, Hkv=0) == h3.H3ATTN_OK


def norm_out(lib, q=FAKE, k=FAKE * 64, q_out=FAKE * 400, k_out=FAKE * 500, wq=FAKE * 200, wk=FAKE * 201,
             cos=FAKE * 202, sin=FAKE * 203, B=1, S=16, Hq=2, Hkv=2, D=128, rot=96, eps=1e-6):
    return lib.h3attn_qk_norm_rope_out(q, k, q_out, k_out, wq, wk, cos, sin, B, S, Hq, Hkv, D, rot, eps, None)


def test_norm_rope_out_validation(lib):
    rows_bytes = 16 * 2 * 128 * 2  # one tensor of B*S*H rows of D bf16
    assert norm_out(lib, q_out=None) == h3.H3ATTN_ERR_INVALID_ARG          # output missing
    assert norm_out(lib, q=None, Hq=0) == h3.H3ATTN_ERR_INVALID_ARG        # output without input
    assert norm_out(lib, q_out=FAKE * 400 + 8) == h3.H3ATTN_ERR_MISALIGNED
    assert norm_out(lib, q_out=FAKE + rows_bytes // 2) == h3.H3ATTN_ERR_INVALID_ARG   # partly over q
    assert norm_out(lib, q_out=FAKE * 64) == h3.H3ATTN_ERR_INVALID_ARG      # writes over input k
    assert norm_out(lib, k_out=FAKE) == h3.H3ATTN_ERR_INVALID_ARG           # writes over input q
    assert norm_out(lib, k_out=FAKE * 400 + 256) == h3.H3ATTN_ERR_INVALID_ARG  # overlaps q_out
    assert norm_out(lib, D=80) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert norm_out(lib, B=0) == h3.H3ATTN_OK
    assert norm_out(lib, q=None, Hq=0, q_out=None, k=None, Hkv=0, k_out=None) == h3.H3ATTN_OK


def modulate(lib, x=FAKE, y=FAKE * 100, w=FAKE * 200, scale=FAKE * 300, shift=FAKE * 400, idx=FAKE * 500, T=16,
             C=256, N=4, eps=1e-6):
    return lib.h3attn_rmsnorm_modulate(x, y, w, scale, shift, idx, T, C, N, eps, None)


def test_rmsnorm_modulate_validation(lib):
    assert modulate(lib, C=12) == h3.H3ATTN_ERR_INVALID_ARG        # not a multiple of 8
    assert modulate(lib, C=8200) == h3.H3ATTN_ERR_INVALID_ARG      # above 8192
    assert modulate(lib, N=0) == h3.H3ATTN_ERR_INVALID_ARG
    assert modulate(lib, eps=-1.0) == h3.H3ATTN_ERR_INVALID_ARG
    assert modulate(lib, scale=None) == h3.H3ATTN_ERR_INVALID_ARG
    assert modulate(lib, x=FAKE + 8) == h3.H3ATTN_ERR_MISALIGNED
    assert modulate(lib, idx=FAKE * 500 + 2) == h3.H3ATTN_ERR_MISALIGNED
    assert modulate(lib, y=FAKE + 512) == h3.H3ATTN_ERR_INVALID_ARG      # partly over x
    assert modulate(lib, y=FAKE * 300) == h3.H3ATTN_ERR_INVALID_ARG      # over the scale table
    assert modulate(lib, T=0) == h3.H3ATTN_OK


def window_call(lib, win=(16, 1, 5, 1), D=128, S=256, mask=None, q=FAKE, o=FAKE * 4):
    w = ctypes.pointer(h3.h3attn_window_t(*win)) if win is not None else None
    return lib.h3attn_prefill_window(q, FAKE * 2, FAKE * 3, o, 1, S, 4, 4, D, 0.088, w, mask, None)


def test_prefill_window_validation(lib):
    assert window_call(lib, win=None) == h3.H3ATTN_ERR_INVALID_ARG
    assert window_call(lib, win=(0, 1, 5, 1)) == h3.H3ATTN_ERR_INVALID_ARG      # frame of no tokens
    assert window_call(lib, win=(16, 1, 0, 1)) == h3.H3ATTN_ERR_INVALID_ARG     # chunk of no frames
    assert window_call(lib, win=(16, -1, 5, 1)) == h3.H3ATTN_ERR_INVALID_ARG
    assert window_call(lib, win=(16, 1, 5, -1)) == h3.H3ATTN_ERR_INVALID_ARG
    assert window_call(lib, win=(1 << 20, 1, 1 << 12, 1)) == h3.H3ATTN_ERR_INVALID_ARG  # chunk tokens overflow
    assert window_call(lib, D=256) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    m = h3.h3attn_mask_t(None, None, FAKE, None)
    assert window_call(lib, mask=ctypes.pointer(m)) == h3.H3ATTN_ERR_UNSUPPORTED_MASK
    m = h3.h3attn_mask_t(None, None, None, FAKE)
    assert window_call(lib, mask=ctypes.pointer(m)) == h3.H3ATTN_ERR_UNSUPPORTED_MASK
    assert window_call(lib, q=FAKE + 8) == h3.H3ATTN_ERR_MISALIGNED
    assert window_call(lib, o=FAKE) == h3.H3ATTN_ERR_INVALID_ARG                 # o aliases q
    assert window_call(lib, S=0) == h3.H3ATTN_OK


def test_binding_rejects_bad_python_arguments(lib):
    """The binding's own checks answer with H3AttnError before any CUDA call
    (CPU tensors are never accepted as device buffers)."""
    import torch
    with pytest.raises(h3.H3AttnError, match="at least one of q and k"):
        h3.h3attn_qk_norm_rope(None, None, None, None, None, None)
    cpu = torch.zeros(1, 4, 2, 128, dtype=torch.bfloat16)
    with pytest.raises(h3.H3AttnError, match="CUDA tensor"):
        h3.h3attn_qk_norm_rope(cpu, None, None, None, None, None)
    with pytest.raises(h3.H3AttnError, match="CUDA tensor"):
        h3.h3attn_prefill(cpu, cpu, cpu, cpu)
    with pytest.raises(h3.H3AttnError, match="CUDA tensor"):
        h3.h3attn_rmsnorm_modulate(cpu[0, :, 0], cpu[0, :, 0], None, cpu[0, :, 0], cpu[0, :, 0])
    with pytest.raises(h3.H3AttnError, match="inference only"):
        h3._check_bf16("q", _GradEnabledBf16())


class _GradEnabledBf16:
    """Stands in for a contiguous 4-D bf16 CUDA tensor that requires grad."""
    dtype = __import__("torch").bfloat16
    is_cuda = True
    requires_grad = True

    def is_contiguous(self):
        return True

    def dim(self):
        return 4


def test_workspace_entry_points_validation(lib):
    n = ctypes.c_size_t(123)
    ws = lib.h3attn_prefill_workspace_size
    assert ws(1, 256, 256, 4, 4, 96, None, 0, ctypes.byref(n)) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert n.value == 0  # cleared before any check that fails
    assert ws(1, 256, 0, 4, 4, 128, None, 0, ctypes.byref(n)) == h3.H3ATTN_ERR_INVALID_ARG
    assert ws(1, 256, 256, 6, 4, 128, None, 0, ctypes.byref(n)) == h3.H3ATTN_ERR_INVALID_ARG
    assert ws(1, 256, 256, 4, 4, 128, None, 0, None) == h3.H3ATTN_ERR_INVALID_ARG
    assert ws(0, 256, 256, 4, 4, 128, None, 0, ctypes.byref(n)) == h3.H3ATTN_OK and n.value == 0

    M = 0x100000  # 1 MiB apart: the [1, 256, 4, 128] tensors do not overlap

    def pws(workspace, q=M, o=4 * M, D=128):
        return lib.h3attn_prefill_ws(q, 2 * M, 3 * M, o, 1, 256, 256, 4, 4, D, 0.088, None, 0,
                                     workspace, 1 << 20, None)
    assert pws(5 * M + 8) == h3.H3ATTN_ERR_MISALIGNED
    assert pws(5 * M, D=96) == h3.H3ATTN_ERR_UNSUPPORTED_HEAD_DIM
    assert pws(5 * M, q=M + 8) == h3.H3ATTN_ERR_MISALIGNED
