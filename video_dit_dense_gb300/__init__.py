"""Thin ctypes binding of libh3attn (the H3 attention step on one GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libh3attn.so``.  PyTorch supplies device memory and streams.
There is no CPU or eager fallback: if the library is missing or the device
is not sm_103, calls raise.

The entry points mirror the C ABI in ``include/h3attn.h``:

* ``h3attn_qk_norm_rope(q, k, wq, wk, cos, sin, rotary_dim, eps, stream)`` --
  fused Q/K RMSNorm, bf16 boundary and partial RoPE, in place (FastVideo
  PR #1832 "Add FlashInfer attention backend support for MiniMax H3",
  section "Preserve H3-specific attention behavior").
* ``h3attn_qk_norm_rope_out(q, k, q_out, k_out, ...)`` -- the same step into
  separate outputs, leaving the raw q and k in place (SGLang PR #37903
  "[diffusion] model: support VDN-H3 ...", section "Modifications": the
  out-of-place variant, bit-equal to the in-place one, keeps the raw q/k).
* ``h3attn_prefill_window(q, k, v, o, window, scale, mask, stream)`` -- the
  chunked window with anchor frames of SGLang PR #37903 ("Modifications",
  hybrid_window_attn_h3), key tiles outside a query block's window skipped.
* ``h3attn_rmsnorm_modulate(x, y, w, scale, shift, idx, eps, stream)`` --
  fused RMSNorm -> indexed AdaLN scale/shift modulation of DiT hidden rows
  with the bf16 boundaries of the unfused path (TeleFuser PR #37, section
  2.5).
* ``h3attn_prefill(q, k, v, o, scale, mask, causal, stream)`` -- dense
  prefill attention on BSHD bf16 tensors with GQA, cross-attention, causal
  and boolean-mask variants (FastVideo PR #1799 "Add opt-in FlashInfer
  attention backend for Wan", section "Implementation").
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libh3attn.so")

H3ATTN_OK = 0
H3ATTN_ERR_INVALID_ARG = 1
H3ATTN_ERR_MISALIGNED = 2
H3ATTN_ERR_UNSUPPORTED_HEAD_DIM = 3
H3ATTN_ERR_UNSUPPORTED_DEVICE = 4
H3ATTN_ERR_UNSUPPORTED_MASK = 5
H3ATTN_ERR_LAUNCH = 6
H3ATTN_ERR_TIMEOUT = 7

# Every symbol include/h3attn.h declares.
EXPORTED = ("h3attn_qk_norm_rope", "h3attn_qk_norm_rope_out", "h3attn_prefill", "h3attn_prefill_ws",
            "h3attn_prefill_workspace_size", "h3attn_prefill_noalloc", "h3attn_prefill_window",
            "h3attn_rmsnorm_modulate",
            "h3attn_status_string", "h3attn_check_device_status", "h3attn_version")


class H3AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.h3attn_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {msg} (status {status})")


class h3attn_mask_t(ctypes.Structure):
    _fields_ = [("kv_len", ctypes.c_void_p), ("q_len", ctypes.c_void_p),
                ("causal_b", ctypes.c_void_p), ("bits", ctypes.c_void_p)]


class h3attn_window_t(ctypes.Structure):
    _fields_ = [("frame_tokens", ctypes.c_int), ("anchor_frames", ctypes.c_int),
                ("chunk_frames", ctypes.c_int), ("radius", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libh3attn.so for sm_103a in this directory."""
    from . import _build
    return _build.build(force=force, verbose=verbose)


def load(path: str = LIB_PATH):
    """Load libh3attn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with video_dit_dense_gb300.build()")
            lib = ctypes.CDLL(path)
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            lib.h3attn_qk_norm_rope.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, P]
            lib.h3attn_qk_norm_rope.restype = I
            lib.h3attn_qk_norm_rope_out.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
            lib.h3attn_qk_norm_rope_out.restype = I
            lib.h3attn_rmsnorm_modulate.argtypes = [P, P, P, P, P, P, I, I, I, F, P]
            lib.h3attn_rmsnorm_modulate.restype = I
            lib.h3attn_prefill.argtypes = [P, P, P, P, I, I, I, I, I, I, F,
                                           ctypes.POINTER(h3attn_mask_t), I, P]
            lib.h3attn_prefill.restype = I
            lib.h3attn_prefill_ws.argtypes = [P, P, P, P, I, I, I, I, I, I, F,
                                              ctypes.POINTER(h3attn_mask_t), I, P, ctypes.c_size_t, P]
            lib.h3attn_prefill_ws.restype = I
            lib.h3attn_prefill_workspace_size.argtypes = [I, I, I, I, I, I, ctypes.POINTER(h3attn_mask_t), I,
                                                          ctypes.POINTER(ctypes.c_size_t)]
            lib.h3attn_prefill_workspace_size.restype = I
            lib.h3attn_prefill_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F,
                                                   ctypes.POINTER(h3attn_mask_t), I, P]
            lib.h3attn_prefill_noalloc.restype = I
            lib.h3attn_prefill_window.argtypes = [P, P, P, P, I, I, I, I, I, F, ctypes.POINTER(h3attn_window_t),
                                                  ctypes.POINTER(h3attn_mask_t), P]
            lib.h3attn_prefill_window.restype = I
            lib.h3attn_status_string.argtypes = [I]
            lib.h3attn_status_string.restype = ctypes.c_char_p
            lib.h3attn_check_device_status.argtypes = [P]
            lib.h3attn_check_device_status.restype = I
            lib.h3attn_version.argtypes = []
            lib.h3attn_version.restype = I
            _lib = lib
    return _lib


def lib():
    return load()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_bf16(name, t):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous 4-D bf16 CUDA tensor (BSHD)")
    if t.requires_grad:
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name}: inference only, grad-enabled inputs are rejected")


def _raise_if(status, where):
    if status != H3ATTN_OK:
        raise H3AttnError(status, where)


def _norm_rope_args(q, k, wq, wk, cos, sin, rotary_dim):
    if q is None and k is None:
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "at least one of q and k must be given")
    ref = q if q is not None else k
    if q is not None:
        _check_bf16("q", q)
    if k is not None:
        _check_bf16("k", k)
    B, S, _, D = ref.shape
    Hq = q.shape[2] if q is not None else 0
    Hkv = k.shape[2] if k is not None else 0
    if k is not None and q is not None and (k.shape[0], k.shape[1], k.shape[3]) != (B, S, D):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "q and k must share batch, sequence and head_dim")
    import torch
    for name, t in (("wq", wq), ("wk", wk), ("cos", cos), ("sin", sin)):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()):
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous float32 CUDA tensor")
    # the kernel reads D weights per row: a shorter tensor would be read past its end
    for name, rows, w in (("wq", q, wq), ("wk", k, wk)):
        if rows is not None and (w is None or w.numel() != D):
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be a [{D}] float32 CUDA tensor")
    if rotary_dim > 0:
        if cos is None or sin is None:
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "cos and sin are required when rotary_dim > 0")
        if cos.shape[-1] != rotary_dim // 2 or cos.numel() < S * (rotary_dim // 2) or sin.shape != cos.shape:
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "cos/sin must be [>=S, rotary_dim/2]")
    return B, S, Hq, Hkv, D


def h3attn_qk_norm_rope(q, k, wq, wk, cos, sin, rotary_dim=96, eps=1e-6, stream=None):
    """In-place fused Q/K RMSNorm + bf16 boundary + partial RoPE.

    q: [B, S, Hq, D] bf16, k: [B, S, Hkv, D] bf16 (either may be None);
    wq, wk: [D] float32; cos, sin: [>=S, rotary_dim/2] float32.
    """
    load()
    B, S, Hq, Hkv, D = _norm_rope_args(q, k, wq, wk, cos, sin, rotary_dim)
    st = _lib.h3attn_qk_norm_rope(_ptr(q), _ptr(k), _ptr(wq), _ptr(wk), _ptr(cos), _ptr(sin),
                                  B, S, Hq, Hkv, D, int(rotary_dim), float(eps), _stream_handle(stream))
    _raise_if(st, "h3attn_qk_norm_rope")


def h3attn_qk_norm_rope_out(q, k, q_out, k_out, wq, wk, cos, sin, rotary_dim=96, eps=1e-6, stream=None):
    """Out-of-place fused Q/K RMSNorm + bf16 boundary + partial RoPE: q and k
    are read only; q_out, k_out (same shapes, preallocated) receive the
    result, bit-identical to the in-place call."""
    load()
    B, S, Hq, Hkv, D = _norm_rope_args(q, k, wq, wk, cos, sin, rotary_dim)
    for name, src, dst in (("q_out", q, q_out), ("k_out", k, k_out)):
        if (src is None) != (dst is None):
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be given exactly when its input is")
        if dst is not None:
            _check_bf16(name, dst)
            if tuple(dst.shape) != tuple(src.shape):
                raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must have the shape of its input")
    st = _lib.h3attn_qk_norm_rope_out(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _ptr(wq), _ptr(wk), _ptr(cos),
                                      _ptr(sin), B, S, Hq, Hkv, D, int(rotary_dim), float(eps),
                                      _stream_handle(stream))
    _raise_if(st, "h3attn_qk_norm_rope_out")
    return q_out, k_out


@dataclass
class Mask:
    """Mask descriptor (device tensors, per batch item): see h3attn_mask_t."""
    kv_len: object = None    # int32 [B]
    q_len: object = None     # int32 [B]
    causal_b: object = None  # uint8 [B]
    bits: object = None      # int32/uint32 [B, Sq, ceil(Sk/32)]


def _mask_struct(mask: Mask, B: int):
    """Checks the per-sample fields of a mask and packs its pointers into an
    h3attn_mask_t (the kernels read B entries of each field given)."""
    import torch
    for name, t, dt in (("kv_len", mask.kv_len, torch.int32), ("q_len", mask.q_len, torch.int32),
                        ("causal_b", mask.causal_b, torch.uint8)):
        if t is not None and (t.dtype != dt or t.numel() != B or not t.is_cuda or not t.is_contiguous()):
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous [{B}] {dt} CUDA tensor")
    return ctypes.pointer(h3attn_mask_t(_ptr(mask.kv_len), _ptr(mask.q_len), _ptr(mask.causal_b), _ptr(mask.bits)))


def h3attn_prefill(q, k, v, o, scale=None, mask: Mask | None = None, causal=False, stream=None, workspace=None):
    """o <- softmax(q k^T * scale) v on BSHD bf16 tensors (o preallocated).

    workspace: None, or a CUDA tensor of at least h3attn_prefill_workspace_size()
    bytes for the split-key tail (the call then goes through h3attn_prefill_ws).
    """
    load()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_bf16(name, t)
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or tuple(o.shape) != tuple(q.shape):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "shape mismatch between q, k, v and o")
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    mptr = None
    if mask is not None:
        if mask.bits is not None:
            if mask.bits.dim() == 4:
                raise H3AttnError(H3ATTN_ERR_UNSUPPORTED_MASK, "per-head [B, H, Q, K] masks are not supported")
            W = (Sk + 31) // 32
            if tuple(mask.bits.shape) != (B, Sq, W) or mask.bits.element_size() != 4 or \
                    not mask.bits.is_cuda or not mask.bits.is_contiguous():
                raise H3AttnError(H3ATTN_ERR_INVALID_ARG,
                                  f"bits must be contiguous 32-bit CUDA words of shape [{B}, {Sq}, {W}]")
        mptr = _mask_struct(mask, B)
    if workspace is None:
        st = _lib.h3attn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Sq, Sk, Hq, Hkv, D, float(scale), mptr,
                                 int(bool(causal)), _stream_handle(stream))
        _raise_if(st, "h3attn_prefill")
    else:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "workspace must be a contiguous CUDA tensor")
        nbytes = workspace.numel() * workspace.element_size()
        st = _lib.h3attn_prefill_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Sq, Sk, Hq, Hkv, D, float(scale), mptr,
                                    int(bool(causal)), _ptr(workspace), nbytes, _stream_handle(stream))
        _raise_if(st, "h3attn_prefill_ws")
    return o


def h3attn_prefill_workspace_size(B, Sq, Sk, Hq, Hkv, D, mask: Mask | None = None, causal=False) -> int:
    """Bytes of workspace the split-key tail needs for this call (0: no split).
    Only the presence of the mask fields matters, not their values."""
    load()
    mptr = None
    if mask is not None:
        mptr = ctypes.pointer(h3attn_mask_t(_ptr(mask.kv_len), _ptr(mask.q_len), _ptr(mask.causal_b),
                                            _ptr(mask.bits)))
    out = ctypes.c_size_t(0)
    st = _lib.h3attn_prefill_workspace_size(B, Sq, Sk, Hq, Hkv, D, mptr, int(bool(causal)), ctypes.byref(out))
    _raise_if(st, "h3attn_prefill_workspace_size")
    return int(out.value)


# Bytes of the fixed scratch array behind h3attn_prefill_noalloc.
NOALLOC_SCRATCH_BYTES = 12 << 20


def h3attn_prefill_noalloc(q, k, v, o, scale=None, mask: Mask | None = None, causal=False, stream=None):
    """h3attn_prefill with the split-key tail's scratch in the library's fixed
    12 MiB device array: the call allocates nothing (for hosts that cannot
    allocate device memory).  Calls whose kernels may overlap must be ordered
    by the caller, since they share the array."""
    load()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_bf16(name, t)
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape) or tuple(o.shape) != tuple(q.shape):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "shape mismatch between q, k, v and o")
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    mptr = None if mask is None else _mask_struct(mask, B)
    need = h3attn_prefill_workspace_size(B, Sq, Sk, Hq, Hkv, D, mask, causal)
    if need > NOALLOC_SCRATCH_BYTES:
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"h3attn_prefill_noalloc: this call needs {need} bytes of "
                                                  f"scratch, more than the fixed {NOALLOC_SCRATCH_BYTES}")
    st = _lib.h3attn_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Sq, Sk, Hq, Hkv, D, float(scale), mptr,
                                     int(bool(causal)), _stream_handle(stream))
    _raise_if(st, "h3attn_prefill_noalloc")
    return o


def prefill_workspace(q, k, mask: Mask | None = None, causal=False):
    """A workspace tensor sized for prefill(q, k, ...) on the current device,
    or None when the call would not split (allocated by torch: the library
    allocates nothing)."""
    import torch
    B, Sq, Hq, D = q.shape
    n = h3attn_prefill_workspace_size(B, Sq, k.shape[1], Hq, k.shape[2], D, mask, causal)
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def h3attn_rmsnorm_modulate(x, y, w, scale, shift, idx=None, eps=1e-6, stream=None):
    """y <- bf16(bf16(bf16(rmsnorm(x) * w) * bf16(1 + scale[idx])) + shift[idx]) row by row.

    x, y: [T, C] bf16 CUDA tensors (y may be x); w: [C] float32 or None;
    scale, shift: [N, C] bf16; idx: [T] int32 or None (table row 0 for all).
    """
    import torch
    load()
    for name, t in (("x", x), ("y", y), ("scale", scale), ("shift", shift)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"{name} must be a contiguous 2-D bf16 CUDA tensor")
    T, C = x.shape
    N = scale.shape[0]
    if tuple(y.shape) != (T, C) or tuple(scale.shape) != (N, C) or tuple(shift.shape) != (N, C):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "shape mismatch between x, y, scale and shift")
    if w is not None and (w.dtype != torch.float32 or not w.is_cuda or w.numel() != C):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"w must be a [{C}] float32 CUDA tensor")
    if idx is not None and (idx.dtype != torch.int32 or not idx.is_cuda or idx.numel() != T):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, f"idx must be a [{T}] int32 CUDA tensor")
    st = _lib.h3attn_rmsnorm_modulate(_ptr(x), _ptr(y), _ptr(w), _ptr(scale), _ptr(shift), _ptr(idx), T, C, N,
                                      float(eps), _stream_handle(stream))
    _raise_if(st, "h3attn_rmsnorm_modulate")
    return y


@dataclass
class Window:
    """Chunked window with anchor frames: see h3attn_window_t."""
    frame_tokens: int
    anchor_frames: int
    chunk_frames: int
    radius: int


def h3attn_prefill_window(q, k, v, o, window: Window, scale=None, mask: Mask | None = None, stream=None):
    """o <- windowed self-attention of q against k, v (BSHD bf16, Sq == Sk)."""
    load()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check_bf16(name, t)
    B, S, Hq, D = q.shape
    if tuple(k.shape[:2]) != (B, S) or k.shape[3] != D or tuple(v.shape) != tuple(k.shape) or \
            tuple(o.shape) != tuple(q.shape):
        raise H3AttnError(H3ATTN_ERR_INVALID_ARG, "shape mismatch between q, k, v and o (self-attention)")
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    mptr = None
    if mask is not None:
        if mask.bits is not None or mask.causal_b is not None:
            raise H3AttnError(H3ATTN_ERR_UNSUPPORTED_MASK, "the window combines with kv_len / q_len only")
        mptr = _mask_struct(mask, B)
    w = h3attn_window_t(int(window.frame_tokens), int(window.anchor_frames), int(window.chunk_frames),
                        int(window.radius))
    st = _lib.h3attn_prefill_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, S, Hq, k.shape[2], D, float(scale),
                                    ctypes.pointer(w), mptr, _stream_handle(stream))
    _raise_if(st, "h3attn_prefill_window")
    return o


def h3attn_check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    load()
    return _lib.h3attn_check_device_status(_stream_handle(stream))


def h3attn_status_string(status: int) -> str:
    return load().h3attn_status_string(status).decode()


def h3attn_version() -> int:
    return load().h3attn_version()


# Short aliases.
qk_norm_rope = h3attn_qk_norm_rope
prefill = h3attn_prefill
check_device_status = h3attn_check_device_status
