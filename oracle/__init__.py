"""CPU oracle of the H3 attention step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The CUDA library does not use
it, and it imports nothing from the CUDA library.

What it computes (all in double precision, from the definitions):

* ``qk_norm_rope_f64`` -- per (token, head) RMSNorm over the D channels of a
  row, a bf16 rounding boundary, then rotate-half RoPE on the first
  ``rotary_dim`` channels (FastVideo PR #1832 "Add FlashInfer attention
  backend support for MiniMax H3", section "Preserve H3-specific attention
  behavior"; TeleFuser PR #37 "perf(minimax-h3): optimize Ulysses attention
  and DiT kernels", section 2.2 steps 1-3).
* ``qk_norm_rope_emulate`` -- the same step in float32 in a fixed operation
  order; the bit-exact contract for the CUDA norm/RoPE kernel (TeleFuser
  PR #37 section 2.5 holds fused kernels to element-wise bit-exactness).
* ``rmsnorm_modulate_f64`` / ``rmsnorm_modulate_emulate`` -- RMSNorm of a DiT
  hidden row, then indexed AdaLN modulation y = n * (1 + scale[idx]) +
  shift[idx] with the bf16 store after every step of the unfused path
  (TeleFuser PR #37 section 2.5); fp64 definition and the float32
  fixed-order contract of the CUDA kernel.
* ``attention_window_f64`` -- self-attention under the chunked window with
  anchor frames of SGLang PR #37903 ("Modifications", hybrid_window_attn_h3):
  anchor rows and keys dense, any other query attends the keys of the chunks
  within the radius of its own (the anchor frames shift the chunk grid).
* ``attention_f64`` -- softmax(Q K^T * scale) V per output row with GQA,
  cross-attention, causal, key-padding and packed boolean [Q, K] masks
  (FastVideo PR #1799 "Add opt-in FlashInfer attention backend for Wan",
  section "Implementation").

Pins (tests under ``tests/test_oracle_*.py``): library routines in float64
(torch ``rms_norm`` and ``scaled_dot_product_attention`` on the CPU), closed
forms (constant rows, a single key, zero scale, quarter-turn rotations),
invariants (unit RMS, pair norms, angle additivity, key permutation, constant
V, poisoned masked keys) and the fp64-vs-emulation rounding bound.
"""
from __future__ import annotations

import contextlib
import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (skipped when the source is unchanged)."""
    stamp = _LIB + ".stamp"
    with open(_SRC, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == h:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    _compile(_SRC, tmp)
    os.replace(tmp, _LIB)
    with open(stamp, "w") as f:
        f.write(h)
    return _LIB


def _compile(src: str, out: str) -> None:
    # -ffp-contract=off: no implicit fused multiply-adds (the emulation's
    # rounding order is part of its contract); no fast-math of any kind.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)


@contextlib.contextmanager
def built_from(source: str, workdir: str):
    """For the tests that plant a mistake in a copy of oracle.c: compile the
    given C source with the flags of build() and route every call of this
    module through that build inside the with-block."""
    global _lib
    src = os.path.join(workdir, "oracle_variant.c")
    out = os.path.join(workdir, "liboracle_variant.so")
    with open(src, "w") as f:
        f.write(source)
    _compile(src, out)
    variant = _bind(ctypes.CDLL(out))
    with _lock:
        saved, _lib = _lib, variant
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    """Declare the argument and result types of the oracle's C entry points."""
    P, I64, I, D, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                       ctypes.c_float)
    lib.oracle_qk_norm_rope_f64.argtypes = [P, P, I64, I, I, I, P, P, P, I, D, I, I]
    lib.oracle_qk_norm_rope_emulate_bf16.argtypes = [P, P, I64, I, I, I, P, P, P, I, F, I]
    lib.oracle_attention_f64.argtypes = [P, P, P, I, I, I, I, I, I, D, I, P, P, P, P, P,
                                         I64, P, I]
    lib.oracle_round_f64_to_bf16.argtypes = [P, P, I64]
    lib.oracle_rmsnorm_modulate_f64.argtypes = [P, P, I64, I, P, P, P, P, I, D, I]
    lib.oracle_rmsnorm_modulate_emulate_bf16.argtypes = [P, P, I64, I, P, P, P, P, I, F, I]
    lib.oracle_rmsnorm_modulate_f64.restype = None
    lib.oracle_rmsnorm_modulate_emulate_bf16.restype = None
    lib.oracle_allowed_pairs.argtypes = [I, I, I, I, P, P, P]
    lib.oracle_allowed_pairs.restype = ctypes.c_int64
    lib.oracle_attention_window_f64.argtypes = [P, P, P, I, I, I, I, I, D, I, I, I, I, P, P, P, I64, P, I]
    lib.oracle_attention_window_f64.restype = None
    lib.oracle_window_allowed_pairs.argtypes = [I, I, I, I, I, I]
    lib.oracle_window_allowed_pairs.restype = ctypes.c_int64
    for fn in ("oracle_qk_norm_rope_f64", "oracle_qk_norm_rope_emulate_bf16",
               "oracle_attention_f64", "oracle_round_f64_to_bf16"):
        getattr(lib, fn).restype = None
    return lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous numpy"
    return a.ctypes.data


def _check_rows(x, D):
    assert x.dtype == np.uint16 and x.shape[-1] == D


def qk_norm_rope_f64(x, w, cos, sin, rotary_dim, eps, round_boundary=True, nthreads=0):
    """x: bf16 bits [B, S, H, D] -> fp64 [B, S, H, D] (the value before the final bf16 store)."""
    B, S, H, D = x.shape
    _check_rows(x, D)
    w = np.ascontiguousarray(w, dtype=np.float32)
    half = rotary_dim // 2
    cos = np.ascontiguousarray(cos, dtype=np.float32).reshape(-1, half) if half else np.zeros((S, 1), np.float32)
    sin = np.ascontiguousarray(sin, dtype=np.float32).reshape(-1, half) if half else np.zeros((S, 1), np.float32)
    assert rotary_dim % 2 == 0 and rotary_dim <= D
    assert half == 0 or cos.shape[0] >= S
    y = np.empty(x.shape, dtype=np.float64)
    _load().oracle_qk_norm_rope_f64(_p(x), _p(y), B * S * H, S, H, D, _p(w), _p(cos), _p(sin),
                                    rotary_dim, float(eps), int(bool(round_boundary)), nthreads)
    return y


def qk_norm_rope_emulate(x, w, cos, sin, rotary_dim, eps, nthreads=0):
    """x: bf16 bits [B, S, H, D] -> bf16 bits, float32 fixed-order emulation (bit-exact contract)."""
    B, S, H, D = x.shape
    _check_rows(x, D)
    assert D % 16 == 0 and D // 16 <= 32 and (D // 16) & (D // 16 - 1) == 0
    assert rotary_dim % 2 == 0 and 0 <= rotary_dim <= D
    half = rotary_dim // 2
    w = np.ascontiguousarray(w, dtype=np.float32)
    cos = np.ascontiguousarray(cos, dtype=np.float32).reshape(-1, half) if half else np.zeros((S, 1), np.float32)
    sin = np.ascontiguousarray(sin, dtype=np.float32).reshape(-1, half) if half else np.zeros((S, 1), np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_qk_norm_rope_emulate_bf16(_p(x), _p(out), B * S * H, S, H, D, _p(w), _p(cos),
                                             _p(sin), rotary_dim, float(np.float32(eps)), nthreads)
    return out


def round_to_bf16(y: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, one rounding to nearest even."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty(y.shape, dtype=np.uint16)
    _load().oracle_round_f64_to_bf16(_p(y), _p(out), y.size)
    return out


def attention_f64(q, k, v, scale, causal=False, kv_len=None, q_len=None, causal_b=None, bits=None,
                  row_ids=None, nthreads=0):
    """Attention rows in fp64.

    q: bf16 bits [B, Sq, Hq, D]; k, v: bf16 bits [B, Sk, Hkv, D].
    row_ids: flat output-row ids ((b*Sq + i)*Hq + h), int64; None = every row.
    Returns fp64 [len(row_ids), D], or [B, Sq, Hq, D] when row_ids is None.
    """
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    assert (Bk, Dk) == (B, D) and v.shape == k.shape and Hq % Hkv == 0
    kv_len = None if kv_len is None else np.ascontiguousarray(kv_len, dtype=np.int32)
    q_len = None if q_len is None else np.ascontiguousarray(q_len, dtype=np.int32)
    causal_b = None if causal_b is None else np.ascontiguousarray(causal_b, dtype=np.uint8)
    if bits is not None:
        bits = np.ascontiguousarray(bits, dtype=np.uint32)
        assert bits.shape == (B, Sq, (Sk + 31) // 32)
    if row_ids is None:
        out = np.empty((B, Sq, Hq, D), dtype=np.float64)
        n = B * Sq * Hq
        rid = None
    else:
        rid = np.ascontiguousarray(row_ids, dtype=np.int64)
        n = rid.size
        out = np.empty((n, D), dtype=np.float64)
    _load().oracle_attention_f64(_p(q), _p(k), _p(v), B, Sq, Sk, Hq, Hkv, D, float(scale), int(bool(causal)),
                                 _p(kv_len), _p(q_len), _p(causal_b), _p(bits), _p(rid), n, _p(out), nthreads)
    return out


def allowed_pairs(B, Sq, Sk, causal=False, kv_len=None, q_len=None, causal_b=None) -> int:
    """Count of allowed (query row, key) pairs over all samples (structured masks only)."""
    kv_len = None if kv_len is None else np.ascontiguousarray(kv_len, dtype=np.int32)
    q_len = None if q_len is None else np.ascontiguousarray(q_len, dtype=np.int32)
    causal_b = None if causal_b is None else np.ascontiguousarray(causal_b, dtype=np.uint8)
    return int(_load().oracle_allowed_pairs(B, Sq, Sk, int(bool(causal)), _p(kv_len), _p(q_len), _p(causal_b)))


def _mod_args(x, w, scale, shift, idx):
    T, C = x.shape
    assert x.dtype == np.uint16 and C % 8 == 0
    N = scale.shape[0]
    assert scale.shape == (N, C) and shift.shape == (N, C) and scale.dtype == np.uint16 and shift.dtype == np.uint16
    w = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    idx = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
    assert idx is None or idx.shape == (T,)
    return T, C, N, np.ascontiguousarray(x), w, np.ascontiguousarray(scale), np.ascontiguousarray(shift), idx


def rmsnorm_modulate_f64(x, w, scale, shift, idx, eps, nthreads=0):
    """x: bf16 bits [T, C]; w: [C] float32 or None; scale, shift: bf16 bits [N, C];
    idx: int32 [T] or None (all rows use index 0).  Returns bf16 bits [T, C]:
    the fp64 definition, each bf16 boundary a single rounding of the exact value."""
    T, C, N, x, w, scale, shift, idx = _mod_args(x, w, scale, shift, idx)
    y = np.empty((T, C), dtype=np.uint16)
    _load().oracle_rmsnorm_modulate_f64(_p(x), _p(y), T, C, _p(w), _p(scale), _p(shift), _p(idx), N,
                                        float(eps), nthreads)
    return y


def rmsnorm_modulate_emulate(x, w, scale, shift, idx, eps, nthreads=0):
    """Same arguments; the float32 fixed-order emulation (bit-exact contract)."""
    T, C, N, x, w, scale, shift, idx = _mod_args(x, w, scale, shift, idx)
    y = np.empty((T, C), dtype=np.uint16)
    _load().oracle_rmsnorm_modulate_emulate_bf16(_p(x), _p(y), T, C, _p(w), _p(scale), _p(shift), _p(idx), N,
                                                 float(np.float32(eps)), nthreads)
    return y


def attention_window_f64(q, k, v, scale, frame_tokens, anchor_frames, chunk_frames, radius, kv_len=None,
                         q_len=None, row_ids=None, nthreads=0):
    """Self-attention rows in fp64 under the chunked window (q, k, v as attention_f64, Sq == Sk)."""
    B, S, Hq, D = q.shape
    assert k.shape[:2] == (B, S) and v.shape == k.shape and Hq % k.shape[2] == 0
    assert frame_tokens > 0 and chunk_frames > 0 and anchor_frames >= 0 and radius >= 0
    kv_len = None if kv_len is None else np.ascontiguousarray(kv_len, dtype=np.int32)
    q_len = None if q_len is None else np.ascontiguousarray(q_len, dtype=np.int32)
    if row_ids is None:
        out = np.empty((B, S, Hq, D), dtype=np.float64)
        n, rid = B * S * Hq, None
    else:
        rid = np.ascontiguousarray(row_ids, dtype=np.int64)
        n = rid.size
        out = np.empty((n, D), dtype=np.float64)
    _load().oracle_attention_window_f64(_p(q), _p(k), _p(v), B, S, Hq, k.shape[2], D, float(scale), frame_tokens,
                                        anchor_frames, chunk_frames, radius, _p(kv_len), _p(q_len), _p(rid), n,
                                        _p(out), nthreads)
    return out


def window_allowed_pairs(S, L, frame_tokens, anchor_frames, chunk_frames, radius) -> int:
    """Allowed (query row, key) pairs of one sample under the window and key padding L."""
    return int(_load().oracle_window_allowed_pairs(S, L, frame_tokens, anchor_frames, chunk_frames, radius))
