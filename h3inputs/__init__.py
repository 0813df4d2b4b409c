"""Seeded synthetic inputs for the H3 attention step.

Shared by the CUDA path's tests/bench and by the CPU oracle's tests.  It draws
numbers and lays them out; it holds none of the method's arithmetic (no norm,
no rotation, no softmax).  The C source (``gen.c``) is compiled on first use
with the host C compiler into ``libh3inputs.so`` next to this file.

Workloads follow the shapes the pages' workloads describe: the MiniMax-H3 /
Wan video-DiT attention (FastVideo PR #1832 "Add FlashInfer attention backend
support for MiniMax H3", section "Summary": BSHD tensors, head_dim 128, dense
non-causal self-attention; section "Performance considerations": one long
packed sequence with attention batch one) and the mask/GQA/cross-attention
variants of FastVideo PR #1799 ("Add opt-in FlashInfer attention backend for
Wan", section "Implementation").
"""
from __future__ import annotations

import ctypes
import dataclasses
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libh3inputs.so")
_lock = threading.Lock()
_lib = None

# Stream ids: each tensor of a workload draws from its own stream.
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_WQ, STREAM_WK = 4, 5
STREAM_KVLEN, STREAM_BITS = 6, 7
STREAM_TEXT_K, STREAM_TEXT_V = 8, 9
STREAM_HIDDEN, STREAM_NORM_W, STREAM_SCALE, STREAM_SHIFT = 10, 11, 12, 13


def _src_hash() -> str:
    with open(_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def build(force: bool = False) -> str:
    """Compile gen.c into libh3inputs.so (skipped when the source is unchanged)."""
    stamp = _LIB + ".stamp"
    h = _src_hash()
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == h:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(stamp, "w") as f:
        f.write(h)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, U64, I, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_double
            lib.h3in_fill_bshd.argtypes = [P, I64, I64, I, I, U64, U64, D, D, I]
            lib.h3in_uniform_f32.argtypes = [P, I64, U64, U64, D, D]
            lib.h3in_uniform_int.argtypes = [P, I64, U64, U64, I64, I64]
            lib.h3in_bernoulli_bits.argtypes = [P, I64, I, U64, U64, D]
            lib.h3in_rope_tables.argtypes = [P, P, I64, I, D]
            for fn in ("h3in_fill_bshd", "h3in_uniform_f32", "h3in_uniform_int",
                       "h3in_bernoulli_bits", "h3in_rope_tables"):
                getattr(lib, fn).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def normal_bshd(B, S, H, D, seed, stream, std=1.0, offset_std=0.0, nthreads=0) -> np.ndarray:
    """bf16 bits (uint16) of shape [B, S, H, D]: std*N(0,1) (+ offset_std*N(0,1) per head/channel)."""
    out = np.empty((B, S, H, D), dtype=np.uint16)
    _load().h3in_fill_bshd(_ptr(out), B, S, H, D, seed, stream, std, offset_std, nthreads)
    return out


def uniform_f32(n, seed, stream, lo, hi) -> np.ndarray:
    out = np.empty((n,), dtype=np.float32)
    _load().h3in_uniform_f32(_ptr(out), n, seed, stream, lo, hi)
    return out


def uniform_int(n, seed, stream, lo, hi) -> np.ndarray:
    """int32 draws in the closed range [lo, hi]."""
    out = np.empty((n,), dtype=np.int32)
    _load().h3in_uniform_int(_ptr(out), n, seed, stream, lo, hi)
    return out


def bernoulli_bits(B, Sq, Sk, seed, stream, p) -> np.ndarray:
    """Packed boolean mask uint32 [B, Sq, ceil(Sk/32)], bit (j&31) of word j>>5; 1 = attend."""
    W = (Sk + 31) // 32
    out = np.empty((B, Sq, W), dtype=np.uint32)
    _load().h3in_bernoulli_bits(_ptr(out), B * Sq, Sk, seed, stream, p)
    return out


def rope_tables(S, rotary_dim, theta=10000.0):
    """(cos, sin) float32 tables [S, rotary_dim/2]; angle = pos * theta^(-2i/rotary_dim)."""
    half = rotary_dim // 2
    c = np.empty((S, half), dtype=np.float32)
    s = np.empty((S, half), dtype=np.float32)
    _load().h3in_rope_tables(_ptr(c), _ptr(s), S, rotary_dim, theta)
    return c, s


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bits to float32 (a layout operation, no rounding)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload of the attention step.

    kv_len_range: per-sample valid key count drawn from U{lo..hi}, or a fixed
    value (lo == hi), or None (all keys valid).  causal_pattern: per-sample
    causal flags, or None.  norm_rope: whether the fused Q/K norm + RoPE runs
    on this workload's q and k before attention.
    """
    name: str
    B: int
    Sq: int
    Sk: int
    Hq: int
    Hkv: int
    D: int
    offset_std: float = 0.0
    kv_len_range: tuple | None = None
    causal_pattern: tuple | None = None
    norm_rope: bool = True
    rotary_dim: int = 96
    eps: float = 1e-6
    theta: float = 10000.0
    cross: bool = False  # K/V are separate raw text tensors (no norm/RoPE on k)

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


# The five workloads (plus sub-cases) of the build's scope.
WORKLOADS = {
    # Tiny multi-head attention.
    "tiny_mha": Workload("tiny_mha", 1, 256, 256, 4, 4, 128),
    # One video-DiT block: S=4096 tokens, 24 heads.
    "dit_block": Workload("dit_block", 1, 4096, 4096, 24, 24, 128),
    # Long video self-attention, 12 heads, peaky softmax from per-head offsets.
    "long_video_h12": Workload("long_video_h12", 1, 32760, 32760, 12, 12, 128, offset_std=0.5),
    # Same length with 24 heads: the shape the headline throughput is quoted on.
    "long_video_h24": Workload("long_video_h24", 1, 32760, 32760, 24, 24, 128, offset_std=0.5),
    # Padded GQA batch: per-sample key padding, causal on samples 0 and 2.
    "padded_gqa": Workload("padded_gqa", 4, 8192, 8192, 16, 4, 128,
                           kv_len_range=(4096, 8192), causal_pattern=(1, 0, 1, 0)),
    "padded_gqa_d64": Workload("padded_gqa_d64", 4, 2048, 2048, 16, 4, 64,
                               kv_len_range=(1024, 2048), causal_pattern=(1, 0, 1, 0), norm_rope=False),
    "padded_gqa_d256": Workload("padded_gqa_d256", 4, 2048, 2048, 16, 4, 256,
                                kv_len_range=(1024, 2048), causal_pattern=(1, 0, 1, 0), norm_rope=False),
    # Packed long clip: 104448 rows, the first 100000 keys valid.
    "packed_clip_self": Workload("packed_clip_self", 1, 104448, 104448, 24, 24, 128,
                                 kv_len_range=(100000, 100000)),
    # Text cross-attention of the packed clip against 512 text keys.
    "packed_clip_cross": Workload("packed_clip_cross", 1, 104448, 512, 24, 24, 128, cross=True),
}


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: np.ndarray            # bf16 bits [B, Sq, Hq, D]
    k: np.ndarray            # bf16 bits [B, Sk, Hkv, D]
    v: np.ndarray            # bf16 bits [B, Sk, Hkv, D]
    wq: np.ndarray | None    # float32 [D]
    wk: np.ndarray | None
    cos: np.ndarray | None   # float32 [max(Sq,Sk), rotary_dim/2]
    sin: np.ndarray | None
    kv_len: np.ndarray | None    # int32 [B]
    causal_b: np.ndarray | None  # uint8 [B]


def make_inputs(wl: Workload, seed: int, nthreads: int = 0) -> Inputs:
    """Draw every input of a workload from (seed, per-tensor stream)."""
    q = normal_bshd(wl.B, wl.Sq, wl.Hq, wl.D, seed, STREAM_Q, 1.0, wl.offset_std, nthreads)
    if wl.cross:
        k = normal_bshd(wl.B, wl.Sk, wl.Hkv, wl.D, seed, STREAM_TEXT_K, 1.0, 0.0, nthreads)
        v = normal_bshd(wl.B, wl.Sk, wl.Hkv, wl.D, seed, STREAM_TEXT_V, 1.0, 0.0, nthreads)
    else:
        k = normal_bshd(wl.B, wl.Sk, wl.Hkv, wl.D, seed, STREAM_K, 1.0, wl.offset_std, nthreads)
        v = normal_bshd(wl.B, wl.Sk, wl.Hkv, wl.D, seed, STREAM_V, 1.0, 0.0, nthreads)
    wq = wk = cos = sin = None
    if wl.norm_rope:
        wq = uniform_f32(wl.D, seed, STREAM_WQ, 0.5, 1.5)
        wk = uniform_f32(wl.D, seed, STREAM_WK, 0.5, 1.5)
        cos, sin = rope_tables(max(wl.Sq, wl.Sk), wl.rotary_dim, wl.theta)
    kv_len = causal_b = None
    if wl.kv_len_range is not None:
        lo, hi = wl.kv_len_range
        kv_len = uniform_int(wl.B, seed, STREAM_KVLEN, lo, hi)
    if wl.causal_pattern is not None:
        causal_b = np.array(wl.causal_pattern, dtype=np.uint8)
    return Inputs(wl, q, k, v, wq, wk, cos, sin, kv_len, causal_b)


# RMSNorm -> indexed AdaLN modulation of DiT hidden rows (TeleFuser PR #37
# section 2.5).  The pages give no shapes for it; the workload takes the
# hidden rows of the long-video clip (T = 32760 tokens) at the hidden size
# of its attention (C = 24 heads x 128 = 3072), one modulation row per latent
# frame (21 frames of 1560 tokens; the index of a token is its frame).
@dataclasses.dataclass(frozen=True)
class ModWorkload:
    name: str
    T: int
    C: int
    frames: int
    eps: float = 1e-6


MOD_WORKLOADS = {
    "dit_hidden_adaln": ModWorkload("dit_hidden_adaln", 32760, 3072, 21),
}


@dataclasses.dataclass
class ModInputs:
    x: np.ndarray      # bf16 bits [T, C]
    w: np.ndarray      # float32 [C]
    scale: np.ndarray  # bf16 bits [N, C]
    shift: np.ndarray  # bf16 bits [N, C]
    idx: np.ndarray    # int32 [T]


def make_modulate_inputs(T, C, N, seed, nthreads: int = 0) -> ModInputs:
    """Hidden rows N(0,1), weight U(0.5,1.5), modulation tables N(0, 0.3^2),
    token t in table row t * N // T (contiguous runs, like frames)."""
    x = normal_bshd(1, T, 1, C, seed, STREAM_HIDDEN, 1.0, 0.0, nthreads)[0, :, 0]
    w = uniform_f32(C, seed, STREAM_NORM_W, 0.5, 1.5)
    scale = normal_bshd(1, N, 1, C, seed, STREAM_SCALE, 0.3)[0, :, 0]
    shift = normal_bshd(1, N, 1, C, seed, STREAM_SHIFT, 0.3)[0, :, 0]
    idx = (np.arange(T, dtype=np.int64) * N // max(T, 1)).astype(np.int32)
    return ModInputs(np.ascontiguousarray(x), w, np.ascontiguousarray(scale), np.ascontiguousarray(shift), idx)


# Chunked-window self-attention (SGLang PR #37903, hybrid_window_attn_h3:
# chunk-5 / radius-1 window with anchor frames).  The page gives the clip
# (~104k packed rows) but not its frame geometry; the workload reads the
# packed clip's 104448 rows as 68 frames of 1536 tokens, one anchor frame,
# chunks of 5 frames, radius 1, 24 heads of 128.
@dataclasses.dataclass(frozen=True)
class WindowWorkload:
    name: str
    B: int
    S: int
    H: int
    D: int
    frame_tokens: int
    anchor_frames: int
    chunk_frames: int
    radius: int


WINDOW_WORKLOADS = {
    "packed_clip_window": WindowWorkload("packed_clip_window", 1, 104448, 24, 128, 1536, 1, 5, 1),
}
