"""Shared test helpers: host <-> device conversion, comparisons, row sampling."""
import numpy as np

# Tolerance for bf16 attention outputs against the fp64 oracle: max |err|
# 2e-2 and relative RMS error 5e-3 (the bound the build is held to; the
# pages report block-level relative L2 errors of 5e-3 to 7e-3 for their
# attention path, SGLang PR #37903 "Accuracy Tests").
MAX_ABS = 2e-2
REL_RMS = 5e-3


def to_dev(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_f32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def to_dev_i32(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def to_dev_u8(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def from_dev(t) -> np.ndarray:
    """bf16 device tensor -> uint16 bits on the host."""
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits: np.ndarray) -> np.ndarray:
    return ((bits.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)


def check_close(got_bits: np.ndarray, ref: np.ndarray, what: str = ""):
    """got: bf16 bits, ref: fp64.  Asserts the max-abs and rel-RMS bounds."""
    got = bf16_f64(got_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - ref
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    denom = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 1.0
    rel_rms = float(np.sqrt(np.mean(err ** 2))) / max(denom, 1e-30) if err.size else 0.0
    assert max_abs <= MAX_ABS, f"{what}: max abs error {max_abs:.3e} > {MAX_ABS}"
    assert rel_rms <= REL_RMS, f"{what}: relative RMS error {rel_rms:.3e} > {REL_RMS}"
    return max_abs, rel_rms


def sample_rows(B, Sq, Hq, per_head, seed, kv_len=None, causal_b=None, extra_rows=()):
    """Flat output-row ids ((b*Sq + i)*Hq + h): first/last rows, tile edges,
    rows around kv_len boundaries and causal diagonals, plus random rows."""
    rng = np.random.default_rng(seed)
    ids = []
    for b in range(B):
        rows = {0, 1, 127, 128, 255, 256, Sq // 2, Sq - 2, Sq - 1}
        rows.update(extra_rows)
        if kv_len is not None:
            L = int(kv_len[b])
            rows.update({L - 129, L - 128, L - 1, L, L + 1})
        rows.update(rng.integers(0, Sq, size=per_head).tolist())
        rows = sorted(r for r in rows if 0 <= r < Sq)
        for h in range(Hq):
            for i in rows:
                ids.append((b * Sq + i) * Hq + h)
    return np.array(sorted(set(ids)), dtype=np.int64)


def assert_convex_bound(dv, do, group: int, what: str):
    """A property of every output element, at any size (checked on the
    device): an attention output row is a softmax-weighted average of value
    rows (or zero), so it is finite and |o[b,i,h,d]| <= max_j |v[b,j,h//group,d]|,
    up to the bf16 rounding of P and of o (a relative slack of 1 %)."""
    import torch
    o = do.float()
    assert bool(torch.isfinite(o).all()), f"{what}: non-finite outputs"
    vmax = dv.float().abs().amax(dim=1)                          # [B, Hkv, D]
    bound = vmax.repeat_interleave(group, dim=1)[:, None]        # [B, 1, Hq, D]
    over = o.abs() > bound * 1.01 + 1e-6
    assert not bool(over.any()), f"{what}: {int(over.sum())} outputs exceed the value range of their column"


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; 2^-133 at zero)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)
