"""Planted mistakes in the oracle, on the CPU.

Each case copies oracle.c, plants one plausible mistake in the copy (a wrong
sign, a dropped term, a wrong or transposed index, a skipped or wrong
rounding, a reordered float32 reduction), builds it with the oracle's own
flags and runs the pins of that part of the oracle against it: at least one
pin must fail.  The unmodified source built the same way passes every pin
(the control), so a failure is the planted mistake's doing.  The oracle
itself is never modified: only the copy is.
"""
import itertools
import os

import pytest

import oracle
import test_golden as golden
import test_oracle_adaln as adaln
import test_oracle_attention as attention
import test_oracle_norm_rope as norm_rope
import test_oracle_rounding as rounding
import test_oracle_window as window

ALL = (norm_rope, attention, adaln, window, rounding, golden)


def _pins(*modules):
    """(name, function, kwargs) for every test of the modules, parametrize
    cases expanded."""
    out = []
    for m in modules:
        for name in sorted(n for n in dir(m) if n.startswith("test_")):
            fn = getattr(m, name)
            marks = [mk for mk in getattr(fn, "pytestmark", []) if mk.name == "parametrize"]
            axes = []
            for mk in marks:
                argnames, argvalues = mk.args[0], mk.args[1]
                if isinstance(argnames, str):
                    argnames = [a.strip() for a in argnames.split(",")]
                cases = []
                for v in argvalues:
                    if hasattr(v, "values") and hasattr(v, "marks"):  # pytest.param
                        v = v.values if len(argnames) > 1 else v.values[0]
                    cases.append(dict(zip(argnames, v)) if len(argnames) > 1 else {argnames[0]: v})
                axes.append(cases)
            for combo in itertools.product(*axes):
                kw = {}
                for c in combo:
                    kw.update(c)
                out.append((f"{m.__name__}.{name}", fn, kw))
    return out


def _first_failing_pin(modules):
    for name, fn, kw in _pins(*modules):
        try:
            fn(**kw)
        except Exception as e:  # an assertion, or an error the mistake provokes
            return f"{name}({kw}): {type(e).__name__}"
    return None


with open(oracle._SRC) as _f:
    SOURCE = _f.read()

# (id, text in oracle.c, the mistake, the pin modules of that part)
MISTAKES = [
    # fp64 RMSNorm -> bf16 boundary -> rotate-half RoPE
    ("rope_sign", "      yr[i] = a * cs - b * sn;", "      yr[i] = a * cs + b * sn;", (norm_rope, golden)),
    ("rope_interleaved_pairs", "      double a = n[i], b = n[i + half];",
     "      double a = n[2 * i], b = n[2 * i + 1];", (norm_rope, golden)),
    ("rope_cos_sin_swapped", "      double cs = (double)c->cos_t[pos * half + i];\n      double sn = (double)c->sin_t[pos * half + i];",
     "      double cs = (double)c->sin_t[pos * half + i];\n      double sn = (double)c->cos_t[pos * half + i];",
     (norm_rope, golden)),
    ("rope_position_from_flat_row", "    int64_t pos = (r / c->H) % c->S; /* row r", "    int64_t pos = r % c->S; /* row r",
     (norm_rope, golden)),
    ("rms_eps_dropped", "    double rinv = 1.0 / sqrt(ms + c->eps);", "    double rinv = 1.0 / sqrt(ms);",
     (norm_rope, golden)),
    ("rms_mean_over_d_minus_1", "    double ms = ss / (double)D;", "    double ms = ss / (double)(D - 1);",
     (norm_rope, golden)),
    ("norm_weight_dropped", "      double v = bf16_to_f64(xr[d]) * rinv * (double)c->w[d];",
     "      double v = bf16_to_f64(xr[d]) * rinv;", (norm_rope, golden)),
    ("bf16_boundary_skipped", "      n[d] = c->round_boundary ? round_f64_to_bf16(v) : v;", "      n[d] = v;",
     (norm_rope, golden)),
    ("pass_through_weighted_twice", "    for (int d = 2 * half; d < D; ++d) yr[d] = n[d];",
     "    for (int d = 2 * half; d < D; ++d) yr[d] = n[d] * (double)c->w[d];", (norm_rope, golden)),
    # fp64 -> bf16 rounding
    ("round_ties_away", "  double r = ldexp(nearbyint(ldexp(ax, -q_exp)), q_exp);",
     "  double r = ldexp(round(ldexp(ax, -q_exp)), q_exp);", (rounding, golden)),
    ("round_9_bit_significand", "  int q_exp = e - 8;", "  int q_exp = e - 9;", (rounding, golden)),
    ("round_no_subnormal_clamp", "  if (q_exp < -133) q_exp = -133;", "", (rounding, golden)),
    ("f32_to_bf16_ties_away", "  u += 0x7FFFu + ((u >> 16) & 1u);", "  u += 0x8000u;", ALL),
    # fp64 attention
    ("scale_dropped", "      s[n] = c->scale * dot;", "      s[n] = dot;", (attention, golden)),
    ("softmax_not_normalised", "      double pw = s[t] / denom;", "      double pw = s[t];", (attention, golden)),
    ("gqa_head_modulo", "    int kvh = h / g;", "    int kvh = h % c->Hkv;", (attention, golden)),
    ("scores_from_v", "      const uint16_t* kr = c->k + (((int64_t)b * c->Sk + j) * c->Hkv + kvh) * D;",
     "      const uint16_t* kr = c->v + (((int64_t)b * c->Sk + j) * c->Hkv + kvh) * D;", (attention, golden)),
    ("value_row_by_rank", "      const uint16_t* vr = c->v + (((int64_t)b * c->Sk + idx[t]) * c->Hkv + kvh) * D;",
     "      const uint16_t* vr = c->v + (((int64_t)b * c->Sk + t) * c->Hkv + kvh) * D;", (attention, golden)),
    ("causal_excludes_diagonal", "  if (causal && j > i) return 0;", "  if (causal && j >= i) return 0;",
     (attention, golden)),
    ("kv_len_off_by_one", "  if (c->kv_len && j >= (int64_t)c->kv_len[b]) return 0;",
     "  if (c->kv_len && j > (int64_t)c->kv_len[b]) return 0;", (attention, golden)),
    ("bits_msb_first", "    if (!((word >> (j & 31)) & 1u)) return 0;",
     "    if (!((word >> (31 - (j & 31))) & 1u)) return 0;", (attention, golden)),
    ("q_len_tail_not_zeroed", "    if (c->q_len && i >= (int64_t)c->q_len[b]) continue; /* zero tail */", "",
     (attention, golden)),
    ("pair_count_causal_off_by_one", "      if (cz && i + 1 < lim) lim = i + 1;", "      if (cz && i < lim) lim = i;",
     (attention,)),
    # chunked window
    ("window_anchor_keys_not_dense", "  if (ct <= 0 || i < af || j < af) return 1;", "  if (ct <= 0 || i < af) return 1;",
     (window,)),
    ("window_one_sided", "  return d <= r && d >= -r;", "  return d <= r && d >= 0;", (window,)),
    ("window_pairs_low_edge", "    int64_t lo = af + (ci - radius) * ct, hi",
     "    int64_t lo = af + (ci - radius + 1) * ct, hi", (window,)),
    # fp64 RMSNorm -> AdaLN modulation
    ("adaln_one_plus_scale_dropped", "      double a = round_f64_to_bf16(1.0 + bf16_to_f64(sc[ch]));",
     "      double a = round_f64_to_bf16(bf16_to_f64(sc[ch]));", (adaln, golden)),
    ("adaln_scale_shift_swapped",
     "    const uint16_t* sc = c->scale + (int64_t)ix * C;\n    const uint16_t* sh = c->shift + (int64_t)ix * C;\n    for (int ch = 0; ch < C; ++ch) {\n      double",
     "    const uint16_t* sc = c->shift + (int64_t)ix * C;\n    const uint16_t* sh = c->scale + (int64_t)ix * C;\n    for (int ch = 0; ch < C; ++ch) {\n      double",
     (adaln, golden)),
    ("adaln_index_ignored",
     "    int32_t ix = c->idx ? c->idx[t] : 0;\n    if (ix < 0 || ix >= c->N) {\n      for (int ch = 0; ch < C; ++ch) yr[ch] = 0;\n      continue;\n    }\n    double ss",
     "    int32_t ix = 0;\n    if (ix < 0 || ix >= c->N) {\n      for (int ch = 0; ch < C; ++ch) yr[ch] = 0;\n      continue;\n    }\n    double ss",
     (adaln, golden)),
    ("adaln_product_boundary_skipped", "      double m = round_f64_to_bf16(n * a);", "      double m = n * a;",
     (adaln, golden)),
    ("adaln_eps_outside_sqrt", "    double rinv = 1.0 / sqrt(ss / (double)C + c->eps);",
     "    double rinv = 1.0 / (sqrt(ss / (double)C) + c->eps);", (adaln, golden)),
    # float32 fixed-order contracts
    ("emulation_rope_sign", "      y[i] = fmaf(a, cs, -bs);", "      y[i] = fmaf(a, cs, bs);", (norm_rope, golden)),
    ("emulation_adaln_one_plus_dropped", "      float a = bf16_to_f32(f32_to_bf16_rne(1.0f + bf16_to_f32(sc[ch])));",
     "      float a = bf16_to_f32(f32_to_bf16_rne(bf16_to_f32(sc[ch])));", (adaln, golden)),
]

# Not in the list, because no CPU pin can see them, by construction:
# * changes of the float32 contracts' operation order alone (the butterfly
#   order, the weight multiplied before 1/rms, lanes taking contiguous
#   groups): both orders stay within the rounding bound of the fp64
#   definition, which is all the pages fix; the order is the kernels'
#   contract, and the GPU tests, bit-exact against the emulation, pin it;
# * dropping the overflow branch of the fp64 -> bf16 rounding: the exported
#   bits come through a float conversion that gives infinity either way.


def test_control_unmodified_source_passes_every_pin(tmp_path):
    with oracle.built_from(SOURCE, str(tmp_path)):
        failing = _first_failing_pin(ALL)
    assert failing is None, failing


@pytest.mark.parametrize("mid,old,new,modules", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_planted_mistake_fails_a_pin(tmp_path, mid, old, new, modules):
    assert SOURCE.count(old) == 1, f"{mid}: the text to change must occur once in oracle.c"
    with oracle.built_from(SOURCE.replace(old, new), str(tmp_path)):
        failing = _first_failing_pin(modules)
    assert failing is not None, f"{mid}: no pin fails with this mistake planted"
