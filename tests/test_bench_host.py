"""Host-side logic of bench.py (no GPU): algorithmic work counts."""
import numpy as np

import bench
import h3inputs as gen
import oracle


def test_allowed_pairs_matches_oracle_count():
    for name in ("padded_gqa", "padded_gqa_d64", "long_video_h12", "packed_clip_self", "packed_clip_cross"):
        wl = gen.WORKLOADS[name]
        kv = None if wl.kv_len_range is None else gen.uniform_int(wl.B, 0, gen.STREAM_KVLEN, *wl.kv_len_range)
        cb = None if wl.causal_pattern is None else np.array(wl.causal_pattern, np.uint8)
        assert bench._allowed_pairs(wl, kv, cb) == oracle.allowed_pairs(wl.B, wl.Sq, wl.Sk, False, kv, None, cb)


def test_nominal_flops_of_headline_shape():
    flops, norm_bytes = bench._workload_numbers(gen.WORKLOADS["long_video_h24"])
    assert flops == 4.0 * 32760 * 32760 * 24 * 128
    assert norm_bytes == 2.0 * (32760 * 48) * 128 * 2 + 2.0 * 32760 * 48 * 4 + 2.0 * 128 * 4


def test_clock_summary_keeps_only_the_timed_window():
    c = bench.ClockSampler(0)
    t0 = c._epoch("2026/12/02 10:00:01.000")
    c.window(t0, t0 + 1.0)

    def row(stamp, mhz, capped):
        return [stamp, "0", str(mhz), "2070", "900.5", "0x0", "Not Active", "Not Active", "Not Active",
                "Active" if capped else "Not Active"]
    rows = [row("2026/12/02 10:00:00.500", 2070, False),      # before the window: idle
            row("2026/12/02 10:00:01.100", 1800, True),
            row("2026/12/02 10:00:01.600", 1700, True),
            row("2026/12/02 10:00:01.900", 1750, False),
            row("2026/12/02 10:00:02.500", 2070, False)]      # after the window
    rec = c.summarise(rows)
    assert rec["samples"] == 3 and rec["sm_mhz"] == 1750 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == ["sw_power_cap"] and rec["window"] == "timed region"


def test_window_pairs_match_oracle_count():
    for S, L, geo in ((104448, 104448, (1536, 1, 5, 1)), (2000, 1500, (100, 1, 5, 1)), (777, 777, (7, 0, 3, 2)),
                      (500, 500, (10, 60, 2, 1))):
        assert bench._window_pairs(S, L, *geo) == oracle.window_allowed_pairs(S, L, *geo)


def test_modulate_shape_label_follows_the_launcher_rule():
    import bench
    # C 3072 with a weight: 14 compute warps x 2 CTAs with the weight staged
    # (28 >= 3/4 of the 32 warps without it); without a weight, 16 x 2
    assert bench._mod_shape(3072, True) == (14, True)
    assert bench._mod_shape(3072, False) == (16, False)
    # C 6144: staging would leave 8 of 16 warps, so the weight is read through L1
    assert bench._mod_shape(6144, True) == (16, False)
    assert bench._mod_shape(8192, True) == (8, True)
