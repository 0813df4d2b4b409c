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
