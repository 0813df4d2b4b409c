"""The oracle against hand-worked examples of the definitions (tests/golden)."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
G = json.load(open(os.path.join(HERE, "golden", "hand_examples.json")))


def _bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_attention_hand_examples():
    for case in G["attention"]:
        q = _bits(case["q"])[None, :, None, :]
        k = _bits(case["k"])[None, :, None, :]
        v = _bits(case["v"])[None, :, None, :]
        o = oracle.attention_f64(q.copy(), k.copy(), v.copy(), case["scale"], case.get("causal", False))
        got = o[0, case.get("row", 0), 0]
        np.testing.assert_allclose(got, case["o"], rtol=1e-14, err_msg=case["name"])


def test_norm_rope_hand_example():
    for case in G["norm_rope"]:
        x = _bits(case["x"])[None, None, None, :]
        half = case["rotary_dim"] // 2
        y = oracle.qk_norm_rope_f64(x.copy(), np.array(case["w"], np.float32),
                                    np.array(case["cos"], np.float32).reshape(1, half),
                                    np.array(case["sin"], np.float32).reshape(1, half),
                                    case["rotary_dim"], case["eps"], round_boundary=False)
        np.testing.assert_allclose(y[0, 0, 0], case["y"], rtol=1e-14, err_msg=case["name"])


def test_rmsnorm_modulate_hand_example():
    for case in G["rmsnorm_modulate"]:
        C = len(case["x"])
        x = _bits(case["x"])[None, :]
        sc = np.full((1, C), _bits([case["scale"]])[0], np.uint16)
        sh = np.full((1, C), _bits([case["shift"]])[0], np.uint16)
        for fn in (oracle.rmsnorm_modulate_f64, oracle.rmsnorm_modulate_emulate):
            y = fn(x.copy(), None, sc, sh, None, case["eps"])
            got = (y.astype(np.uint32) << 16).view(np.float32)[0]
            np.testing.assert_array_equal(got, np.array(case["y"], np.float32), err_msg=f"{case['name']} {fn.__name__}")
