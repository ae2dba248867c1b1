"""Golden fixtures: a hand-derived closed-form case and an oracle regression set."""
import json
import math
import os

import numpy as np
import torch

import oracle
from hybrid_sliding_window_02_b300 import inputs as gen

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def test_hand_derived_three_tokens():
    g = _load("hand_derived_t3.json")
    T, D = g["T"], g["D"]
    q = torch.tensor(g["q"], dtype=torch.float64).reshape(1, T, 1, D)
    k = torch.tensor(g["k"], dtype=torch.float64).reshape(1, T, 1, D)
    v = torch.tensor(g["v"], dtype=torch.float64).reshape(1, T, 1, D)
    o, l = oracle.swa_sink_fwd(q, k, v, torch.tensor(g["sink"], dtype=torch.float64), g["W"])
    env = {"e": math.e, "log": math.log}
    want_o = np.array([[eval(s, {}, env) for s in row] for row in g["out_expr"]])
    want_l = np.array([eval(s, {}, env) for s in g["lse_expr"]])
    np.testing.assert_allclose(o[0, :, 0, :], want_o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l[0, 0], want_l, rtol=0, atol=1e-15)


def test_oracle_tiny_regression():
    g = _load("oracle_tiny_rows.json")
    x = gen.prefill_inputs(1, 512, 4, 1, 64, seed=0, dtype=torch.float32)
    o, l = oracle.swa_sink_fwd_rows(x.q, x.k, x.v, x.sink, 128, g["rows"])
    np.testing.assert_allclose(o[:, :8], np.array(g["out_first8"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(o.sum(axis=1), np.array(g["out_sum"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, np.array(g["lse"]), rtol=0, atol=1e-13)


def test_rope_hand_derived_angles_and_pairs():
    """RoPE frequency schedule and pair layout, pinned by hand-derived values:
    the angle of pair i is p * theta^(-2i/rot_dim), the pairs are (i, i+rot_dim/2),
    and token t of sequence b sits at position pos0[b] + t."""
    g = _load("rope_hand_derived.json")
    env = {"cos": math.cos, "sin": math.sin}
    for case in g["cases"]:
        x = torch.tensor(case["x"], dtype=torch.float64)
        pos0 = torch.tensor(case["pos0"], dtype=torch.int64)
        y = oracle.rope(x, pos0, case["rot_dim"], case["theta"])
        want = np.vectorize(lambda s: float(eval(s, {}, env)))(np.array(case["y_expr"]))
        assert y.shape == want.shape, case["name"]
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-12, err_msg=case["name"])
