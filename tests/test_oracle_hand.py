"""The oracle against a four-token example derived by hand.

The fixture holds the inputs, the derivation and the expected values as
closed-form expressions (see tests/golden/hand_example.json).
"""

import json
import math
import os

import numpy as np

import oracle

_FIX = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def _ev(x):
    return float(eval(str(x), {"__builtins__": {}}, {"e": math.e, "sqrt": math.sqrt}))


def test_hand_example():
    fx = json.load(open(_FIX))
    i = fx["inputs"]
    arr = lambda x: np.array(x, np.float32)[None, None]
    q, k, v = arr(i["q"]), arr(i["k"]), arr(i["v"])
    g = np.full((1, 1, 4), np.float32(math.log(0.5)))
    beta = arr(i["beta"])[0]
    w_s = np.array(i["w_s"], np.float32)[None]
    b_s = np.array(i["b_s"], np.float32)[None]
    w_g = np.array([[math.log(3.0), 0.0]], np.float32)
    b_g = np.zeros(1, np.float32)
    r = oracle.forward(q, k, v, g, beta, w_s, b_s, w_g, b_g, chunk=i["chunk"], scale=i["scale"],
                       eps=i["eps"])
    ex = fx["expected"]
    assert r["sel"][0].tolist() == ex["sel"]
    np.testing.assert_allclose(r["scores"][0], np.vectorize(_ev)(np.array(ex["scores"])), atol=1e-7)
    # a = exp(float32(ln 1/2)) differs from 1/2 by ~1e-8; ln 3 is rounded to float32 too
    for key, tol in (("o_s", 1e-13), ("o_l", 1e-7), ("state", 1e-7), ("out", 1e-6)):
        want = np.vectorize(_ev)(np.array(ex[key], dtype=object)).astype(np.float64)
        np.testing.assert_allclose(r[key][0], want, rtol=tol, atol=tol, err_msg=key)
