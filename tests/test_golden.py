"""Oracle against hand-derived worked examples stored in tests/golden/ (each
fixture states its derivation and citation). No GPU needed."""
import json
import math
import os
from fractions import Fraction

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _fr(xs):
    return np.array([float(Fraction(x)) for x in xs])


def test_causal_powers_of_two():
    with open(os.path.join(GOLDEN, "causal_powers_of_two.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    Q, K, V, dO = (np.array(inp[k], dtype=np.float64) for k in ("Q", "K", "V", "dO"))
    ln2 = math.log(2.0)
    r = oracle.attn_bwd(Q, K, V, dO, inp["causal"], ln2)
    e = g["expected_rational"]
    np.testing.assert_allclose(r["O"][:, 0], _fr(e["O"]), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(np.exp(r["LSE"]), _fr(e["LSE_exp"]), rtol=1e-14)
    np.testing.assert_allclose(r["dQ"][:, 0], ln2 * _fr(e["dQ_over_ln2"]), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["dK"][:, 0], ln2 * _fr(e["dK_over_ln2"]), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(r["dV"][:, 0], _fr(e["dV"]), rtol=1e-14, atol=1e-14)


def test_cross_attention_powers_of_two():
    with open(os.path.join(GOLDEN, "cross_attention_powers_of_two.json")) as f:
        g = json.load(f)
    ln2 = math.log(2.0)
    for case in g["cases"]:
        inp = case["inputs"]
        Q, K, V, dO = (np.array(inp[k], dtype=np.float64) for k in ("Q", "K", "V", "dO"))
        r = oracle.attn_bwd_ex(Q, K, V, dO, inp["mask"], ln2)
        e = case["expected_rational"]
        name = case["name"]
        np.testing.assert_allclose(r["O"][:, 0], _fr(e["O"]), rtol=1e-14, atol=1e-14, err_msg=name)
        np.testing.assert_allclose(np.exp(r["LSE"]), _fr(e["LSE_exp"]), rtol=1e-14, err_msg=name)
        np.testing.assert_allclose(r["dQ"][:, 0], ln2 * _fr(e["dQ_over_ln2"]), rtol=1e-13,
                                   atol=1e-14, err_msg=name)
        np.testing.assert_allclose(r["dK"][:, 0], ln2 * _fr(e["dK_over_ln2"]), rtol=1e-13,
                                   atol=1e-14, err_msg=name)
        np.testing.assert_allclose(r["dV"][:, 0], _fr(e["dV"]), rtol=1e-14, atol=1e-14,
                                   err_msg=name)
