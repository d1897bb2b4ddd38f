"""Pins for the oracle's scalar tape against the worked examples the pages
print (microcrad page, NumPy framework page) and textbook derivatives."""
import json
import math
import os

import pytest

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_product_example(oracle):
    g = _gold("scalar_tape.json")
    V = oracle.Value
    oracle.value_reset()
    a, b = V.leaf(g["a"]), V.leaf(g["b"])
    c = a * b
    assert c.backward() == 0
    assert c.data == g["c"]
    assert a.grad == g["dc_da"]
    assert b.grad == g["dc_db"]


def test_accumulation_over_shared_input(oracle):
    g = _gold("grad_accumulation.json")
    V = oracle.Value
    oracle.value_reset()
    x = V.leaf(0.7)
    y = x * V.leaf(g["coef_y"])
    z = x * V.leaf(g["coef_z"])
    L = y + z
    assert L.backward() == 0
    assert x.grad == g["dx"]


def test_graph_trace(oracle):
    g = _gold("graph_trace.json")
    V = oracle.Value
    oracle.value_reset()
    x1, x2, x3 = V.leaf(g["x1"]), V.leaf(g["x2"]), V.leaf(g["x3"])
    y = (x1 + x2) * x3
    assert y.backward() == 0
    assert y.data == g["y"]
    assert (x1.grad, x2.grad, x3.grad) == (g["dy_dx1"], g["dy_dx2"], g["dy_dx3"])


def test_diamond_and_reuse(oracle):
    """x used along several paths and twice in one op: d(x*x + x)/dx = 2x + 1."""
    V = oracle.Value
    oracle.value_reset()
    x = V.leaf(3.0)
    y = x * x + x
    assert y.backward() == 0
    assert x.grad == 7.0


def test_unary_ops_textbook_derivatives(oracle):
    V = oracle.Value
    oracle.value_reset()
    x = V.leaf(1.3)
    f = x.pow(3.0)
    assert f.backward() == 0
    assert math.isclose(x.grad, 3 * 1.3 ** 2, rel_tol=1e-15)
    oracle.value_reset()
    x = V.leaf(0.4)
    f = x.exp()
    f.backward()
    assert math.isclose(x.grad, math.exp(0.4), rel_tol=1e-15)
    oracle.value_reset()
    x = V.leaf(2.5)
    f = x.log()
    f.backward()
    assert math.isclose(x.grad, 1 / 2.5, rel_tol=1e-15)
    # softmax-CE over two logits built from scalars: d/dz0 = p0 - 1
    oracle.value_reset()
    z0, z1 = V.leaf(0.3), V.leaf(-1.1)
    s = z0.exp() + z1.exp()
    loss = s.log() + (z0 * V.leaf(-1.0))
    loss.backward()
    p0 = math.exp(0.3) / (math.exp(0.3) + math.exp(-1.1))
    assert math.isclose(z0.grad, p0 - 1.0, rel_tol=1e-13)
    assert math.isclose(z1.grad, 1.0 - p0, rel_tol=1e-13)


def test_bad_root_returns_minus_one(oracle):
    oracle.value_reset()
    assert oracle.value_backward_raw(12345) == -1
    assert oracle.value_backward_raw(-1) == -1


def test_mlp_matches_finite_difference(oracle):
    """A 2-3-1 tanh-free MLP built from scalars (the page's small-net advice,
    NumPy framework page 4.2): tape gradients vs central differences."""
    fd = _gold("finite_difference.json")
    V = oracle.Value
    w = [0.3, -0.2, 0.5, 0.1, -0.4, 0.25, 0.6, -0.3, 0.2]

    def build(ws):
        oracle.value_reset()
        leaves = [V.leaf(v) for v in ws]
        x = [V.leaf(0.5), V.leaf(-1.5)]
        h = []
        for j in range(3):
            a = leaves[2 * j] * x[0] + leaves[2 * j + 1] * x[1]
            h.append(a.exp())
        out = h[0] * leaves[6] + h[1] * leaves[7] + h[2] * leaves[8]
        return leaves, out.pow(2.0)

    leaves, out = build(w)
    out.backward()
    grads = [l.grad for l in leaves]
    for i in range(len(w)):
        wp = list(w); wp[i] += fd["eps"]
        wm = list(w); wm[i] -= fd["eps"]
        fp = build(wp)[1].data
        fm = build(wm)[1].data
        num = (fp - fm) / (2 * fd["eps"])
        assert abs(num - grads[i]) <= fd["tolerance"] * max(1.0, abs(num))
