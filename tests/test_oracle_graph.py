"""Pins for the oracle's generic tensor ops and the small SGD classifier
(tinytorch page 三.3-三.5, 八.1, 八.5).

Each function is checked against something other than itself: a product
worked by hand, numpy's matmul, closed forms of the softmax and the cross
entropy, the oracle's fused log-softmax cross entropy (pinned on its own in
test_oracle_ops against torch), and central finite differences for every
backward, including the whole classifier's gradient."""
import math

import numpy as np
import pytest

from autograd_arena_allocated_gb300 import synth

rng = np.random.default_rng(11)


def _fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + eps
        fp = f()
        x[i] = old - eps
        fm = f()
        x[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


def _rel(a, b):
    return np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300)


def test_matmul_worked_example_and_library(oracle):
    A = np.array([[1.0, 2, 3], [4, 5, 6]])
    B = np.array([[7.0, 8], [9, 10], [11, 12]])
    assert np.array_equal(oracle.matmul(A, B), [[58, 64], [139, 154]])
    for M, K, N in [(1, 3, 32), (5, 7, 3), (17, 33, 9)]:
        A, B = rng.standard_normal((M, K)), rng.standard_normal((K, N))
        assert _rel(oracle.matmul(A, B), A @ B) < 1e-14


def test_matmul_backward_finite_differences(oracle):
    A, B = rng.standard_normal((4, 5)), rng.standard_normal((5, 3))
    R = rng.standard_normal((4, 3))
    dA, dB = oracle.matmul_bwd(A, B, R)
    f = lambda: float(np.sum(R * oracle.matmul(A, B)))
    assert _rel(dA, _fd(f, A)) < 1e-8
    assert _rel(dB, _fd(f, B)) < 1e-8
    # the shapes of the transposed products
    assert dA.shape == A.shape and dB.shape == B.shape


def test_add_row(oracle):
    A, b = rng.standard_normal((3, 4)), rng.standard_normal(4)
    assert np.array_equal(oracle.add_row(A, b), A + b[None, :])
    dC = rng.standard_normal((3, 4))
    dA, db = oracle.add_row_bwd(dC)
    assert np.array_equal(dA, dC)
    assert np.allclose(db, dC.sum(axis=0), rtol=0, atol=1e-15)


def test_softmax_closed_forms(oracle):
    P = oracle.softmax_rows(np.array([[0.0, math.log(2.0)], [5.0, 5.0]]))
    assert np.allclose(P, [[1 / 3, 2 / 3], [0.5, 0.5]], rtol=0, atol=1e-15)
    Z = rng.standard_normal((6, 9)) * 4
    P = oracle.softmax_rows(Z)
    assert np.allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.allclose(oracle.softmax_rows(Z + 100.0), P, rtol=0, atol=1e-14)  # shift invariance
    assert np.all(np.argmax(P, axis=1) == np.argmax(Z, axis=1))


def test_softmax_backward_finite_differences(oracle):
    Z = rng.standard_normal((3, 5))
    R = rng.standard_normal((3, 5))
    P = oracle.softmax_rows(Z)
    dZ = oracle.softmax_rows_bwd(P, R)
    assert _rel(dZ, _fd(lambda: float(np.sum(R * oracle.softmax_rows(Z))), Z)) < 1e-8


def test_xent_probs_closed_forms(oracle):
    for Cc in (3, 10):
        P = np.full((4, Cc), 1.0 / Cc)
        loss, _ = oracle.xent_probs(P, np.arange(4) % Cc)
        assert abs(loss - math.log(Cc)) < 1e-14
    P = np.eye(3)
    loss, _ = oracle.xent_probs(P, np.arange(3))
    assert loss == 0.0


def test_xent_probs_backward_finite_differences(oracle):
    P = oracle.softmax_rows(rng.standard_normal((5, 4)))
    y = np.array([0, 3, 1, 1, 2], dtype=np.int32)
    _, dP = oracle.xent_probs(P, y, dloss=0.7)
    g = _fd(lambda: 0.7 * oracle.xent_probs(P, y)[0], P)
    assert _rel(dP, g) < 1e-8


def test_softmax_then_xent_equals_fused_log_softmax(oracle):
    """The chain softmax -> CE of probabilities gives the fused log-softmax
    cross entropy and its gradient (probs - onehot)/R (tinytorch 三.5)."""
    Z = rng.standard_normal((6, 7)) * 3
    y = rng.integers(0, 7, 6).astype(np.int32)
    P = oracle.softmax_rows(Z)
    loss, dP = oracle.xent_probs(P, y)
    dZ = oracle.softmax_rows_bwd(P, dP)
    fl, _, fdz = oracle.xent(Z, y, want_grad=True)
    assert abs(loss - fl) < 1e-13
    onehot = np.eye(7)[y]
    assert _rel(dZ, fdz) < 1e-12
    assert _rel(dZ, (P - onehot) / 6) < 1e-12


def _mlp_loss(oracle, x, y, W1, b1, W2, b2):
    losses, _, _ = oracle.mlp_sgd(x, y, W1, b1, W2, b2, 0.0, 1)
    return float(losses[0])


def test_mlp_gradient_finite_differences(oracle):
    x, y = synth.fruit_batch(6, seed=3)
    W1, b1, W2, b2 = (a.astype(np.float64) for a in synth.mlp_init(3, 5, 3, seed=4, std=0.8))
    _, _, (gW1, gb1, gW2, gb2) = oracle.mlp_sgd(x, y, W1, b1, W2, b2, 0.0, 1)
    f = lambda: _mlp_loss(oracle, x, y, W1, b1, W2, b2)
    for g, p in [(gW1, W1), (gb1, b1), (gW2, W2), (gb2, b2)]:
        assert _rel(g, _fd(f, p)) < 1e-7


def test_mlp_sgd_update_and_closed_form_start(oracle):
    x, y = synth.fruit_batch(8, seed=5)
    W1, b1, W2, b2 = (a.astype(np.float64) for a in synth.mlp_init(3, 32, 3, seed=6))
    # zero output layer: every class has probability 1/3
    losses, _, _ = oracle.mlp_sgd(x, y, W1, b1, np.zeros_like(W2), np.zeros_like(b2), 0.0, 1)
    assert abs(losses[0] - math.log(3.0)) < 1e-14
    # one step is p - lr g, with g the step's own gradient
    lr = 0.05
    _, (W1n, b1n, W2n, b2n), (gW1, gb1, gW2, gb2) = oracle.mlp_sgd(x, y, W1, b1, W2, b2, lr, 1)
    for new, old, g in [(W1n, W1, gW1), (b1n, b1, gb1), (W2n, W2, gW2), (b2n, b2, gb2)]:
        assert np.allclose(new, old - lr * g, rtol=0, atol=1e-15)
    # training reduces the loss on its batch
    losses, _, _ = oracle.mlp_sgd(x, y, W1, b1, W2, b2, 0.1, 300)
    assert losses[-1] < 0.5 * losses[0]
