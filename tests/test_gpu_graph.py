"""The generic tensor graph (tt_graph.h) on the GPU against the oracle.

Every op's forward and backward is compared with the oracle's float64
functions on the same seeded inputs (fp32 arithmetic: relative L2 error
<= 1e-5, a few hundred ulps of float32 on sums of up to a few hundred
terms).  The backward of an op is driven through an elementwise product with
a random leaf R, so that the op sees a general output gradient R.  The
classifier of the tinytorch page's example (three features, 32 hidden GELU
units, three classes, SGD) trains on the device and its losses and weights
follow the oracle's float64 run.  The microcrad scalar example c = a * b
gives (6, 3, 2) exactly."""
import math

import numpy as np
import pytest

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import build as native_build

pytestmark = pytest.mark.gpu
rng = np.random.default_rng(5)


@pytest.fixture(scope="module")
def ctx():
    native_build.build()
    c = api.Context(256 << 20)
    yield c
    c.close()


def _rel(a, b):
    return float(np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-30))


def _leaf(ctx, a, dtype="f32"):
    a = np.ascontiguousarray(a, dtype=np.int32 if dtype == "i32" else np.float32)
    return ctx.tensor(*a.shape, dtype=dtype).fill(a)


def test_scalar_product_and_fan_out(ctx):
    ctx.reset()
    a, b = _leaf(ctx, [2.0]), _leaf(ctx, [3.0])
    c = a * b
    c.forward()
    c.backward()
    assert c.numpy()[0] == 6.0 and a.grad()[0] == 3.0 and b.grad()[0] == 2.0
    # y = 2x, z = 3x, L = y + z: dL/dx = 5 (a node with two consumers gets both gradients)
    x, two, three = _leaf(ctx, [1.5]), _leaf(ctx, [2.0]), _leaf(ctx, [3.0])
    L = two * x + three * x
    L.forward()
    L.backward()
    assert L.numpy()[0] == 7.5 and x.grad()[0] == 5.0
    # y = (x1 + x2) * x3
    x1, x2, x3 = _leaf(ctx, [1.0]), _leaf(ctx, [2.0]), _leaf(ctx, [4.0])
    y = (x1 + x2) * x3
    y.forward()
    y.backward()
    assert y.numpy()[0] == 12.0
    assert (x1.grad()[0], x2.grad()[0], x3.grad()[0]) == (4.0, 4.0, 3.0)
    # leaf gradients accumulate across backward calls until zeroed
    y.backward()
    assert x3.grad()[0] == 6.0
    y.zero_grad()
    assert x3.grad()[0] == 0.0


@pytest.mark.parametrize("M,K,N", [(1, 3, 32), (37, 70, 45), (64, 64, 64), (5, 1, 3)])
def test_matmul_matches_oracle(ctx, oracle, M, K, N):
    ctx.reset()
    A, B, R = rng.standard_normal((M, K)), rng.standard_normal((K, N)), rng.standard_normal((M, N))
    a, b, r = _leaf(ctx, A), _leaf(ctx, B), _leaf(ctx, R)
    c = a @ b
    out = c * r
    out.forward()
    out.backward()
    A32, B32, R32 = (x.astype(np.float32).astype(np.float64) for x in (A, B, R))
    assert _rel(c.numpy(), oracle.matmul(A32, B32)) <= 1e-5
    dA, dB = oracle.matmul_bwd(A32, B32, R32)
    assert _rel(a.grad(), dA) <= 1e-5
    assert _rel(b.grad(), dB) <= 1e-5


@pytest.mark.parametrize("rows,cols", [(1, 3), (33, 257), (128, 10)])
def test_elementwise_and_row_ops_match_oracle(ctx, oracle, rows, cols):
    ctx.reset()
    A, Bf, b, R = (rng.standard_normal(s) for s in [(rows, cols), (rows, cols), (cols,), (rows, cols)])
    A32, B32, b32, R32 = (x.astype(np.float32).astype(np.float64) for x in (A, Bf, b, R))
    for name in ["add", "add_row", "mul", "gelu", "softmax"]:
        ctx.reset()
        a, bb, brow, r = _leaf(ctx, A), _leaf(ctx, Bf), _leaf(ctx, b), _leaf(ctx, R)
        y = {"add": lambda: a + bb, "add_row": lambda: a + brow, "mul": lambda: a * bb,
             "gelu": lambda: a.gelu(), "softmax": lambda: a.softmax()}[name]()
        out = y * r
        out.forward()
        out.backward()
        if name == "add":
            ref, ga, gb = A32 + B32, R32, R32
        elif name == "add_row":
            ref = oracle.add_row(A32, b32)
            ga, gb = oracle.add_row_bwd(R32)
        elif name == "mul":
            ref, ga, gb = A32 * B32, R32 * B32, R32 * A32
        elif name == "gelu":
            ref, ga, gb = oracle.gelu_fwd(A32), oracle.gelu_bwd(A32, R32), None
        else:
            ref = oracle.softmax_rows(A32)
            ga, gb = oracle.softmax_rows_bwd(ref, R32), None
        assert _rel(y.numpy(), ref) <= 1e-5, name
        assert _rel(a.grad(), ga) <= 1e-5, name
        if gb is not None:
            got = brow.grad() if name == "add_row" else bb.grad()
            assert _rel(got, gb) <= 1e-5, name


@pytest.mark.parametrize("rows,cols", [(1, 3), (70, 11), (300, 5)])
def test_cross_entropy_both_backward_routes(ctx, oracle, rows, cols):
    Z = rng.standard_normal((rows, cols)) * 2
    y = rng.integers(0, cols, rows).astype(np.int32)
    Z32 = Z.astype(np.float32).astype(np.float64)
    P = oracle.softmax_rows(Z32)
    loss_ref, dP = oracle.xent_probs(P, y)
    dZ = oracle.softmax_rows_bwd(P, dP)
    # softmax -> cross entropy: the pair's gradient (p - onehot) / R
    ctx.reset()
    z, lab = _leaf(ctx, Z), _leaf(ctx, y, "i32")
    loss = z.softmax().cross_entropy(lab)
    loss.forward()
    loss.backward()
    assert abs(float(loss.numpy()[0]) - loss_ref) <= 1e-5 * abs(loss_ref)
    assert _rel(z.grad(), dZ) <= 1e-5
    # the same through the separate backward of each op (the softmax has a second consumer)
    ctx.reset()
    z, lab = _leaf(ctx, Z), _leaf(ctx, y, "i32")
    p = z.softmax()
    loss = p.cross_entropy(lab)
    _ = p * p  # another consumer of p, not on loss's path
    loss.forward()
    loss.backward()
    assert abs(float(loss.numpy()[0]) - loss_ref) <= 1e-5 * abs(loss_ref)
    assert _rel(z.grad(), dZ) <= 1e-5
    # cross entropy of a probability leaf
    ctx.reset()
    pl, lab = _leaf(ctx, P), _leaf(ctx, y, "i32")
    loss = pl.cross_entropy(lab)
    loss.forward()
    loss.backward()
    assert _rel(pl.grad(), oracle.xent_probs(P.astype(np.float32).astype(np.float64), y)[1]) <= 1e-5


def _fruit_graph(ctx, x, y, params):
    W1, b1, W2, b2 = (_leaf(ctx, p) for p in params)
    xn, yn = _leaf(ctx, x), _leaf(ctx, y, "i32")
    hidden = (xn @ W1 + b1).gelu()
    logits = hidden @ W2 + b2
    probs = logits.softmax()
    loss = probs.cross_entropy(yn)
    return (W1, b1, W2, b2), xn, yn, probs, loss


@pytest.mark.parametrize("R,steps,lr", [(64, 200, 0.1), (1, 50, 0.05)])
def test_classifier_sgd_matches_oracle(ctx, oracle, R, steps, lr):
    """The tinytorch page's example loop: the graph is built once; each step
    runs Forward, ZeroGrad, Backward and SGD on the device."""
    if R == 1:  # the page's single sample: colour 0.5, size 0.3, weight 0.8, label 1
        x, y = np.array([[0.5, 0.3, 0.8]], dtype=np.float32), np.array([1], dtype=np.int32)
    else:
        x, y = synth.fruit_batch(R)
    params = synth.mlp_init(*synth.FRUIT_SHAPE)
    ctx.reset()
    P, xn, yn, probs, loss = _fruit_graph(ctx, x, y, params)
    losses = []
    for _ in range(steps):
        loss.forward()
        losses.append(float(loss.numpy()[0]))
        loss.zero_grad()
        loss.backward()
        ctx.sgd(P, lr)
    ref, new_params, _ = oracle.mlp_sgd(x, y, *params, lr, steps)
    assert losses[-1] < losses[0]
    assert _rel(np.array(losses), ref) <= 1e-4
    for got, want in zip(P, new_params):
        assert _rel(got.numpy(), want) <= 1e-4
    # inference on the trained weights
    probs.forward()
    pr = probs.numpy()
    assert np.allclose(pr.sum(axis=1), 1.0, atol=1e-6)


def test_graph_is_deterministic(ctx):
    x, y = synth.fruit_batch(64)
    params = synth.mlp_init(*synth.FRUIT_SHAPE)
    runs = []
    for _ in range(2):
        ctx.reset()
        P, _, _, _, loss = _fruit_graph(ctx, x, y, params)
        for _ in range(20):
            loss.forward()
            loss.zero_grad()
            loss.backward()
            ctx.sgd(P, 0.1)
        runs.append(np.concatenate([p.numpy().ravel() for p in P]))
    assert np.array_equal(runs[0], runs[1])


def test_graph_errors(ctx):
    ctx.reset()
    a = _leaf(ctx, np.ones((2, 3)))
    b = _leaf(ctx, np.ones((4, 5)))
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        a @ b
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        a + b
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.tensor(2, 0)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        a.fill(np.ones(5, dtype=np.float32))
    # labels out of range are reported at the next sync
    lab = _leaf(ctx, [0, 7], "i32")
    loss = a.softmax().cross_entropy(lab)
    loss.forward()
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.sync()
    # a reset makes every earlier handle stale
    ctx.reset()
    with pytest.raises(api.TTError, match="TT_ERR_STALE"):
        a.forward()
    # and a handle of another context is refused
    with api.Context(1 << 20) as other:
        o = other.tensor(1)
        with pytest.raises(api.TTError, match="TT_ERR_STALE"):
            api.Node(ctx, o.h).forward()
    # an arena too small for a node
    with api.Context(4096) as small:
        with pytest.raises(api.TTError, match="TT_ERR_ARENA_OOM"):
            small.tensor(1024, 1024)
        small.tensor(8)  # still usable


def test_recorded_step_replays_the_loop(ctx, oracle):
    """One step recorded as a CUDA graph and replayed gives the directly run
    loop's weights bit for bit, and follows the oracle."""
    x, y = synth.fruit_batch(64)
    params = synth.mlp_init(*synth.FRUIT_SHAPE)
    steps = 200
    ctx.reset()
    P, _, _, _, loss = _fruit_graph(ctx, x, y, params)

    def step():
        loss.forward()
        loss.zero_grad()
        loss.backward()
        ctx.sgd(P, 0.1)

    for _ in range(steps):
        step()
    direct = [p.numpy() for p in P]
    ctx.reset()
    P, _, _, _, loss = _fruit_graph(ctx, x, y, params)
    step()
    n0 = ctx.launches
    ctx.record(step)  # recorded, not run
    assert ctx.launches == n0
    ctx.replay(steps - 1)
    assert ctx.launches > n0
    replayed = [p.numpy() for p in P]
    for a, b in zip(direct, replayed):
        assert np.array_equal(a, b)
    _, new_params, _ = oracle.mlp_sgd(x, y, *params, 0.1, steps)
    for got, want in zip(replayed, new_params):
        assert _rel(got, want) <= 1e-4
    # calls that wait for the device, or make nodes, are refused while recording
    ctx.capture_begin()
    for call in (lambda: loss.numpy(), ctx.sync, ctx.reset, lambda: ctx.tensor(3),
                 lambda: P[0].fill(np.zeros(P[0].shape, dtype=np.float32))):
        with pytest.raises(api.TTError, match="TT_ERR_STATE"):
            call()
    with pytest.raises(api.TTError, match="TT_ERR_STATE"):
        ctx.capture_begin()
    ctx.capture_end()
    ctx.replay(0)
    # a reset drops the recording
    ctx.reset()
    with pytest.raises(api.TTError, match="TT_ERR_STATE"):
        ctx.replay(1)
    with pytest.raises(api.TTError, match="TT_ERR_STATE"):
        ctx.capture_end()
