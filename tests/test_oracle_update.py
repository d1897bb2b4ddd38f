"""Pins for the oracle's update-side variants: the global gradient norm and
its clip (dl-scratch page 3.2), AdamW on the clipped, unscaled gradient with
the step skipped on overflow, the dynamic loss scale (3.4), and gradient
accumulation over micro-batches (the += of the tinytorch page 三.3).

Checked against torch's own clip_grad_norm_ and AdamW in float64, numpy's
norm, sequences worked by hand, and the linearity of the mean loss."""
import math

import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import synth

rng = np.random.default_rng(17)


def _rel(a, b):
    return np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300)


def test_grad_norm_library_and_scale(oracle):
    g = rng.standard_normal(1000)
    n, bad = oracle.grad_norm(g)
    assert bad == 0 and abs(n - np.linalg.norm(g)) <= 1e-12 * n
    assert oracle.grad_norm([3.0, 4.0]) == (5.0, 0)
    n2, _ = oracle.grad_norm(g * 1024.0, scale=1024.0)
    assert n2 == n  # a power-of-two scale divides out exactly
    for poison in (np.inf, -np.inf, np.nan):
        h = g.copy()
        h[17] = poison
        assert oracle.grad_norm(h)[1] == 1
    assert oracle.grad_norm(np.array([1e200, 1.0]))[1] == 1  # the square overflows


def test_clip_matches_torch(oracle):
    for max_norm in (0.1, 1.0, 100.0):
        parts = [torch.from_numpy(rng.standard_normal(s)) for s in [(7, 5), (11,), (3, 3)]]
        for p in parts:
            p.grad = p.clone()
        flat = np.concatenate([p.grad.numpy().ravel() for p in parts])
        total = torch.nn.utils.clip_grad_norm_(parts, max_norm)
        n, _ = oracle.grad_norm(flat)
        assert abs(n - float(total)) <= 1e-12 * n
        k = oracle.clip_coef(n, max_norm)
        got = np.concatenate([p.grad.numpy().ravel() for p in parts])
        assert _rel(flat * k, got) < 1e-14
        assert k <= 1.0 and (k == 1.0) == (max_norm / (n + 1e-6) >= 1.0)


def test_adamw_ex_against_torch_clip_then_adamw(oracle):
    n, steps = 64, 3
    p0 = rng.standard_normal(n)
    lr, b1, b2, eps, wd, max_norm, scale = 1e-2, 0.9, 0.95, 1e-8, 0.1, 0.5, 256.0
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    tp = torch.from_numpy(p0.copy()).requires_grad_(True)
    opt = torch.optim.AdamW([tp], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    for t in range(1, steps + 1):
        g = rng.standard_normal(n) * 3.0
        p, m, v, skipped = oracle.adamw_ex(p, g * scale, m, v, lr, b1, b2, eps, wd, t, scale=scale,
                                           max_norm=max_norm)
        assert not skipped
        tp.grad = torch.from_numpy(g.copy())
        torch.nn.utils.clip_grad_norm_([tp], max_norm)
        opt.step()
        assert _rel(p, tp.detach().numpy()) < 1e-12
    # no scale and no clip: the plain AdamW step
    g = rng.standard_normal(n)
    a = oracle.adamw_ex(p, g, m, v, lr, b1, b2, eps, wd, 4)
    b = oracle.adamw(p, g, m, v, lr, b1, b2, eps, wd, 4)
    for x, y in zip(a[:3], b):
        assert np.array_equal(x, y)


def test_adamw_ex_skips_on_overflow(oracle):
    p, g, m, v = (rng.standard_normal(16) for _ in range(4))
    g[3] = np.inf
    p2, m2, v2, skipped = oracle.adamw_ex(p, g, m, v, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, max_norm=1.0)
    assert skipped
    assert np.array_equal(p2, p) and np.array_equal(m2, m) and np.array_equal(v2, v)


def test_loss_scale_sequence_by_hand(oracle):
    s, c = 65536.0, 0
    s, c = oracle.loss_scale_update(s, c, True)
    assert (s, c) == (32768.0, 0)
    for i in range(999):
        s, c = oracle.loss_scale_update(s, c, False)
    assert (s, c) == (32768.0, 999)
    s, c = oracle.loss_scale_update(s, c, False)  # the 1000th clean step in a row
    assert c == 0 and abs(s - 32768.0 * 1.001) < 1e-9
    s, c = oracle.loss_scale_update(s, 500, True)  # an overflow restarts the count
    assert c == 0 and abs(s - 32768.0 * 1.001 / 2) < 1e-9
    s, c = oracle.loss_scale_update(8.0, 1, False, window=2, growth=2.0)
    assert (s, c) == (16.0, 0)


def test_accumulated_micro_batches_equal_the_full_batch(oracle):
    """Mean losses: the gradients of two equal micro-batches, added, are
    twice the gradient of the batch they make up."""
    sh = synth.WORKLOADS["tiny_fp32"].shape
    p = synth.init_params(sh, jitter=0.05).astype(np.float64)
    tok, tgt = synth.token_stream(4, 16, sh.V, "uniform", seed=9)
    _, g_full, _ = oracle.gpt2_step(sh, p, tok, tgt)
    _, g_a, _ = oracle.gpt2_step(sh, p, tok[:2], tgt[:2])
    _, g_b, _ = oracle.gpt2_step(sh, p, tok[2:], tgt[2:])
    assert _rel(g_a + g_b, 2.0 * g_full) < 1e-12
