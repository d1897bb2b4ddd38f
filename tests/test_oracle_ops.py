"""Pins for the oracle's op arithmetic.

Each op is checked against something other than itself: torch float64
library routines (F.linear, F.layer_norm, F.gelu, scaled_dot_product_attention,
F.cross_entropy, torch.optim.AdamW), closed forms and invariants the pages
name (softmax rows sum to 1, uniform logits give ln V, LN output has mean 0
and variance 1), and central finite differences for every backward."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

rng = np.random.default_rng(7)


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _fd(f, x, eps=1e-6):
    """central finite difference of scalar f w.r.t. every element of x (in place)."""
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


# ----------------------------------------------------------------- linear
def test_linear_matches_library(oracle):
    x, W, b = rng.normal(size=(7, 5)), rng.normal(size=(3, 5)), rng.normal(size=3)
    y = oracle.linear_fwd(x, W, b)
    ref = F.linear(_t(x), _t(W), _t(b)).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(oracle.linear_fwd(x, W), (_t(x) @ _t(W).T).numpy(), rtol=1e-14, atol=1e-14)


def test_linear_backward_fd(oracle):
    x, W, b = rng.normal(size=(4, 3)), rng.normal(size=(5, 3)), rng.normal(size=5)
    R = rng.normal(size=(4, 5))  # loss = sum(R * y)
    dx, dW, db = oracle.linear_bwd(x, W, R)
    f = lambda: float(np.sum(R * oracle.linear_fwd(x, W, b)))
    assert _rel(dx, _fd(f, x)) < 1e-8
    assert _rel(dW, _fd(f, W)) < 1e-8
    assert _rel(db, _fd(f, b)) < 1e-8


# ----------------------------------------------------------------- layernorm
def test_layernorm_matches_library_and_invariants(oracle):
    x = rng.normal(size=(6, 16)) * 3 + 1.5
    w, b = rng.normal(size=16), rng.normal(size=16)
    y, mean, rstd = oracle.layernorm_fwd(x, w, b)
    ref = F.layer_norm(_t(x), (16,), _t(w), _t(b), eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # before the affine: mean 0, (biased) variance 1 up to eps
    yh, _, _ = oracle.layernorm_fwd(x, np.ones(16), np.zeros(16))
    assert np.max(np.abs(yh.mean(axis=1))) < 1e-12
    var = (x.var(axis=1))
    np.testing.assert_allclose(yh.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13)


def test_layernorm_backward_fd(oracle):
    x = rng.normal(size=(3, 8))
    w, b = rng.normal(size=8), rng.normal(size=8)
    R = rng.normal(size=(3, 8))
    _, mean, rstd = oracle.layernorm_fwd(x, w, b)
    dx, dw, db = oracle.layernorm_bwd(x, w, mean, rstd, R)
    f = lambda: float(np.sum(R * oracle.layernorm_fwd(x, w, b)[0]))
    assert _rel(dx, _fd(f, x)) < 1e-7
    assert _rel(dw, _fd(f, w)) < 1e-8
    assert _rel(db, _fd(f, b)) < 1e-8


# ----------------------------------------------------------------- gelu
def test_gelu_matches_library_and_closed_forms(oracle):
    u = np.linspace(-8, 8, 1001)
    g = oracle.gelu_fwd(u)
    ref = F.gelu(_t(u), approximate="tanh").numpy()
    np.testing.assert_allclose(g, ref, rtol=1e-14, atol=1e-15)
    assert oracle.gelu_fwd(np.array([0.0]))[0] == 0.0
    assert oracle.gelu_bwd(np.array([0.0]), np.array([1.0]))[0] == 0.5
    big = oracle.gelu_fwd(np.array([30.0, -30.0]))
    assert big[0] == 30.0 and big[1] == 0.0


def test_gelu_backward_fd_and_library(oracle):
    u = rng.normal(size=50) * 3
    d = oracle.gelu_bwd(u, np.ones_like(u))
    ut = _t(u).requires_grad_(True)
    F.gelu(ut, approximate="tanh").sum().backward()
    np.testing.assert_allclose(d, ut.grad.numpy(), rtol=1e-12, atol=1e-14)
    f = lambda: float(np.sum(oracle.gelu_fwd(u)))
    assert _rel(d, _fd(f, u)) < 1e-8


# ----------------------------------------------------------------- attention
def _split(qkv, B, T, C, H):
    hd = C // H
    q = qkv[:, :C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    k = qkv[:, C:2 * C].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    v = qkv[:, 2 * C:].reshape(B, T, H, hd).transpose(0, 2, 1, 3)
    return q, k, v


@pytest.mark.parametrize("B,T,C,H", [(2, 5, 8, 2), (1, 9, 12, 3), (3, 1, 4, 1)])
def test_attention_matches_library(oracle, B, T, C, H):
    qkv = rng.normal(size=(B * T, 3 * C))
    y, P = oracle.attention_fwd(qkv, B, T, C, H)
    q, k, v = (_t(a) for a in _split(qkv, B, T, C, H))
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    ref = ref.transpose(1, 2).reshape(B * T, C).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-13)
    # softmax rows sum to 1; the future has zero weight
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.triu(P, k=1) == 0.0)


def test_attention_special_cases(oracle):
    # T = 1: each position attends only to itself, y = v
    B, T, C, H = 3, 1, 8, 2
    qkv = rng.normal(size=(B * T, 3 * C))
    y, _ = oracle.attention_fwd(qkv, B, T, C, H)
    np.testing.assert_allclose(y, qkv[:, 2 * C:], rtol=0, atol=1e-15)
    # zero queries: uniform weights over the causal window, y_t = mean(v_0..v_t)
    B, T = 2, 6
    qkv = rng.normal(size=(B * T, 3 * C))
    qkv[:, :C] = 0.0
    y, _ = oracle.attention_fwd(qkv, B, T, C, H)
    v = qkv[:, 2 * C:].reshape(B, T, C)
    cm = np.cumsum(v, axis=1) / np.arange(1, T + 1)[None, :, None]
    np.testing.assert_allclose(y.reshape(B, T, C), cm, rtol=1e-13, atol=1e-14)


def test_attention_lse(oracle):
    """The saved log-sum-exp: torch's float64 logsumexp of the masked, scaled
    scores; with T = 1 the single score q.k/sqrt(hd); with zero queries every
    visible score is 0, so row t gives ln(t + 1)."""
    B, T, C, H = 2, 7, 12, 3
    hd = C // H
    qkv = rng.normal(size=(B * T, 3 * C))
    _, P, lse = oracle.attention_fwd(qkv, B, T, C, H, want_lse=True)
    q, k, _ = (_t(a) for a in _split(qkv, B, T, C, H))
    s = (q @ k.transpose(-1, -2)) / np.sqrt(hd)
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-13, atol=1e-13)
    # P is rebuilt from the scores and lse alone: exp(s - lse)
    np.testing.assert_allclose(P, torch.exp(s - _t(lse)[..., None]).numpy(), rtol=1e-12, atol=1e-15)
    # T = 1
    B, T = 3, 1
    qkv = rng.normal(size=(B * T, 3 * C))
    _, _, lse = oracle.attention_fwd(qkv, B, T, C, H, want_lse=True)
    qh = qkv[:, :C].reshape(B, H, hd)
    kh = qkv[:, C:2 * C].reshape(B, H, hd)
    np.testing.assert_allclose(lse[:, :, 0], np.sum(qh * kh, axis=-1) / np.sqrt(hd), rtol=1e-14, atol=1e-14)
    # zero queries
    B, T = 2, 9
    qkv = rng.normal(size=(B * T, 3 * C))
    qkv[:, :C] = 0.0
    _, _, lse = oracle.attention_fwd(qkv, B, T, C, H, want_lse=True)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, T + 1)), (B, H, T)), rtol=0,
                               atol=1e-15)


def test_attention_backward_fd(oracle):
    B, T, C, H = 2, 4, 6, 2
    qkv = rng.normal(size=(B * T, 3 * C))
    R = rng.normal(size=(B * T, C))
    _, P = oracle.attention_fwd(qkv, B, T, C, H)
    d = oracle.attention_bwd(qkv, P, R, B, T, C, H)
    f = lambda: float(np.sum(R * oracle.attention_fwd(qkv, B, T, C, H)[0]))
    assert _rel(d, _fd(f, qkv)) < 1e-7


# ----------------------------------------------------------------- cross entropy
def test_xent_matches_library(oracle):
    z = rng.normal(size=(9, 13)) * 4
    t = rng.integers(0, 13, size=9).astype(np.int32)
    loss, rl, dz = oracle.xent(z, t, want_grad=True)
    zt = _t(z).requires_grad_(True)
    ref = F.cross_entropy(zt, torch.from_numpy(t.astype(np.int64)))
    ref.backward()
    assert math.isclose(loss, ref.item(), rel_tol=1e-14)
    np.testing.assert_allclose(dz, zt.grad.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(rl, F.cross_entropy(_t(z), torch.from_numpy(t.astype(np.int64)),
                                                   reduction="none").numpy(), rtol=1e-13)


@pytest.mark.parametrize("V", [256, 65, 50257])
def test_xent_uniform_logits_is_log_v(oracle, V):
    z = np.zeros((3, V))
    t = np.array([0, V - 1, V // 2], dtype=np.int32)
    loss, rl, dz = oracle.xent(z, t, want_grad=True)
    assert abs(loss - math.log(V)) <= 4e-16 * math.log(V) * 4
    # gradient rows sum to zero (probabilities sum to 1, minus the one-hot)
    assert np.max(np.abs(dz.sum(axis=1))) < 1e-15


def test_xent_large_logits_stable(oracle):
    z = np.array([[1000.0, 0.0, -1000.0]])
    loss, _, dz = oracle.xent(z, np.array([0], dtype=np.int32), want_grad=True)
    assert loss == 0.0 and np.all(np.isfinite(dz))


# ----------------------------------------------------------------- embedding
def test_embedding_gather_and_scatter(oracle):
    B, T, V, C, maxT = 2, 3, 5, 4, 4
    wte, wpe = rng.normal(size=(V, C)), rng.normal(size=(maxT, C))
    tok = np.array([[1, 1, 4], [0, 1, 2]], dtype=np.int32)
    x = oracle.embed_fwd(wte, wpe, tok, B, T)
    ref = (F.embedding(torch.from_numpy(tok.astype(np.int64)), _t(wte))
           + _t(wpe)[:T][None]).reshape(B * T, C).numpy()
    np.testing.assert_array_equal(x, ref)
    dx = rng.normal(size=(B * T, C))
    dwte, dwpe = oracle.embed_bwd(dx, tok, B, T, V, maxT)
    # token 1 appears at positions (0,0), (0,1), (1,1)
    np.testing.assert_allclose(dwte[1], dx[0] + dx[1] + dx[4], rtol=1e-15)
    assert np.all(dwte[3] == 0.0)
    np.testing.assert_allclose(dwpe[:T], dx.reshape(B, T, C).sum(axis=0), rtol=1e-15)
    assert np.all(dwpe[T:] == 0.0)


# ----------------------------------------------------------------- adamw
def test_adamw_matches_library_over_steps(oracle):
    n = 37
    p0 = rng.normal(size=n)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    pt = _t(p0.copy()).requires_grad_(True)
    opt = torch.optim.AdamW([pt], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 6):
        g = rng.normal(size=n)
        pt.grad = _t(g)
        opt.step()
        p, m, v = oracle.adamw(p, g, m, v, lr, b1, b2, eps, wd, t)
        np.testing.assert_allclose(p, pt.detach().numpy(), rtol=1e-14, atol=1e-16)


def test_adamw_first_step_closed_form(oracle):
    p0 = np.array([0.5, -0.25, 2.0])
    g = np.array([0.1, -3.0, 1e-9])
    lr, wd, eps = 1e-3, 0.1, 1e-8
    p, m, v = oracle.adamw(p0, g, np.zeros(3), np.zeros(3), lr, 0.9, 0.95, eps, wd, 1)
    expect = p0 - lr * (g / (np.abs(g) + eps) + wd * p0)
    np.testing.assert_allclose(p, expect, rtol=1e-15)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v, 0.05 * g * g, rtol=1e-15)
