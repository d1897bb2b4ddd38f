"""Pins for the oracle's whole GPT-2 step.

- parameter counts (the tinytorch page prints 124,475,904 with the vocabulary
  padded to 50304);
- every gradient element of a small model against central finite
  differences (NumPy framework page, 4.2), and a sample of the tiny model's;
- loss = ln V when the (tied) embedding is zero;
- two reductions to library routines that pin the block wiring: T = 1
  (attention returns v) and all-zero weight matrices (blocks add constants);
- the per-position losses average to the loss.
"""
import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from autograd_arena_allocated_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


class Shape:
    def __init__(self, L, C, H, V, maxT):
        self.L, self.C, self.H, self.V, self.maxT = L, C, H, V, maxT


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _slices(o, sh):
    """name -> (offset, numel) from the oracle's own layout."""
    out = {"wte": o.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 0),
           "wpe": o.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 1)}
    names = ["ln1_w", "ln1_b", "qkv_w", "qkv_b", "proj_w", "proj_b", "ln2_w", "ln2_b",
             "fc_w", "fc_b", "fcproj_w", "fcproj_b"]
    for l in range(sh.L):
        for j, nm in enumerate(names):
            out[f"h{l}.{nm}"] = o.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, l, 2 + j)
    out["lnf_w"] = o.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 14)
    out["lnf_b"] = o.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 15)
    return out


def test_param_counts(oracle):
    g = _gold("gpt2_124m.json")
    L, C, H, V, T = g["num_layers"], g["channels"], g["num_heads"], g["vocab_size"], g["max_seq_len"]
    n = oracle.num_params(L, C, H, V, T)
    assert n == 124_439_808
    assert n + (g["padded_vocab_size"] - V) * C == g["num_parameters_padded"]
    # the layout is contiguous and in the documented order
    sh = Shape(L, C, H, V, T)
    sl = _slices(oracle, sh)
    at = 0
    for name, numel, _ in synth.param_table(synth.GPT2Shape(L, C, H, V, T)):
        assert sl[name] == (at, numel), name
        at += numel
    assert at == n
    assert oracle.num_params(24, 1024, 16, 50257, 1024) == 354_823_168
    assert oracle.num_params(6, 384, 6, 65, 256) == 10_770_816
    assert oracle.num_params(2, 64, 4, 256, 32) == 118_528


def _inputs(sh, B, T, seed=3, jitter=0.05, kind="uniform"):
    p = synth.init_params(synth.GPT2Shape(sh.L, sh.C, sh.H, sh.V, sh.maxT), jitter=jitter)
    tok, tgt = synth.token_stream(B, T, sh.V, kind, seed=seed)
    return p.astype(np.float64), tok, tgt


def test_every_gradient_matches_finite_difference(oracle):
    """Small model (L=1, C=16, H=2, V=17, B=2, T=5): all 3,664 parameters."""
    fd = _gold("finite_difference.json")
    sh = Shape(1, 16, 2, 17, 5)
    p, tok, tgt = _inputs(sh, 2, 5, jitter=0.3)
    p *= 3.0  # larger weights so that every path carries signal
    loss, g, _ = oracle.gpt2_step(sh, p, tok, tgt)
    eps = fd["eps"]
    num = np.zeros_like(p)
    for i in range(p.size):
        old = p[i]
        p[i] = old + eps
        fp = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False)[0]
        p[i] = old - eps
        fm = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False)[0]
        p[i] = old
        num[i] = (fp - fm) / (2 * eps)
    # element-wise: the page's bar (1e-5)
    assert np.max(np.abs(num - g)) <= fd["tolerance"]
    # per tensor: relative L2 error far below it
    for name, (off, n) in _slices(oracle, sh).items():
        ref = num[off:off + n]
        err = np.linalg.norm(g[off:off + n] - ref) / max(np.linalg.norm(ref), 1e-12)
        assert err < 1e-6, (name, err)


def test_tiny_model_gradient_sample(oracle):
    """Tiny config (L=2, C=64, H=4, V=256, B=4, T=32): 6 elements of every tensor."""
    sh = Shape(2, 64, 4, 256, 32)
    p, tok, tgt = _inputs(sh, 4, 32, jitter=0.1)
    _, g, _ = oracle.gpt2_step(sh, p, tok, tgt)
    rs = np.random.default_rng(11)
    eps = 1e-5
    for name, (off, n) in _slices(oracle, sh).items():
        idx = off + rs.choice(n, size=min(6, n), replace=False)
        if name == "wte":  # include rows of tokens that do and do not occur
            idx = np.concatenate([idx, off + tok[0, :2] * sh.C + 5])
        for i in idx:
            old = p[i]
            p[i] = old + eps
            fp = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False)[0]
            p[i] = old - eps
            fm = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False)[0]
            p[i] = old
            num = (fp - fm) / (2 * eps)
            assert abs(num - g[i]) <= 1e-8 + 1e-6 * abs(num), (name, i, num, g[i])


def test_zero_embedding_gives_log_v(oracle):
    for sh, B, T in [(Shape(2, 64, 4, 256, 32), 2, 8), (Shape(1, 16, 2, 65, 8), 3, 8),
                     (Shape(1, 16, 2, 50257, 4), 1, 4)]:
        p, tok, tgt = _inputs(sh, B, T)
        off, n = oracle.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 0)
        p[off:off + n] = 0.0
        loss, g, rl = oracle.gpt2_step(sh, p, tok, tgt, want_row_loss=True)
        assert abs(loss - math.log(sh.V)) < 1e-14 * math.log(sh.V) * 8
        np.testing.assert_allclose(rl, math.log(sh.V), rtol=1e-14)


def _lib_tensors(oracle, sh, p):
    return {k: torch.from_numpy(p[o:o + n].copy()) for k, (o, n) in _slices(oracle, sh).items()}


def test_single_position_reduces_to_library_mlp(oracle):
    """With T = 1 causal attention returns v, so each pre-LN block is
    x1 = x + proj(v(LN1 x)), x2 = x1 + fcproj(gelu(fc(LN2 x1))): a stack of
    library calls, written here from the block structure the tinytorch page
    gives (LN -> Attn -> + -> LN -> MLP -> +)."""
    sh = Shape(2, 16, 2, 23, 4)
    B, T = 3, 1
    p, tok, tgt = _inputs(sh, B, T, jitter=0.2)
    p *= 5.0
    loss, _, rl = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False, want_row_loss=True)
    W = _lib_tensors(oracle, sh, p)
    C = sh.C
    x = F.embedding(torch.from_numpy(tok[:, 0].astype(np.int64)), W["wte"].view(sh.V, C)) \
        + W["wpe"].view(sh.maxT, C)[0]
    for l in range(sh.L):
        h = F.layer_norm(x, (C,), W[f"h{l}.ln1_w"], W[f"h{l}.ln1_b"], eps=1e-5)
        qkv = F.linear(h, W[f"h{l}.qkv_w"].view(3 * C, C), W[f"h{l}.qkv_b"])
        a = qkv[:, 2 * C:]
        x = x + F.linear(a, W[f"h{l}.proj_w"].view(C, C), W[f"h{l}.proj_b"])
        h2 = F.layer_norm(x, (C,), W[f"h{l}.ln2_w"], W[f"h{l}.ln2_b"], eps=1e-5)
        u = F.linear(h2, W[f"h{l}.fc_w"].view(4 * C, C), W[f"h{l}.fc_b"])
        x = x + F.linear(F.gelu(u, approximate="tanh"), W[f"h{l}.fcproj_w"].view(C, 4 * C),
                         W[f"h{l}.fcproj_b"])
    hf = F.layer_norm(x, (C,), W["lnf_w"], W["lnf_b"], eps=1e-5)
    z = F.linear(hf, W["wte"].view(sh.V, C))
    ref = F.cross_entropy(z, torch.from_numpy(tgt[:, 0].astype(np.int64)), reduction="none")
    np.testing.assert_allclose(rl, ref.numpy(), rtol=1e-12)
    assert math.isclose(loss, ref.mean().item(), rel_tol=1e-12)


def test_zero_matrices_reduce_blocks_to_constants(oracle):
    """With every block matrix zero, attention averages the constant v = b_v,
    so block l adds c_l = proj(b_v) + fcproj(gelu(b_fc)) to every position and
    the logits are LN_f(wte[tok] + wpe[t] + sum_l c_l) wte^T."""
    sh = Shape(2, 16, 4, 29, 6)
    B, T = 2, 6
    p, tok, tgt = _inputs(sh, B, T, jitter=0.3)
    sl = _slices(oracle, sh)
    for l in range(sh.L):
        for nm in ("qkv_w", "fc_w"):
            o, n = sl[f"h{l}.{nm}"]
            p[o:o + n] = 0.0
    loss, _, rl = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False, want_row_loss=True)
    W = _lib_tensors(oracle, sh, p)
    C = sh.C
    x = F.embedding(torch.from_numpy(tok.astype(np.int64)), W["wte"].view(sh.V, C)) \
        + W["wpe"].view(sh.maxT, C)[:T][None]
    for l in range(sh.L):
        bv = W[f"h{l}.qkv_b"][2 * C:]
        c = F.linear(bv, W[f"h{l}.proj_w"].view(C, C), W[f"h{l}.proj_b"])
        g = F.gelu(W[f"h{l}.fc_b"], approximate="tanh")
        c = c + F.linear(g, W[f"h{l}.fcproj_w"].view(C, 4 * C), W[f"h{l}.fcproj_b"])
        x = x + c
    hf = F.layer_norm(x, (C,), W["lnf_w"], W["lnf_b"], eps=1e-5)
    z = F.linear(hf, W["wte"].view(sh.V, C)).reshape(B * T, sh.V)
    ref = F.cross_entropy(z, torch.from_numpy(tgt.reshape(-1).astype(np.int64)), reduction="none")
    np.testing.assert_allclose(rl, ref.numpy(), rtol=1e-12)
    assert math.isclose(loss, float(np.mean(rl)), rel_tol=1e-14)


def test_bad_arguments_give_nan(oracle):
    sh = Shape(1, 16, 2, 17, 5)
    p, tok, tgt = _inputs(sh, 1, 5)
    bad = tok.copy()
    bad[0, 0] = 17
    assert math.isnan(oracle.gpt2_step(sh, p, bad, tgt)[0])
    p2, tok2, tgt2 = _inputs(sh, 1, 5)
    tok6, tgt6 = synth.token_stream(1, 6, 17, "uniform")
    assert math.isnan(oracle.gpt2_step(sh, p2, tok6, tgt6)[0])


def test_thread_count_does_not_change_results(oracle):
    sh = Shape(2, 32, 2, 41, 8)
    p, tok, tgt = _inputs(sh, 2, 8, jitter=0.1)
    n0 = oracle.get_threads()
    oracle.set_threads(1)
    l1, g1, _ = oracle.gpt2_step(sh, p, tok, tgt)
    oracle.set_threads(max(2, n0))
    l2, g2, _ = oracle.gpt2_step(sh, p, tok, tgt)
    oracle.set_threads(n0)
    assert l1 == l2
    np.testing.assert_array_equal(g1, g2)


def test_last_position_logits_agree_with_the_step(oracle):
    """or_gpt2_logits_last against the pinned step: for every prefix length t,
    log-sum-exp(z) - z[target] of the last-position logits of tokens[:, :t] is
    the step's per-position loss at position t - 1 of the full sequence (which
    also pins causality: later tokens do not change earlier positions)."""
    sh = Shape(2, 32, 4, 97, 16)
    B, T = 2, 9
    p, tok, tgt = _inputs(sh, B, T)
    p = p + 0.05 * synth.normals(7, 0, p.size)  # no constant tensors
    _, _, rl = oracle.gpt2_step(sh, p, tok, tgt, want_grads=False, want_row_loss=True)
    rl = rl.reshape(B, T)
    for t in range(1, T + 1):
        z = oracle.gpt2_logits_last(sh, p, tok[:, :t])
        assert z.shape == (B, sh.V)
        zmax = z.max(axis=1, keepdims=True)
        lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
        ce = lse - z[np.arange(B), tgt[:, t - 1]]
        np.testing.assert_allclose(ce, rl[:, t - 1], rtol=1e-12, atol=1e-13)


def test_last_position_logits_zero_embedding_and_bad_arguments(oracle):
    sh = Shape(1, 16, 2, 33, 8)
    p, tok, _ = _inputs(sh, 2, 5)
    off, n = oracle.param_offset(sh.L, sh.C, sh.H, sh.V, sh.maxT, 0, 0)
    p[off:off + n] = 0.0  # tied head: logits = hf wte^T = 0
    assert np.all(oracle.gpt2_logits_last(sh, p, tok) == 0.0)
    bad = tok.copy()
    bad[0, 0] = sh.V
    try:
        oracle.gpt2_logits_last(sh, p, bad)
    except ValueError:
        pass
    else:
        raise AssertionError("an out-of-range token must be rejected")
