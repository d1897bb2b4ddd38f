"""The step in IEEE half storage (TT_FP16) against the oracle, and the reason
the dl-scratch page (3.4) pairs half precision with a dynamic loss scale.

Half keeps a 10-bit mantissa, three bits more than bf16, so a scaled step's
rounding error is an eighth of the bf16 step's: the tolerances here are the
bf16 ones divided by 8 (loss 2.5e-4 relative, gradients rel-L2 2.5e-3; the
cosine's distance from 1 goes as the square of the error, so 1 - 1e-3/64).
But half keeps only 5 exponent bits: below 2^-14 values lose precision and
below 2^-25 they vanish.  The char model's logit gradients are about
p / (B T) ~ 6e-5 before any scale, right at that edge, and the activation
gradients below them are smaller still; a loss scale of 2^12 lifts them clear.
Too large a scale overflows (beyond 65504 a half is infinite): the step is
then skipped on the device and the scale halves until it fits."""
import os

import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import build as native_build

from test_gpu_step import Run, compare_grads, make_inputs, oracle_params

pytestmark = pytest.mark.gpu
DEV = "cuda"
LOSS_TOL, GRAD_TOL, MIN_COS = 2e-3 / 8, 2e-2 / 8, 1.0 - 1e-3 / 64


@pytest.fixture(scope="module", autouse=True)
def _threads(oracle):
    oracle.set_threads(os.cpu_count() or 1)


@pytest.fixture(scope="module")
def ctx():
    native_build.build()
    c = api.Context(2 << 30)
    yield c
    c.close()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(B=4, T=64):
    w = synth.WORKLOADS["char_bf16"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, B, T, w.tokens, jitter=0.05)
    return sh, p, tok, tgt


@pytest.fixture(scope="module")
def reference(oracle):
    sh, p, tok, tgt = _case()
    rl, rg, _ = oracle.gpt2_step(sh, oracle_params(oracle, p, "fp16"), tok, tgt)
    return rl, rg


def _grad_err(run, g, rg):
    worst = 0.0
    from test_gpu_step import tensor_slices
    for name, off, n in tensor_slices(run.cfg, run.sh.L):
        a, b = g[off:off + n], rg[off:off + n]
        worst = max(worst, float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)))
    return worst


def test_scaled_fp16_step_matches_oracle(ctx, oracle, reference):
    sh, p, tok, tgt = _case()
    run = Run(ctx, sh, "fp16", p)
    B, T = tok.shape
    scale = torch.tensor([4096.0], device=DEV)
    ctx.reset()
    loss = ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
    rl, rg = reference
    assert abs(loss - rl) <= LOSS_TOL * rl, (loss, rl)
    g = run.grads.cpu().numpy().astype(np.float64) / 4096.0
    compare_grads(run.cfg, sh.L, g, rg, GRAD_TOL, MIN_COS, label="fp16 scaled 2^12")
    # the forward alone gives the same loss
    ctx.reset()
    assert ctx.eval(run.params, _dev(tok), _dev(tgt), B, T) == loss


def test_fp16_small_heads_and_accumulation(ctx, oracle):
    """The tiny model (head dim 16) in half: two accumulated micro-batches
    against the oracle's summed gradients, scaled by 2^10."""
    w = synth.WORKLOADS["tiny_fp32"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 4, w.T, w.tokens, jitter=0.05)
    run = Run(ctx, sh, "fp16", p)
    B, T = tok.shape
    h = B // 2
    scale = torch.tensor([1024.0], device=DEV)
    ctx.reset()
    la = ctx.step_ex(run.params, run.grads, _dev(tok[:h]), _dev(tgt[:h]), h, T, loss_scale=scale)
    ctx.reset()
    lb = ctx.step_ex(run.params, run.grads, _dev(tok[h:]), _dev(tgt[h:]), h, T, accumulate=True, loss_scale=scale)
    po = oracle_params(oracle, p, "fp16")
    ra, ga, _ = oracle.gpt2_step(sh, po, tok[:h], tgt[:h])
    rb, gb, _ = oracle.gpt2_step(sh, po, tok[h:], tgt[h:])
    assert abs(la - ra) <= LOSS_TOL * ra and abs(lb - rb) <= LOSS_TOL * rb
    g = run.grads.cpu().numpy().astype(np.float64) / 1024.0
    compare_grads(run.cfg, sh.L, g, ga + gb, GRAD_TOL, MIN_COS, label="fp16 tiny accumulated")


def test_unscaled_fp16_gradients_underflow(ctx, oracle):
    """A larger batch (B T = 2048) makes the logit gradients p / (B T) about
    7e-6, subnormal in half, and the activation gradients below them a few
    dozen subnormal steps (2^-24) each.  Without a scale they keep only their
    top bits and the gradients are markedly further from the oracle than with a
    scale of 2^15.  (At the 124M model's B T = 32768 and V = 50257 most logit
    gradients, about 6e-10, would round to zero.)"""
    sh, p, tok, tgt = _case(B=8, T=256)
    run = Run(ctx, sh, "fp16", p)
    B, T = tok.shape
    rl, rg, _ = oracle.gpt2_step(sh, oracle_params(oracle, p, "fp16"), tok, tgt)
    ctx.reset()
    l0 = ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T)
    e0 = _grad_err(run, run.grads.cpu().numpy().astype(np.float64), rg)
    scale = torch.tensor([2.0 ** 15], device=DEV)
    ctx.reset()
    l1 = ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
    e1 = _grad_err(run, run.grads.cpu().numpy().astype(np.float64) / 2.0 ** 15, rg)
    print(f"[fp16 B T = 2048] worst gradient rel-L2: unscaled {e0:.3e}, scaled 2^15 {e1:.3e}")
    assert l0 == l1 and abs(l1 - rl) <= LOSS_TOL * rl
    assert e1 <= GRAD_TOL
    assert e0 > GRAD_TOL and e0 > 4.0 * e1


def test_fp16_overflow_backs_off_until_the_step_fits(ctx, oracle, reference):
    """Start from a scale so large that the scaled logit gradients exceed the
    largest half: each such step is skipped on the device (master, moments
    and step count unchanged) and the scale halves, following the oracle's
    loss-scale rule on the device's own overflow flags, until a step fits; that
    step is the oracle's clipped AdamW step on the unscaled gradients."""
    sh, p, tok, tgt = _case()
    run = Run(ctx, sh, "fp16", p)
    B, T = tok.shape
    rl, rg = reference
    s_ref, c_ref = 2.0 ** 28, 0
    scale = torch.tensor([s_ref], device=DEV)
    clean = torch.zeros(1, device=DEV, dtype=torch.int32)
    step = torch.zeros(1, device=DEV, dtype=torch.int32)
    stats = torch.zeros(2, device=DEV)
    p0 = run.master.clone()
    args = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    skipped = 0
    for _ in range(32):
        s_used = float(scale.item())
        ctx.reset()
        ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
        ctx.grad_stats(run.grads, stats, loss_scale=scale)
        ctx.adamw_ex(run.master, run.lowp, run.grads, run.m, run.v, step=step, stats=stats, max_norm=1.0,
                     loss_scale=scale, **args)
        ctx.loss_scale_update(scale, clean, stats)
        over = float(stats[1].item()) != 0.0
        s_ref, c_ref = oracle.loss_scale_update(s_ref, c_ref, over)
        assert float(scale.item()) == s_ref and int(clean.item()) == c_ref
        if not over:
            break
        skipped += 1
        assert torch.equal(run.master, p0) and not run.m.any() and int(step.item()) == 0
    else:
        pytest.fail("the loss scale never came down to a step that fits")
    print(f"[fp16] {skipped} overflow steps skipped; the first clean step used scale 2^{np.log2(s_used):.0f}")
    assert skipped >= 4  # a target logit gradient is about -2^s / (B T) = -2^(s-8): infinite in half for s >= 25
    assert int(step.item()) == 1
    norm, _ = oracle.grad_norm(rg)
    assert abs(float(stats[0].item()) - norm) <= GRAD_TOL * norm
    rp, _, _, sk = oracle.adamw_ex(p.astype(np.float64), rg, np.zeros(p.size), np.zeros(p.size), args["lr"],
                                   args["beta1"], args["beta2"], args["eps"], args["weight_decay"], 1, max_norm=1.0)
    assert not sk
    got = run.master.cpu().numpy().astype(np.float64)
    d_got, d_ref = got - p, rp - p
    # Adam's first step moves each weight by about lr sign(g): the direction matches where the gradients do
    assert np.dot(d_got, d_ref) >= 0.99 * np.linalg.norm(d_got) * np.linalg.norm(d_ref)
    # the half copy is the rounded master
    assert np.array_equal(run.lowp.cpu().numpy().astype(np.float64), oracle.f16_values(run.master.cpu().numpy()))


def test_fp16_adamw_copy_and_cast(ctx, oracle):
    sh, p, _, _ = _case()
    run = Run(ctx, sh, "fp16", p)
    assert np.array_equal(run.lowp.cpu().numpy().astype(np.float64), oracle.f16_values(p))
    n = 100_003
    big = (synth.normals(31, 0, n) * 3e4).astype(np.float32)  # reaches past 65504: the copy saturates to inf
    P = _dev(big.copy())
    low = torch.empty(n, device=DEV, dtype=torch.float16)
    G = _dev((synth.normals(32, 0, n) * 0.01).astype(np.float32))
    Mm, Vv = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    ctx.adamw(P, low, G, Mm, Vv, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    want = oracle.f16_values(P.cpu().numpy())
    assert np.isinf(want).any()
    assert np.array_equal(low.cpu().numpy().astype(np.float64), want)


def test_fp16_generation_is_refused(ctx):
    sh, p, tok, _ = _case(B=1, T=8)
    run = Run(ctx, sh, "fp16", p)
    assert api.generate_arena_bytes(run.cfg, 1, 8, 4) == 0
    out = torch.zeros(1, 12, dtype=torch.int32, device=DEV)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.generate(run.params, _dev(tok), 1, 8, 4, out)
