"""The step variants on the GPU against the oracle: gradient accumulation over
micro-batches (tt_gpt2_step_ex with TT_STEP_ACCUMULATE), the device loss
scale that seeds the backward, the global gradient statistics, AdamW on the
clipped, unscaled gradient with the update skipped on overflow, and the
dynamic loss scale, all decided on the device.

Tolerances are the step's: fp32 mode rel-L2 <= 1e-4 per gradient tensor,
bf16 mode <= 2e-2 (with cosine >= 0.999); AdamW in fp32 arithmetic within a
few ulps (1e-6 relative plus 1e-6 of the operands' rms).  A power-of-two loss
scale multiplies every product and sum of the backward exactly, so the scaled
gradients are the unscaled ones times the scale, bit for bit."""
import os

import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import build as native_build

from test_gpu_step import Run, compare_grads, make_inputs, oracle_params

pytestmark = pytest.mark.gpu
DEV = "cuda"


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


@pytest.mark.parametrize("name,dtype,tol,cos", [("tiny_fp32", "fp32", 1e-4, None),
                                                ("char_bf16", "bf16", 2e-2, 0.999)])
def test_accumulated_micro_batches_match_oracle(ctx, oracle, name, dtype, tol, cos):
    w = synth.WORKLOADS[name]
    sh = w.shape
    B, T = 4, min(w.T, 64)
    p, tok, tgt = make_inputs(sh, B, T, w.tokens, jitter=0.05)
    run = Run(ctx, sh, dtype, p)
    h = B // 2
    ctx.reset()
    la = ctx.step_ex(run.params, run.grads, _dev(tok[:h]), _dev(tgt[:h]), h, T)
    g_first = run.grads.clone()
    ctx.reset()
    lb = ctx.step_ex(run.params, run.grads, _dev(tok[h:]), _dev(tgt[h:]), h, T, accumulate=True)
    g = run.grads.cpu().numpy().astype(np.float64)
    po = oracle_params(oracle, p, dtype)
    ra, ga, _ = oracle.gpt2_step(sh, po, tok[:h], tgt[:h])
    rb, gb, _ = oracle.gpt2_step(sh, po, tok[h:], tgt[h:])
    rtol = 1e-5 if dtype == "fp32" else 2e-3
    assert abs(la - ra) <= rtol * ra and abs(lb - rb) <= rtol * rb
    compare_grads(run.cfg, sh.L, g, ga + gb, tol, cos, label=f"{name} accumulated")
    # accumulating into zeros gives the plain step's gradients bit for bit
    run.grads.zero_()
    ctx.reset()
    ctx.step_ex(run.params, run.grads, _dev(tok[:h]), _dev(tgt[:h]), h, T, accumulate=True)
    assert torch.equal(run.grads, g_first)


@pytest.mark.parametrize("name,dtype", [("tiny_fp32", "fp32"), ("char_bf16", "bf16")])
def test_power_of_two_loss_scale_is_exact(ctx, name, dtype):
    w = synth.WORKLOADS[name]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 4, min(w.T, 64), w.tokens, jitter=0.05)
    run = Run(ctx, sh, dtype, p)
    B, T = tok.shape
    ctx.reset()
    l1 = ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T)
    g1 = run.grads.clone()
    scale = torch.tensor([1024.0], device=DEV)
    ctx.reset()
    l2 = ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
    assert l2 == l1  # the reported loss is unscaled
    assert torch.equal(run.grads, g1 * 1024.0)


def test_grad_stats_match_oracle(ctx, oracle):
    n = 3_000_001
    g = (synth.normals(77, 0, n) * 0.01).astype(np.float32)
    G = _dev(g)
    stats = torch.zeros(2, device=DEV)
    ctx.grad_stats(G, stats)
    ref, bad = oracle.grad_norm(g.astype(np.float64))
    s = stats.cpu().numpy()
    assert bad == 0 and s[1] == 0.0
    assert abs(s[0] - ref) <= 1e-6 * ref
    scale = torch.tensor([512.0], device=DEV)
    ctx.grad_stats(G * 512.0, stats, loss_scale=scale)
    assert abs(stats.cpu().numpy()[0] - ref) <= 1e-6 * ref
    # deterministic
    s2 = torch.zeros(2, device=DEV)
    ctx.grad_stats(G, s2)
    ctx.grad_stats(G, stats)
    assert torch.equal(s2, stats)
    # an Inf, a NaN (host-made inputs) and a gradient whose square overflows float
    for poison in (np.inf, np.nan, 3e19):
        h = g.copy()
        h[n - 1] = poison  # in the tail of the float4 groups
        ctx.grad_stats(_dev(h), stats)
        assert stats.cpu().numpy()[1] == 1.0


@pytest.mark.parametrize("max_norm,scale", [(0.0, None), (0.5, None), (0.5, 256.0), (1e9, 4096.0)])
def test_adamw_ex_matches_oracle(ctx, oracle, max_norm, scale):
    n = 1_000_003
    rnd = lambda seed, s=1.0: (synth.normals(seed, 0, n) * s).astype(np.float32)
    p0, g, m0, v0 = rnd(1), rnd(2, 0.01), rnd(3, 0.01), np.abs(rnd(4, 0.01))
    gs = g * np.float32(scale) if scale else g
    P, G, Mm, Vv = (_dev(a.copy()) for a in (p0, gs, m0, v0))
    low = torch.empty(n, device=DEV, dtype=torch.bfloat16)
    step = torch.tensor([2], device=DEV, dtype=torch.int32)
    sc = torch.tensor([scale], device=DEV) if scale else None
    stats = torch.zeros(2, device=DEV)
    ctx.grad_stats(G, stats, loss_scale=sc)
    args = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    ctx.adamw_ex(P, low, G, Mm, Vv, step=step, stats=stats, max_norm=max_norm, loss_scale=sc, **args)
    rp, rm, rv, skipped = oracle.adamw_ex(p0, gs, m0, v0, args["lr"], args["beta1"], args["beta2"], args["eps"],
                                          args["weight_decay"], 3, scale=scale or 1.0, max_norm=max_norm)
    assert not skipped and int(step.item()) == 3
    from test_gpu_ops import assert_close, host
    assert_close(host(P), rp, 1e-6, 1e-6, "master")
    assert_close(host(Mm), rm, 1e-6, 1e-6, "m")
    assert_close(host(Vv), rv, 1e-6, 1e-6, "v")
    assert np.array_equal(host(low), oracle.bf16_values(P.cpu().numpy()))


def test_overflow_skips_update_and_backs_off_scale(ctx, oracle):
    n = 4099
    p0 = synth.normals(5, 0, n).astype(np.float32)
    g = (synth.normals(6, 0, n) * 0.01).astype(np.float32)
    g[100] = np.inf
    P, G = _dev(p0.copy()), _dev(g)
    Mm, Vv = torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)
    step = torch.tensor([7], device=DEV, dtype=torch.int32)
    scale = torch.tensor([65536.0], device=DEV)
    clean = torch.tensor([123], device=DEV, dtype=torch.int32)
    stats = torch.zeros(2, device=DEV)
    ctx.grad_stats(G, stats, loss_scale=scale)
    ctx.adamw_ex(P, None, G, Mm, Vv, 1e-3, 0.9, 0.95, 1e-8, 0.1, step, stats=stats, max_norm=1.0, loss_scale=scale)
    ctx.loss_scale_update(scale, clean, stats)
    assert torch.equal(P, _dev(p0)) and not Mm.any() and not Vv.any()
    assert int(step.item()) == 7 and float(scale.item()) == 32768.0 and int(clean.item()) == 0
    # clean steps: the step count advances, the scale grows on the window-th one
    G.copy_(_dev(np.nan_to_num(g, posinf=0.0)))
    s_ref, c_ref = 32768.0, 0
    for i in range(3):
        ctx.grad_stats(G, stats, loss_scale=scale)
        ctx.adamw_ex(P, None, G, Mm, Vv, 1e-3, 0.9, 0.95, 1e-8, 0.1, step, stats=stats, loss_scale=scale)
        ctx.loss_scale_update(scale, clean, stats, window=2, growth=2.0)
        s_ref, c_ref = oracle.loss_scale_update(s_ref, c_ref, False, window=2, growth=2.0)
        assert float(scale.item()) == s_ref and int(clean.item()) == c_ref
    assert int(step.item()) == 10


def test_scaled_training_loop_recovers_from_overflow(ctx, oracle):
    """A step whose scaled gradients overflow (an infinite scale makes that
    certain) is skipped on the device; with a sane scale the loop then trains
    as the unscaled, clipped oracle step does."""
    w = synth.WORKLOADS["tiny_fp32"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, w.B, w.T, w.tokens, jitter=0.05)
    run = Run(ctx, sh, "fp32", p)
    B, T = tok.shape
    scale = torch.tensor([float("inf")], device=DEV)
    clean = torch.zeros(1, device=DEV, dtype=torch.int32)
    step = torch.zeros(1, device=DEV, dtype=torch.int32)
    stats = torch.zeros(2, device=DEV)
    p_before = run.master.clone()
    ctx.reset()
    ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
    ctx.grad_stats(run.grads, stats, loss_scale=scale)
    ctx.adamw_ex(run.master, None, run.grads, run.m, run.v, 1e-3, 0.9, 0.95, 1e-8, 0.1, step, stats=stats,
                 max_norm=1.0, loss_scale=scale)
    ctx.loss_scale_update(scale, clean, stats)
    assert float(stats[1].item()) == 1.0
    assert torch.equal(run.master, p_before) and int(step.item()) == 0 and int(clean.item()) == 0
    # a sane scale: one clean step equals the unscaled oracle step with clipping
    scale.fill_(1024.0)
    ctx.reset()
    ctx.step_ex(run.params, run.grads, _dev(tok), _dev(tgt), B, T, loss_scale=scale)
    ctx.grad_stats(run.grads, stats, loss_scale=scale)
    ctx.adamw_ex(run.master, None, run.grads, run.m, run.v, 1e-3, 0.9, 0.95, 1e-8, 0.1, step, stats=stats,
                 max_norm=1.0, loss_scale=scale)
    ctx.loss_scale_update(scale, clean, stats)
    assert float(stats[1].item()) == 0.0 and int(step.item()) == 1 and int(clean.item()) == 1
    _, rg, _ = oracle.gpt2_step(sh, p.astype(np.float64), tok, tgt)
    norm, _ = oracle.grad_norm(rg)
    assert abs(float(stats[0].item()) - norm) <= 1e-4 * norm
    rp, _, _, skipped = oracle.adamw_ex(p.astype(np.float64), rg, np.zeros(p.size), np.zeros(p.size), 1e-3, 0.9,
                                        0.95, 1e-8, 0.1, 1, max_norm=1.0)
    assert not skipped
    got = run.master.cpu().numpy().astype(np.float64)
    d_got, d_ref = got - p, rp - p
    assert np.linalg.norm(d_got - d_ref) <= 1e-3 * np.linalg.norm(d_ref)


def test_step_ex_errors(ctx):
    w = synth.WORKLOADS["tiny_fp32"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 2, 8, w.tokens)
    run = Run(ctx, sh, "fp32", p)
    ctx.reset()
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        from autograd_arena_allocated_gb300._native import lib
        import ctypes as C
        rc = lib().tt_gpt2_step_ex(ctx.h, run.params.data_ptr(), run.grads.data_ptr(), _dev(tok).data_ptr(),
                                   _dev(tgt).data_ptr(), 2, 8, 4, None, None)
        ctx._check(rc)
    stats = torch.zeros(2, device=DEV)
    step = torch.zeros(1, device=DEV, dtype=torch.int32)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):  # clipping without statistics
        ctx.adamw_ex(run.master, None, run.grads, run.m, run.v, 1e-3, 0.9, 0.95, 1e-8, 0.1, step, max_norm=1.0)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.loss_scale_update(torch.ones(1, device=DEV), step, stats, window=0)
