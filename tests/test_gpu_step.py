"""Whole-step parity: tt_gpt2_step (+ tt_adamw) against the oracle on the same
seeded inputs, with the tolerances of the spec:
  fp32 mode: loss rel err <= 1e-5, every gradient tensor rel-L2 <= 1e-4;
  bf16 mode: loss rel err <= 2e-3, gradient rel-L2 <= 2e-2 and cosine >= 0.999,
             AdamW-updated parameters rel-L2 <= 1e-3.
At the full batch sizes the oracle cannot run, whole sequences are sampled:
sequences are independent, so the GPU's per-position losses for sequence b
must equal the oracle's on that sequence alone.  Also: run-to-run bitwise
determinism, host vs device token buffers, and the boundary's error paths."""
import math
import os

import numpy as np
import pytest
import torch

from autograd_arena_allocated_gb300 import api, synth
from autograd_arena_allocated_gb300 import build as native_build

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _threads(oracle):
    oracle.set_threads(os.cpu_count() or 1)


def make_inputs(sh, B, T, kind, jitter=0.0):
    p = synth.init_params(sh, jitter=jitter)
    tok, tgt = synth.token_stream(B, T, sh.V, kind)
    return p, tok, tgt


class Run:
    """Device state of one model: master fp32, compute copy, grads, moments."""

    def __init__(self, ctx, sh, dtype, p):
        self.ctx, self.sh, self.dtype = ctx, sh, dtype
        self.cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, dtype)
        ctx.set_model(self.cfg)
        self.n = api.num_params(self.cfg)
        assert self.n == p.size
        self.master = torch.from_numpy(p).to(DEV)
        if dtype == "bf16":
            self.lowp = torch.empty(self.n, device=DEV, dtype=torch.bfloat16)
            ctx.cast_bf16(self.master, self.lowp)
            self.params = self.lowp
        elif dtype == "fp16":
            self.lowp = torch.empty(self.n, device=DEV, dtype=torch.float16)
            ctx.cast_f16(self.master, self.lowp)
            self.params = self.lowp
        else:
            self.lowp = None
            self.params = self.master
        self.grads = torch.empty(self.n, device=DEV)
        self.m = torch.zeros(self.n, device=DEV)
        self.v = torch.zeros(self.n, device=DEV)

    def step(self, tok, tgt):
        B, T = tok.shape
        self.ctx.reset()
        td = torch.from_numpy(tok).to(DEV) if isinstance(tok, np.ndarray) else tok
        gd = torch.from_numpy(tgt).to(DEV) if isinstance(tgt, np.ndarray) else tgt
        return self.ctx.step(self.params, self.grads, td, gd, B, T)


def oracle_params(oracle, p, dtype):
    if dtype == "bf16":
        return oracle.bf16_values(p)
    if dtype == "fp16":
        return oracle.f16_values(p)
    return p.astype(np.float64)


def tensor_slices(cfg, L):
    out = [("wte",) + api.param_offset(cfg, 0, 0), ("wpe",) + api.param_offset(cfg, 0, 1)]
    names = ["ln1_w", "ln1_b", "qkv_w", "qkv_b", "proj_w", "proj_b", "ln2_w", "ln2_b",
             "fc_w", "fc_b", "fcproj_w", "fcproj_b"]
    for l in range(L):
        for j, nm in enumerate(names):
            out.append((f"h{l}.{nm}",) + api.param_offset(cfg, l, 2 + j))
    out += [("lnf_w",) + api.param_offset(cfg, 0, 14), ("lnf_b",) + api.param_offset(cfg, 0, 15)]
    return out


def compare_grads(cfg, L, g, rg, rel_l2, min_cos=None, T=None, maxT=None, label=""):
    worst = []
    for name, off, n in tensor_slices(cfg, L):
        a, b = g[off:off + n], rg[off:off + n]
        if name == "wpe" and T is not None and T < maxT:
            C_ = n // maxT
            assert np.all(a[T * C_:] == 0.0), "unused position rows must have zero gradient"
            a, b = a[:T * C_], b[:T * C_]
        nb = np.linalg.norm(b)
        err = np.linalg.norm(a - b) / max(nb, 1e-30)
        cos = float(np.dot(a, b) / max(np.linalg.norm(a) * nb, 1e-30))
        worst.append((err, name, cos))
        assert err <= rel_l2, f"{name}: rel-L2 {err:.3e} > {rel_l2}"
        if min_cos is not None:
            assert cos >= min_cos, f"{name}: cosine {cos:.6f} < {min_cos}"
    w = max(worst)
    print(f"[{label}] worst gradient rel-L2 {w[0]:.3e} ({w[1]}), min cosine "
          f"{min(c for _, _, c in worst):.6f}")
    return w


@pytest.fixture(scope="module")
def ctx():
    native_build.build()
    c = api.Context(8 << 30)
    yield c
    c.close()


# ----------------------------------------------------------------- fp32 mode
def test_tiny_fp32_step_matches_oracle(ctx, oracle):
    w = synth.WORKLOADS["tiny_fp32"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, w.B, w.T, w.tokens, jitter=0.05)
    run = Run(ctx, sh, "fp32", p)
    loss = run.step(tok, tgt)
    rl, rg, _ = oracle.gpt2_step(sh, p.astype(np.float64), tok, tgt)
    assert abs(loss - rl) <= 1e-5 * abs(rl), (loss, rl)
    g = run.grads.cpu().numpy().astype(np.float64)
    compare_grads(run.cfg, sh.L, g, rg, 1e-4, label="tiny fp32")
    print(f"[tiny fp32] loss {loss:.7f} oracle {rl:.7f} rel {abs(loss - rl) / rl:.2e}")
    # AdamW on the master (fp32 mode trains the master directly)
    lr, b1, b2, eps, wd = w.lr, w.beta1, w.beta2, w.eps, w.weight_decay
    ctx.adamw(run.master, None, run.grads, run.m, run.v, lr, b1, b2, eps, wd, 1)
    torch.cuda.synchronize()
    rp, _, _ = oracle.adamw(p.astype(np.float64), rg, np.zeros(p.size), np.zeros(p.size), lr, b1, b2,
                            eps, wd, 1)
    got = run.master.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - rp) / np.linalg.norm(rp) <= 1e-5


def test_tiny_fp32_short_sequences(ctx, oracle):
    """T < maxT (unused position rows get zero gradient) and B = 1, T = 1."""
    sh = synth.WORKLOADS["tiny_fp32"].shape
    for B, T in [(3, 17), (1, 1)]:
        p, tok, tgt = make_inputs(sh, B, T, "uniform", jitter=0.05)
        run = Run(ctx, sh, "fp32", p)
        loss = run.step(tok, tgt)
        rl, rg, _ = oracle.gpt2_step(sh, p.astype(np.float64), tok, tgt)
        assert abs(loss - rl) <= 1e-5 * abs(rl)
        compare_grads(run.cfg, sh.L, run.grads.cpu().numpy().astype(np.float64), rg, 1e-4,
                      T=T, maxT=sh.maxT)


# ----------------------------------------------------------------- bf16 mode
def _bf16_parity(ctx, oracle, sh, B, T, kind, jitter, label):
    p, tok, tgt = make_inputs(sh, B, T, kind, jitter=jitter)
    run = Run(ctx, sh, "bf16", p)
    loss = run.step(tok, tgt)
    po = oracle_params(oracle, p, "bf16")
    rl, rg, _ = oracle.gpt2_step(sh, po, tok, tgt)
    print(f"[{label}] loss {loss:.6f} oracle {rl:.6f} rel {abs(loss - rl) / rl:.2e}")
    assert abs(loss - rl) <= 2e-3 * abs(rl), (loss, rl)
    g = run.grads.cpu().numpy().astype(np.float64)
    compare_grads(run.cfg, sh.L, g, rg, 2e-2, min_cos=0.999, T=T, maxT=sh.maxT, label=label)
    return run, p, rg


def test_char_bf16_step_matches_oracle(ctx, oracle):
    """The char workload at its full batch (B=64, T=256): loss, every gradient
    tensor, and the AdamW-updated parameters."""
    w = synth.WORKLOADS["char_bf16"]
    assert (w.B, w.T) == (64, 256)
    run, p, rg = _bf16_parity(ctx, oracle, w.shape, w.B, w.T, "zipf", jitter=0.05, label="char bf16")
    lr, b1, b2, eps, wd = w.lr, w.beta1, w.beta2, w.eps, w.weight_decay
    rp, _, _ = oracle.adamw(p.astype(np.float64), rg, np.zeros(p.size), np.zeros(p.size), lr, b1, b2,
                            eps, wd, 1)
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))
    # (1) AdamW-updated parameters from identical inputs (the oracle's gradient
    #     given to the GPU's tt_adamw): the fp32 master within 1e-3 (it is at
    #     ~1e-7); the bf16 compute copy is exactly the nearest bf16 of the
    #     master (its distance to the exact update is bf16 rounding, ~2e-3)
    g_or = torch.from_numpy(rg.astype(np.float32)).to(DEV)
    master = torch.from_numpy(p).to(DEV)
    low = torch.empty_like(run.lowp)
    ctx.adamw(master, low, g_or, torch.zeros_like(master), torch.zeros_like(master), lr, b1, b2,
              eps, wd, 1)
    torch.cuda.synchronize()
    e_master = rel(master.cpu().numpy().astype(np.float64), rp)
    e_low = rel(low.float().cpu().numpy().astype(np.float64), rp)
    print(f"[char bf16] AdamW from identical inputs: master rel-L2 {e_master:.2e}, bf16 copy {e_low:.2e}")
    assert e_master <= 1e-6
    assert np.array_equal(low.float().cpu().numpy().astype(np.float64),
                          oracle.bf16_values(master.cpu().numpy()))
    # (2) end to end: the update of the GPU's own bf16-mode gradient.  At step 1
    #     the bias-corrected moments are m = g and v = g^2, so AdamW moves each
    #     component by lr * (g / (|g| + eps) + wd * p): a step function of g.
    #     A gradient within the bf16 tolerance can still have the other sign
    #     where |g| is near zero, and there the update jumps by up to 2 * lr
    #     whatever the gradient's accuracy.  So the 1e-3 bound on updated
    #     parameters is applied to the components whose two gradients agree in
    #     sign (where the update is continuous in g); each other component must
    #     be within the 2 * lr jump; the whole vector's rel-L2 is printed.
    ctx.adamw(run.master, run.lowp, run.grads, run.m, run.v, lr, b1, b2, eps, wd, 1)
    torch.cuda.synchronize()
    got = run.master.cpu().numpy().astype(np.float64)
    g = run.grads.cpu().numpy().astype(np.float64)
    agree = np.sign(g) == np.sign(rg)
    flips = float(np.mean(~agree))
    e_agree = rel(got[agree], rp[agree])
    e_all = rel(got, rp)
    jump = float(np.max(np.abs(got[~agree] - rp[~agree]))) if flips > 0 else 0.0
    print(f"[char bf16] AdamW after the bf16 step: params rel-L2 {e_all:.2e} over all "
          f"{p.size} components, {e_agree:.2e} over the {int(agree.sum())} whose gradient signs agree; "
          f"sign disagreements {100 * flips:.3f}%, largest jump there {jump:.2e} (2*lr = {2 * lr:.1e})")
    assert e_agree <= 1e-3
    assert jump <= 2 * lr * (1 + 1e-6) + 1e-7
    assert flips <= 0.05
    assert np.array_equal(run.lowp.float().cpu().numpy().astype(np.float64),
                          oracle.bf16_values(run.master.cpu().numpy()))


def test_gpt2_124m_bf16_reduced_batch(ctx, oracle):
    """GPT-2 124M architecture at B=1, T=64 (the oracle's reduced size)."""
    _bf16_parity(ctx, oracle, synth.GPT2_124M, 1, 64, "zipf", jitter=0.0, label="124M B=1 T=64")


def _sampled_sequences(ctx, oracle, w, seqs):
    sh = w.shape
    p, tok, tgt = make_inputs(sh, w.B, w.T, w.tokens)
    cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, "bf16")
    big = api.Context(api.arena_bytes(cfg, w.B, w.T))
    ctx = big
    run = Run(ctx, sh, "bf16", p)
    loss = run.step(tok, tgt)
    rl_gpu = torch.empty(w.B * w.T, device=DEV)
    ctx.row_losses(rl_gpu)
    rl_gpu = rl_gpu.cpu().numpy().reshape(w.B, w.T).astype(np.float64)
    assert math.isfinite(loss)
    assert abs(loss - rl_gpu.mean()) <= 1e-4 * abs(loss)
    po = oracle_params(oracle, p, "bf16")
    for b in seqs:
        _, _, rl = oracle.gpt2_step(sh, po, tok[b:b + 1], tgt[b:b + 1], want_grads=False,
                                    want_row_loss=True)
        err = np.abs(rl_gpu[b] - rl)
        print(f"[{w.name}] sequence {b}: per-position loss max abs err {np.max(err):.2e}, "
              f"mean abs err {np.mean(err):.2e} (mean loss {np.mean(rl):.4f})")
        # the spec's bf16 loss bound (2e-3 relative) on the sequence's mean loss;
        # single positions within 5e-3 relative
        assert abs(np.mean(rl_gpu[b]) - np.mean(rl)) <= 2e-3 * np.mean(rl)
        assert np.max(err) <= 5e-3 * np.mean(rl) and np.mean(err) <= 2e-3 * np.mean(rl), (b, np.max(err))
    g = run.grads.clone()
    big.close()
    return g


def test_gpt2_350m_bf16_reduced_batch(ctx, oracle):
    """GPT-2 medium (L=24, C=1024, H=16) at B=1, T=64: every gradient tensor."""
    _bf16_parity(ctx, oracle, synth.GPT2_350M, 1, 64, "zipf", jitter=0.0, label="350M B=1 T=64")


def test_gpt2_124m_b8_full_batch_sampled(ctx, oracle):
    _sampled_sequences(ctx, oracle, synth.WORKLOADS["gpt2_124m_b8"], [0, 7])


def test_gpt2_350m_b8_full_batch_sampled(ctx, oracle):
    g = _sampled_sequences(ctx, oracle, synth.WORKLOADS["gpt2_350m_b8"], [5])
    assert torch.isfinite(g).all()


def test_char_bf16_full_batch_sampled(ctx, oracle):
    _sampled_sequences(ctx, oracle, synth.WORKLOADS["char_bf16"], [0, 37, 63])


def test_gpt2_124m_full_batch_sampled(ctx, oracle):
    """The benchmark's workload (B=32, T=1024): one whole sequence sampled."""
    g = _sampled_sequences(ctx, oracle, synth.WORKLOADS["gpt2_124m_b32"], [31])
    assert torch.isfinite(g).all()


# ----------------------------------------------------------------- determinism & inputs
def test_step_is_bitwise_deterministic_and_host_tokens_match(ctx):
    w = synth.WORKLOADS["char_bf16"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 8, 256, "zipf", jitter=0.05)
    run = Run(ctx, sh, "bf16", p)
    l1 = run.step(tok, tgt)
    g1 = run.grads.clone()
    l2 = run.step(tok, tgt)
    assert l1 == l2 and torch.equal(g1, run.grads)
    # host (pageable) token buffers are staged by the library
    ctx.reset()
    l3 = ctx.step(run.params, run.grads, tok, tgt, 8, 256)
    assert l3 == l1 and torch.equal(g1, run.grads)


_PDL_OFF_STEP = r"""
import sys
import numpy as np, torch
from autograd_arena_allocated_gb300 import api, synth
w = synth.WORKLOADS["char_bf16"]
sh = w.shape
p = synth.init_params(sh, jitter=0.05)
tok, tgt = synth.token_stream(8, 256, sh.V, "zipf")
with api.Context(1 << 30) as ctx:
    cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, "bf16")
    ctx.set_model(cfg)
    master = torch.from_numpy(p).cuda()
    low = torch.empty(master.numel(), device="cuda", dtype=torch.bfloat16)
    ctx.cast_bf16(master, low)
    grads = torch.empty(master.numel(), device="cuda")
    ctx.reset()
    loss = ctx.step(low, grads, torch.from_numpy(tok).cuda(), torch.from_numpy(tgt).cuda(), 8, 256)
    np.savez(sys.argv[1], loss=np.array([loss]), grads=grads.cpu().numpy())
"""


def test_step_is_the_same_without_dependent_launch(ctx, tmp_path):
    """Programmatic dependent launch changes when a kernel's CTAs are
    scheduled, never what they compute: each waits for its predecessor before
    touching global memory.  The same bf16 step in a process with TT_PDL=0
    (every kernel launched in plain stream order) gives the same bits."""
    import subprocess
    import sys

    w = synth.WORKLOADS["char_bf16"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 8, 256, "zipf", jitter=0.05)
    run = Run(ctx, sh, "bf16", p)
    loss = run.step(tok, tgt)
    g = run.grads.cpu().numpy()
    out = tmp_path / "pdl_off.npz"
    env = dict(os.environ, TT_PDL="0")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    subprocess.run([sys.executable, "-c", _PDL_OFF_STEP, str(out)], check=True, env=env, cwd=root, timeout=600)
    r = np.load(out)
    assert float(r["loss"][0]) == loss
    assert np.array_equal(r["grads"], g)


# ----------------------------------------------------------------- boundary
def test_arena_oom_is_detected_before_launch():
    sh = synth.WORKLOADS["tiny_fp32"].shape
    cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, "fp32")
    need = api.arena_bytes(cfg, 4, 32)
    p, tok, tgt = make_inputs(sh, 4, 32, "uniform")
    with api.Context(need // 2) as c:
        run = Run(c, sh, "fp32", p)
        launches = c.launches
        with pytest.raises(api.TTError, match="TT_ERR_ARENA_OOM"):
            run.step(tok, tgt)
        assert c.launches == launches
        # usable afterwards with a batch that fits
        tok2, tgt2 = synth.token_stream(1, 8, sh.V, "uniform")
        assert math.isfinite(run.step(tok2, tgt2))
    with api.Context(need) as c:
        run = Run(c, sh, "fp32", p)
        assert math.isfinite(run.step(tok, tgt))
        assert c.high_water <= need


def test_boundary_errors(ctx):
    sh = synth.WORKLOADS["tiny_fp32"].shape
    p, tok, tgt = make_inputs(sh, 2, 8, "uniform")
    run = Run(ctx, sh, "fp32", p)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.step(run.params, run.grads, tok, tgt, 2, sh.maxT + 1)
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.step(run.params, run.grads, tok, tgt, 0, 8)
    bad = tok.copy()
    bad[1, 3] = sh.V
    ctx.reset()
    with pytest.raises(api.TTError, match="TT_ERR_ARG"):
        ctx.step(run.params, run.grads, bad, tgt, 2, 8)
    # usable after the error
    assert math.isfinite(run.step(tok, tgt))
    c2 = api.Context(1 << 20)
    h = c2.h
    c2.close()
    from autograd_arena_allocated_gb300 import _native
    assert _native.lib().tt_ctx_reset(h) == -7  # TT_ERR_STALE
    with api.Context(1 << 20) as c3:
        with pytest.raises(api.TTError, match="TT_ERR_STATE"):
            c3.step(run.params, run.grads, tok, tgt, 2, 8)


def test_nonfinite_parameter_is_reported_and_context_recovers(ctx):
    """A NaN planted on the host in one parameter (the final LayerNorm's first
    bias) reaches every logit, so the step's loss is NaN: the step must return
    TT_ERR_NONFINITE (read from the device flag at its sync), and the context
    must run a clean step normally after a reset."""
    w = synth.WORKLOADS["char_bf16"]
    sh = w.shape
    p, tok, tgt = make_inputs(sh, 2, 64, "zipf", jitter=0.05)
    cfg = api.make_config(sh.L, sh.C, sh.H, sh.V, sh.maxT, "bf16")
    off, _ = api.param_offset(cfg, 0, 15)  # lnf_b
    bad = p.copy()
    bad[off] = np.nan
    run = Run(ctx, sh, "bf16", bad)
    with pytest.raises(api.TTError, match="TT_ERR_NONFINITE"):
        run.step(tok, tgt)
    clean = Run(ctx, sh, "bf16", p)
    loss = clean.step(tok, tgt)
    assert math.isfinite(loss)
    assert torch.isfinite(clean.grads).all()
